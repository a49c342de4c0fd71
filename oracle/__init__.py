"""CPU oracle for the centroid-masked sparse LM head: test infrastructure only."""
