"""Centroid-masked sparse LM head for GB300 (placeholder, filled in with the binding)."""
