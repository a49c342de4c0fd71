"""Seeded synthetic inputs for the centroid-masked sparse LM head.

This module only draws random numbers: it holds none of the head's arithmetic
(no projection, no top-K, no dot product).  Both the CUDA path (tests, bench)
and the CPU oracle read their inputs from here, so it is the one module they
share.

Workloads (shapes follow the Gemma4 MTP drafter head: ``num_centroids`` 2048 and
``centroid_intermediate_top_k`` 32 are the defaults in ``Gemma4MTP.__init__`` of
"Add Gemma4 MTP speculative decoding with centroids masking", vLLM
``gemma4_mtp.py``; batch sizes 1..64 are the CUDA-graph sizes of
``Gemma4Proposer._setup_centroids_cuda_graphs`` in vLLM ``gemma4.py``):

* ``tiny``     V=4096 as 64 clusters of 64, H=64, C=64, K=4, B=1, N(0, 0.05^2) tables
* ``uniform``  V=262144 as 2048 clusters of 128, H=1536, K=32, B in 1..64, N(0, 0.02^2)
* ``variable`` V=262144 as 2048 lognormal-sized clusters, H=2560, K=32, B=64
* ``scatter``  the ``uniform`` tables at B=64, full-vocab output
* ``shared``   V=262144 as 4096 clusters of 64, H=2048, K=128, B=256, hidden rows
               are 8 prototypes plus N(0, 0.1^2) noise so rows share centroids

Generator: numpy PCG64.  Seed = 20261202 + 1000*workload_index + stream, with
streams 0 = centroid table, 1 = embedding table, 2 = permutation, 3 = hidden,
4 = cluster sizes, 5 = prototypes.  Tables are drawn in fp32 and rounded to
bf16 with round-to-nearest-even; bf16 arrays are carried as ``uint16`` bit
patterns.  Hidden row ``r`` at redraw attempt ``a`` comes from its own
sub-stream ``(seed_hidden, r, a)`` so one row can be redrawn without touching
the others.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BASE_SEED = 20261202

STREAM_CENTROIDS = 0
STREAM_EMBED = 1
STREAM_PERM = 2
STREAM_HIDDEN = 3
STREAM_SIZES = 4
STREAM_PROTO = 5


@dataclass(frozen=True)
class Workload:
    name: str
    index: int              # fixes the seeds
    vocab: int              # V
    hidden: int             # H
    centroids: int          # C
    top_k: int              # K
    batch: int              # default B
    table_std: float
    variable_clusters: bool = False
    prototypes: int = 0     # >0: hidden rows = prototype + noise
    noise_std: float = 0.0
    table_from: str = ""    # reuse another workload's tables
    batches: tuple = field(default_factory=tuple)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4096, 64, 64, 4, 1, 0.05),
    "uniform": Workload("uniform", 2, 262144, 1536, 2048, 32, 64, 0.02,
                        batches=(1, 2, 4, 8, 16, 32, 64)),
    "variable": Workload("variable", 3, 262144, 2560, 2048, 32, 64, 0.02,
                         variable_clusters=True),
    "scatter": Workload("scatter", 4, 262144, 1536, 2048, 32, 64, 0.02,
                        table_from="uniform"),
    "shared": Workload("shared", 5, 262144, 2048, 4096, 128, 256, 0.02,
                       prototypes=8, noise_std=0.1),
    # the draft-dimension sweep point: a drafter whose hidden size is 256
    "draft256": Workload("draft256", 6, 262144, 256, 2048, 32, 64, 0.02,
                         batches=(1, 8, 64)),
}


def seed_for(w: Workload, stream: int) -> int:
    return BASE_SEED + 1000 * w.index + stream


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_table_bf16(rows: int, cols: int, std: float, seed: int,
                      block_rows: int = 8192) -> np.ndarray:
    """[rows, cols] bf16 bits of N(0, std^2), drawn in row blocks.

    Block j uses PCG64 seeded with (seed, j) so the result does not depend on
    the number of threads.
    """
    out = np.empty((rows, cols), dtype=np.uint16)
    nblk = (rows + block_rows - 1) // block_rows

    def work(j: int) -> None:
        r0 = j * block_rows
        r1 = min(rows, r0 + block_rows)
        g = np.random.Generator(np.random.PCG64([seed, j]))
        x = g.standard_normal((r1 - r0, cols), dtype=np.float32)
        x *= np.float32(std)
        out[r0:r1] = bf16_bits(x)

    if nblk == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nblk)))
    return out


def lognormal_cluster_sizes(vocab: int, clusters: int, seed: int,
                            mu: float = float(np.log(128.0)), sigma: float = 0.6) -> np.ndarray:
    """Cluster sizes: lognormal, rounded, at least 1, summing exactly to vocab.

    s_i = max(1, round(x_i * V / sum(x))); the residual is then removed one
    token at a time on clusters taken in (size desc, index asc) order, never
    taking a cluster below 1.
    """
    g = np.random.Generator(np.random.PCG64(seed))
    x = np.exp(g.normal(mu, sigma, size=clusters))
    s = np.maximum(1, np.rint(x * vocab / x.sum())).astype(np.int64)
    resid = int(vocab - s.sum())
    order = sorted(range(clusters), key=lambda i: (-int(s[i]), i))
    step = 1 if resid > 0 else -1
    i = 0
    guard = 0
    while resid != 0:
        c = order[i % clusters]
        if step > 0 or s[c] > 1:
            s[c] += step
            resid -= step
        i += 1
        guard += 1
        if guard > 100 * clusters + abs(resid) * clusters:
            raise RuntimeError("cannot balance cluster sizes")
    assert int(s.sum()) == vocab and int(s.min()) >= 1
    return s.astype(np.int32)


def offsets_from_sizes(sizes: np.ndarray) -> np.ndarray:
    off = np.zeros(len(sizes) + 1, dtype=np.int64)
    np.cumsum(sizes, out=off[1:])
    return off.astype(np.int32)


@dataclass
class Tables:
    workload: Workload
    centroid_w: np.ndarray       # uint16 [C, H] bf16 bits
    embed_w: np.ndarray          # uint16 [V, H] bf16 bits, token-id order
    token_ordering: np.ndarray   # int32 [V]: ordered position -> token id
    cluster_offsets: np.ndarray | None  # int32 [C+1] or None (uniform)
    prototypes: np.ndarray | None = None  # float32 [P, H]


def _table_workload(w: Workload) -> Workload:
    return WORKLOADS[w.table_from] if w.table_from else w


def make_tables(w: Workload | str) -> Tables:
    if isinstance(w, str):
        w = WORKLOADS[w]
    tw = _table_workload(w)
    cw = normal_table_bf16(tw.centroids, tw.hidden, tw.table_std, seed_for(tw, STREAM_CENTROIDS))
    ew = normal_table_bf16(tw.vocab, tw.hidden, tw.table_std, seed_for(tw, STREAM_EMBED))
    perm = np.random.Generator(np.random.PCG64(seed_for(tw, STREAM_PERM))).permutation(tw.vocab)
    perm = perm.astype(np.int32)
    offs = None
    if tw.variable_clusters:
        offs = offsets_from_sizes(lognormal_cluster_sizes(tw.vocab, tw.centroids,
                                                          seed_for(tw, STREAM_SIZES)))
    protos = None
    if w.prototypes:
        g = np.random.Generator(np.random.PCG64(seed_for(w, STREAM_PROTO)))
        protos = g.standard_normal((w.prototypes, w.hidden), dtype=np.float32)
    return Tables(w, cw, ew, perm, offs, protos)


def hidden_row(w: Workload | str, row: int, attempt: int = 0,
               prototypes: np.ndarray | None = None) -> np.ndarray:
    """One draft hidden state as bf16 bits [H].

    Plain workloads: N(0, 1).  Prototype workloads: prototype (row mod P)
    plus N(0, noise_std^2); a redraw changes only the noise.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    g = np.random.Generator(np.random.PCG64([seed_for(w, STREAM_HIDDEN), row, attempt]))
    if w.prototypes:
        if prototypes is None:
            gp = np.random.Generator(np.random.PCG64(seed_for(w, STREAM_PROTO)))
            prototypes = gp.standard_normal((w.prototypes, w.hidden), dtype=np.float32)
        x = prototypes[row % w.prototypes] + np.float32(w.noise_std) * g.standard_normal(
            w.hidden, dtype=np.float32)
    else:
        x = g.standard_normal(w.hidden, dtype=np.float32)
    return bf16_bits(x)


def hidden_batch(w: Workload | str, batch: int, attempts: np.ndarray | None = None,
                 prototypes: np.ndarray | None = None, row0: int = 0) -> np.ndarray:
    """[batch, H] bf16 bits; row i is hidden_row(w, row0 + i, attempts[i])."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    if attempts is None:
        attempts = np.zeros(batch, dtype=np.int64)
    return np.stack([hidden_row(w, row0 + i, int(attempts[i]), prototypes)
                     for i in range(batch)])


def custom_tables(vocab: int, hidden: int, centroids: int, seed: int, std: float = 0.05,
                  sizes: np.ndarray | None = None, identity: bool = False) -> Tables:
    """Small ad-hoc tables for edge cases (ragged sizes, empty clusters, identity order)."""
    w = Workload(f"custom{seed}", 100 + seed % 900, vocab, hidden, centroids, 1, 1, std)
    cw = normal_table_bf16(centroids, hidden, std, seed * 7 + 1)
    ew = normal_table_bf16(vocab, hidden, std, seed * 7 + 2)
    if identity:
        perm = np.arange(vocab, dtype=np.int32)
    else:
        perm = np.random.Generator(np.random.PCG64(seed * 7 + 3)).permutation(vocab).astype(np.int32)
    offs = None if sizes is None else offsets_from_sizes(np.asarray(sizes))
    return Tables(w, cw, ew, perm, offs)


def random_hidden(batch: int, hidden: int, seed: int, std: float = 1.0) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(seed))
    return bf16_bits(np.float32(std) * g.standard_normal((batch, hidden), dtype=np.float32))
