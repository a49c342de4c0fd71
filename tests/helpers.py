"""Shared helpers of the parity tests: near-tie-free inputs and tolerance checks.

Tolerances: selected centroid sets and token ids must match the oracle exactly
whenever the oracle's K-th/(K+1)-th centroid-score margin and its top-1/top-2
logit margin both exceed 1e-3 (rows closer than that are redrawn from their
next sub-stream, up to 64 times); fp32 scores and logits must satisfy
|gpu - oracle| <= 2e-3 + 1e-2 * |oracle| against the oracle's fp64 values;
-inf entries must match exactly.
"""
from __future__ import annotations

import numpy as np

from centroid_masked_sparse_gb300 import synth
from oracle import oracle

MARGIN = 1e-3
ATOL = 2e-3
RTOL = 1e-2

_TABLES = {}


def tables(name: str) -> synth.Tables:
    """Host tables of a named workload (generated once per process)."""
    w = synth.WORKLOADS[name]
    key = w.table_from or name
    if key not in _TABLES:
        _TABLES[key] = synth.make_tables(key)
    return _TABLES[key]


def clean_batch(name: str, head: oracle.Head, batch: int, need_logit_margin: bool = True,
                max_attempts: int = 64, row0: int = 0):
    """Hidden rows of a workload whose oracle margins all exceed MARGIN.

    Returns (hidden uint16 [B, H], oracle result dict, number of redraws)."""
    w = synth.WORKLOADS[name]
    t = tables(name)
    attempts = np.zeros(batch, dtype=np.int64)
    hidden = synth.hidden_batch(w, batch, attempts, t.prototypes, row0=row0)
    res = oracle.masked_topk_tokens(head, hidden)
    redraws = 0
    for _ in range(max_attempts):
        bad = res["score_margin"] <= MARGIN
        if need_logit_margin:
            bad |= res["logit_margin"] <= MARGIN
        idx = np.nonzero(bad)[0]
        if idx.size == 0:
            break
        redraws += idx.size
        attempts[idx] += 1
        for i in idx:
            hidden[i] = synth.hidden_row(w, row0 + int(i), int(attempts[i]), t.prototypes)
        sub = oracle.masked_topk_tokens(head, hidden[idx])
        for k in res:
            res[k][idx] = sub[k]
    else:
        raise RuntimeError("could not draw rows away from near-ties")
    return hidden, res, redraws


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    ninf_ref = np.isneginf(ref)
    ninf_gpu = np.isneginf(gpu)
    if not np.array_equal(ninf_ref, ninf_gpu):
        n = int((ninf_ref != ninf_gpu).sum())
        raise AssertionError(f"{what}: -inf pattern differs at {n} entries")
    fin = ~ninf_ref
    err = np.abs(gpu[fin] - ref[fin])
    bound = ATOL + RTOL * np.abs(ref[fin])
    bad = err > bound
    if bad.any():
        i = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: {int(bad.sum())} entries out of tolerance; worst |d|="
                             f"{err[i]:.3e} bound {bound[i]:.3e}")
    assert np.all(np.isfinite(gpu[fin])), f"{what}: non-finite values where finite expected"


def bf16_tensor(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
