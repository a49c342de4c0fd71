"""Python face of the CPU oracle (``mtp_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg are the only users.  The product library never
imports this module and this module never imports the product library; the
two meet only through the seeded generator (``synth``).

The C file is compiled with gcc into ``oracle/_build/libmtp_oracle.so`` by
``build()`` (also called lazily on first use).  Calls over a batch can be split
over threads by row: the C functions take a row range and ctypes releases the
GIL during a foreign call.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mtp_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmtp_oracle.so")
_lock = threading.Lock()
_lib = None

_p = ctypes.c_void_p
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math, no -march)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fno-fast-math",
                        "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_SIGS = {
    "orc_centroid_scores": [_p, _i64, _i64, _i64, _p, _i64, _p],
    "orc_topk_row": [_p, _i64, _i64, _p, _p],
    "orc_masked_topk_tokens": [_p, _i64, _i64, _i64, _p, _i64, _i64, _p, _i64, _i64,
                               _p, _p, _p, _p, _p, _p, _p, _p, _i64],
    "orc_masked_scatter_logits": [_p, _i64, _i64, _i64, _p, _i64, _i64, _p, _i64,
                                  _i64, _p, _p, _p, _i64],
    "orc_select_and_score_row": [_p, _i64, _i64, _p, _i64, _i64, _p, _i64, _i64,
                                 _p, _p, _p, _p, _i64, _p, _i64],
    "orc_dense_logits": [_p, _i64, _i64, _i64, _p, _i64, _i64, _p, _i64, ctypes.c_double],
    "orc_dense_logits_at": [_p, _i64, _p, _i64, _p, _p, _i64, _p],
    "orc_is_permutation": [_p, _i64],
}


def load_library(path: str):
    """Load an oracle shared library and declare its C signatures."""
    L = ctypes.CDLL(path)
    for name, args in _SIGS.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.orc_round_bf16.argtypes = [ctypes.c_double]
    L.orc_round_bf16.restype = ctypes.c_double
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load_library(_LIB_PATH)
    return _lib


FLAG_FILL_FINFO_MIN = 1
FLAG_BF16_SCORES = 2
FLAG_BF16_LOGITS = 4


def round_bf16(x: float) -> float:
    """x rounded to the nearest bf16 value, ties to even (the oracle's own rounding)."""
    return float(lib().orc_round_bf16(float(x)))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _threads(threads: int | None) -> int:
    return max(1, threads if threads else (os.cpu_count() or 1))


def _row_split(B: int, threads: int):
    n = max(1, min(threads, B))
    step = (B + n - 1) // n
    return [(b, min(B, b + step)) for b in range(0, B, step)]


class Head:
    """The head's tables as the oracle sees them (all host numpy arrays).

    centroid_w   uint16 [C, H]   bf16 bits
    embed_w      uint16 [V', ld] bf16 bits, token-id order, V' >= V, ld >= H
    ordering     int32  [V]      ordered position -> token id
    offsets      int32  [C+1] or None (uniform clusters of V/C)
    flags        FLAG_* reference-fidelity options (0: fp64 scores and logits, -inf fill)
    softcap      the dense comparator's final logit softcap (0: none)
    """

    def __init__(self, centroid_w, embed_w, ordering, offsets, top_k, vocab=None, flags=0,
                 softcap=0.0):
        self.centroid_w = np.ascontiguousarray(centroid_w, dtype=np.uint16)
        self.embed_w = np.ascontiguousarray(embed_w, dtype=np.uint16)
        self.ordering = np.ascontiguousarray(ordering, dtype=np.int32)
        self.offsets = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.int32)
        self.C, self.H = self.centroid_w.shape
        self.ld = self.embed_w.shape[1]
        self.V = int(vocab) if vocab is not None else int(self.ordering.shape[0])
        self.K = int(top_k)
        self.flags = int(flags)
        self.softcap = float(softcap)

    @classmethod
    def from_tables(cls, t, top_k=None):
        return cls(t.centroid_w, t.embed_w, t.token_ordering, t.cluster_offsets,
                   top_k if top_k is not None else t.workload.top_k)

    def cluster_range(self, c: int):
        if self.offsets is None:
            s = self.V // self.C
            return c * s, (c + 1) * s
        return int(self.offsets[c]), int(self.offsets[c + 1])


def centroid_scores(head: Head, hidden: np.ndarray, threads: int | None = None) -> np.ndarray:
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    B = hidden.shape[0]
    out = np.empty((B, head.C), dtype=np.float64)
    L = lib()

    def run(r):
        _check(L.orc_centroid_scores(_ptr(hidden), r[0], r[1], head.H, _ptr(head.centroid_w),
                                     head.C, _ptr(out)), "centroid_scores")

    with ThreadPoolExecutor(_threads(threads)) as ex:
        list(ex.map(run, _row_split(B, _threads(threads))))
    return out


def topk_row(scores_row: np.ndarray, K: int):
    s = np.ascontiguousarray(scores_row, dtype=np.float64)
    sel = np.empty(K, dtype=np.int32)
    margin = ctypes.c_double()
    _check(lib().orc_topk_row(_ptr(s), s.shape[0], K, _ptr(sel), ctypes.byref(margin)), "topk")
    return sel, margin.value


def masked_topk_tokens(head: Head, hidden: np.ndarray, threads: int | None = None) -> dict:
    """Sparse argmax per row plus the selection and the near-tie margins."""
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    B = hidden.shape[0]
    res = dict(tokens=np.empty(B, np.int32), max_logit=np.empty(B, np.float64),
               score_margin=np.empty(B, np.float64), logit_margin=np.empty(B, np.float64),
               sel=np.empty((B, head.K), np.int32), n_cand=np.empty(B, np.int64))
    L = lib()

    def run(r):
        _check(L.orc_masked_topk_tokens(
            _ptr(hidden), r[0], r[1], head.H, _ptr(head.centroid_w), head.C, head.K,
            _ptr(head.embed_w), head.ld, head.V, _ptr(head.ordering), _ptr(head.offsets),
            _ptr(res["tokens"]), _ptr(res["max_logit"]), _ptr(res["score_margin"]),
            _ptr(res["logit_margin"]), _ptr(res["sel"]), _ptr(res["n_cand"]), head.flags),
            "masked_topk_tokens")

    nt = _threads(threads)
    if nt == 1 or B == 1:
        run((0, B))
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(run, [(b, b + 1) for b in range(B)]))
    return res


def masked_scatter_logits(head: Head, hidden: np.ndarray, threads: int | None = None) -> np.ndarray:
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    B = hidden.shape[0]
    out = np.empty((B, head.V), dtype=np.float64)
    L = lib()

    def run(r):
        _check(L.orc_masked_scatter_logits(
            _ptr(hidden), r[0], r[1], head.H, _ptr(head.centroid_w), head.C, head.K,
            _ptr(head.embed_w), head.ld, head.V, _ptr(head.ordering), _ptr(head.offsets),
            _ptr(out), head.flags), "masked_scatter_logits")

    nt = _threads(threads)
    with ThreadPoolExecutor(nt) as ex:
        list(ex.map(run, [(b, b + 1) for b in range(B)]))
    return out


def select_and_score_row(head: Head, hidden: np.ndarray, b: int):
    """(logits, token ids) of row b's candidates in the page's order."""
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    cap = head.V
    toks = np.empty(cap, np.int32)
    logs = np.empty(cap, np.float64)
    n = ctypes.c_int64()
    _check(lib().orc_select_and_score_row(
        _ptr(hidden), b, head.H, _ptr(head.centroid_w), head.C, head.K, _ptr(head.embed_w),
        head.ld, head.V, _ptr(head.ordering), _ptr(head.offsets), _ptr(toks), _ptr(logs),
        cap, ctypes.byref(n), head.flags), "select_and_score_row")
    return logs[:n.value].copy(), toks[:n.value].copy()


def dense_logits(head: Head, hidden: np.ndarray, threads: int | None = None) -> np.ndarray:
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    B = hidden.shape[0]
    out = np.empty((B, head.V), dtype=np.float64)
    L = lib()

    def run(r):
        _check(L.orc_dense_logits(_ptr(hidden), r[0], r[1], head.H, _ptr(head.embed_w),
                                  head.ld, head.V, _ptr(out), head.flags, head.softcap),
               "dense_logits")

    nt = _threads(threads)
    with ThreadPoolExecutor(nt) as ex:
        list(ex.map(run, _row_split(B, nt)))
    return out


def dense_logits_at(head: Head, hidden: np.ndarray, rows, tokens,
                    threads: int | None = None) -> np.ndarray:
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    n = rows.shape[0]
    out = np.empty(n, dtype=np.float64)
    L = lib()
    nt = _threads(threads)
    parts = _row_split(n, nt) if n else []

    def run(r):
        _check(L.orc_dense_logits_at(_ptr(hidden), head.H, _ptr(head.embed_w), head.ld,
                                     _ptr(rows[r[0]:r[1]]), _ptr(tokens[r[0]:r[1]]),
                                     r[1] - r[0], _ptr(out[r[0]:r[1]])), "dense_logits_at")

    with ThreadPoolExecutor(nt) as ex:
        list(ex.map(run, parts))
    return out


def is_permutation(ordering: np.ndarray) -> bool:
    o = np.ascontiguousarray(ordering, dtype=np.int32)
    return bool(lib().orc_is_permutation(_ptr(o), o.shape[0]))
