"""ctypes loader and signatures for ``libmtp_head.so`` (the C ABI of include/mtp_head.h).

There is no fallback: if the library has not been built the import of the
binding fails with a message saying how to build it.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmtp_head.so")

MTP_OK = 0
STATUS_NAMES = {0: "MTP_OK", -1: "MTP_ERR_NULL", -2: "MTP_ERR_SHAPE", -3: "MTP_ERR_ALIGN",
                -4: "MTP_ERR_WORKSPACE", -5: "MTP_ERR_CUDA", -6: "MTP_ERR_UNSUPPORTED"}
MTP_DEVERR_TOKEN_RANGE = 0x1
MTP_DEVERR_OFFSETS = 0x2
MTP_DEVERR_TIMEOUT = 0x4
MTP_MAX_HIDDEN = 4096
MTP_MAX_CENTROIDS = 16384
MTP_MAX_BATCH = 1024

KERNEL_IDS = {"projection": 0, "topk": 1, "gather_score": 2, "fill": 3, "dense": 4}

# Every function declared in include/mtp_head.h, with its ctypes signature.
_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t


class MtpHeadDesc(ctypes.Structure):
    _fields_ = [
        ("vocab_size", ctypes.c_int32),
        ("hidden_size", ctypes.c_int32),
        ("num_centroids", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("device", ctypes.c_int32),
        ("flags", ctypes.c_int32),
        ("centroid_w", ctypes.c_void_p),
        ("embed_w", ctypes.c_void_p),
        ("ld_embed", ctypes.c_int64),
        ("token_ordering", ctypes.c_void_p),
        ("cluster_offsets", ctypes.c_void_p),
        ("embed_packed", ctypes.c_void_p),
        ("cluster_begin", ctypes.c_int32),
        ("cluster_end", ctypes.c_int32),
        ("final_logit_softcap", ctypes.c_float),
    ]


_DP = ctypes.POINTER(MtpHeadDesc)

SIGNATURES = {
    "mtp_workspace_bytes": (_sz, [_DP, _i32]),
    "mtp_centroid_scores": (_i32, [_DP, _p, _i32, _p, _p, _p]),
    "mtp_masked_topk_tokens": (_i32, [_DP, _p, _i32, _p, _p, _p, _sz, _p]),
    "mtp_masked_scatter_logits": (_i32, [_DP, _p, _i32, _p, _p, _sz, _p]),
    "mtp_dense_lm_head": (_i32, [_DP, _p, _i32, _p, _p, _p, _p, _sz, _p]),
    "mtp_masked_topk_tokens_noalloc": (_i32, [_DP, _p, _i32, _p, _p, _p]),
    "mtp_noalloc_read_device_error": (_i32, [_i32, ctypes.POINTER(ctypes.c_uint32), _p]),
    "mtp_packed_embeddings_bytes": (ctypes.c_size_t, [_DP]),
    "mtp_pack_embeddings": (_i32, [_DP, _p, ctypes.c_size_t, _p, _p]),
    "mtp_gather_plan": (_i32, [_DP, _i32]),
    "mtp_select_and_score": (_i32, [_DP, _p, _i32, _p, _p, _p, ctypes.c_size_t, _p]),
    "mtp_masked_topk_keys": (_i32, [_DP, _p, _i32, _p, _p, ctypes.c_size_t, _p]),
    "mtp_decode_keys": (_i32, [_p, _i32, _p, _p, _p]),
    "mtp_graph_capture": (_i32, [_DP, _i32, _p, _i32, _p, _p, _p, ctypes.c_size_t, _p,
                                 ctypes.POINTER(ctypes.c_void_p)]),
    "mtp_graph_launch": (_i32, [_p, _p]),
    "mtp_graph_destroy": (_i32, [_p]),
    "mtp_read_device_error": (_i32, [_p, ctypes.POINTER(ctypes.c_uint32), _p]),
    "mtp_status_string": (ctypes.c_char_p, [_i32]),
    "mtp_version": (_i32, []),
    "mtp_profile_events": (_i32, [_i32, _p, _p]),
    "mtp_force_gather": (_i32, [_i32]),
    "mtp_wait_test": (_i32, [ctypes.c_int64, _i32]),
}

_lib = None


class MtpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        msg = lib().mtp_status_string(status).decode() if _lib is not None else name
        super().__init__(f"{where}: {name} ({msg})")


def lib():
    """The loaded library (loaded once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"CUDA library not built ({LIB_PATH} missing): run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def check(status: int, where: str) -> None:
    if status != MTP_OK:
        raise MtpError(status, where)
