"""The C ABI on the host: the library loads, exports every declared entry point,
and rejects bad arguments before touching the GPU (no kernel is launched here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def L():
    from centroid_masked_sparse_gb300 import build
    build.build()
    from centroid_masked_sparse_gb300 import _lib
    return _lib.lib()


def _declared():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            names |= set(re.findall(r"MTP_API\s+[\w\s\*]*?\b(mtp_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(L):
    from centroid_masked_sparse_gb300 import _lib
    names = _declared()
    assert {"mtp_centroid_scores", "mtp_masked_topk_tokens", "mtp_masked_scatter_logits",
            "mtp_dense_lm_head", "mtp_workspace_bytes"} <= names
    for n in names:
        assert hasattr(L, n), n
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature in the binding"


def test_status_strings_and_version(L):
    for code in range(-6, 1):
        assert L.mtp_status_string(code)
    assert L.mtp_status_string(-99) == b"unknown status"
    assert L.mtp_version() >= 100


def _desc(V=262144, H=1536, C=2048, K=32, cw=0x1000, ew=0x2000, ordering=0x3000, offsets=None,
          ld=None):
    from centroid_masked_sparse_gb300._lib import MtpHeadDesc
    return MtpHeadDesc(vocab_size=V, hidden_size=H, num_centroids=C, top_k=K, device=0,
                       reserved0=0, centroid_w=cw, embed_w=ew, ld_embed=ld if ld else H,
                       token_ordering=ordering, cluster_offsets=offsets)


def test_workspace_bytes(L):
    d = _desc()
    b1 = L.mtp_workspace_bytes(ctypes.byref(d), 1)
    b64 = L.mtp_workspace_bytes(ctypes.byref(d), 64)
    assert 0 < b1 < b64
    # scores [B, C] fp32 dominate the batch-dependent part
    assert b64 - b1 >= 63 * 2048 * 4
    assert L.mtp_workspace_bytes(ctypes.byref(d), 0) == 0
    assert L.mtp_workspace_bytes(ctypes.byref(d), 1025) == 0
    bad = _desc(K=4096)
    assert L.mtp_workspace_bytes(ctypes.byref(bad), 8) == 0


FAKE = ctypes.c_void_p(0x7000)
WS = ctypes.c_void_p(0x9000)


@pytest.mark.parametrize("kw,expect", [
    (dict(K=0), -2), (dict(K=2049), -2), (dict(H=12), -2), (dict(H=4104), -6),
    (dict(C=20000, K=4), -6), (dict(V=262145), -2), (dict(ld=1540), -3), (dict(ld=1000), -2),
    (dict(cw=0x1008), -3), (dict(ew=0x2004), -3), (dict(cw=None), -1), (dict(ordering=None), -1),
])
def test_masked_call_rejects_bad_descriptor(L, kw, expect):
    d = _desc(**kw)
    out = ctypes.c_void_p(0x8000)
    st = L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, out, None, WS, 1 << 30, None)
    assert st == expect


def test_masked_call_rejects_bad_arguments(L):
    d = _desc()
    out = ctypes.c_void_p(0x8000)
    assert L.mtp_masked_topk_tokens(None, FAKE, 4, out, None, WS, 1 << 30, None) == -1
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), None, 4, out, None, WS, 1 << 30, None) == -1
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, None, None, WS, 1 << 30, None) == -1
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, -1, out, None, WS, 1 << 30, None) == -2
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 2000, out, None, WS, 1 << 30, None) == -6
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), ctypes.c_void_p(0x7002), 4, out, None, WS,
                                    1 << 30, None) == -3
    need = L.mtp_workspace_bytes(ctypes.byref(d), 4)
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, out, None, WS, need - 1, None) == -4
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, out, None, None, need, None) == -4
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, out, None, ctypes.c_void_p(0x9004),
                                    need, None) == -3
    # an empty batch is a no-op
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), None, 0, None, None, None, 0, None) == 0
    # scatter: output must be 16-byte aligned
    assert L.mtp_masked_scatter_logits(ctypes.byref(d), FAKE, 4, ctypes.c_void_p(0x8004), WS,
                                       1 << 30, None) == -3


def test_dense_and_scores_reject_bad_arguments(L):
    d = _desc()
    assert L.mtp_dense_lm_head(ctypes.byref(d), FAKE, 4, None, None, None, None, 0, None) == -1
    assert L.mtp_dense_lm_head(ctypes.byref(d), FAKE, 4, None, ctypes.c_void_p(0x8000), None, None,
                               0, None) == -4
    assert L.mtp_dense_lm_head(ctypes.byref(d), FAKE, 4, ctypes.c_void_p(0x8000), None,
                               ctypes.c_void_p(0x8100), None, 0, None) == -1
    nd = _desc(ew=None)
    assert L.mtp_dense_lm_head(ctypes.byref(nd), FAKE, 4, ctypes.c_void_p(0x8000), None, None, None,
                               0, None) == -1
    assert L.mtp_centroid_scores(ctypes.byref(d), FAKE, 4, None, None, None) == -1
    assert L.mtp_centroid_scores(ctypes.byref(_desc(K=0)), FAKE, 4, ctypes.c_void_p(0x8000), None,
                                 None) == -2
    assert L.mtp_read_device_error(None, None, None) == -1
    assert L.mtp_profile_events(7, None, None) == -2
    assert L.mtp_profile_events(0, None, None) == 0


def test_ordered_table_checks(L):
    # the optional cluster-ordered table must be 16-byte aligned like the embedding table
    d = _desc()
    d.embed_ordered = 0xA004
    out = ctypes.c_void_p(0x8000)
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, out, None, WS, 1 << 30, None) == -3
    # building it: null, misaligned and overlapping tables are refused before any launch
    d = _desc(V=1024, H=64, ew=0x100000)
    assert L.mtp_reorder_embeddings(ctypes.byref(d), None, None, None) == -1
    assert L.mtp_reorder_embeddings(None, ctypes.c_void_p(0x800000), None, None) == -1
    assert L.mtp_reorder_embeddings(ctypes.byref(_desc(V=1024, H=64, ordering=None)),
                                    ctypes.c_void_p(0x800000), None, None) == -1
    assert L.mtp_reorder_embeddings(ctypes.byref(d), ctypes.c_void_p(0x800008), None, None) == -3
    assert L.mtp_reorder_embeddings(ctypes.byref(d), ctypes.c_void_p(0x800000),
                                    ctypes.c_void_p(0x9004), None) == -3
    # [V, H] bf16 at 0x100000 spans 128 KiB: an output inside that range overlaps it
    assert L.mtp_reorder_embeddings(ctypes.byref(d), ctypes.c_void_p(0x110000), None, None) == -2
    assert L.mtp_reorder_embeddings(ctypes.byref(_desc(V=1024, H=12, ew=0x100000)),
                                    ctypes.c_void_p(0x800000), None, None) == -2
