"""The allocation-free sparse argmax (mtp_masked_topk_tokens_noalloc).

Callers that are handed only input and output buffers (no allocator), or that
cannot afford cudaMalloc, use this entry point: it keeps its scratch in a
fixed-size array inside the library's device memory instead of a caller
workspace.  Its results must equal those of mtp_masked_topk_tokens, which runs
the same kernels on a workspace allocated by the caller, and the oracle's, on
consecutive calls that share the array while the shapes, the gather kernel and
the array's layout change from call to call.  This file is collected last on
purpose.
"""
import ctypes

import numpy as np
import pytest

from centroid_masked_sparse_gb300 import synth
from oracle import oracle
from tests import helpers

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _lib_and_module():
    from centroid_masked_sparse_gb300 import build
    build.build()
    import centroid_masked_sparse_gb300 as m
    from centroid_masked_sparse_gb300 import _lib
    return m, _lib.lib()


_HEADS = {}


def _head(m, name):
    if name not in _HEADS:
        t = helpers.tables(name)
        w = synth.WORKLOADS[name]
        _HEADS[name] = (oracle.Head.from_tables(t, w.top_k),
                        m.MaskedHead.from_host(t.centroid_w, t.embed_w, t.token_ordering, t.cluster_offsets,
                                               w.top_k))
    return _HEADS[name]


def _noalloc(L, dh, h, B, stream, host_out=False):
    kw = dict(dtype=torch.int32)
    if host_out:
        tok = torch.full((B,), -7, **kw).pin_memory()
        mx = torch.full((B,), 7.0, dtype=torch.float32).pin_memory()
    else:
        tok = torch.full((B,), -7, device="cuda", **kw)
        mx = torch.full((B,), 7.0, dtype=torch.float32, device="cuda")
    st = L.mtp_masked_topk_tokens_noalloc(ctypes.byref(dh.desc), ctypes.c_void_p(h.data_ptr()), B,
                                          ctypes.c_void_p(tok.data_ptr()), ctypes.c_void_p(mx.data_ptr()),
                                          stream)
    assert st == 0, L.mtp_status_string(st)
    return tok, mx


def _device_error(L, stream):
    word = ctypes.c_uint32(0xFFFFFFFF)
    assert L.mtp_noalloc_read_device_error(torch.cuda.current_device(), ctypes.byref(word), stream) == 0
    torch.cuda.synchronize()
    return word.value


# name, batch, oracle check: each call changes the scratch layout (scores, work items and
# the staging region move with the batch and the tables), and the gather kernel with it
SEQUENCE = [
    ("shared", 256, True),      # tensor-core-sized buckets, C=4096, K=128
    ("uniform", 64, True),      # pipelined CUDA-core gather (token-order table)
    ("uniform", 8, True),       # fused small-batch kernel
    ("uniform", 1, True),
    ("variable", 64, True),     # lognormal clusters, H=2560
    ("uniform", 943, False),    # the largest batch whose workspace fits the 8 MiB array
    ("uniform", 3, True),
]


def test_noalloc_matches_workspace_call_and_oracle_on_consecutive_calls():
    m, L = _lib_and_module()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for i, (name, B, with_oracle) in enumerate(SEQUENCE):
        oh, dh = _head(m, name)
        assert L.mtp_workspace_bytes(ctypes.byref(dh.desc), B) <= 8 << 20
        if with_oracle:
            hidden, ref, _ = helpers.clean_batch(name, oh, B, row0=7000 + 1000 * i)
        else:
            hidden = synth.hidden_batch(name, B, row0=7000 + 1000 * i)
        h = helpers.bf16_tensor(hidden)
        ref_tok, ref_max = m.mtp_masked_topk_tokens(dh, h, workspace=dh.workspace(B))
        tok, mx = _noalloc(L, dh, h, B, stream)
        torch.cuda.synchronize()
        what = f"call {i}: {name} B={B}"
        np.testing.assert_array_equal(tok.cpu().numpy(), ref_tok.cpu().numpy(), err_msg=what)
        np.testing.assert_array_equal(mx.cpu().numpy(), ref_max.cpu().numpy(), err_msg=what)
        if with_oracle:
            np.testing.assert_array_equal(tok.cpu().numpy(), ref["tokens"], err_msg=what)
            helpers.assert_close(mx.cpu().numpy(), ref["max_logit"], what)
        assert _device_error(L, stream) == 0, what


def test_noalloc_host_resident_hidden_states():
    """MTP_FLAG_HOST_HIDDEN stages the pinned batch at the end of the scratch layout; token
    ids and max logits go straight to pinned host memory."""
    m, L = _lib_and_module()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    oh, dh = _head(m, "uniform")
    hh = dh.with_flags(m.MTP_FLAG_HOST_HIDDEN)
    for B in (64, 5):
        hidden, ref, _ = helpers.clean_batch("uniform", oh, B, row0=31000 + B)
        h_host = helpers.bf16_tensor(hidden).cpu().pin_memory()
        tok, mx = _noalloc(L, hh, h_host, B, stream, host_out=True)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(tok.numpy(), ref["tokens"])
        helpers.assert_close(mx.numpy(), ref["max_logit"], f"host hidden B={B}")
        assert _device_error(L, stream) == 0


def test_noalloc_reports_device_errors():
    """A token id outside [0, V) in token_ordering is reported through the array's error
    word (mtp_noalloc_read_device_error), and the next clean call resets it."""
    m, L = _lib_and_module()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t = synth.custom_tables(1024, 64, 16, 5, std=0.05)
    bad = t.token_ordering.copy()
    bad[10] = 1024 + 7       # owned by centroid 0, selected since K = C
    cw, ew = helpers.bf16_tensor(t.centroid_w), helpers.bf16_tensor(t.embed_w)
    dbad = m.MaskedHead(cw, ew, torch.from_numpy(bad).cuda(), 16, vocab_size=1024)
    dok = m.MaskedHead(cw, ew, torch.from_numpy(t.token_ordering).cuda(), 16, vocab_size=1024)
    h = helpers.bf16_tensor(synth.random_hidden(4, 64, 6))
    _noalloc(L, dbad, h, 4, stream)
    assert _device_error(L, stream) & m.MTP_DEVERR_TOKEN_RANGE
    tok, _ = _noalloc(L, dok, h, 4, stream)
    assert _device_error(L, stream) == 0
    ref, _ = m.mtp_masked_topk_tokens(dok, h)
    torch.cuda.synchronize()
    assert torch.equal(tok, ref)


def test_noalloc_rejects_requests_beyond_its_scratch():
    m, L = _lib_and_module()
    from centroid_masked_sparse_gb300._lib import MtpHeadDesc
    # 1024 rows x 4096 centroids of fp32 scores alone need 16 MiB
    d = MtpHeadDesc(vocab_size=262144, hidden_size=2048, num_centroids=4096, top_k=128, device=0,
                    flags=0, centroid_w=0x1000, embed_w=0x2000, ld_embed=2048,
                    token_ordering=0x3000, cluster_offsets=None)
    assert L.mtp_workspace_bytes(ctypes.byref(d), 1024) > 8 << 20
    out = ctypes.c_void_p(0x8000)
    assert L.mtp_masked_topk_tokens_noalloc(ctypes.byref(d), ctypes.c_void_p(0x7000), 1024, out,
                                            None, None) == -6
