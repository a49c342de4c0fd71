"""The allocation-free sparse argmax (mtp_masked_topk_tokens_noalloc).

Callers that are handed only input and output buffers (no allocator), or that
cannot afford cudaMalloc, use this entry point: it keeps its scratch in a
fixed-size array inside the library's device memory instead of a caller
workspace.  Its results must equal those of mtp_masked_topk_tokens, which runs
the same kernels on a workspace allocated by the caller, on consecutive calls
that share the array.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from centroid_masked_sparse_gb300 import synth
from tests import helpers

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _lib_and_module():
    from centroid_masked_sparse_gb300 import build
    build.build()
    import centroid_masked_sparse_gb300 as m
    from centroid_masked_sparse_gb300 import _lib
    return m, _lib.lib()


def test_noalloc_matches_workspace_call_on_consecutive_calls():
    m, L = _lib_and_module()
    t = helpers.tables("uniform")
    dh = m.MaskedHead.from_host(t.centroid_w, t.embed_w, t.token_ordering, t.cluster_offsets, 32)
    B = 64
    assert L.mtp_workspace_bytes(ctypes.byref(dh.desc), B) <= 8 << 20
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        hidden = synth.hidden_batch("uniform", B, row0=7000 + call * B)
        h = helpers.bf16_tensor(hidden)
        ref_tok, ref_max = m.mtp_masked_topk_tokens(dh, h)
        tok = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        mx = torch.full((B,), 7.0, dtype=torch.float32, device="cuda")
        st = L.mtp_masked_topk_tokens_noalloc(ctypes.byref(dh.desc), ctypes.c_void_p(h.data_ptr()),
                                              B, ctypes.c_void_p(tok.data_ptr()),
                                              ctypes.c_void_p(mx.data_ptr()), stream)
        assert st == 0, L.mtp_status_string(st)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(tok.cpu().numpy(), ref_tok.cpu().numpy())
        helpers.assert_close(mx.cpu().numpy(), ref_max.cpu().numpy(), f"noalloc call {call}")


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
