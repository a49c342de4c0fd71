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


def test_exports_nothing_beyond_the_header(L):
    """The library's dynamic symbols are the header's entry points; everything else is
    hidden (built with -fvisibility=hidden), apart from the C++ standard library's own
    template instantiations, which the toolchain exports as weak symbols."""
    import shutil
    import subprocess
    from centroid_masked_sparse_gb300 import _lib
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    names = {line.split()[-1] for line in out.splitlines() if line.strip()}
    extra = {n for n in names - _declared() if not re.match(r"_Z(NK?)?St", n)}
    assert not extra, sorted(extra)


def test_status_strings_and_version(L):
    for code in range(-6, 1):
        assert L.mtp_status_string(code)
    assert L.mtp_status_string(-99) == b"unknown status"
    assert L.mtp_version() >= 100


def _desc(V=262144, H=1536, C=2048, K=32, cw=0x1000, ew=0x2000, ordering=0x3000, offsets=None,
          ld=None):
    from centroid_masked_sparse_gb300._lib import MtpHeadDesc
    return MtpHeadDesc(vocab_size=V, hidden_size=H, num_centroids=C, top_k=K, device=0,
                       flags=0, centroid_w=cw, embed_w=ew, ld_embed=ld if ld else H,
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


def test_packed_table_sizes_and_checks(L):
    # uniform clusters of 128: no padding, exactly V*H*2 bytes of blocks + poff[C+1]
    d = _desc()
    assert L.mtp_packed_embeddings_bytes(ctypes.byref(d)) == 262144 * 1536 * 2 + 2049 * 4
    # explicit offsets: bound with 31 padding rows per cluster
    d = _desc(offsets=0x5000)
    groups = (262144 + 31 * 2048 + 31) // 32
    assert L.mtp_packed_embeddings_bytes(ctypes.byref(d)) == (groups + 3) // 4 * 24 * 16384 + 2049 * 4
    # a K tail (H = 72: two k-blocks) and clusters of 40 (two groups of 32 each): 16 groups
    # make 4 blocks of 128 rows per k-block
    d = _desc(V=40 * 8, H=72, C=8, K=2)
    assert L.mtp_packed_embeddings_bytes(ctypes.byref(d)) == 4 * 2 * 16384 + 9 * 4
    d = _desc(V=40 * 9, H=72, C=9, K=2)   # 18 groups -> 5 super-groups
    assert L.mtp_packed_embeddings_bytes(ctypes.byref(d)) == 5 * 2 * 16384 + 10 * 4
    assert L.mtp_packed_embeddings_bytes(ctypes.byref(_desc(H=12))) == 0
    assert L.mtp_packed_embeddings_bytes(None) == 0
    # the packed table must be 256-byte aligned when attached
    d = _desc()
    d.embed_packed = 0xA010
    out = ctypes.c_void_p(0x8000)
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, out, None, WS, 1 << 30, None) == -3
    # building it: null, misaligned, small and overlapping buffers are refused before any launch
    d = _desc(V=1024, H=64, C=16, ew=0x100000)
    need = L.mtp_packed_embeddings_bytes(ctypes.byref(d))
    big = ctypes.c_void_p(0x4000000)
    assert L.mtp_pack_embeddings(ctypes.byref(d), None, need, None, None) == -1
    assert L.mtp_pack_embeddings(None, big, need, None, None) == -1
    assert L.mtp_pack_embeddings(ctypes.byref(_desc(V=1024, H=64, C=16, ordering=None)), big, need,
                                 None, None) == -1
    assert L.mtp_pack_embeddings(ctypes.byref(d), ctypes.c_void_p(0x4000010), need, None, None) == -3
    assert L.mtp_pack_embeddings(ctypes.byref(d), big, need, ctypes.c_void_p(0x9004), None) == -3
    assert L.mtp_pack_embeddings(ctypes.byref(d), big, need - 1, None, None) == -4
    # [V, H] bf16 at 0x100000 spans 128 KiB: a packed buffer starting inside it overlaps
    assert L.mtp_pack_embeddings(ctypes.byref(d), ctypes.c_void_p(0x110000), need, None, None) == -2
    assert L.mtp_pack_embeddings(ctypes.byref(_desc(V=1000, H=64, C=16, ew=0x100000)), big, need,
                                 None, None) == -2


def test_gather_plan(L):
    d = _desc()
    assert L.mtp_gather_plan(ctypes.byref(d), 64) == 0      # B*K = C: CUDA-core gather
    assert L.mtp_gather_plan(ctypes.byref(d), 13) == 0
    assert L.mtp_gather_plan(ctypes.byref(d), 12) == 2      # a dozen rows: the direct one
    assert L.mtp_gather_plan(ctypes.byref(d), 11) == 2
    assert L.mtp_gather_plan(ctypes.byref(d), 10) == 3      # up to 10 rows (uniform clusters,
    assert L.mtp_gather_plan(ctypes.byref(d), 8) == 3       # H <= 1536): the fused kernel
    assert L.mtp_gather_plan(ctypes.byref(d), 1) == 3
    assert L.mtp_gather_plan(ctypes.byref(_desc(K=1025, C=2048)), 1) == 2   # fused: K <= 1024
    assert L.mtp_gather_plan(ctypes.byref(d), 256) == 1     # B*K = 4C: large buckets
    assert L.mtp_gather_plan(ctypes.byref(d), 0) == 0
    assert L.mtp_gather_plan(ctypes.byref(d), -1) == -2
    assert L.mtp_gather_plan(ctypes.byref(d), 2000) == -6
    assert L.mtp_gather_plan(ctypes.byref(_desc(K=0)), 8) == -2
    d.embed_packed = 0xA000                                  # packed table: from B*K >= C/5
    assert L.mtp_gather_plan(ctypes.byref(d), 64) == 1
    assert L.mtp_gather_plan(ctypes.byref(d), 16) == 1
    assert L.mtp_gather_plan(ctypes.byref(d), 13) == 1
    assert L.mtp_gather_plan(ctypes.byref(d), 12) == 2       # below: up to 12 rows direct
    d = _desc(K=16)                                          # the same rule at any batch size
    d.embed_packed = 0xA000
    assert L.mtp_gather_plan(ctypes.byref(d), 25) == 0
    assert L.mtp_gather_plan(ctypes.byref(d), 26) == 1
    assert L.mtp_gather_plan(ctypes.byref(d), 65) == 1
    assert L.mtp_gather_plan(ctypes.byref(d), 128) == 1
    d = _desc(H=256)                                         # small hidden size, token order:
    assert L.mtp_gather_plan(ctypes.byref(d), 20) == 2       # the direct gather up to 20 rows,
    assert L.mtp_gather_plan(ctypes.byref(d), 13) == 2
    assert L.mtp_gather_plan(ctypes.byref(d), 21) == 1       # then tensor cores (B*K >= C/4)
    assert L.mtp_gather_plan(ctypes.byref(d), 64) == 1
    d = _desc(H=256)                                         # and packed: from B*K >= C/16
    d.embed_packed = 0xA000
    assert L.mtp_gather_plan(ctypes.byref(d), 11) == 1
    assert L.mtp_gather_plan(ctypes.byref(d), 10) == 2      # up to 10 rows of 512 bytes: direct
    assert L.mtp_gather_plan(ctypes.byref(d), 8) == 2
    assert L.mtp_gather_plan(ctypes.byref(d), 3) == 2
    assert L.mtp_gather_plan(ctypes.byref(_desc(H=512)), 8) == 3   # above H=256: fused
    d = _desc(offsets=0x5000)                                # ragged clusters: the same rules but C/4
    assert L.mtp_gather_plan(ctypes.byref(d), 64) == 0
    assert L.mtp_gather_plan(ctypes.byref(d), 9) == 2        # and the fused kernel to 8 rows
    assert L.mtp_gather_plan(ctypes.byref(_desc(H=2048)), 9) == 2   # (also above H=1536)
    d.embed_packed = 0xA000
    assert L.mtp_gather_plan(ctypes.byref(d), 64) == 1
    assert L.mtp_gather_plan(ctypes.byref(d), 16) == 1
    assert L.mtp_gather_plan(ctypes.byref(d), 15) == 0       # packed, ragged: from B*K >= C/4
    assert L.mtp_gather_plan(ctypes.byref(d), 8) == 3
    assert L.mtp_gather_plan(ctypes.byref(d), 256) == 1


def test_forced_gather(L):
    d = _desc()
    try:
        for kind in (0, 1, 2, 3):
            assert L.mtp_force_gather(kind) == 0
            assert L.mtp_gather_plan(ctypes.byref(d), 4) == kind
        assert L.mtp_force_gather(2) == 0                   # the direct kernel: at most 32 rows
        assert L.mtp_gather_plan(ctypes.byref(d), 33) == -6
        assert L.mtp_force_gather(3) == 0                   # the fused kernel: K <= 1024
        assert L.mtp_gather_plan(ctypes.byref(_desc(K=1025, C=2048)), 4) == -6
        assert L.mtp_force_gather(4) == -2
        assert L.mtp_force_gather(-2) == -2
    finally:
        assert L.mtp_force_gather(-1) == 0
    assert L.mtp_gather_plan(ctypes.byref(d), 4) == 3


def test_wait_test_control(L):
    assert L.mtp_wait_test(-1, 0) == -2
    assert L.mtp_wait_test(1000000, 1) == 0
    assert L.mtp_wait_test(0, 0) == 0                       # back to the default


def test_graph_capture_rejects_bad_arguments(L):
    d = _desc()
    g = ctypes.c_void_p(0x1234)
    out = ctypes.c_void_p(0x8000)
    assert L.mtp_graph_capture(ctypes.byref(d), 0, FAKE, 4, out, None, WS, 1 << 30, None,
                               ctypes.byref(g)) == -1          # the legacy stream cannot be captured
    assert g.value is None                                    # *graph is cleared on every failure
    st = ctypes.c_void_p(0x77)
    assert L.mtp_graph_capture(ctypes.byref(d), 3, FAKE, 4, out, None, WS, 1 << 30, st,
                               ctypes.byref(g)) == -2          # unknown finish
    assert L.mtp_graph_capture(ctypes.byref(d), 0, FAKE, 0, out, None, WS, 1 << 30, st,
                               ctypes.byref(g)) == -2          # nothing to record
    assert L.mtp_graph_capture(ctypes.byref(d), 0, FAKE, 4, out, None, WS, 1 << 30, st, None) == -1
    # the eager call's own checks come first (misaligned hidden states)
    assert L.mtp_graph_capture(ctypes.byref(d), 0, ctypes.c_void_p(0x7002), 4, out, None, WS,
                               1 << 30, st, ctypes.byref(g)) == -3
    assert L.mtp_graph_launch(None, None) == -1
    assert L.mtp_graph_destroy(None) == 0


def test_select_and_score_rejects_bad_arguments(L):
    d = _desc()
    out = ctypes.c_void_p(0x8000)
    ids = ctypes.c_void_p(0x9000000)
    # the pair's width K*S needs uniform clusters
    assert L.mtp_select_and_score(ctypes.byref(_desc(offsets=0x5000)), FAKE, 4, out, ids, WS,
                                  1 << 30, None) == -6
    assert L.mtp_select_and_score(ctypes.byref(d), None, 4, out, ids, WS, 1 << 30, None) == -1
    assert L.mtp_select_and_score(ctypes.byref(d), FAKE, 4, None, ids, WS, 1 << 30, None) == -1
    assert L.mtp_select_and_score(ctypes.byref(d), ctypes.c_void_p(0x7002), 4, out, ids, WS,
                                  1 << 30, None) == -3
    assert L.mtp_select_and_score(ctypes.byref(d), FAKE, 4, out, ids, WS, 16, None) == -4
    assert L.mtp_select_and_score(ctypes.byref(d), FAKE, -2, out, ids, WS, 1 << 30, None) == -2
    assert L.mtp_select_and_score(ctypes.byref(d), None, 0, None, None, None, 0, None) == 0


def test_key_exchange_rejects_bad_arguments(L):
    """The sharded head's key export and decode check their arguments on the host, in the
    header's order, before any device work; an empty batch is a no-op."""
    d = _desc()
    keys = ctypes.c_void_p(0x8000)
    tok = ctypes.c_void_p(0xA000)
    big = 1 << 30
    assert L.mtp_masked_topk_keys(None, FAKE, 4, keys, WS, big, None) == -1
    assert L.mtp_masked_topk_keys(ctypes.byref(d), None, 4, keys, WS, big, None) == -1
    assert L.mtp_masked_topk_keys(ctypes.byref(d), FAKE, 4, None, WS, big, None) == -1
    assert L.mtp_masked_topk_keys(ctypes.byref(d), ctypes.c_void_p(0x7001), 4, keys, WS, big, None) == -3
    assert L.mtp_masked_topk_keys(ctypes.byref(d), FAKE, 4, keys, None, 0, None) == -4
    assert L.mtp_masked_topk_keys(ctypes.byref(d), FAKE, 4, keys, WS, 16, None) == -4
    assert L.mtp_masked_topk_keys(ctypes.byref(d), FAKE, -1, keys, WS, big, None) == -2
    assert L.mtp_masked_topk_keys(ctypes.byref(d), FAKE, 1025, keys, WS, big, None) == -6
    assert L.mtp_masked_topk_keys(ctypes.byref(d), None, 0, None, None, 0, None) == 0
    assert L.mtp_decode_keys(None, 4, tok, None, None) == -1
    assert L.mtp_decode_keys(keys, 4, None, None, None) == -1
    assert L.mtp_decode_keys(keys, -3, tok, None, None) == -2
    assert L.mtp_decode_keys(keys, 1025, tok, None, None) == -6
    assert L.mtp_decode_keys(None, 0, None, None, None) == 0


def test_noalloc_host_checks(L):
    """The allocation-free entry point refuses, before any device work, requests whose
    workspace would exceed its fixed 8 MiB scratch: 943 rows of the V=262144, C=2048, K=32
    head fit, 944 do not; empty and negative batches behave as in the workspace call."""
    d = _desc()
    out = ctypes.c_void_p(0x8000)
    assert L.mtp_workspace_bytes(ctypes.byref(d), 943) <= 8 << 20 < L.mtp_workspace_bytes(ctypes.byref(d), 944)
    assert L.mtp_masked_topk_tokens_noalloc(None, FAKE, 4, out, None, None) == -1
    assert L.mtp_masked_topk_tokens_noalloc(ctypes.byref(d), FAKE, 0, out, None, None) == 0
    assert L.mtp_masked_topk_tokens_noalloc(ctypes.byref(d), FAKE, -1, out, None, None) == -2
    assert L.mtp_masked_topk_tokens_noalloc(ctypes.byref(d), FAKE, 944, out, None, None) == -6
    # the workspace call's checks come first, with its statuses, whatever the size
    assert L.mtp_masked_topk_tokens_noalloc(ctypes.byref(_desc(ew=0)), FAKE, 944, out, None, None) == -1
    assert L.mtp_masked_topk_tokens_noalloc(ctypes.byref(d), ctypes.c_void_p(0x7008), 944, out, None,
                                            None) == -3
    assert L.mtp_masked_topk_tokens_noalloc(ctypes.byref(d), FAKE, 4, None, None, None) == -1
    assert L.mtp_masked_topk_tokens_noalloc(ctypes.byref(_desc(K=0)), FAKE, 944, out, None, None) == -2
    word = ctypes.c_uint32(0)
    assert L.mtp_noalloc_read_device_error(0, None, None) == -1
    assert L.mtp_noalloc_read_device_error(-1, ctypes.byref(word), None) == -2


def test_cluster_range_checks_and_packed_size(L):
    out = ctypes.c_void_p(0x8000)
    for b, e in ((5, 3), (-1, 4), (0, 2049)):
        d = _desc()
        d.cluster_begin, d.cluster_end = b, e
        assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, out, None, WS, 1 << 30, None) == -2
        assert L.mtp_packed_embeddings_bytes(ctypes.byref(d)) == 0
    # a shard of half the clusters packs half the blocks (poff still covers all C)
    d = _desc()
    d.cluster_begin, d.cluster_end = 0, 1024
    assert L.mtp_packed_embeddings_bytes(ctypes.byref(d)) == 1024 * 24 * 16384 + 2049 * 4
    d.cluster_begin, d.cluster_end = 1024, 2048
    assert L.mtp_packed_embeddings_bytes(ctypes.byref(d)) == 1024 * 24 * 16384 + 2049 * 4
    # keys: argument checks
    keys = ctypes.c_void_p(0xB000)
    d = _desc()
    assert L.mtp_masked_topk_keys(ctypes.byref(d), FAKE, 4, None, WS, 1 << 30, None) == -1
    assert L.mtp_masked_topk_keys(ctypes.byref(d), FAKE, 4, keys, WS, 16, None) == -4
    assert L.mtp_masked_topk_keys(ctypes.byref(d), FAKE, 0, None, None, 0, None) == 0
    assert L.mtp_decode_keys(None, 4, out, None, None) == -1
    assert L.mtp_decode_keys(keys, 4, None, None, None) == -1
    assert L.mtp_decode_keys(keys, -1, out, None, None) == -2
    assert L.mtp_decode_keys(None, 0, None, None, None) == 0


def test_unknown_flags_are_refused(L):
    out = ctypes.c_void_p(0x8000)
    d = _desc()
    for bad in (16, 1 << 30, 15 | 32):
        d.flags = bad
        assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, out, None, WS, 1 << 30, None) == -6
        assert L.mtp_dense_lm_head(ctypes.byref(d), FAKE, 4, out, None, None, None, 0, None) == -6
    d.flags = 7
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, out, None, WS, 16, None) == -4


def test_host_hidden_flag_host_checks(L):
    """MTP_FLAG_HOST_HIDDEN: the workspace grows by the staged rows (B * H * 2 bytes,
    with the layout's 256-byte rounding), calls without a workspace refuse the flag, and
    a short workspace is refused before anything else happens."""
    out = ctypes.c_void_p(0x8000)
    d = _desc()
    plain = [L.mtp_workspace_bytes(ctypes.byref(d), b) for b in (1, 7, 64)]
    d.flags = 8
    staged = [L.mtp_workspace_bytes(ctypes.byref(d), b) for b in (1, 7, 64)]
    for b, p0, p1 in zip((1, 7, 64), plain, staged):
        assert p1 - p0 == (b * 1536 * 2 + 255) // 256 * 256
    scores = ctypes.c_void_p(0x9000)
    assert L.mtp_centroid_scores(ctypes.byref(d), FAKE, 4, scores, None, None) == -6
    assert L.mtp_centroid_scores(ctypes.byref(d), FAKE, 0, scores, None, None) == 0
    # the dense head needs the workspace for the staged rows even without an argmax
    assert L.mtp_dense_lm_head(ctypes.byref(d), FAKE, 4, out, None, None, None, 0, None) == -4
    need = L.mtp_workspace_bytes(ctypes.byref(d), 4)
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, out, None, WS, need - 1, None) == -4
    d.flags = 8 | 7   # combines with the fidelity options
    assert L.mtp_masked_topk_tokens(ctypes.byref(d), FAKE, 4, out, None, WS, 16, None) == -4


def test_softcap_checks(L):
    out = ctypes.c_void_p(0x8000)
    for cap in (-1.0, float("nan")):
        d = _desc()
        d.final_logit_softcap = cap
        assert L.mtp_dense_lm_head(ctypes.byref(d), FAKE, 4, out, None, None, None, 0, None) == -2
    d = _desc()
    d.final_logit_softcap = 30.0
    assert L.mtp_dense_lm_head(ctypes.byref(d), FAKE, 4, None, None, None, None, 0, None) == -1
