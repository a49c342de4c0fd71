"""Parity of the CUDA library against the CPU oracle, element by element.

Every workload of the head is covered at its full size: the tiny head, the
Gemma-scale uniform clusters at batches 1..64, lognormal variable clusters, the
full-vocabulary scatter, and the shared-centroid stress case (both finishes),
plus the dense comparator and edge cases (ragged and maximum batches, small and
maximum hidden sizes, empty and oversized clusters, padded tables, exact
integer inputs with forced ties, corrupt orderings caught on the device).
Tolerances are those of tests/helpers.py.
"""
import numpy as np
import pytest

from centroid_masked_sparse_gb300 import synth
from oracle import oracle
from tests import helpers

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="session")
def build_lib():
    from centroid_masked_sparse_gb300 import build
    build.build()
    import centroid_masked_sparse_gb300 as m
    return m


_DEV = {}


def device_head(m, name, top_k=None):
    w = synth.WORKLOADS[name]
    key = (w.table_from or name, top_k)
    if key not in _DEV:
        t = helpers.tables(name)
        k = top_k if top_k is not None else w.top_k
        _DEV[key] = (oracle.Head.from_tables(t, k),
                     m.MaskedHead.from_host(t.centroid_w, t.embed_w, t.token_ordering,
                                            t.cluster_offsets, k))
    return _DEV[key]


def run_topk(m, dh, hidden_np):
    h = helpers.bf16_tensor(hidden_np)
    tok, mx = m.mtp_masked_topk_tokens(dh, h)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), mx.cpu().numpy()


def check_topk(m, name, B, row0=0):
    oh, dh = device_head(m, name)
    hidden, ref, _ = helpers.clean_batch(name, oh, B, row0=row0)
    tok, mx = run_topk(m, dh, hidden)
    np.testing.assert_array_equal(tok, ref["tokens"])
    helpers.assert_close(mx, ref["max_logit"], f"{name} B={B} max logit")
    return hidden, ref


def check_selection(m, dh, oh, hidden, ref_sel=None):
    h = helpers.bf16_tensor(hidden)
    scores, topk = m.mtp_centroid_scores(dh, h)
    torch.cuda.synchronize()
    ref_scores = oracle.centroid_scores(oh, hidden)
    helpers.assert_close(scores.cpu().numpy(), ref_scores, "centroid scores")
    topk = topk.cpu().numpy()
    if ref_sel is not None:
        for b in range(hidden.shape[0]):
            assert set(topk[b].tolist()) == set(ref_sel[b].tolist()), f"row {b} selection"
            # order: wherever consecutive oracle scores are well separated, it is the same
            gaps = ref_scores[b, ref_sel[b][:-1]] - ref_scores[b, ref_sel[b][1:]]
            sep = np.nonzero(gaps > helpers.MARGIN)[0]
            for i in sep:
                assert ref_scores[b, topk[b][i]] >= ref_scores[b, topk[b][i + 1]]
    return scores, topk


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B", [1, 8])
def test_tiny_every_call(build_lib, B):
    m = build_lib
    oh, dh = device_head(m, "tiny")
    hidden, ref = check_topk(m, "tiny", B)
    check_selection(m, dh, oh, hidden, ref["sel"])
    h = helpers.bf16_tensor(hidden)
    sc = m.mtp_masked_scatter_logits(dh, h)
    logits, dtok, dmax = m.mtp_dense_lm_head(dh, h, want_tokens=True)
    torch.cuda.synchronize()
    helpers.assert_close(sc.cpu().numpy(), oracle.masked_scatter_logits(oh, hidden), "tiny scatter")
    dref = oracle.dense_logits(oh, hidden)
    helpers.assert_close(logits.cpu().numpy(), dref, "tiny dense")
    top2 = np.sort(dref, axis=1)[:, -2:]
    clear = (top2[:, 1] - top2[:, 0]) > helpers.MARGIN
    np.testing.assert_array_equal(dtok.cpu().numpy()[clear], np.argmax(dref, axis=1)[clear])
    helpers.assert_close(dmax.cpu().numpy(), dref.max(axis=1), "tiny dense max")


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16, 32, 64])
def test_uniform_topk_tokens(build_lib, B):
    m = build_lib
    hidden, ref = check_topk(m, "uniform", B)
    if B in (1, 64):
        oh, dh = device_head(m, "uniform")
        check_selection(m, dh, oh, hidden, ref["sel"])


def test_variable_clusters_topk_tokens(build_lib):
    m = build_lib
    hidden, ref = check_topk(m, "variable", 64)
    oh, dh = device_head(m, "variable")
    check_selection(m, dh, oh, hidden, ref["sel"])


def test_full_vocab_scatter(build_lib):
    m = build_lib
    oh, dh = device_head(m, "scatter")
    hidden, ref, _ = helpers.clean_batch("scatter", oh, 64)
    h = helpers.bf16_tensor(hidden)
    sc = m.mtp_masked_scatter_logits(dh, h)
    tok, _ = m.mtp_masked_topk_tokens(dh, h)
    torch.cuda.synchronize()
    sc_np = sc.cpu().numpy()
    helpers.assert_close(sc_np, oracle.masked_scatter_logits(oh, hidden), "scatter B=64")
    # invariants: exactly K*S finite entries per row; argmax(scatter row) == sparse argmax
    assert (np.isfinite(sc_np).sum(axis=1) == 32 * 128).all()
    np.testing.assert_array_equal(np.argmax(sc_np, axis=1), tok.cpu().numpy())
    np.testing.assert_array_equal(tok.cpu().numpy(), ref["tokens"])


@pytest.mark.parametrize("mode", ["argmax", "scatter"])
def test_shared_centroids(build_lib, mode):
    m = build_lib
    oh, dh = device_head(m, "shared")
    hidden, ref, _ = helpers.clean_batch("shared", oh, 256, need_logit_margin=(mode == "argmax"))
    h = helpers.bf16_tensor(hidden)
    if mode == "argmax":
        tok, mx = m.mtp_masked_topk_tokens(dh, h)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(tok.cpu().numpy(), ref["tokens"])
        helpers.assert_close(mx.cpu().numpy(), ref["max_logit"], "shared max")
    else:
        sc = m.mtp_masked_scatter_logits(dh, h)
        torch.cuda.synchronize()
        helpers.assert_close(sc.cpu().numpy(), oracle.masked_scatter_logits(oh, hidden),
                             "shared scatter")
    # heavy overlap is what this workload is for
    assert len(np.unique(ref["sel"])) < 256 * 128 / 4


def test_dense_head_full_size_sampled(build_lib):
    m = build_lib
    oh, dh = device_head(m, "uniform")
    hidden = synth.hidden_batch("scatter", 64)
    h = helpers.bf16_tensor(hidden)
    logits, dtok, dmax = m.mtp_dense_lm_head(dh, h, want_tokens=True)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    g = np.random.default_rng(5)
    rows = g.integers(0, 64, 20000)
    toks = g.integers(0, oh.V, 20000)
    helpers.assert_close(lg[rows, toks], oracle.dense_logits_at(oh, hidden, rows, toks),
                         "dense sampled")
    # the fused argmax agrees with the logits it wrote (lower id on ties)
    np.testing.assert_array_equal(dtok.cpu().numpy(), np.argmax(lg, axis=1))
    np.testing.assert_array_equal(dmax.cpu().numpy(), lg.max(axis=1))
    # and with the oracle on rows whose dense top-2 gap is clear
    ref4 = oracle.dense_logits(oh, hidden[:4])
    top2 = np.sort(ref4, axis=1)[:, -2:]
    clear = (top2[:, 1] - top2[:, 0]) > helpers.MARGIN
    np.testing.assert_array_equal(dtok.cpu().numpy()[:4][clear], np.argmax(ref4, axis=1)[clear])


def test_k_equals_c_is_dense(build_lib):
    m = build_lib
    oh, dh = device_head(m, "tiny", top_k=64)
    hidden = synth.hidden_batch("tiny", 5)
    h = helpers.bf16_tensor(hidden)
    sc = m.mtp_masked_scatter_logits(dh, h)
    dl, _, _ = m.mtp_dense_lm_head(dh, h)
    torch.cuda.synchronize()
    ref = oracle.dense_logits(oh, hidden)
    helpers.assert_close(sc.cpu().numpy(), ref, "masked K=C")
    helpers.assert_close(dl.cpu().numpy(), ref, "dense")
    # the masked path (CUDA cores) and the dense head (tensor cores) agree
    helpers.assert_close(sc.cpu().numpy(), dl.cpu().numpy().astype(np.float64), "masked vs dense")


def test_projection_paths_agree(build_lib):
    """Batches of at most 8 rows use the CUDA-core projection (which reduces 1, 2, 4 or
    8 rows at once, the last group padded), larger ones at H=1536 the tensor-core GEMM
    with a cluster split-K: the same rows must score alike either way, and the CUDA-core
    scores of a row must not depend on the batch it came in (the same bits)."""
    m = build_lib
    oh, dh = device_head(m, "uniform")
    hidden = synth.hidden_batch("uniform", 24, row0=900)
    h = helpers.bf16_tensor(hidden)
    big, big_top = m.mtp_centroid_scores(dh, h)
    small = torch.cat([m.mtp_centroid_scores(dh, h[i:i + 1])[0] for i in range(24)])
    cuts = [0, 8, 13, 16, 18, 24]   # batches of 8, 5, 3, 2 and 6 rows
    grouped = torch.cat([m.mtp_centroid_scores(dh, h[a:b])[0] for a, b in zip(cuts, cuts[1:])])
    torch.cuda.synchronize()
    ref = oracle.centroid_scores(oh, hidden)
    helpers.assert_close(big.cpu().numpy(), ref, "tensor-core projection")
    helpers.assert_close(small.cpu().numpy(), ref, "CUDA-core projection")
    helpers.assert_close(grouped.cpu().numpy(), ref, "CUDA-core projection, row groups")
    assert torch.equal(grouped, small)
    d = np.abs(big.cpu().numpy().astype(np.float64) - small.cpu().numpy())
    assert d.max() < 1e-3


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B", [3, 17, 63, 65])
def test_ragged_batches(build_lib, B):
    check_topk(build_lib, "uniform", B, row0=1000)


@pytest.mark.parametrize("name,B", [("uniform", 10), ("uniform", 11), ("draft256", 10), ("draft256", 20),
                                    ("draft256", 64), ("draft256", 65)])
def test_projection_plan_boundary(build_lib, name, B):
    """Either side of the projection plan's switch (the CUDA-core GEMV up to B*H = 16384,
    tensor cores beyond it): H=1536 at 10 rows (GEMV, a padded second group of 8; the fused
    kernel's last batch size) and 11 (tensor cores, the direct gather), H=256 on the
    token-order table at 10 and 20 rows (the direct gather, 20 its last batch size there),
    64 (GEMV, eight groups of 8) and 65 (tensor cores); selections and tokens against the
    oracle."""
    m = build_lib
    hidden, ref = check_topk(m, name, B, row0=3000)
    oh, dh = device_head(m, name)
    check_selection(m, dh, oh, hidden, ref["sel"])


def test_maximum_batch(build_lib):
    check_topk(build_lib, "tiny", 1024)


def _custom(m, V, H, C, K, seed, sizes=None, identity=False, pad_rows=0, pad_cols=0):
    t = synth.custom_tables(V, H, C, seed, std=0.05, sizes=sizes, identity=identity)
    ew = t.embed_w
    if pad_rows or pad_cols:
        big = np.zeros((V + pad_rows, H + pad_cols), dtype=np.uint16)
        big[:V, :H] = ew
        big[V:, :] = 0x7FC0  # NaN padding: must never be read
        big[:, H:] = 0x7FC0
        ew = big
    oh = oracle.Head(t.centroid_w, ew, t.token_ordering, t.cluster_offsets, K, vocab=V)
    torch_ew = helpers.bf16_tensor(ew)
    dh = m.MaskedHead(helpers.bf16_tensor(t.centroid_w), torch_ew,
                      torch.from_numpy(t.token_ordering).cuda(), K,
                      None if t.cluster_offsets is None else torch.from_numpy(t.cluster_offsets).cuda(),
                      vocab_size=V)
    return t, oh, dh


def _full_check(m, oh, dh, hidden, what):
    ref = oracle.masked_topk_tokens(oh, hidden)
    clear = (ref["score_margin"] > helpers.MARGIN) & (ref["logit_margin"] > helpers.MARGIN)
    h = helpers.bf16_tensor(hidden)
    tok, mx = m.mtp_masked_topk_tokens(dh, h)
    sc = m.mtp_masked_scatter_logits(dh, h)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tok.cpu().numpy()[clear], ref["tokens"][clear])
    sref = oracle.masked_scatter_logits(oh, hidden)
    sc_np = sc.cpu().numpy()
    sel_clear = ref["score_margin"] > helpers.MARGIN
    helpers.assert_close(sc_np[sel_clear], sref[sel_clear], what)
    helpers.assert_close(mx.cpu().numpy()[sel_clear], ref["max_logit"][sel_clear], what + " max")
    # the dense head (tensor-core GEMM) on the same tables
    dl, dtok, _ = m.mtp_dense_lm_head(dh, h, want_tokens=True)
    torch.cuda.synchronize()
    dref = oracle.dense_logits(oh, hidden)
    helpers.assert_close(dl.cpu().numpy(), dref, what + " dense")
    np.testing.assert_array_equal(dtok.cpu().numpy(), np.argmax(dl.cpu().numpy(), axis=1))
    return ref


@pytest.mark.parametrize("H", [8, 72, 256, 264, 4096])
def test_hidden_sizes(build_lib, H):
    m = build_lib
    t, oh, dh = _custom(m, 2048, H, 32, 3, seed=H)
    hidden = synth.random_hidden(7, H, H + 1)
    _full_check(m, oh, dh, hidden, f"H={H}")


@pytest.mark.parametrize("H,B", [(3072, 8), (1536, 16), (2048, 12)])
def test_shared_memory_at_the_default_limit(build_lib, H, B):
    """Kernels whose dynamic shared memory is at or just under the default 48 KB (the
    direct gather keeps B x H bf16 hidden rows: exactly 48 KB for the first two cases)
    still launch, since their static shared memory counts against the same limit."""
    m = build_lib
    t, oh, dh = _custom(m, 4096, H, 64, 2, seed=H + B)
    hidden = synth.random_hidden(B, H, H + B)
    _full_check(m, oh, dh, hidden, f"H={H} B={B}")


@pytest.mark.parametrize("H", [72, 264, 1536])
def test_hidden_sizes_tensor_core_gather(build_lib, H):
    """B*K >= 4C: large buckets, gathered onto the tensor cores (K tails at 72, 264)."""
    m = build_lib
    t, oh, dh = _custom(m, 4096, H, 32, 8, seed=H + 5)
    hidden = synth.random_hidden(64, H, H + 6)
    _full_check(m, oh, dh, hidden, f"tc H={H}")


@pytest.mark.parametrize("B", [9, 41])
def test_variable_clusters_empty_and_oversized(build_lib, B):
    m = build_lib
    sizes = [0] * 5 + [1, 2, 3] + [700, 1] + [37] * 20 + [0, 19]
    V = int(sum(sizes))
    t, oh, dh = _custom(m, V, 64, len(sizes), 6, seed=77, sizes=sizes)
    hidden = synth.random_hidden(B, 64, 78)
    assert (B * V) % 4 != 0  # the -inf fill ends in a scalar tail
    _full_check(m, oh, dh, hidden, f"ragged clusters B={B}")


@pytest.mark.parametrize("B", [2, 8])
def test_only_empty_clusters_selected(build_lib, B):
    m = build_lib
    sizes = [0, 0, 10, 6]
    t, oh, dh = _custom(m, 16, 8, 4, 2, seed=3, sizes=sizes)
    # make the empty clusters win: their centroid rows point along the hidden state
    hidden = synth.bf16_bits(np.ones((B, 8), np.float32))
    cw = np.zeros((4, 8), np.float32)
    cw[0] = 1.0
    cw[1] = 0.5
    cw[2] = -1.0
    cw[3] = -2.0
    cwb = synth.bf16_bits(cw)
    oh = oracle.Head(cwb, t.embed_w, t.token_ordering, t.cluster_offsets, 2, vocab=16)
    dh = m.MaskedHead(helpers.bf16_tensor(cwb), dh.embed_w, dh.token_ordering, 2, dh.cluster_offsets,
                      vocab_size=16)
    h = helpers.bf16_tensor(hidden)
    tok, mx = m.mtp_masked_topk_tokens(dh, h)
    sc = m.mtp_masked_scatter_logits(dh, h)
    torch.cuda.synchronize()
    assert tok.cpu().tolist() == [-1] * B
    assert np.isneginf(mx.cpu().numpy()).all()
    assert np.isneginf(sc.cpu().numpy()).all()
    assert oracle.masked_topk_tokens(oh, hidden)["tokens"].tolist() == [-1] * B


def test_padded_table_and_identity_ordering(build_lib):
    m = build_lib
    t, oh, dh = _custom(m, 4096, 128, 64, 5, seed=21, identity=True, pad_rows=64, pad_cols=8)
    hidden = synth.random_hidden(6, 128, 22)
    _full_check(m, oh, dh, hidden, "padded")


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("B,K", [(12, 3), (32, 8)])
def test_integer_inputs_bit_exact_with_ties(build_lib, B, K, packed):
    """Small-integer inputs make every sum exact in fp32 and fp64: logits must be
    bit-identical, and forced ties exercise both tie-break rules.  B*K >= 4C sends
    the second case through the tensor-core gather; with the packed table both do."""
    m = build_lib
    g = np.random.default_rng(11)
    V, C, H = 512, 16, 64
    cw = g.integers(-2, 3, size=(C, H)).astype(np.float32)
    cw[5] = cw[9]          # centroids 5 and 9 always tie
    ew = g.integers(-2, 3, size=(V, H)).astype(np.float32)
    perm = g.permutation(V).astype(np.int32)
    S = V // C
    for c in range(C):     # duplicate rows inside each cluster: argmax ties between token ids
        toks = perm[c * S:(c + 1) * S]
        ew[toks[1]] = ew[toks[0]]
    hid = g.integers(-2, 3, size=(B, H)).astype(np.float32)
    cwb, ewb, hb = synth.bf16_bits(cw), synth.bf16_bits(ew), synth.bf16_bits(hid)
    oh = oracle.Head(cwb, ewb, perm, None, K)
    dh = m.MaskedHead(helpers.bf16_tensor(cwb), helpers.bf16_tensor(ewb),
                      torch.from_numpy(perm).cuda(), K)
    if packed:
        dh.use_packed_table()
    h = helpers.bf16_tensor(hb)
    scores, topk = m.mtp_centroid_scores(dh, h)
    tok, mx = m.mtp_masked_topk_tokens(dh, h)
    sc = m.mtp_masked_scatter_logits(dh, h)
    torch.cuda.synchronize()
    ref = oracle.masked_topk_tokens(oh, hb)
    np.testing.assert_array_equal(scores.cpu().numpy(), oracle.centroid_scores(oh, hb))
    np.testing.assert_array_equal(topk.cpu().numpy(), ref["sel"])
    np.testing.assert_array_equal(tok.cpu().numpy(), ref["tokens"])
    np.testing.assert_array_equal(mx.cpu().numpy(), ref["max_logit"])
    np.testing.assert_array_equal(sc.cpu().numpy(), oracle.masked_scatter_logits(oh, hb))


@pytest.mark.parametrize("name", ["tiny", "uniform"])
def test_all_equal_scores(build_lib, name):
    """Zero hidden states make every centroid score and every logit 0: the selection is
    the K lowest centroid indices and the token the lowest id among their candidates.
    At C=2048 every score lands in one bucket, which exercises the radix fallback of
    the top-K kernel; at C=64 the bucketed fast path handles the ties."""
    m = build_lib
    oh, dh = device_head(m, name)
    hidden = np.zeros((5, oh.H), dtype=np.uint16)
    h = helpers.bf16_tensor(hidden)
    scores, topk = m.mtp_centroid_scores(dh, h)
    tok, mx = m.mtp_masked_topk_tokens(dh, h)
    torch.cuda.synchronize()
    ref = oracle.masked_topk_tokens(oh, hidden)
    np.testing.assert_array_equal(topk.cpu().numpy(), np.tile(np.arange(oh.K), (5, 1)))
    np.testing.assert_array_equal(topk.cpu().numpy(), ref["sel"])
    np.testing.assert_array_equal(tok.cpu().numpy(), ref["tokens"])
    assert (mx.cpu().numpy() == 0).all()


@pytest.mark.parametrize("B", [2, 8])
def test_corrupt_ordering_sets_device_error(build_lib, B):
    m = build_lib
    t, oh, dh = _custom(m, 1024, 64, 16, 16, seed=5)
    bad = t.token_ordering.copy()
    bad[10] = 1024 + 7       # out of range id, owned by centroid 0 (selected: K = C)
    dbad = m.MaskedHead(dh.centroid_w, dh.embed_w, torch.from_numpy(bad).cuda(), 16, vocab_size=1024)
    hidden = synth.random_hidden(B, 64, 6)
    h = helpers.bf16_tensor(hidden)
    ws = dbad.workspace(B)
    tok, _ = m.mtp_masked_topk_tokens(dbad, h, workspace=ws)
    assert m.mtp_read_device_error(ws) & m.MTP_DEVERR_TOKEN_RANGE
    # a clean call on the same workspace clears the word
    m.mtp_masked_topk_tokens(dh, h, workspace=ws)
    assert m.mtp_read_device_error(ws) == 0


def test_corrupt_offsets_set_device_error(build_lib):
    m = build_lib
    sizes = [4, 4, 4, 4]
    t, oh, dh = _custom(m, 16, 8, 4, 4, seed=8, sizes=sizes)
    off = t.cluster_offsets.copy()
    off[2] = 40              # beyond V and not ascending
    dbad = m.MaskedHead(dh.centroid_w, dh.embed_w, dh.token_ordering, 4,
                        torch.from_numpy(off).cuda(), vocab_size=16)
    h = helpers.bf16_tensor(synth.random_hidden(1, 8, 9))
    ws = dbad.workspace(1)
    m.mtp_masked_topk_tokens(dbad, h, workspace=ws)
    assert m.mtp_read_device_error(ws) & m.MTP_DEVERR_OFFSETS


def test_overlapping_offsets_overflow_the_item_list(build_lib):
    """Cluster ranges that overlap (possible only beside an invalid range: clusters 0, 2, 4
    and 6 below each own all of V, 1, 3, 5 and 7 are reversed) ask for 4 x 32 work items of
    8 positions, more than the list holds (V/8 + C + 1 = 41).  The top-K drops every cluster
    whose items do not fit instead of writing past the list, the call reports
    MTP_DEVERR_OFFSETS, and a clean call on the same workspace runs clean."""
    m = build_lib
    V, H, C, K = 256, 8, 8, 8
    t, oh, dh = _custom(m, V, H, C, K, seed=11, sizes=[32] * C)
    off = np.array([0, V, 0, V, 0, V, 0, V, 0], dtype=np.int32)
    dbad = m.MaskedHead(dh.centroid_w, dh.embed_w, dh.token_ordering, K, torch.from_numpy(off).cuda(),
                        vocab_size=V)
    h = helpers.bf16_tensor(synth.random_hidden(1, H, 12))
    ws = dbad.workspace(1)
    ref = oracle.masked_topk_tokens(oh, synth.random_hidden(1, H, 12))
    # the work-item list belongs to the top-K kernel + gather path; the fused kernel has none
    # (it only reports the reversed ranges)
    for kind in ("cuda_core_direct", "fused"):
        m.mtp_force_gather(kind)
        try:
            tok, _ = m.mtp_masked_topk_tokens(dbad, h, workspace=ws)
            torch.cuda.synchronize()
            assert m.mtp_read_device_error(ws) & m.MTP_DEVERR_OFFSETS
            assert 0 <= int(tok.cpu()[0]) < V
            tok, _ = m.mtp_masked_topk_tokens(dh, h, workspace=ws)
            torch.cuda.synchronize()
        finally:
            m.mtp_force_gather(None)
        assert m.mtp_read_device_error(ws) == 0
        if ref["score_margin"][0] > helpers.MARGIN and ref["logit_margin"][0] > helpers.MARGIN:
            assert int(tok.cpu()[0]) == int(ref["tokens"][0])


# ---------------------------------------------------------------------------
# every gather kernel at the drafter's small batches; the fused small-batch kernel


@pytest.mark.parametrize("B", [1, 3, 8, 10])
@pytest.mark.parametrize("kind", ["fused", "cuda_core_direct", "cuda_core", "tensor_core"])
def test_every_gather_kernel_small_batches(build_lib, B, kind):
    """The uniform workload at small batches through each gather kernel (forced): token
    ids equal the oracle's, max logits and full-vocabulary rows within the tolerance."""
    m = build_lib
    oh, dh = device_head(m, "uniform")
    hidden, ref, _ = helpers.clean_batch("uniform", oh, B, row0=7000 + B)
    h = helpers.bf16_tensor(hidden)
    ws = dh.workspace(B)
    m.mtp_force_gather(kind)
    try:
        assert m.mtp_gather_plan(dh, B) == kind
        tok, mx = m.mtp_masked_topk_tokens(dh, h, workspace=ws)
        sc = m.mtp_masked_scatter_logits(dh, h, workspace=ws)
        torch.cuda.synchronize()
    finally:
        m.mtp_force_gather(None)
    assert m.mtp_read_device_error(ws) == 0
    np.testing.assert_array_equal(tok.cpu().numpy(), ref["tokens"])
    helpers.assert_close(mx.cpu().numpy(), ref["max_logit"], f"{kind} B={B} max")
    sc_np = sc.cpu().numpy()
    helpers.assert_close(sc_np, oracle.masked_scatter_logits(oh, hidden), f"{kind} B={B} scatter")
    assert (np.isfinite(sc_np).sum(axis=1) == 32 * 128).all()


@pytest.mark.parametrize("name,B", [("variable", 1), ("variable", 8), ("shared", 8), ("draft256", 4)])
def test_fused_kernel_other_workloads(build_lib, name, B):
    """The fused kernel on lognormal clusters, on K=128 of 4096 small clusters and at H=256
    (where the library runs the direct gather instead, so the kernel is forced), both
    finishes, against the oracle."""
    m = build_lib
    oh, dh = device_head(m, name)
    small_h = oh.H <= 256
    assert m.mtp_gather_plan(dh, B) == ("cuda_core_direct" if small_h else "fused")
    if small_h:
        m.mtp_force_gather("fused")
    try:
        assert m.mtp_gather_plan(dh, B) == "fused"
        hidden, ref = check_topk(m, name, B, row0=6100)
        sc = m.mtp_masked_scatter_logits(dh, helpers.bf16_tensor(hidden))
        torch.cuda.synchronize()
    finally:
        m.mtp_force_gather(None)
    helpers.assert_close(sc.cpu().numpy(), oracle.masked_scatter_logits(oh, hidden), f"fused {name} scatter")


@pytest.mark.parametrize("K", [1024, 1025])
def test_fused_kernel_at_its_k_limit(build_lib, K):
    """K up to 1024 selections per row run the fused kernel (here K of C = 1100 centroids,
    most of the vocabulary a candidate; H = 512, above the sizes that take the direct
    gather instead); one more falls back to the direct gather."""
    m = build_lib
    t, oh, dh = _custom(m, 1100 * 8, 512, 1100, K, seed=K)
    assert m.mtp_gather_plan(dh, 3) == ("fused" if K <= 1024 else "cuda_core_direct")
    hidden = synth.random_hidden(3, 512, K + 1)
    _full_check(m, oh, dh, hidden, f"K={K}")


def test_bounded_wait_gives_up_cleanly(build_lib):
    """A wait that runs out: the pipelined gather's first hidden-row buffer wait is made to
    wait for a barrier phase that nothing completes, with a 20 ms limit (the wait test).
    The producer gives up before it has issued any copy, the consumer warps' waits run out
    next, and the call finishes with MTP_DEVERR_TIMEOUT and the site of the first wait that
    gave up in the workspace; the next call on the same workspace runs clean and right."""
    import time
    m = build_lib
    oh, dh = device_head(m, "uniform")
    hidden, ref, _ = helpers.clean_batch("uniform", oh, 8, row0=8800)
    h = helpers.bf16_tensor(hidden)
    ws = dh.workspace(8)
    m.mtp_force_gather("cuda_core")
    try:
        m.mtp_masked_topk_tokens(dh, h, workspace=ws)     # module loaded, nothing pending
        torch.cuda.synchronize()
        m.mtp_wait_test(20_000_000, stall=True)
        try:
            t0 = time.time()
            m.mtp_masked_topk_tokens(dh, h, workspace=ws)
            torch.cuda.synchronize()
            elapsed = time.time() - t0
        finally:
            m.mtp_wait_test(0, stall=False)
        word = m.mtp_read_device_error(ws)
        ctrl = ws[:32].view(torch.int32).cpu().tolist()
        assert word & m.MTP_DEVERR_TIMEOUT, f"error word {word:#x}"
        assert ctrl[4] in (1, 4), f"wait site {ctrl[4]}"     # consumer slot / producer h buffer
        assert elapsed < 1.0, f"{elapsed:.3f} s: the waits did not give up after 20 ms"
        tok, mx = m.mtp_masked_topk_tokens(dh, h, workspace=ws)
        torch.cuda.synchronize()
        assert m.mtp_read_device_error(ws) == 0
    finally:
        m.mtp_force_gather(None)
    np.testing.assert_array_equal(tok.cpu().numpy(), ref["tokens"])
    helpers.assert_close(mx.cpu().numpy(), ref["max_logit"], "after the wait test")


def test_repeat_calls_are_deterministic(build_lib):
    m = build_lib
    oh, dh = device_head(m, "uniform")
    hidden = synth.hidden_batch("uniform", 64, row0=5000)
    h = helpers.bf16_tensor(hidden)
    ws = dh.workspace(64)
    outs = [m.mtp_masked_topk_tokens(dh, h, workspace=ws) for _ in range(3)]
    sc = [m.mtp_masked_scatter_logits(dh, h[:8], workspace=ws) for _ in range(2)]
    torch.cuda.synchronize()
    for t_, x_ in outs[1:]:
        assert torch.equal(t_, outs[0][0]) and torch.equal(x_, outs[0][1])
    assert torch.equal(sc[0], sc[1])


@pytest.mark.parametrize("name,B,calls", [("uniform", 64, 60), ("shared", 256, 12)])
def test_repeated_calls_stay_identical(build_lib, name, B, calls):
    """Many consecutive calls on one workspace, in both finishes: every call must report
    a clean device error word (no pipeline wait gave up) and reproduce the first call's
    output bit for bit (no stale shared-memory metadata, no lost work item)."""
    m = build_lib
    oh, dh = device_head(m, name)
    t = helpers.tables(name)
    hidden = synth.hidden_batch(name, B, None, t.prototypes, row0=3000)
    h = helpers.bf16_tensor(hidden)
    ws = dh.workspace(B)
    first_tok, first_max = m.mtp_masked_topk_tokens(dh, h, workspace=ws)
    first_sc = m.mtp_masked_scatter_logits(dh, h, workspace=ws)
    assert m.mtp_read_device_error(ws) == 0
    tok = torch.empty_like(first_tok)
    mx = torch.empty_like(first_max)
    sc = torch.empty_like(first_sc)
    for i in range(calls):
        m.mtp_masked_topk_tokens(dh, h, out_tokens=tok, out_max=mx, workspace=ws)
        assert m.mtp_read_device_error(ws) == 0, f"argmax call {i}"
        assert torch.equal(tok, first_tok) and torch.equal(mx, first_max), f"argmax call {i}"
        m.mtp_masked_scatter_logits(dh, h, out=sc, workspace=ws)
        assert m.mtp_read_device_error(ws) == 0, f"scatter call {i}"
        assert torch.equal(sc, first_sc), f"scatter call {i}"


@pytest.mark.parametrize("name,B,calls", [("uniform", 64, 120), ("shared", 256, 40)])
def test_scatter_calls_with_profiling_events(build_lib, name, B, calls):
    """The bench's per-kernel breakdown loop: consecutive scatter calls with the library
    recording events around every kernel.  Each call must finish without any wait giving
    up (the workspace records which wait and where if one does) and well under a second."""
    m = build_lib
    oh, dh = device_head(m, name)
    t = helpers.tables(name)
    hidden = synth.hidden_batch(name, B, None, t.prototypes, row0=5000)
    h = helpers.bf16_tensor(hidden)
    ws = dh.workspace(B)
    out = torch.empty(B, oh.V, dtype=torch.float32, device="cuda")
    first = m.mtp_masked_scatter_logits(dh, h, workspace=ws).clone()
    kernels = ["projection", "topk", "gather_score", "fill"]
    evs = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for k in kernels}
    for a, b in evs.values():
        a.record()
        b.record()
    call_s, call_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        for k in kernels:
            m.mtp_profile_events(k, *evs[k])
        for i in range(calls):
            call_s.record()
            m.mtp_masked_scatter_logits(dh, h, out=out, workspace=ws)
            call_e.record()
            word = m.mtp_read_device_error(ws)
            ctrl = ws[:32].view(torch.int32).cpu().tolist()
            assert word == 0, f"call {i}: error {word:#x}, wait site/cta/seq {ctrl[4:7]}"
            assert call_s.elapsed_time(call_e) < 1000.0, f"call {i} took too long"
            assert torch.equal(out, first), f"call {i}"
    finally:
        for k in kernels:
            m.mtp_profile_events(k, None, None)


def test_empty_batch_is_noop(build_lib):
    m = build_lib
    oh, dh = device_head(m, "tiny")
    h = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    tok, mx = m.mtp_masked_topk_tokens(dh, h)
    assert tok.numel() == 0


# ---------------------------------------------------------------------------
# the packed embedding table (tensor-core gather operand tiles)


def _unpack(packed, V, H, C, sizes):
    """The packed layout read back with numpy: (padded table [poff[C], H], poff [C+1])."""
    KB = (H + 63) // 64
    if sizes is None:
        groups = C * ((V // C + 31) // 32)
    else:
        groups = (V + 31 * C + 31) // 32
    SG = (groups + 3) // 4
    off = SG * KB * 16384
    buf = packed.cpu().numpy()
    poff = buf[off:off + 4 * (C + 1)].view(np.int32)
    blocks = buf[:off].reshape(SG, KB, 128, 8, 16)
    r = np.arange(128)[:, None]
    j = np.arange(8)[None, :]
    un = blocks[:, :, r, j ^ (r & 7)]                        # undo the 128-byte swizzle
    rows = un.reshape(SG, KB, 128, 128).view(np.uint16)      # [SG, KB, 128, 64]
    table = rows.transpose(0, 2, 1, 3).reshape(SG * 128, KB * 64)[:int(poff[-1])]
    assert not table[:, H:].any(), "elements past H must be zero"
    return table[:, :H], poff


@pytest.mark.parametrize("H,sizes", [(264, "ragged"), (128, None)])
def test_pack_embeddings_layout(build_lib, H, sizes):
    m = build_lib
    if sizes == "ragged":
        sz = [0] * 5 + [1, 2, 3] + [700, 1] + [37] * 20 + [0, 19]
        t, oh, dh = _custom(m, int(sum(sz)), H, len(sz), 6, seed=77, sizes=sz, pad_cols=8)
        sizes = np.array(sz)
    else:
        t, oh, dh = _custom(m, 4096, H, 64, 5, seed=21)
        sizes = None
    V, C = oh.V, t.centroid_w.shape[0]
    ws = dh.workspace(1)
    ws.zero_()
    n = m.mtp_packed_embeddings_bytes(dh)
    packed = torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")
    m.mtp_pack_embeddings(dh, packed, workspace=ws)
    assert m.mtp_read_device_error(ws) == 0
    table, poff = _unpack(packed, V, H, C, sizes)
    off = t.cluster_offsets if t.cluster_offsets is not None else np.arange(C + 1) * (V // C)
    size = np.diff(off)
    np.testing.assert_array_equal(poff, np.concatenate([[0], np.cumsum((size + 31) // 32 * 32)]))
    ew = t.embed_w[:, :H]
    for c in range(C):
        blk = table[poff[c]:poff[c + 1]]
        np.testing.assert_array_equal(blk[:size[c]], ew[t.token_ordering[off[c]:off[c + 1]]])
        assert not blk[size[c]:].any(), f"cluster {c}: padding rows must be zero"


def test_pack_embeddings_flags_bad_inputs(build_lib):
    m = build_lib
    t, oh, dh = _custom(m, 1024, 64, 16, 4, seed=5)
    bad = t.token_ordering.copy()
    bad[10] = 1024 + 7
    dbad = m.MaskedHead(dh.centroid_w, dh.embed_w, torch.from_numpy(bad).cuda(), 4, vocab_size=1024)
    ws = dbad.workspace(1)
    ws.zero_()
    packed = dbad.use_packed_table()
    m.mtp_pack_embeddings(dbad, packed, workspace=ws)
    assert m.mtp_read_device_error(ws) & m.MTP_DEVERR_TOKEN_RANGE
    table, _ = _unpack(packed, 1024, 64, 16, None)
    keep = np.arange(1024) != 10
    np.testing.assert_array_equal(table[keep], t.embed_w[bad[keep]])
    assert not table[10].any()   # the bad id becomes a zero row
    # overlapping clusters (each in range on its own) whose padded sizes overflow the
    # table's bound: flagged, every cluster recorded as empty, and later calls read nothing
    off = np.array([0, 1024] * 8 + [1024], dtype=np.int32)
    dov = m.MaskedHead(dh.centroid_w, dh.embed_w, dh.token_ordering, 4, torch.from_numpy(off).cuda(),
                       vocab_size=1024)
    ws2 = dov.workspace(64)
    ws2.zero_()
    p2 = torch.empty(m.mtp_packed_embeddings_bytes(dov), dtype=torch.uint8, device="cuda")
    m.mtp_pack_embeddings(dov, p2, workspace=ws2)
    assert m.mtp_read_device_error(ws2) & m.MTP_DEVERR_OFFSETS
    dov.use_packed_table(p2)
    h = helpers.bf16_tensor(synth.random_hidden(64, 64, 3))
    m.mtp_masked_topk_tokens(dov, h, workspace=ws2)
    assert m.mtp_read_device_error(ws2) & m.MTP_DEVERR_OFFSETS


def _same_outputs(m, dh, h):
    tok, mx = m.mtp_masked_topk_tokens(dh, h)
    sc = m.mtp_masked_scatter_logits(dh, h)
    torch.cuda.synchronize()
    return tok.clone(), mx.clone(), sc.clone()


@pytest.mark.parametrize("H,B,sizes", [
    (264, 7, None),                # few pairs: the CUDA-core gather either way
    (264, 64, None),               # large buckets: the tensor-core gather either way, K tail
    (264, 4, None),                # B*K = C: packed -> tensor cores, token order -> CUDA cores
    (64, 41, "ragged"),            # empty and oversized clusters, padding groups, table end
    (64, 13, "ragged"),            # the same at B*K >= C: packed -> tensor cores, copies
                                   # that stop short of a group's end
])
def test_packed_table_parity(build_lib, H, B, sizes):
    """With the packed table attached every finish matches the oracle; where both
    layouts run the same gather kernel the outputs are bit-identical."""
    m = build_lib
    if sizes == "ragged":
        sz = [0] * 5 + [1, 2, 3] + [700, 1] + [37] * 20 + [0, 19]
        t, oh, dh = _custom(m, int(sum(sz)), H, len(sz), 6, seed=77, sizes=sz)
    else:
        t, oh, dh = _custom(m, 4096, H, 32, 8, seed=H + 5)
    hidden = synth.random_hidden(B, H, H + 6)
    h = helpers.bf16_tensor(hidden)
    base = _same_outputs(m, dh, h)
    dh.use_packed_table()
    try:
        _full_check(m, oh, dh, hidden, f"packed H={H} B={B}")
        got = _same_outputs(m, dh, h)
        same_kernel = B * 8 >= 4 * 32 or B * 8 < 32
        if same_kernel and sizes is None:
            for a, b in zip(base, got):
                assert torch.equal(a, b)
        else:
            np.testing.assert_array_equal(got[0].cpu().numpy(), base[0].cpu().numpy())
            helpers.assert_close(got[2].cpu().numpy(), base[2].cpu().numpy(), "packed vs token order")
    finally:
        dh.drop_packed_table()


@pytest.mark.parametrize("name,B", [("shared", 256), ("uniform", 64), ("uniform", 32), ("uniform", 20),
                                    ("uniform", 16), ("uniform", 8), ("variable", 64), ("variable", 32)])
def test_packed_table_full_size(build_lib, name, B):
    """Full-size tables with the packed table: token ids match the oracle and the
    token-order path exactly, logits within the fp32 tolerance (the packed call may run
    the tensor-core gather where the token-order call runs the CUDA-core one).  Uniform
    B=16 and 20 run the tensor-core gather with two CTAs per SM (a full last round of
    units), the other uniform batches with three."""
    m = build_lib
    oh, dh = device_head(m, name)
    hidden, ref, _ = helpers.clean_batch(name, oh, B)
    h = helpers.bf16_tensor(hidden)
    base = _same_outputs(m, dh, h)
    dh.use_packed_table()
    try:
        got = _same_outputs(m, dh, h)
        np.testing.assert_array_equal(got[0].cpu().numpy(), ref["tokens"])
        np.testing.assert_array_equal(got[0].cpu().numpy(), base[0].cpu().numpy())
        helpers.assert_close(got[1].cpu().numpy(), ref["max_logit"], f"packed {name} max")
        sc = got[2].cpu().numpy()
        helpers.assert_close(sc[:4], oracle.masked_scatter_logits(oh, hidden[:4]), f"packed {name} scatter")
        helpers.assert_close(sc, base[2].cpu().numpy(), f"packed {name} scatter vs token order")
    finally:
        dh.drop_packed_table()


# ---------------------------------------------------------------------------
# CUDA graphs of the calls (fixed sizes, pad-up replay)


def test_captured_calls_match_eager_calls(build_lib):
    """Replays at padded sizes give the eager call's outputs bit for bit (each row's
    result does not depend on the other rows), a replay reads the current contents of
    the static input, and batches above the largest size fall back to the eager call."""
    m = build_lib
    oh, dh = device_head(m, "uniform")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = m.CapturedCalls(dh, sizes=(1, 2, 4, 8, 16, 32, 64))
        try:
            for B in (1, 3, 5, 8, 17, 64, 70):
                hidden = synth.hidden_batch("uniform", B, row0=9000 + 100 * B)
                h = helpers.bf16_tensor(hidden)
                tok, mx = g(h)
                tok, mx = tok.clone(), mx.clone()
                etok, emx = m.mtp_masked_topk_tokens(dh, h)
                s.synchronize()
                assert torch.equal(tok, etok) and torch.equal(mx, emx), f"B={B}"
                if B in (5, 64):
                    ref = oracle.masked_topk_tokens(oh, hidden)
                    clear = (ref["score_margin"] > helpers.MARGIN) & (ref["logit_margin"] > helpers.MARGIN)
                    np.testing.assert_array_equal(tok.cpu().numpy()[clear], ref["tokens"][clear])
            assert m.mtp_read_device_error(g.ws, stream=s) == 0
        finally:
            g.close()


def test_captured_scatter_and_packed_graphs(build_lib):
    m = build_lib
    # scatter finish on the tiny head
    oh, dh = device_head(m, "tiny")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = m.CapturedCalls(dh, sizes=(1, 2), finish="scatter")
        try:
            hidden = synth.hidden_batch("tiny", 2, row0=77)
            out = g(helpers.bf16_tensor(hidden)).clone()
            s.synchronize()
            helpers.assert_close(out.cpu().numpy(), oracle.masked_scatter_logits(oh, hidden), "graph scatter")
        finally:
            g.close()
    # the packed table's tensor-core gather inside a graph (B*K = C on uniform clusters)
    oh, dh = device_head(m, "uniform")
    packed = dh.use_packed_table()
    try:
        with torch.cuda.stream(s):
            g = m.CapturedCalls(dh, sizes=(64,))
            try:
                assert m.mtp_gather_plan(dh, 64) == "tensor_core"
                hidden = synth.hidden_batch("uniform", 64, row0=4242)
                h = helpers.bf16_tensor(hidden)
                tok, mx = g(h)
                tok, mx = tok.clone(), mx.clone()
                etok, emx = m.mtp_masked_topk_tokens(dh, h)
                s.synchronize()
                assert torch.equal(tok, etok) and torch.equal(mx, emx)
            finally:
                g.close()
    finally:
        dh.drop_packed_table()
        del packed


# ---------------------------------------------------------------------------
# the sparse pair of _select_and_score


@pytest.mark.parametrize("name,B,packed,rows", [
    ("tiny", 1, False, None),
    ("uniform", 1, False, None),
    ("uniform", 8, False, None),
    ("uniform", 64, False, [0, 17, 40, 63]),
    ("uniform", 64, True, [1, 30, 62]),        # packed table: the tensor-core gather
    ("shared", 256, False, [0, 99, 255]),      # large buckets: the tensor-core gather (gather4)
    ("shared", 256, True, [3, 128, 200]),
])
def test_select_and_score_pair(build_lib, name, B, packed, rows):
    """Every row's K*S candidates in selection order with their token ids: ids exact where
    the oracle's K/(K+1) margin is clear, logits within the fp32 tolerance."""
    m = build_lib
    oh, dh = device_head(m, name)
    hidden, ref, _ = helpers.clean_batch(name, oh, B, need_logit_margin=False)
    if packed:
        dh.use_packed_table()
    try:
        logits, ids = m.mtp_select_and_score(dh, helpers.bf16_tensor(hidden))
        torch.cuda.synchronize()
    finally:
        if packed:
            dh.drop_packed_table()
    logits, ids = logits.cpu().numpy(), ids.cpu().numpy()
    assert logits.shape == (B, oh.K * (oh.V // oh.C)) and ids.shape == logits.shape
    for b in (rows if rows is not None else range(B)):
        rlog, rtok = oracle.select_and_score_row(oh, hidden, b)
        np.testing.assert_array_equal(ids[b], rtok, err_msg=f"{name} row {b} ids")
        helpers.assert_close(logits[b], rlog, f"{name} row {b} logits")
    # every row's ids are the union of its selected clusters: a set of K*S distinct tokens
    for b in range(B):
        assert len(np.unique(ids[b])) == ids.shape[1]


def test_select_and_score_matches_the_scatter(build_lib):
    """The pair scattered into a -inf row is the full-vocabulary scatter finish."""
    m = build_lib
    oh, dh = device_head(m, "uniform")
    h = helpers.bf16_tensor(synth.hidden_batch("uniform", 16, row0=777))
    logits, ids = m.mtp_select_and_score(dh, h)
    sc = m.mtp_masked_scatter_logits(dh, h)
    torch.cuda.synchronize()
    rebuilt = torch.full_like(sc, float("-inf"))
    rebuilt.scatter_(1, ids.long(), logits)
    assert torch.equal(rebuilt, sc)


def test_captured_pair_graph(build_lib):
    m = build_lib
    oh, dh = device_head(m, "uniform")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = m.CapturedCalls(dh, sizes=(4, 8), finish="pair")
        try:
            h = helpers.bf16_tensor(synth.hidden_batch("uniform", 6, row0=31337))
            lg, ids = g(h)
            lg, ids = lg.clone(), ids.clone()
            elg, eids = m.mtp_select_and_score(dh, h)
            s.synchronize()
            assert torch.equal(lg, elg) and torch.equal(ids, eids)
        finally:
            g.close()


@pytest.mark.parametrize("B,packed", [(1, False), (8, False), (64, False), (64, True)])
def test_draft256_full_size(build_lib, B, packed):
    """The H=256 draft-dimension workload at Gemma scale (V=262144, C=2048, K=32)."""
    m = build_lib
    oh, dh = device_head(m, "draft256")
    if packed:
        dh.use_packed_table()
    try:
        hidden, ref = check_topk(m, "draft256", B)
        if B == 64:
            check_selection(m, dh, oh, hidden, ref["sel"])
    finally:
        if packed:
            dh.drop_packed_table()


# ---------------------------------------------------------------------------
# cluster-sharded head (shards emulated on one GPU, combined by an elementwise max)


@pytest.mark.parametrize("name,B,packed,shards", [
    ("uniform", 8, False, 2),
    ("uniform", 64, False, 3),
    ("uniform", 64, True, 2),       # per-shard packed tables: the tensor-core gather
    ("shared", 256, False, 2),      # large buckets
    ("variable", 64, False, 3),
])
def test_sharded_head_equals_unsharded(build_lib, name, B, packed, shards):
    """Each shard gathers only its clusters; the max of the shards' keys decodes to the
    unsharded argmax and the max of their scatter rows is the unsharded scatter, bit
    for bit (every candidate's logit is computed by one shard, with the same arithmetic),
    and both equal the oracle (token ids exactly, logits within the tolerance)."""
    m = build_lib
    oh, dh = device_head(m, name)
    hidden, oref, _ = helpers.clean_batch(name, oh, B, row0=123)
    h = helpers.bf16_tensor(hidden)
    C = oh.C
    cuts = [round(i * C / shards) for i in range(shards + 1)]
    heads = [m.MaskedHead(dh.centroid_w, dh.embed_w, dh.token_ordering, oh.K, dh.cluster_offsets,
                          vocab_size=oh.V, cluster_range=(cuts[i], cuts[i + 1])) for i in range(shards)]
    if packed:
        dh.use_packed_table()
        full = m.mtp_packed_embeddings_bytes(dh)
        for sh in heads:
            sh.use_packed_table()
            assert sh.embed_packed.numel() < full / shards + 2 * 16384 * 24 + 4 * (C + 1)
    try:
        ref_tok, ref_max = m.mtp_masked_topk_tokens(dh, h)
        ref_sc = m.mtp_masked_scatter_logits(dh, h)
        keys = [m.mtp_masked_topk_keys(sh, h) for sh in heads]
        scs = [m.mtp_masked_scatter_logits(sh, h) for sh in heads]
        combined = keys[0].clone()
        for k in keys[1:]:
            combined = torch.maximum(combined, k)
        tok, mx = m.mtp_decode_keys(combined)
        sc = scs[0].clone()
        for x in scs[1:]:
            sc = torch.maximum(sc, x)
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok) and torch.equal(mx, ref_max)
        assert torch.equal(sc, ref_sc)
        # and the combined shards against the oracle: token ids, max logits, scatter rows
        np.testing.assert_array_equal(tok.cpu().numpy(), oref["tokens"])
        helpers.assert_close(mx.cpu().numpy(), oref["max_logit"], f"sharded {name} max")
        rows = [0, B // 2, B - 1]
        helpers.assert_close(sc.cpu().numpy()[rows], oracle.masked_scatter_logits(oh, hidden[rows]),
                             f"sharded {name} scatter rows")
        # each shard wrote only its own clusters' tokens
        finite = [torch.isfinite(x).sum().item() for x in scs]
        assert sum(finite) == torch.isfinite(ref_sc).sum().item()
        for sh in heads:
            assert m.mtp_read_device_error(sh.workspace(B)) == 0
    finally:
        if packed:
            dh.drop_packed_table()


# ---------------------------------------------------------------------------
# reference-fidelity options (bf16 scores and logits, finite fill)


@pytest.mark.parametrize("flags", [2, 4, 6, 7])
@pytest.mark.parametrize("B,K,packed", [(12, 3, False), (32, 8, False), (32, 8, True)])
def test_fidelity_flags_integer_inputs(build_lib, flags, B, K, packed):
    """Integer inputs large enough for bf16 rounding to bite (|sums| up to 8192, bf16
    spacing up to 32): every sum is exact in fp32 and fp64 and both sides round the same
    values to nearest even, so selection, argmax, scatter, pair and dense head must equal
    the oracle bit for bit, many ties included."""
    m = build_lib
    g = np.random.default_rng(21 + flags)
    V, C, H = 512, 16, 64
    cw = synth.bf16_bits(g.integers(-8, 9, size=(C, H)).astype(np.float32))
    ew = synth.bf16_bits(g.integers(-8, 9, size=(V, H)).astype(np.float32))
    perm = g.permutation(V).astype(np.int32)
    hid = synth.bf16_bits(g.integers(-16, 17, size=(B, H)).astype(np.float32))
    oh = oracle.Head(cw, ew, perm, None, K, flags=flags)
    dh = m.MaskedHead(helpers.bf16_tensor(cw), helpers.bf16_tensor(ew), torch.from_numpy(perm).cuda(), K,
                      flags=flags)
    if packed:
        dh.use_packed_table()
    h = helpers.bf16_tensor(hid)
    scores, topk = m.mtp_centroid_scores(dh, h)
    tok, mx = m.mtp_masked_topk_tokens(dh, h)
    sc = m.mtp_masked_scatter_logits(dh, h)
    plog, pids = m.mtp_select_and_score(dh, h)
    dl, dtok, dmax = m.mtp_dense_lm_head(dh, h, want_tokens=True)
    torch.cuda.synchronize()
    ref = oracle.masked_topk_tokens(oh, hid)
    np.testing.assert_array_equal(scores.cpu().numpy(), oracle.centroid_scores(oh, hid))   # unrounded
    np.testing.assert_array_equal(topk.cpu().numpy(), ref["sel"])
    np.testing.assert_array_equal(tok.cpu().numpy(), ref["tokens"])
    np.testing.assert_array_equal(mx.cpu().numpy(), ref["max_logit"])
    np.testing.assert_array_equal(sc.cpu().numpy(), oracle.masked_scatter_logits(oh, hid).astype(np.float32))
    for b in range(B):
        rl, rt = oracle.select_and_score_row(oh, hid, b)
        np.testing.assert_array_equal(pids[b].cpu().numpy(), rt)
        np.testing.assert_array_equal(plog[b].cpu().numpy(), rl.astype(np.float32))
    dref = oracle.dense_logits(oh, hid)
    np.testing.assert_array_equal(dl.cpu().numpy(), dref.astype(np.float32))
    np.testing.assert_array_equal(dtok.cpu().numpy(), np.argmax(dref, axis=1))
    # the rounding really acts on these inputs: many scores and logits are not bf16 values
    raw = oracle.centroid_scores(oh, hid)
    assert sum(oracle.round_bf16(x) != x for x in raw.ravel()) > raw.size // 10
    if flags & 4:
        raw_d = oracle.dense_logits(oracle.Head(cw, ew, perm, None, K), hid)
        assert (dref != raw_d).mean() > 0.1


# ---------------------------------------------------------------------------
# seeded random shapes through every finish


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes(build_lib, seed):
    """Random V, C, H, K, B, uniform or ragged clusters (empty ones included), with or without
    the packed table: every finish against the oracle (token ids exact on rows whose margins
    are clear, logits within the tolerance)."""
    m = build_lib
    g = np.random.default_rng(900 + seed)
    C = int(g.integers(2, 65))
    K = int(g.integers(1, C + 1))
    H = 8 * int(g.integers(1, 65))
    B = int(g.integers(1, 81))
    ragged = bool(g.integers(0, 2))
    if ragged:
        sizes = g.integers(0, 200, size=C)
        sizes[g.integers(0, C)] = 0
        sizes[g.integers(0, C)] += 1
        V = int(sizes.sum())
    else:
        sizes = None
        V = C * int(g.integers(1, 160))
    t, oh, dh = _custom(m, V, H, C, K, seed=1000 + seed, sizes=sizes)
    packed = bool(g.integers(0, 2))
    if packed:
        dh.use_packed_table()
    hidden = synth.random_hidden(B, H, 2000 + seed)
    h = helpers.bf16_tensor(hidden)
    tok, mx = m.mtp_masked_topk_tokens(dh, h)
    sc = m.mtp_masked_scatter_logits(dh, h)
    torch.cuda.synchronize()
    ref = oracle.masked_topk_tokens(oh, hidden)
    sel_ok = ref["score_margin"] > helpers.MARGIN
    clear = sel_ok & (ref["logit_margin"] > helpers.MARGIN)
    what = f"seed {seed}: V={V} C={C} K={K} H={H} B={B} ragged={ragged} packed={packed}"
    np.testing.assert_array_equal(tok.cpu().numpy()[clear], ref["tokens"][clear], err_msg=what)
    helpers.assert_close(mx.cpu().numpy()[sel_ok], ref["max_logit"][sel_ok], what + " max")
    helpers.assert_close(sc.cpu().numpy()[sel_ok], oracle.masked_scatter_logits(oh, hidden)[sel_ok],
                         what + " scatter")
    if not ragged:
        plog, pids = m.mtp_select_and_score(dh, h)
        torch.cuda.synchronize()
        for b in np.nonzero(sel_ok)[0][:8]:
            rl, rt = oracle.select_and_score_row(oh, hidden, int(b))
            np.testing.assert_array_equal(pids[b].cpu().numpy(), rt, err_msg=what)
            helpers.assert_close(plog[b].cpu().numpy(), rl, what + " pair")
    assert m.mtp_read_device_error(dh.workspace(B)) == 0, what


@pytest.mark.parametrize("cap,flags", [(3.0, 0), (30.0, 0), (3.0, 4)])
def test_dense_softcap(build_lib, cap, flags):
    """The dense head's final logit softcap against the oracle's cap * tanh(logit / cap);
    the masked calls ignore it."""
    m = build_lib
    t = synth.custom_tables(4096, 128, 32, 55, std=0.2)
    oh = oracle.Head(t.centroid_w, t.embed_w, t.token_ordering, None, 4, flags=flags, softcap=cap)
    dh = m.MaskedHead(helpers.bf16_tensor(t.centroid_w), helpers.bf16_tensor(t.embed_w),
                      torch.from_numpy(t.token_ordering).cuda(), 4, flags=flags, softcap=cap)
    hidden = synth.random_hidden(8, 128, 56)
    h = helpers.bf16_tensor(hidden)
    dl, dtok, dmax = m.mtp_dense_lm_head(dh, h, want_tokens=True)
    tok, _ = m.mtp_masked_topk_tokens(dh, h)
    torch.cuda.synchronize()
    ref = oracle.dense_logits(oh, hidden)
    got = dl.cpu().numpy()
    helpers.assert_close(got, ref, f"softcap {cap}")
    assert np.abs(got).max() <= cap
    np.testing.assert_array_equal(dtok.cpu().numpy(), np.argmax(got, axis=1))
    np.testing.assert_array_equal(dmax.cpu().numpy(), got.max(axis=1))
    # the masked argmax is uncapped: same as without the cap
    plain = m.MaskedHead(dh.centroid_w, dh.embed_w, dh.token_ordering, 4, flags=flags)
    ptok, _ = m.mtp_masked_topk_tokens(plain, h)
    torch.cuda.synchronize()
    assert torch.equal(tok, ptok)


# ---------------------------------------------------------------------------
# hidden states in pinned host memory, staged by the call itself


@pytest.mark.parametrize("name,B,packed", [("uniform", 64, True), ("uniform", 8, False), ("variable", 32, True),
                                           ("tiny", 1, False)])
def test_host_hidden_equals_device_hidden(build_lib, name, B, packed):
    """With MTP_FLAG_HOST_HIDDEN a call reads a pinned CPU batch through its staging kernel;
    every finish then gives the same bits as the same call on a device copy of the batch,
    with outputs on the device or in pinned host memory, and graphs capture the staging."""
    m = build_lib
    oh, dh = device_head(m, name)
    if packed:
        dh.use_packed_table()
    try:
        hh = dh.with_flags(m.MTP_FLAG_HOST_HIDDEN)
        hidden = synth.hidden_batch(name, B, row0=777)
        h_dev = helpers.bf16_tensor(hidden)
        h_host = h_dev.cpu().pin_memory()
        tok, mx = m.mtp_masked_topk_tokens(dh, h_dev)
        sc = m.mtp_masked_scatter_logits(dh, h_dev)
        keys = m.mtp_masked_topk_keys(dh, h_dev)
        dl, dtok, dmax = m.mtp_dense_lm_head(dh, h_dev, want_tokens=True)
        tok2, mx2 = m.mtp_masked_topk_tokens(hh, h_host)
        tok3 = torch.empty(B, dtype=torch.int32).pin_memory()
        mx3 = torch.empty(B, dtype=torch.float32).pin_memory()
        m.mtp_masked_topk_tokens(hh, h_host, out_tokens=tok3, out_max=mx3)
        sc2 = m.mtp_masked_scatter_logits(hh, h_host)
        keys2 = m.mtp_masked_topk_keys(hh, h_host)
        dl2, dtok2, dmax2 = m.mtp_dense_lm_head(hh, h_host, want_tokens=True)
        dl3, _, _ = m.mtp_dense_lm_head(hh, h_host)          # no argmax: workspace for the staging only
        torch.cuda.synchronize()
        for a, b in ((tok, tok2), (mx, mx2), (sc, sc2), (keys, keys2), (dl, dl2), (dtok, dtok2), (dmax, dmax2),
                     (dl, dl3)):
            assert torch.equal(a, b)
        assert torch.equal(tok.cpu(), tok3) and torch.equal(mx.cpu(), mx3)
        ref = oracle.masked_topk_tokens(oh, hidden)
        np.testing.assert_array_equal(tok2.cpu().numpy(), ref["tokens"])
        if not synth.WORKLOADS[name].variable_clusters:
            pl, pi = m.mtp_select_and_score(dh, h_dev)
            pl2, pi2 = m.mtp_select_and_score(hh, h_host)
            torch.cuda.synchronize()
            assert torch.equal(pl, pl2) and torch.equal(pi, pi2)
        assert m.mtp_read_device_error(hh.workspace(B)) == 0
        # the staging kernel inside a captured graph (its static input is device memory,
        # which the flag accepts as well)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            g = m.CapturedCalls(hh, sizes=(B,))
            try:
                gt, gm = g(h_dev)
                torch.cuda.synchronize()
                assert torch.equal(gt[:B], tok) and torch.equal(gm[:B], mx)
            finally:
                g.close()
    finally:
        dh.drop_packed_table()


def test_host_hidden_refuses_memory_the_device_cannot_read(build_lib):
    """A pageable (unregistered) CPU buffer with MTP_FLAG_HOST_HIDDEN is refused by the
    library's pointer check (MTP_ERR_UNSUPPORTED, nothing launched) and by the binding."""
    import ctypes
    m = build_lib
    _, dh = device_head(m, "tiny")
    hh = dh.with_flags(m.MTP_FLAG_HOST_HIDDEN)
    h = torch.zeros(2, dh.hidden_size, dtype=torch.bfloat16)
    assert not h.is_pinned()
    out = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    ws = hh.workspace(2)
    st = m._lib.lib().mtp_masked_topk_tokens(ctypes.byref(hh.desc), ctypes.c_void_p(h.data_ptr()), 2,
                                             ctypes.c_void_p(out.data_ptr()), None,
                                             ctypes.c_void_p(ws.data_ptr()), ws.numel(), None)
    assert st == -6
    torch.cuda.synchronize()
    assert (out.cpu() == -7).all()
    with pytest.raises(AssertionError):
        m.mtp_masked_topk_tokens(hh, h)
    with pytest.raises(AssertionError):
        m.mtp_masked_topk_tokens(dh, helpers.bf16_tensor(np.zeros((2, dh.hidden_size), np.uint16)),
                                 out_tokens=torch.empty(2, dtype=torch.int32))   # pageable output


# ---------------------------------------------------------------------------
# buckets larger than one unit of the tensor-core gather


@pytest.mark.parametrize("B,K,C,packed", [(64, 4, 128, True), (128, 4, 128, False), (48, 8, 192, True),
                                         (256, 4, 512, True), (200, 16, 64, True)])
def test_buckets_split_over_units(build_lib, B, K, C, packed):
    """Rows that share a hidden state share their selection, so the clusters they pick get
    buckets larger than a unit of the tensor-core gather (32 rows when B*K <= 2C, 64 above),
    split over several units whose candidate tiles repeat: every finish must still match the
    oracle, and the pair's rows agree with the scatter."""
    m = build_lib
    V, H = C * 64, 192
    t, oh, dh = _custom(m, V, H, C, K, seed=B + 7 * K)
    g = np.random.default_rng(B * 1000 + K)
    base = synth.random_hidden(1, H, B + K)[0]
    hidden = synth.random_hidden(B, H, 2 * B + K)
    crowd = g.choice(B, size=(3 * B) // 4, replace=False)
    hidden[crowd] = base
    if packed:
        dh.use_packed_table()
    assert m.mtp_gather_plan(dh, B) == "tensor_core"
    ref = _full_check(m, oh, dh, hidden, f"split buckets B={B} K={K} C={C}")
    # the crowd's rows all select the same clusters: one bucket of len(crowd) rows each
    assert len(set(tuple(r) for r in ref["sel"][crowd])) == 1
    h = helpers.bf16_tensor(hidden)
    plog, pids = m.mtp_select_and_score(dh, h)
    sc = m.mtp_masked_scatter_logits(dh, h)
    torch.cuda.synchronize()
    pl, pi, scn = plog.cpu().numpy(), pids.cpu().numpy(), sc.cpu().numpy()
    for b in range(B):
        np.testing.assert_array_equal(scn[b][pi[b]], pl[b])
    assert m.mtp_read_device_error(dh.workspace(B)) == 0


@pytest.mark.parametrize("B", [64, 128])
def test_tensor_core_gather_one_k_block_large_buckets(build_lib, B):
    """H = 64: every unit of the tensor-core gather is one k-block, and B*K >= 4C makes the
    item hand-out ticketed (the next item claimed once the previous one is consumed).  The
    B warps must settle the stages they still owe a signal before they block on the next
    unit, or the claim never comes (the call then ended in the bounded waits' timeout).
    Argmax and sparse pair against the oracle, the device error word clear."""
    m = build_lib
    g = np.random.default_rng(300 + B)
    V, C, H, K = 65536, 256, 64, 32
    cw = synth.bf16_bits(g.integers(-8, 9, size=(C, H)).astype(np.float32))
    ew = synth.bf16_bits(g.integers(-8, 9, size=(V, H)).astype(np.float32))
    perm = g.permutation(V).astype(np.int32)
    hid = synth.bf16_bits(g.integers(-16, 17, size=(B, H)).astype(np.float32))
    oh = oracle.Head(cw, ew, perm, None, K)
    dh = m.MaskedHead(helpers.bf16_tensor(cw), helpers.bf16_tensor(ew), torch.from_numpy(perm).cuda(), K)
    assert m.mtp_gather_plan(dh, B) == "tensor_core"
    h = helpers.bf16_tensor(hid)
    tok, mx = m.mtp_masked_topk_tokens(dh, h)
    torch.cuda.synchronize()
    assert m.mtp_read_device_error(dh.workspace(B)) == 0
    ref = oracle.masked_topk_tokens(oh, hid)
    np.testing.assert_array_equal(tok.cpu().numpy(), ref["tokens"])
    np.testing.assert_array_equal(mx.cpu().numpy(), ref["max_logit"].astype(np.float32))
    plog, pids = m.mtp_select_and_score(dh, h)
    torch.cuda.synchronize()
    assert m.mtp_read_device_error(dh.workspace(B)) == 0
    for b in range(0, B, 17):
        rl, rt = oracle.select_and_score_row(oh, hid, b)
        np.testing.assert_array_equal(pids[b].cpu().numpy(), rt)
        np.testing.assert_array_equal(plog[b].cpu().numpy(), rl.astype(np.float32))


@pytest.mark.parametrize("V,C,H,K,B,packed,protos", [
    (65536, 256, 128, 32, 128, False, 0),     # two k-blocks per unit, ticketed hand-out
    (65536, 256, 192, 16, 64, True, 0),       # three k-blocks, packed table, ticketed
    (32768, 512, 64, 64, 96, True, 0),        # 64-position clusters: paired short chunks, one k-block
    (32768, 512, 256, 32, 40, True, 0),       # paired chunks, round-robin, 32-row units
    (65536, 1024, 64, 16, 20, True, 0),       # paired chunks, tiny buckets, round-robin
    (131072, 1024, 320, 8, 256, False, 4),    # five k-blocks; four prototypes x 64 rows: 64-row
                                              # buckets span two 32-row units
    (32768, 512, 128, 32, 256, True, 4),      # ticketed, paired short chunks beside buckets of
])                                            # several 64-row blocks (items per block)
def test_tensor_core_gather_shape_matrix(build_lib, V, C, H, K, B, packed, protos):
    """Integer inputs (every sum exact, so bit-for-bit against the oracle) over shapes that
    cross the tensor-core gather's switches: units of one to five k-blocks against the B
    warps' signal lag, ticketed and round-robin hand-out, paired short chunks, bucket-row
    caps of 16 to 64 rows and buckets spanning several units (one work item per block of
    a bucket's rows).  Argmax, scatter and sparse
    pair; the device error word must stay clear (a stalled pipeline ends in a timeout)."""
    m = build_lib
    g = np.random.default_rng(V + C + H + K + B)
    cw = synth.bf16_bits(g.integers(-8, 9, size=(C, H)).astype(np.float32))
    ew = synth.bf16_bits(g.integers(-8, 9, size=(V, H)).astype(np.float32))
    perm = g.permutation(V).astype(np.int32)
    rows = g.integers(-16, 17, size=(protos or B, H)).astype(np.float32)
    hid = synth.bf16_bits(np.repeat(rows, B // protos, axis=0) if protos else rows)
    oh = oracle.Head(cw, ew, perm, None, K)
    dh = m.MaskedHead(helpers.bf16_tensor(cw), helpers.bf16_tensor(ew), torch.from_numpy(perm).cuda(), K)
    if packed:
        dh.use_packed_table()
    m.mtp_force_gather("tensor_core")
    try:
        h = helpers.bf16_tensor(hid)
        tok, mx = m.mtp_masked_topk_tokens(dh, h)
        torch.cuda.synchronize()
        assert m.mtp_read_device_error(dh.workspace(B)) == 0
        sc = m.mtp_masked_scatter_logits(dh, h)
        torch.cuda.synchronize()
        assert m.mtp_read_device_error(dh.workspace(B)) == 0
        plog, pids = m.mtp_select_and_score(dh, h)
        torch.cuda.synchronize()
        assert m.mtp_read_device_error(dh.workspace(B)) == 0
    finally:
        m.mtp_force_gather(None)
    ref = oracle.masked_topk_tokens(oh, hid)
    np.testing.assert_array_equal(tok.cpu().numpy(), ref["tokens"])
    np.testing.assert_array_equal(mx.cpu().numpy(), ref["max_logit"].astype(np.float32))
    some = list(range(0, B, max(1, B // 6)))
    np.testing.assert_array_equal(sc[some].cpu().numpy(),
                                  oracle.masked_scatter_logits(oh, hid[some]).astype(np.float32))
    for b in some:
        rl, rt = oracle.select_and_score_row(oh, hid, b)
        np.testing.assert_array_equal(pids[b].cpu().numpy(), rt)
        np.testing.assert_array_equal(plog[b].cpu().numpy(), rl.astype(np.float32))


def test_smoke_entry_point(build_lib):
    """The smoke run the package entry point offers (one small invocation of every gather
    against the oracle) passes: it asserts which gather each of its calls runs, so a change
    of the library's plan shows here first."""
    import __graft_entry__
    __graft_entry__.smoke()
