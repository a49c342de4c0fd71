"""Pins for the CPU oracle: checks against things other than the oracle itself.

* hand-worked examples (tests/golden/worked_examples.json), derived from the
  definition of Gemma4MTPMaskedEmbedder ("Add Gemma4 MTP speculative decoding
  with centroids masking", vLLM gemma4_mtp.py) with exact integer values;
* the top-K set found by enumerating every K-subset;
* closed forms: with K = C, or with a single centroid, the masked head is the
  dense head (whose logits are checked against numpy's matmul);
* integer-valued inputs, where every sum is exact, against integer matmul;
* invariants of the method: candidate counts, the -inf count of the full-vocab
  row, argmax(full-vocab row) == sparse argmax, identity ordering.
"""
import itertools
import json
import os

import numpy as np
import pytest

from centroid_masked_sparse_gb300 import synth
from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _num(v):
    return -np.inf if v == "-inf" else float(v)


def _bits(a):
    return synth.bf16_bits(np.asarray(a, dtype=np.float32))


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)["examples"]


def _head_from_example(ex):
    offs = None if ex["cluster_offsets"] is None else np.array(ex["cluster_offsets"], np.int32)
    return oracle.Head(_bits(ex["centroid_w"]), _bits(ex["embed_w"]),
                       np.array(ex["token_ordering"], np.int32), offs, ex["K"], vocab=ex["V"])


@pytest.mark.parametrize("ex", _golden(), ids=lambda e: e["name"])
def test_worked_examples(ex):
    head = _head_from_example(ex)
    hidden = _bits(ex["hidden"])
    e = ex["expect"]
    res = oracle.masked_topk_tokens(head, hidden, threads=1)
    np.testing.assert_array_equal(res["sel"], np.array(e["selection"]))
    np.testing.assert_array_equal(res["tokens"], np.array(e["token"]))
    np.testing.assert_array_equal(res["max_logit"], np.array([_num(v) for v in e["max_logit"]]))
    if "score_margin" in e:
        np.testing.assert_array_equal(res["score_margin"], np.array(e["score_margin"], float))
    if "logit_margin" in e:
        np.testing.assert_array_equal(res["logit_margin"], np.array(e["logit_margin"], float))
    for b in range(hidden.shape[0]):
        logs, toks = oracle.select_and_score_row(head, hidden, b)
        np.testing.assert_array_equal(toks, np.array(e["candidate_tokens"][b], dtype=np.int32))
        np.testing.assert_array_equal(logs, np.array(e["candidate_logits"][b], dtype=float))
    sc = oracle.masked_scatter_logits(head, hidden, threads=1)
    np.testing.assert_array_equal(sc, np.array([[_num(v) for v in row] for row in e["scatter"]]))
    de = oracle.dense_logits(head, hidden, threads=1)
    np.testing.assert_array_equal(de, np.array(e["dense"], dtype=float))
    # dense argmax with the lower-id tie rule
    np.testing.assert_array_equal(np.argmax(de, axis=1), np.array(e["dense_argmax"]))


def _topk_bruteforce(scores, K):
    """The unique K-subset S with (s_i > s_j) or (s_i == s_j and i < j) for i in S, j not in S."""
    C = len(scores)
    found = []
    for S in itertools.combinations(range(C), K):
        Sset = set(S)
        ok = all((scores[i] > scores[j]) or (scores[i] == scores[j] and i < j)
                 for i in S for j in range(C) if j not in Sset)
        if ok:
            found.append(Sset)
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("seed", range(12))
def test_topk_matches_subset_enumeration(seed):
    g = np.random.default_rng(seed)
    C = int(g.integers(2, 11))
    K = int(g.integers(1, C + 1))
    if seed % 2:
        scores = g.integers(-2, 3, size=C).astype(float)   # many exact ties
    else:
        scores = g.standard_normal(C)
    sel, margin = oracle.topk_row(scores, K)
    assert set(sel.tolist()) == _topk_bruteforce(scores.tolist(), K)
    # sorted by (score desc, index asc)
    for a, b in zip(sel[:-1], sel[1:]):
        assert scores[a] > scores[b] or (scores[a] == scores[b] and a < b)
    if K < C:
        rest = [scores[j] for j in range(C) if j not in set(sel.tolist())]
        assert margin == scores[sel[-1]] - max(rest)
    else:
        assert margin == np.inf


def _small_tables(seed, V=96, C=8, H=16, sizes=None, identity=False):
    return synth.custom_tables(V, H, C, seed, std=0.25, sizes=sizes, identity=identity)


def _dense_numpy(head, hidden):
    E = synth.bf16_to_f32(head.embed_w[:head.V, :head.H]).astype(np.float64)
    X = synth.bf16_to_f32(hidden).astype(np.float64)
    return X @ E.T


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_dense_matches_numpy_matmul(seed):
    t = _small_tables(seed)
    head = oracle.Head.from_tables(t, top_k=3)
    hidden = synth.random_hidden(5, head.H, seed)
    np.testing.assert_allclose(oracle.dense_logits(head, hidden), _dense_numpy(head, hidden),
                               rtol=1e-12, atol=1e-12)
    rows = np.array([0, 4, 2, 2]); toks = np.array([0, 95, 17, 3])
    np.testing.assert_allclose(oracle.dense_logits_at(head, hidden, rows, toks),
                               _dense_numpy(head, hidden)[rows, toks], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed,sizes", [(4, None), (5, [1, 30, 7, 0, 20, 11, 2, 25])])
def test_k_equals_c_is_dense(seed, sizes):
    t = _small_tables(seed, sizes=sizes)
    head = oracle.Head.from_tables(t, top_k=8)
    hidden = synth.random_hidden(6, head.H, seed + 100)
    dense = oracle.dense_logits(head, hidden)
    sc = oracle.masked_scatter_logits(head, hidden)
    np.testing.assert_array_equal(sc, dense)
    res = oracle.masked_topk_tokens(head, hidden)
    np.testing.assert_array_equal(res["tokens"], np.argmax(dense, axis=1))
    np.testing.assert_array_equal(res["max_logit"], dense.max(axis=1))
    np.testing.assert_array_equal(res["n_cand"], np.full(6, head.V))


def test_single_centroid_is_dense():
    t = synth.custom_tables(64, 16, 1, 9, std=0.25)
    head = oracle.Head.from_tables(t, top_k=1)
    hidden = synth.random_hidden(3, 16, 9)
    dense = _dense_numpy(head, hidden)
    np.testing.assert_allclose(oracle.masked_scatter_logits(head, hidden), dense, rtol=1e-12)
    np.testing.assert_array_equal(oracle.masked_topk_tokens(head, hidden)["tokens"],
                                  np.argmax(dense, axis=1))


def test_integer_inputs_are_exact():
    g = np.random.default_rng(7)
    V, C, H, K = 128, 16, 32, 5
    cw = g.integers(-4, 5, size=(C, H))
    ew = g.integers(-4, 5, size=(V, H))
    hid = g.integers(-4, 5, size=(4, H))
    perm = g.permutation(V).astype(np.int32)
    head = oracle.Head(_bits(cw), _bits(ew), perm, None, K)
    hidden = _bits(hid)
    dense_exact = (hid.astype(np.int64) @ ew.T.astype(np.int64)).astype(np.float64)
    scores_exact = (hid.astype(np.int64) @ cw.T.astype(np.int64)).astype(np.float64)
    np.testing.assert_array_equal(oracle.centroid_scores(head, hidden), scores_exact)
    np.testing.assert_array_equal(oracle.dense_logits(head, hidden), dense_exact)
    res = oracle.masked_topk_tokens(head, hidden)
    S = V // C
    for b in range(4):
        assert set(res["sel"][b].tolist()) == _topk_bruteforce(scores_exact[b].tolist(), K)
        cand = np.concatenate([perm[c * S:(c + 1) * S] for c in res["sel"][b]])
        best = dense_exact[b, cand].max()
        assert res["max_logit"][b] == best
        assert res["tokens"][b] == cand[dense_exact[b, cand] == best].min()


@pytest.mark.parametrize("identity", [False, True])
def test_invariants_tiny(identity):
    w = synth.WORKLOADS["tiny"]
    t = synth.make_tables(w)
    if identity:
        t.token_ordering = np.arange(w.vocab, dtype=np.int32)
    head = oracle.Head.from_tables(t)
    hidden = synth.hidden_batch(w, 8)
    res = oracle.masked_topk_tokens(head, hidden)
    sc = oracle.masked_scatter_logits(head, hidden)
    S = w.vocab // w.centroids
    assert oracle.is_permutation(t.token_ordering)
    for b in range(8):
        assert res["n_cand"][b] == w.top_k * S
        assert np.isneginf(sc[b]).sum() == w.vocab - w.top_k * S
        fin = np.isfinite(sc[b])
        # the finite entries are exactly the tokens of the selected clusters
        expect = np.zeros(w.vocab, bool)
        for c in res["sel"][b]:
            expect[t.token_ordering[c * S:(c + 1) * S]] = True
        np.testing.assert_array_equal(fin, expect)
        if identity:
            # identity ordering: the candidates are the contiguous ranges
            for c in res["sel"][b]:
                assert fin[c * S:(c + 1) * S].all()
        assert np.argmax(sc[b]) == res["tokens"][b]
        assert sc[b].max() == res["max_logit"][b]


def test_variable_cluster_candidate_counts():
    sizes = [3, 0, 9, 1, 14, 5, 0, 28]
    t = synth.custom_tables(60, 16, 8, 11, std=0.25, sizes=sizes)
    head = oracle.Head.from_tables(t, top_k=3)
    hidden = synth.random_hidden(7, 16, 11)
    res = oracle.masked_topk_tokens(head, hidden)
    sc = oracle.masked_scatter_logits(head, hidden)
    for b in range(7):
        n = sum(sizes[c] for c in res["sel"][b])
        assert res["n_cand"][b] == n
        assert np.isfinite(sc[b]).sum() == n


def test_second_formulation_tiny():
    """Cross-check (not a pin): a vectorised numpy float64 restatement."""
    w = synth.WORKLOADS["tiny"]
    t = synth.make_tables(w)
    head = oracle.Head.from_tables(t)
    hidden = synth.hidden_batch(w, 16)
    X = synth.bf16_to_f32(hidden).astype(np.float64)
    Wc = synth.bf16_to_f32(t.centroid_w).astype(np.float64)
    E = synth.bf16_to_f32(t.embed_w).astype(np.float64)
    scores = X @ Wc.T
    S = w.vocab // w.centroids
    res = oracle.masked_topk_tokens(head, hidden)
    for b in range(16):
        order = np.lexsort((np.arange(w.centroids), -scores[b]))[:w.top_k]
        cand = t.token_ordering.reshape(w.centroids, S)[order].reshape(-1)
        logits = E[cand] @ X[b]
        np.testing.assert_array_equal(order, res["sel"][b])
        best = logits.max()
        assert res["tokens"][b] == cand[logits == best].min()
        assert abs(res["max_logit"][b] - best) < 1e-12


def test_permutation_check():
    assert oracle.is_permutation(np.array([2, 0, 1], np.int32))
    assert not oracle.is_permutation(np.array([2, 0, 2], np.int32))
    assert not oracle.is_permutation(np.array([3, 0, 1], np.int32))


def test_generator_basics():
    # bf16 round-to-nearest-even
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5, 0.0], dtype=np.float32)
    assert synth.bf16_bits(x).tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000]
    s = synth.lognormal_cluster_sizes(262144, 2048, 123)
    assert s.sum() == 262144 and s.min() >= 1 and s.max() > 2 * 128
    off = synth.offsets_from_sizes(s)
    assert off[0] == 0 and off[-1] == 262144 and np.all(np.diff(off) >= 1)
    # row redraws are independent of the other rows
    a = synth.hidden_batch("uniform", 4)
    b = synth.hidden_batch("uniform", 4, attempts=np.array([0, 1, 0, 0]))
    assert (a[0] == b[0]).all() and (a[2] == b[2]).all() and not (a[1] == b[1]).all()


def test_round_bf16_values():
    """Round-to-nearest-even to bf16 (8 significant bits), values worked by hand."""
    r = oracle.round_bf16
    assert r(256.0) == 256.0
    assert r(257.0) == 256.0            # midpoint of 256 and 258: the even mantissa (256)
    assert r(259.0) == 260.0            # midpoint of 258 and 260: 260 is even
    assert r(-257.0) == -256.0
    assert r(257.5) == 258.0            # above the midpoint
    assert r(1 + 2 ** -8) == 1.0        # midpoint of 1 and 1 + 2^-7
    assert r(1 + 3 * 2 ** -8) == 1 + 2 ** -6
    assert r(0.1) == 0.10009765625      # bf16 0x3DCD
    assert r(2.0 ** -140) == 0.0        # below half the smallest subnormal 2^-133
    assert r(3 * 2.0 ** -134) == 2 * 2.0 ** -133   # 1.5 quanta: the even multiple
    assert r(3.3895313892515355e38) == 3.3895313892515355e38
    assert r(3.4e38) == float("inf")
    assert r(0.0) == 0.0


def _flag_head(flags):
    # C = 2 centroids of H = 2: h = (1, 1) scores 256 and 257; clusters of 2 positions,
    # ordering [3, 0, 1, 2]: centroid 0 owns tokens 3 and 0, centroid 1 tokens 1 and 2
    one, big = 0x3F80, 0x4380          # bf16 1.0 and 256.0
    cw = np.array([[big, 0], [big, one]], np.uint16)
    ew = np.array([[big, 0], [one, 0], [0, one], [big, one]], np.uint16)   # token rows 0..3
    return oracle.Head(cw, ew, np.array([3, 0, 1, 2], np.int32), None, 1, flags=flags)


def test_fidelity_flags_hand_example():
    h = np.array([[0x3F80, 0x3F80]], np.uint16)
    # plain reading: centroid 1 (257 > 256), tokens 1 and 2 both score 1: lower id
    r = oracle.masked_topk_tokens(_flag_head(0), h, threads=1)
    assert r["sel"].tolist() == [[1]] and r["tokens"].tolist() == [1] and r["max_logit"][0] == 1.0
    # bf16 scores: 257 rounds to 256, a tie with centroid 0, whose lower index wins; its
    # tokens 3 and 0 score 257 and 256
    f = oracle.FLAG_BF16_SCORES
    r = oracle.masked_topk_tokens(_flag_head(f), h, threads=1)
    assert r["sel"].tolist() == [[0]] and r["tokens"].tolist() == [3] and r["max_logit"][0] == 257.0
    # bf16 logits too: 257 -> 256 ties with token 0, the lower id
    f = oracle.FLAG_BF16_SCORES | oracle.FLAG_BF16_LOGITS
    r = oracle.masked_topk_tokens(_flag_head(f), h, threads=1)
    assert r["tokens"].tolist() == [0] and r["max_logit"][0] == 256.0
    logs, toks = oracle.select_and_score_row(_flag_head(f), h, 0)
    assert toks.tolist() == [3, 0] and logs.tolist() == [256.0, 256.0]
    # finite fill: bf16's largest negative value where the page's code puts finfo.min
    f = oracle.FLAG_BF16_SCORES | oracle.FLAG_FILL_FINFO_MIN
    sc = oracle.masked_scatter_logits(_flag_head(f), h, threads=1)
    m = -3.3895313892515355e38
    assert sc.tolist() == [[256.0, m, m, 257.0]]
    # dense logits with bf16 rounding
    d = oracle.dense_logits(_flag_head(oracle.FLAG_BF16_LOGITS), h, threads=1)
    assert d.tolist() == [[256.0, 1.0, 1.0, 256.0]]


def test_dense_softcap_hand_example():
    """cap * tanh(logit / cap) on the dense comparator: with cap 2 the logits 256 and 1 of the
    two-centroid example become 2 tanh(128) and 2 tanh(1/2), worked by hand."""
    import math
    h = np.array([[0x3F80, 0x3F80]], np.uint16)
    head = _flag_head(0)
    head.softcap = 2.0
    d = oracle.dense_logits(head, h, threads=1)
    want = [2 * math.tanh(128.0), 2 * math.tanh(0.5), 2 * math.tanh(0.5), 2 * math.tanh(128.5)]
    assert d.tolist() == [want]
    assert abs(d[0, 1] - 0.9242343145200195) < 1e-15   # 2 tanh(1/2)
    head.softcap = 0.0
    assert oracle.dense_logits(head, h, threads=1).tolist() == [[256.0, 1.0, 1.0, 257.0]]
