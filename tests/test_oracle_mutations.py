"""Planted mistakes: each plausible slip in the oracle must fail one of its pins.

A mutated copy of the oracle's C source is compiled into a temporary library
(on the CPU) and the pins of test_oracle_pins.py are run against it; at least
one of them has to fail.  The real oracle is never modified.
"""
import os
import subprocess

import pytest

from oracle import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mtp_oracle.c")

# (name, text in the oracle, planted replacement)
MUTATIONS = [
    ("embedding row indexed by ordered position instead of token id",
     "embed_w + (int64_t)t * ld_embed, H);", "embed_w + (int64_t)p * ld_embed, H);"),
    ("top-K ties go to the higher centroid index",
     "return (a->index > b->index) - (a->index < b->index);",
     "return (a->index < b->index) - (a->index > b->index);"),
    ("top-K keeps the smallest scores",
     "if (a->score > b->score) return -1;", "if (a->score < b->score) return -1;"),
    ("argmax ties go to the higher token id",
     "(v == best && t < best_t)", "(v == best && t > best_t)"),
    ("last term of every dot product dropped",
     "for (int64_t i = 0; i < n; ++i)", "for (int64_t i = 0; i + 1 < n; ++i)"),
    ("subtracted products (wrong sign)",
     "s += bf16_value(x[i]) * bf16_value(w[i]);", "s -= bf16_value(x[i]) * bf16_value(w[i]);"),
    ("full-vocab fill of 0 instead of -inf",
     "? -ORC_BF16_MAX : -INFINITY;", "? -ORC_BF16_MAX : 0.0;"),
    ("dense softcap without dividing by the cap",
     "softcap * tanh(out[b * V + t] / softcap)", "softcap * tanh(out[b * V + t])"),
    ("bf16 rounding with ties away from zero",
     "ldexp(nearbyint(ldexp(x, -q)), q)", "ldexp(round(ldexp(x, -q)), q)"),
    ("bf16-score option rounds the logits instead",
     "        if (flags & ORC_FLAG_BF16_SCORES)\n                scores[c] = orc_round_bf16(scores[c]);\n        }\n        double smargin;",
     "        if (flags & ORC_FLAG_BF16_LOGITS)\n                scores[c] = orc_round_bf16(scores[c]);\n        }\n        double smargin;"),
    ("uniform clusters one position short",
     "*hi = (c + 1) * s;", "*hi = (c + 1) * s - 1;"),
    ("variable clusters read one offset too far",
     "*hi = off[c + 1];", "*hi = off[c + 1] + (c + 2 < C ? 1 : 0);"),
    ("bf16 decoded with the wrong shift",
     "uint32_t u = ((uint32_t)bits) << 16;", "uint32_t u = ((uint32_t)bits) << 15;"),
    ("sparse pair lists a cluster's positions in reverse",
     "        for (int64_t p = lo; p < hi; ++p) {\n            int32_t t = ordering[p];\n            tokens[j] = t;",
     "        for (int64_t p = hi - 1; p >= lo; --p) {\n            int32_t t = ordering[p];\n            tokens[j] = t;"),
    ("sparse pair reports ordered positions as token ids",
     "            tokens[j] = t;\n            logits[j] =", "            tokens[j] = (int32_t)p;\n            logits[j] ="),
    ("sparse pair reports one candidate fewer than it lists",
     "        *n = candidate_count(sel, K, V, C, off);", "        *n = candidate_count(sel, K, V, C, off) - 1;"),
    ("full-vocab scatter stores at the candidate's list index, not its token id",
     "row[cand_tok[j]] = cand_log[j];", "row[j] = cand_log[j];"),
    ("finite-minimum fill takes fp32's minimum instead of bf16's",
     "? -ORC_BF16_MAX : -INFINITY;", "? -3.4028234663852886e38 : -INFINITY;"),
    ("score margin taken between the (K-1)-th and K-th picks",
     "all[K - 1].score - all[K].score", "all[K > 1 ? K - 2 : 0].score - all[K - 1].score"),
    ("logit margin forgets the best it displaces",
     "                if (best_t >= 0)\n                    second = best;",
     "                if (0)\n                    second = best;"),
    ("sampled dense logits read the table row of the batch row, not of the token",
     "embed_w + tokens[i] * ld_embed", "embed_w + rows[i] * ld_embed"),
    ("permutation check accepts repeated token ids",
     "if (t < 0 || t >= V || seen[t])", "if (t < 0 || t >= V)"),
    ("centroid table read transposed",
     "scores[c] = dot_bf16(h_row, centroid_w + c * H, H);",
     "{ scores[c] = 0; for (int64_t i = 0; i < H; ++i) scores[c] += bf16_value(h_row[i]) * "
     "bf16_value(centroid_w[i * C + c]); }"),
]


def _pin_calls():
    ex = pins._golden()
    calls = [(f"golden:{e['name']}", (lambda e=e: pins.test_worked_examples(e))) for e in ex]
    calls += [(f"topk:{s}", (lambda s=s: pins.test_topk_matches_subset_enumeration(s)))
              for s in range(12)]
    calls += [("integer", pins.test_integer_inputs_are_exact),
              ("k_eq_c", lambda: pins.test_k_equals_c_is_dense(5, [1, 30, 7, 0, 20, 11, 2, 25])),
              ("dense_numpy", lambda: pins.test_dense_matches_numpy_matmul(1)),
              ("single", pins.test_single_centroid_is_dense),
              ("variable", pins.test_variable_cluster_candidate_counts),
              ("round_bf16", pins.test_round_bf16_values),
              ("flags", pins.test_fidelity_flags_hand_example),
              ("softcap", pins.test_dense_softcap_hand_example),
              ("permutation", pins.test_permutation_check)]
    return calls


@pytest.mark.parametrize("name,orig,planted", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, monkeypatch, name, orig, planted):
    src = open(SRC).read()
    assert src.count(orig) >= 1, f"mutation anchor not found: {orig}"
    mutated = src.replace(orig, planted)
    path = tmp_path / "mut.c"
    path.write_text(mutated)
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-o", str(so), str(path), "-lm"],
                   check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.load_library(str(so)))
    failed = []
    for label, call in _pin_calls():
        try:
            call()
        except Exception:  # noqa: BLE001 - any failure counts as caught
            failed.append(label)
    assert failed, f"planted mistake '{name}' passed every pin"
