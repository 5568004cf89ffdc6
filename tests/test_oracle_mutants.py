"""Mutation check of the oracle's pins.

Each mutant is a copy of the oracle source with one plausible mistake
planted on the CPU (a swapped operand, a flipped comparison, a dropped term,
a wrong row or index, a wrong scale). The test compiles the copy and runs the
pins against it: at least one pin must fail. A mutant that passes every pin
would mean the pins leave that part of the oracle unchecked.
"""
import os
import shutil

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "specverify_oracle.c")

SAMPLED_TARGET_ROW = ("load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)i, V, s->lt);\n"
                      "        double m_p, logZ_p, m_q, logZ_q;\n"
                      "        softmax_T2(s->lt, V, T, s->p, &m_p, &logZ_p);\n        load_row(s->draft")
SAMPLED_BONUS_ROW = ("load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)G, V, s->lt);\n"
                     "        softmax_T")

MUTANTS = [
    ("alpha_q_over_p", "const double lr = ((lt_x - m_p) - (ld_x - m_q)) / T - (logZ_p - logZ_q);",
     "const double lr = ((ld_x - m_q) - (lt_x - m_p)) / T - (logZ_q - logZ_p);"),
    ("alpha_from_unshifted_logits", "const double lr = ((lt_x - m_p) - (ld_x - m_q)) / T - (logZ_p - logZ_q);",
     "const double lr = (lt_x / T - (m_p / T + logZ_p)) - (ld_x / T - (m_q / T + logZ_q));"),
    ("accept_flipped", "return u < alpha || u == 0.0;", "return u > alpha || u == 0.0;"),
    ("zero_uniform_rejects_underflowed_alpha", "return u < alpha || u == 0.0;", "return u < alpha;"),
    ("temperature_floor", "        double T = (double)temperature[b];\n        for (int j = 0; j <= gamma; ++j)",
     "        double T = (temperature[b] > 0.0f && temperature[b] < 0x1p-16f) ? 0x1p-16 : (double)temperature[b];\n"
     "        for (int j = 0; j <= gamma; ++j)"),
    ("logit_magnitude_limit", "            has_finite = 1;",
     "            has_finite = 1;\n            if (fabs(l[x]) >= 1.5e9) return 0;"),
    ("residual_q_minus_p", "double diff = s->p[x] - s->q[x];", "double diff = s->q[x] - s->p[x];"),
    ("temperature_multiplied", "p[x] = exp((l[x] - m) / T);", "p[x] = exp((l[x] - m) * T);"),
    ("tie_to_highest_index", "if (l[x] > l[a]) a = x;", "if (l[x] >= l[a]) a = x;"),
    ("bonus_from_row_gamma_minus_1", SAMPLED_BONUS_ROW,
     SAMPLED_BONUS_ROW.replace("(size_t)G, V", "(size_t)(G - 1), V")),
    ("draw_without_W", "double t = u * W;", "double t = u;"),
    ("normaliser_drops_a_term", "        Z += p[x];", "        if (x > 0) Z += p[x];"),
    ("q_read_from_target", "double px = s->p[x], qx = s->q[x];", "double px = s->p[x], qx = s->p[x];"),
    ("gather_off_by_one", "        int x = tok[i];", "        int x = (tok[i] + 1) % V;"),
    ("greedy_keeps_draft_token", "            out[i] = a;\n            return i;",
     "            out[i] = tok[i];\n            return i;"),
    ("greedy_count_off_by_one", "            out[i] = a;\n            return i;",
     "            out[i] = a;\n            return i + 1;"),
    ("target_row_stride_gamma", SAMPLED_TARGET_ROW,
     SAMPLED_TARGET_ROW.replace("(size_t)b * (size_t)(G + 1) + (size_t)i", "(size_t)b * (size_t)G + (size_t)i")),
    ("draft_rows_reversed", "load_row(s->draft, s->dtype, r, V, s->ld);\n        softmax_T2(s->ld, V, T, s->q, &m_q, &logZ_q);",
     "load_row(s->draft, s->dtype, (size_t)b * (size_t)G + (size_t)(G - 1 - i), V, s->ld);\n"
     "        softmax_T2(s->ld, V, T, s->q, &m_q, &logZ_q);"),
    ("bf16_decoded_wrong", "[idx]) << 16;", "[idx]) << 15;"),
    ("accepted_token_not_copied", "            out[i] = x;\n        } else {", "            out[i] = tok[0];\n        } else {"),
    ("no_padding_after_n", "for (int j = 0; j <= gamma; ++j) out[j] = -1;",
     "for (int j = 0; j < gamma; ++j) out[j] = -1;"),
    ("residual_from_next_row", "            n = i;\n            break;",
     "            n = i;\n            if (i + 1 < G) {\n"
     "                load_row(s->target, s->dtype, (size_t)b * (size_t)(G + 1) + (size_t)(i + 1), V, s->lt);\n"
     "                softmax_T(s->lt, V, T, s->p);\n            }\n            break;"),
    ("q_zero_rejects", "    if (ld_x == -INFINITY) return 1.0;", "    if (ld_x == -INFINITY) return 0.0;"),
    ("nan_not_detected", "if (isnan(l[x])) return 0;", "if (0) return 0;"),
    ("draw_from_first_token", "        if (C > t) {", "        if (C >= 0.0) {"),
    # the checker's tie measure
    ("tie_measure_adds_overlaps", "        if (a <= hi) {\n            if (b > hi) hi = b;\n        } else {",
     "        if (0) {\n            if (b > hi) hi = b;\n        } else {"),
    ("tie_measure_wide_margin", "    const double delta = ORACLE_TIE_MARGIN * W;", "    const double delta = 10.0 * ORACLE_TIE_MARGIN * W;"),
    # deterministic (one-hot) proposals
    ("onehot_residual_keeps_x", "double diff = s->p[x] - (x == tok[n] ? 1.0 : 0.0);", "double diff = s->p[x];"),
    ("onehot_alpha_always_one", "double alpha = fmin(1.0, px / qx);", "double alpha = 1.0;"),
    ("onehot_bonus_from_row_gamma", "(size_t)b * (size_t)(G + 1) + (size_t)k, V, s->lt);\n        softmax_T",
     "(size_t)b * (size_t)(G + 1) + (size_t)G, V, s->lt);\n        softmax_T"),
    ("onehot_count_ignored", "        int k = num_draft[b];", "        int k = gamma;"),
    # early exit
    ("early_alpha_ignores_q", "            alpha = accept_alpha(s->lt[x], m_p, logZ_p, s->ld[x], m_q, logZ_q, T);",
     "            alpha = fmin(px, 1.0);"),
    ("early_greedy_keeps_draft_token", "                out[i] = a;\n                return i;",
     "                out[i] = x;\n                return i;"),
    ("early_extra_token_from_row_k_minus_1", "    for (int i = 0; i <= k; ++i) {\n        size_t tr",
     "    for (int i = 0; i < k + (k == 0); ++i) {\n        size_t tr"),
    ("early_onehot_residual_keeps_x", "const double qy = onehot ? (y == x ? 1.0 : 0.0) : s->q[y];",
     "const double qy = onehot ? 0.0 : s->q[y];"),
    # tree verification
    ("tree_alpha_not_renormalised", "const double alpha = rest > 0.0 ? fmin(1.0, px / rest) : 0.0;",
     "const double alpha = rest > 0.0 ? fmin(1.0, px) : 0.0;"),
    ("tree_children_of_the_root_only", "            if (par[c - 1] != u) continue;",
     "            if (par[c - 1] != 0) continue;"),
    ("tree_residual_keeps_rejected", "            s->w[y] = ex ? 0.0 : s->p[y];", "            s->w[y] = s->p[y];"),
    ("tree_greedy_takes_first_child", "if (par[c - 1] == u && tok[c - 1] == a) next = c;",
     "if (par[c - 1] == u) next = c;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_fails_a_pin(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mdir = tmp_path / "oracle_mutant"
    mdir.mkdir()
    shutil.copy(os.path.join(os.path.dirname(SRC), "specverify_oracle.h"), mdir)
    msrc = mdir / "specverify_oracle.c"
    msrc.write_text(src.replace(old, new))
    lib = oracle.load_path(oracle.build(force=True, src=str(msrc), out=str(mdir / "lib.so")))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib, quick=True)
        except AssertionError:
            failed.append(pin.__name__)
            break
    assert failed, f"mutant {name} passed every pin"
