"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Every mutant is the committed oracle source with one textual edit, compiled
into a temporary directory on the CPU.  A mutant that passes every pin would
mean the pins cannot tell that mistake from the correct oracle.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "maxsim_oracle.c")

# (name, exact text in the source, replacement)
MUTANTS = [
    ("ignore_doc_mask", "if (dm && !dm[j]) continue;", ";"),
    ("ignore_query_mask", "if (qm && !qm[i]) {", "if (0) {"),
    ("ties_go_high", "if (s > best) {", "if (s >= best) {"),
    ("empty_doc_scores_zero", "return ORACLE_EMPTY_DOC_SCORE;", "return 0.0;"),
    ("reversed_dim_index", "q[i * dim + k] * d[j * dim + k]", "q[i * dim + k] * d[j * dim + (dim - 1 - k)]"),
    ("sum_keeps_last_term", "score += best;", "score = best;"),
    ("max_starts_at_zero", "double best = -INFINITY, second = -INFINITY;",
     "double best = 0.0, second = -INFINITY;"),
    ("gap_against_worst", "} else if (s > second) {", "} else if (s < second) {"),
    ("gQ_drops_upstream", "g[p] * widen(D, dtype", "widen(D, dtype"),
    ("gD_wrong_row", "gD[(dd * Ld + a) * dim + k]", "gD[(dd * Ld + (Ld - 1 - a)) * dim + k]"),
    ("gQ_wrong_token", "gQ[(qq * Lq + i) * dim + k]", "gQ[(qq * Lq + (Lq - 1 - i)) * dim + k]"),
    ("bf16_shift", "(uint32_t)h << 16", "(uint32_t)h << 15"),
    ("f16_bias", "e - 25", "e - 24"),
    ("f16_subnormal_scale", "ldexp((double)m, -24)", "ldexp((double)m, -25)"),
    ("ce_loss_not_mean", "*loss = rows > 0 ? total / (double)rows : 0.0;", "*loss = total;"),
    ("ce_grad_no_onehot", "(c == t ? 1.0 : 0.0)", "(c == t ? 0.0 : 0.0)"),
    ("ce_grad_no_scale", "gr[c] = scale * (exp", "gr[c] = (exp"),
    ("ce_wrong_target_logit", "row_loss[r] = lse - scale * s[t];", "row_loss[r] = lse - scale * s[0];"),
    ("ce_grad_not_mean", "/ (double)rows;", ";"),
    ("kd_wrong_candidate", "score_blocks(Q, D, dtype, b, p, Lq", "score_blocks(Q, D, dtype, b, b, Lq"),
    ("pairwise_wrong_doc", "scores[b] = score_blocks(Q, D, dtype, b, b,",
     "scores[b] = score_blocks(Q, D, dtype, b, (b + 1) % B,"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation target for {name} must occur exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_oracle(str(path), str(tmp_path / f"lib{name}.so"))
    mutant = oracle.Oracle(oracle.load_library(lib))
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(mutant)
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin catches mutant {name}"
