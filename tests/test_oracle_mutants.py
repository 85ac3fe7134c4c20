"""Plant one plausible mistake at a time in a copy of the oracle's C source,
compile the copy on the CPU, and check that at least one pin rejects it.

This is the evidence that the pins constrain every part of the oracle: a
dropped scale, a wrong alignment offset, a window off by one, a global
offset used as a position, a wrong head grouping, a missing denominator term
in the backward and so on
("attention-algorithm-error-and-complexity-tests", first and fourth
paragraphs; "formal-correctness", "The Counterexample": a missing rescale is
correct whenever the maximum does not move, so pins must hit the slice where
it is wrong).  Mistakes are planted only in the CPU oracle copy, never in the
CUDA path.
"""
import os

import pytest

import oracle
from tests import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "dropped_scale": ("return p->scale * dot(qi, kj, p->d) +", "return dot(qi, kj, p->d) +"),
    "lse_without_max": ("double lse_i = m + log(l);", "double lse_i = log(l);"),
    "no_max_subtraction": ("if (mrow[u]) l += exp(srow[u] - m);",
                           "if (mrow[u]) l += exp(srow[u]);"),
    "top_left_strict": ("bound = i;", "bound = i - 1;"),
    "bottom_right_off_by_one": ("bound = i + nk - nq;", "bound = i + nk - nq + 1;"),
    "bottom_right_as_top_left": ("bound = i + nk - nq;", "bound = i;"),
    "window_off_by_one": ("bound - j >= p->window", "bound - j > p->window"),
    "window_ignored": ("if (p->window > 0 && bound - j >= p->window) return 0;", ""),
    "window_from_query_position": ("bound - j >= p->window", "i - j >= p->window"),
    "bias_sign_flipped": ("return -p->slopes[h] * fabs((double)dist);",
                          "return p->slopes[h] * fabs((double)dist);"),
    "bias_without_offset": ("int off = p->mask_kind == ORACLE_MASK_BOTTOM_RIGHT ? nk - nq : 0;",
                            "int off = 0;"),
    "bias_signed_distance": ("return -p->slopes[h] * fabs((double)dist);",
                             "return -p->slopes[h] * (double)dist;"),
    "bias_global_positions": ("int dist = p->pos_q[tq] + off - p->pos_k[tk];",
                              "int dist = tq + off - tk;"),
    "bias_missing_in_backward": ("double s = logit(p, qi, kj, t, u, h);",
                                 "double s = p->scale * dot(qi, kj, p->d);"),
    "tab_bias_sign_flipped": ("return p->btab[", "return -p->btab["),
    "tab_bias_head_ignored": ("(int64_t)h * p->bhs", "0 * p->bhs"),
    "tab_bias_sequence_ignored": ("s * p->bss", "0 * p->bss"),
    "tab_bias_in_log2_units": ("+ tab_bias(p, tq, tk, h);", "+ 1.4426950408889634 * tab_bias(p, tq, tk, h);"),
    "tab_masked_row_not_empty": ("if (m == -INFINITY) { /* every allowed logit masked by the bias tensor */",
                                 "if (0) {"),
    "window_accepted_without_causal": (
        "if (window > 0 && mask_kind == ORACLE_MASK_NONE) return -1;", ""),
    "global_offset_as_position": ("pos[t] = t - cu[s];", "pos[t] = t;"),
    "cross_sequence_pairs": ("if (s < 0 || p->seq_k[tk] != s) return 0;", "if (s < 0) return 0;"),
    "interleaved_gqa": ("int hk = h / (p->hq / p->hkv);", "int hk = h % p->hkv;"),
    "empty_row_lse_zero": ("*lse = -INFINITY;", "*lse = 0.0;"),
    "dq_missing_scale": ("dq_row[c] += p->scale * ds * kj[c];", "dq_row[c] += ds * kj[c];"),
    "ds_missing_D": ("double ds = pij * (dpij - D_i);", "double ds = pij * dpij;"),
    "dk_missing_scale": ("dk[c] += p->scale * ds * qi[c];", "dk[c] += ds * qi[c];"),
    "dv_missing_p": ("dv[c] += pij * doi[c];", "dv[c] += doi[c];"),
    "gqa_grad_not_summed": ("for (int r = 0; r < g; r++) {", "for (int r = 0; r < 1; r++) {"),
    "p_not_normalised": ("double pij = exp(srow[u] - lse_i);", "double pij = exp(srow[u] - m);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    path = tmp_path / "attn_oracle_mutant.c"
    path.write_text(mutated)
    lib = oracle.compile_library(str(path), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
            break
    assert failed, f"no pin rejects the mutant {name}"
