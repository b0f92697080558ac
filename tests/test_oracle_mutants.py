"""Planted mistakes in copies of the oracle must each fail a pin.

Each mutant is the committed oracle source with one plausible mistake (a
dropped term, a wrong sign, a wrong index or operand), compiled with gcc into
a temporary directory. The committed oracle itself is never changed. CPU only.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "no_max_shift": ("t += exp((double)x[j] - r.m);", "t += exp((double)x[j]);"),
    "label_sign": ("(st.m - (double)x[label]) + log1p(st.t)", "(st.m + (double)x[label]) + log1p(st.t)"),
    "max_counted_twice": ("if (j == r.jmax)\n            continue;", ""),
    "log_not_log1p": ("loss_out[i] = (st.m - (double)x[label]) + log1p(st.t);",
                      "loss_out[i] = (st.m - (double)x[label]) + log(1.0 + st.t);"),
    "softmax_over_t": ("double p = exp((double)x[j] - st.m) / s;",
                       "double p = exp((double)x[j] - st.m) / st.t;"),
    "grad_sign": ("g[j] = (p - onehot) * scale;", "g[j] = (onehot - p) * scale;"),
    "onehot_off_by_one": ("(label_ok && j == label)", "(label_ok && j == label + 1)"),
    "scale_dropped": ("g[j] = (p - onehot) * scale;", "g[j] = (p - onehot);"),
    "mean_divisor": ("return sum / (double)rows;", "return sum / (double)(rows - 1);"),
    "stride_ignored": ("const float *x = logits + i * stride;\n        double *g",
                       "const float *x = logits + i * vocab;\n        double *g"),
    "argmax_last_of_equals": ("if (!seen || v > best_v) {", "if (!seen || v >= best_v) {"),
    "argmax_nan_wins": ("            if (isnan(v))\n                continue;\n            if (!seen || v > best_v)",
                        "            if (!seen || v > best_v || isnan(v))"),
    "nan_rows_not_flagged": ("if (any_nan || !seen || isinf(r.m))", "if (!seen)"),
    "grad_transposed": ("double *g = grad_out + i * vocab;", "double *g = grad_out + i;"),
    "softmax_no_shift": ("o[j] = st.degenerate ? NAN : exp((double)x[j] - st.m) / (1.0 + st.t);",
                         "o[j] = st.degenerate ? NAN : exp((double)x[j]) / (1.0 + st.t);"),
    "softmax_sum_is_t": ("exp((double)x[j] - st.m) / (1.0 + st.t);", "exp((double)x[j] - st.m) / st.t;"),
    "log_softmax_cancels": ("((double)x[j] - st.m) - log1p(st.t);", "(double)x[j] - (st.m + log1p(st.t));"),
    "log_softmax_log_t": ("((double)x[j] - st.m) - log1p(st.t);", "((double)x[j] - st.m) - log(st.t);"),
    "cand_last_of_equals": ("while (pos < kept && kv[pos] >= v)", "while (pos < kept && kv[pos] > v)"),
    "cand_ascending": ("while (pos < kept && kv[pos] >= v)", "while (pos < kept && kv[pos] <= v)"),
    "cand_nan_kept": ("                if (isnan(v))\n                    continue;\n                /* where", "                /* where"),
    "cand_blocked_columns": ("for (int64_t j = t; j < vocab; j += CAND_THREADS) {",
                             "for (int64_t j = t * 4; j < vocab && j < t * 4 + 4; ++j) {"),
    "cand_keeps_three": ("if (pos >= CAND_KEEP)\n                    continue;", "if (pos >= CAND_KEEP - 1)\n                    continue;"),
    "cand_empty_token_zero": ("slot[1] = k < kept ? (float)kc[k] : -1.0f;", "slot[1] = k < kept ? (float)kc[k] : 0.0f;"),
    "cand_thread_major_swapped": ("float *slot = out + 2 * (CAND_KEEP * t + k);", "float *slot = out + 2 * (CAND_THREADS * k + t);"),
    "split_sum_add_ignored": ("double acc = add ? (double)y_in[i] : 0.0;", "double acc = 0.0;"),
    "split_sum_drops_last_part": ("for (int64_t s = 0; s < splits; ++s)", "for (int64_t s = 0; s + 1 < splits; ++s)"),
    "split_sum_transposed": ("acc += (double)p[s * total + i];", "acc += (double)p[i * splits + s];"),
    "stats_t_counts_max": ("                if (j != jmax)\n                    t += exp((double)x[j] - m);",
                           "                t += exp((double)x[j] - m);"),
    "stats_top_local": ("o[2] = jmax < 0 ? -1.0 : (double)(col0 + jmax);", "o[2] = jmax < 0 ? -1.0 : (double)jmax;"),
    "stats_xl_unowned": ("o[3] = (local >= 0 && local < vocab) ? (double)x[local] : 0.0;",
                         "o[3] = (local >= 0 && local < vocab) ? (double)x[local] : (double)x[0];"),
    "combine_no_rescale": ("T += (1.0 + st[1]) * exp(st[0] - M);", "T += (1.0 + st[1]);"),
    "combine_drops_tied_max": ("T += (1.0 + st[1]) * exp(st[0] - M);", "T += st[1] * exp(st[0] - M);"),
    "combine_last_top": ("(top < 0.0 || st[2] < top)", "(top < 0.0 || st[2] > top)"),
    "combine_nan_ignored": ("int degenerate = any_nan_t || isinf(M) || star < 0;", "int degenerate = isinf(M) || star < 0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle.build(path, os.path.join(tmp_path, "libmutant.so"), force=True)
    caught = oracle_pins.failing_pins(oracle.load(lib))
    assert caught, f"no pin catches mutant {name}"
