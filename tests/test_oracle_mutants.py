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
