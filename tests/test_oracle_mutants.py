"""Plants plausible mistakes in copies of the oracle (on the CPU) and checks
that the pins catch every one of them."""
import os

import pytest

from oracle import oracle as O
from tests import oracle_pins as P

SRC = open(os.path.join(os.path.dirname(O.__file__), "ss_oracle.c")).read()

WRITE = "double write = delta * B[(b * N + n) * L + t] * xr[t];"
READ = "out += C[(b * N + n) * L + t] * h[n];"
SKIP = "out += (D ? D[d] : 0.0) * xr[t];"
GATE = "out *= zr[t] * sigmoid(zr[t]);"
DELTA = "double delta = delta_softplus ? oracle_softplus(v) : v;"
DECAY = "double a_bar = exp(delta * A[d * N + n]);"
BIAS = "double v = dtr[t] + (dt_bias ? dt_bias[d] : 0.0);"

MUTANTS = {
    "drop_skip_term": [(SKIP, "")],
    "read_before_write": [(READ, "out += C[(b * N + n) * L + t] * (h[n] - delta * B[(b * N + n) * L + t]"
                                 " * xr[t]) / exp(delta * A[d * N + n]);")],
    "softplus_twice": [(DELTA, "double delta = delta_softplus ? oracle_softplus(oracle_softplus(v)) : v;")],
    "gate_before_skip": [(SKIP, ""), (GATE, GATE + " out += (D ? D[d] : 0.0) * xr[t];")],
    "swap_B_and_C": [(WRITE, "double write = delta * C[(b * N + n) * L + t] * xr[t];"),
                     (READ, "out += B[(b * N + n) * L + t] * h[n];")],
    "A_transposed": [(DECAY, "double a_bar = exp(delta * A[n * d_inner + d]);")],
    "bias_ignored": [(BIAS, "double v = dtr[t];")],
    "zoh_write": [(WRITE, "double write = (a_bar - 1.0) / A[d * N + n] * B[(b * N + n) * L + t] * xr[t];")],
    "decay_sign": [(DECAY, "double a_bar = exp(-delta * A[d * N + n]);")],
    "gate_without_z": [(GATE, "out *= sigmoid(zr[t]);")],
    "B_one_step_late": [(WRITE, "double write = delta * B[(b * N + n) * L + (t > 0 ? t - 1 : 0)] * xr[t];")],
    "x_missing_in_write": [(WRITE, "double write = delta * B[(b * N + n) * L + t];")],
    "final_state_stale": [("final_state[r * N + n] = h[n];", "final_state[r * N + n] = h[n] * (L > 1 ? 0.5 : 1.0);")],
    "conv_taps_reversed": [("acc += w[d * k + i] * v;", "acc += w[d * k + (k - 1 - i)] * v;")],
    "conv_lag_off_by_one": [("const int64_t s = t - i;   /* input i steps back */",
                             "const int64_t s = t - i - 1;")],
    "conv_silu_before_bias": [("double acc = bias ? bias[d] : 0.0;", "double acc = 0.0;"),
                              ("out[r * L + t] = silu ? acc * sigmoid(acc) : acc;",
                               "out[r * L + t] = (silu ? acc * sigmoid(acc) : acc) + (bias ? bias[d] : 0.0);")],
    "conv_history_newest_first": [("v = state[(b * (k - 1) + (k - 1 + s)) * d_inner + d];\n                else\n                    v = 0.0;\n                acc",
                                   "v = state[(b * (k - 1) + (-1 - s)) * d_inner + d];\n                else\n                    v = 0.0;\n                acc")],
    "ex_start_zeroed_on_wrong_side": [("if (starts && !reverse)\n                for (int64_t n = 0; n < N; ++n)\n                    h[n] = 0.0;",
                                       "if (starts && reverse)\n                for (int64_t n = 0; n < N; ++n)\n                    h[n] = 0.0;"),
                                      ("if (starts && reverse)\n                for (int64_t n = 0; n < N; ++n)\n                    h[n] = 0.0;\n        }",
                                       "if (starts && !reverse)\n                for (int64_t n = 0; n < N; ++n)\n                    h[n] = 0.0;\n        }")],
    "ex_reverse_walks_forward": [("const int64_t t = reverse ? L - 1 - i : i;", "const int64_t t = i;")],
    "ex_starts_ignored": [("const int starts = seq_start && seq_start[b * L + t];", "const int starts = 0;")],
    "ex_h0_ignored": [("            h[n] = h0 ? h0[r * N + n] : 0.0;\n        for (int64_t i = 0; i < L; ++i) {",
                       "            h[n] = 0.0;\n        for (int64_t i = 0; i < L; ++i) {")],
    "ssd_group_index_wrong": [("const int64_t g = h / (H / G);", "const int64_t g = h % G;")],
    "ssd_read_before_write": [("S[p * N + n] = alpha * S[p * N + n] + delta * xv * Bt[n];\n                    out += Ct[n] * S[p * N + n];",
                               "out += Ct[n] * S[p * N + n];\n                    S[p * N + n] = alpha * S[p * N + n] + delta * xv * Bt[n];")],
    "ssd_decay_without_step": [("const double alpha = exp(delta * A[h]);", "const double alpha = exp(A[h]);")],
    "ssd_state_transposed": [("final_state[r * P * N + i] = S[i];", "final_state[r * P * N + i] = S[(i % N) * P + i / N];")],
    "bwd_adjoint_without_decay": [("lam[n] *= as[(t + 1) * N + n];", "lam[n] *= 1.0;")],
    "bwd_dA_uses_new_state": [("const double ah = as[t * N + n] * hs[t * N + n];  /* a_t h_{t-1} */",
                               "const double ah = as[t * N + n] * hs[(t + 1) * N + n];")],
    "bwd_dfinal_ignored": [("lam[n] = dfinal ? dfinal[r * N + n] : 0.0;", "lam[n] = 0.0;")],
    "bwd_gate_derivative_short": [("dz[r * L + t] = gr[t] * y * s * (1.0 + zr[t] * (1.0 - s));",
                                   "dz[r * L + t] = gr[t] * y * s;")],
    "bwd_softplus_derivative_at_step": [("const double dv = delta_softplus ? ddel * sigmoid(v) : ddel;",
                                         "const double dv = delta_softplus ? ddel * sigmoid(del[t]) : ddel;")],
    "bwd_dC_uses_old_state": [("dC[(b * N + n) * L + t] += gy * hs[(t + 1) * N + n];",
                               "dC[(b * N + n) * L + t] += gy * hs[t * N + n];")],
    "bwd_dB_without_step": [("dB[(b * N + n) * L + t] += lam[n] * del[t] * xr[t];",
                             "dB[(b * N + n) * L + t] += lam[n] * xr[t];")],
    "bwd_skip_gradient_missing": [("double dxt = Dd * gy;", "double dxt = 0.0;")],
    "bwd_dh0_without_decay": [("dh0[r * N + n] = as[n] * lam[n];", "dh0[r * N + n] = lam[n];")],
    "bwd_ex_cut_ignored_in_adjoint": [("lam[n] = cut ? 0.0 : lam[n] * as[(i + 1) * N + n];",
                                       "lam[n] = lam[n] * as[(i + 1) * N + n];")],
    "bwd_ex_dfinal_through_cut": [("            if (CUT_AFTER(i))\n                for (int64_t n = 0; n < N; ++n)\n                    lam[n] = 0.0;\n            double y",
                                   "            double y")],
    "bwd_ex_state_before_cut": [("                hin[i * N + n] = h[n];", "                hin[i * N + n] = i > 0 ? out[(i - 1) * N + n] : h[n];")],
    "bwd_ex_walks_forward": [("#define TW(i) (reverse ? L - 1 - (i) : (i))", "#define TW(i) (i)")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = SRC
    for old, new in MUTANTS[name]:
        assert old in src, (name, old)
        src = src.replace(old, new, 1)
    path = tmp_path / ("mutant_%s.c" % name)
    path.write_text(src)
    lib = O.load(O.build(force=True, src=str(path), out=str(tmp_path / ("lib%s.so" % name))))
    failed = []
    for check in P.ALL_CHECKS:
        try:
            check(lib)
        except (AssertionError, FloatingPointError, OverflowError, ValueError):
            failed.append(check.__name__)
    assert failed, "no pin caught mutant %s" % name
