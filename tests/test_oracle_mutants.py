"""Planted mistakes: each plausible bug, planted in a COPY of the oracle source, must fail at least one pin.

This shows the pins are strong enough to trust the oracle: a dropped term, a
wrong sign or index, a swapped operand anywhere in it is caught.  Runs on CPU.
"""
import os

import pytest

import oracle as O
from tests import pins

MUTANTS = {
    "nibble_order": ("int code = (k % 2 == 0) ? (byte & 15) : (byte >> 4);",
                     "int code = (k % 2 == 0) ? (byte >> 4) : (byte & 15);"),
    "zero_nibble_order": ("int zero = (g % 2 == 0) ? (zb & 15) : (zb >> 4);",
                          "int zero = (g % 2 == 0) ? (zb >> 4) : (zb & 15);"),
    "scale_group_index": ("orc_f16_to_double(sr[g])", "orc_f16_to_double(sr[0])"),
    "zero_point_dropped": ("w[k] = (double)(code - zero) * orc_f16_to_double(sr[g]);",
                           "w[k] = (double)(code) * orc_f16_to_double(sr[g]);"),
    "int8_zero_sign": ("w[k] = (double)((int)qr[k] - zero) * scale;", "w[k] = (double)((int)qr[k] + zero) * scale;"),
    "f16_exponent_bias": ("v = ldexp(1024.0 + (double)m, e - 25);", "v = ldexp(1024.0 + (double)m, e - 24);"),
    "f16_subnormal": ("if (e == 0) v = ldexp((double)m, -24);", "if (e == 0) v = ldexp((double)m, -25);"),
    "silu_on_up": ("h[n] = silu(a) * c;", "h[n] = silu(c) * a;"),
    "silu_missing": ("h[n] = silu(a) * c;", "h[n] = a * c;"),
    "down_index": ("for (int n = 0; n < F; ++n) acc += w[n] * h[n];",
                   "for (int n = 0; n < F; ++n) acc += w[n] * h[F - 1 - n];"),
    "sigmoid_sign": ("s[e] = 1.0 / (1.0 + exp(-z));", "s[e] = 1.0 / (1.0 + exp(z));"),
    "bias_in_weights": ("for (j = 0; j < k; ++j) g[j] = rho * s[sel[j]] / ssum;",
                        "for (j = 0; j < k; ++j) g[j] = rho * u[sel[j]] / ssum;"),
    "select_unbiased": ("u[e] = s[e] + (double)b[e];", "u[e] = s[e];"),
    "tie_to_higher_id": ("if (!taken[e] && (best < 0 || u[e] > u[best])) best = e;",
                         "if (!taken[e] && (best < 0 || u[e] >= u[best])) best = e;"),
    "no_renormalise": ("if (taken[e]) { sel[j++] = e; ssum += s[e]; }", "if (taken[e]) { sel[j++] = e; ssum = 1.0; }"),
    "routed_scale_missing": ("for (j = 0; j < k; ++j) g[j] = rho * s[sel[j]] / ssum;",
                             "for (j = 0; j < k; ++j) g[j] = s[sel[j]] / ssum;"),
    "shared_weighted": ("for (int i = 0; i < d; ++i) o[i] += y[i];", "for (int i = 0; i < d; ++i) o[i] += D->rho * y[i];"),
    "unstable_grouping": ("int pos = offsets[e] + fill[e]++;",
                          "int pos = offsets[e + 1] - 1 - fill[e]++;"),
    "gap_off_by_one": ("*gap = kth - u[nxt];", "*gap = kth - u[nxt] + 1e-9;"),
    "rms_sum_not_mean": ("double r = sqrt(ss / (double)d + eps);", "double r = sqrt(ss + eps);"),
    "bf16_truncates": ("return nearbyint(v / quantum) * quantum;", "return trunc(v / quantum) * quantum;"),
    "logit_drops_last_input": ("for (int i = 0; i < d; ++i) z += xt[i] * (double)we[i];",
                               "for (int i = 0; i < d - 1; ++i) z += xt[i] * (double)we[i];"),
    "mx8_exponent_high": ("e = ex - 1 > -100 ? ex - 1 : -100;", "e = ex > -100 ? ex : -100;"),
    "mx8_clamp_128": ("if (q > 127.0) q = 127.0;", "if (q > 128.0) q = 128.0;"),
    "mx8_ties_away": ("double q = nearbyint(s);        /* the default rounding mode: half to even */",
                      "double q = round(s);"),
    "mx8_truncates": ("double q = nearbyint(s);        /* the default rounding mode: half to even */",
                      "double q = trunc(s);"),
    "idot_x_unquantised": ("for (int i = 0; i < d; ++i) a += w[i] * xq[i];",
                           "for (int i = 0; i < d; ++i) a += w[i] * x[i];"),
    "idot_h_unquantised": ("acc += w[n] * hq[n];", "acc += w[n] * h[n];"),
    "idot_hidden_skips_block": ("for (int b = 0; b < F; b += 32) orc_mx8_block(32, h + b, tau, hq + b, amb + b);",
                                "for (int b = 0; b < F - 32; b += 32) orc_mx8_block(32, h + b, tau, hq + b, amb + b);"),
    "idot_bound_signed": ("bnd += fabs(w[n]) * amb[n];", "bnd += w[n] * amb[n];"),
    "idot_block_tie_one_side": ("block_amb = (r - 1.0 < tau / 64.0) || (2.0 - r < tau / 64.0);",
                                "block_amb = (r - 1.0 < tau / 64.0);"),
    "idot_shared_bound_dropped": ("for (int i = 0; i < d; ++i) { o[i] += y[i]; ob[i] += yb[i]; }",
                                  "for (int i = 0; i < d; ++i) { o[i] += y[i]; }"),
}


@pytest.fixture(scope="module")
def src():
    return O.source()


def test_mutations_apply(src):
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, f"mutation {name}: anchor not found exactly once"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, src, tmp_path):
    old, new = MUTANTS[name]
    path = O.compile_source(src.replace(old, new), os.path.join(str(tmp_path), f"liboracle_{name}.so"))
    L = O.load(path)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(L)
        except (AssertionError, RuntimeError, ValueError, IndexError):
            caught.append(pin.__name__)
            break
    assert caught, f"planted mistake '{name}' passed every pin"
