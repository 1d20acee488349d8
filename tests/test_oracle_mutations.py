"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each one.

Every mutation keeps all memory accesses in bounds; it only changes arithmetic
or indexing inside the arrays' extents.
"""
import os

import pytest

import oracle
import pins

MUTATIONS = {
    "linear_drops_bias": ("s += bias[n];", ";"),
    "linear_transposed_w": ("double t = x[m * K + k] * w[n * K + k];",
                            "double t = x[m * K + k] * w[k * N + n];"),
    "matmul_transposed_b": ("double t = a[m * K + k] * b[k * N + n];\n                s += t;\n                r += fabs(t);\n            }\n            y[m * N + n] = s;",
                            "double t = a[m * K + k] * b[n * K + k];\n                s += t;\n                r += fabs(t);\n            }\n            y[m * N + n] = s;"),
    "addmm_sign": ("beta * cv + alpha * s", "beta * cv - alpha * s"),
    "addmm_alpha_beta_swapped": ("beta * cv + alpha * s", "alpha * cv + beta * s"),
    "sdpa_gqa_map": ("const int64_t hk = h / group;", "const int64_t hk = h % Hkv;"),
    "sdpa_causal_off_by_one": ("else if (causal) visible = j <= q_offset + i;",
                               "else if (causal) visible = j <= q_offset + i + 1;"),
    "sdpa_sink_not_in_denominator": ("double den = sinks ? exp(sinks[h] - mx) : 0.0;",
                                     "double den = 0.0;"),
    "sdpa_mask_ignored": ("if (mask) visible = mask[((b * H + h) * Lq + i) * Lkv + j] != 0;",
                          "if (mask) visible = 1;"),
    "sdpa_mask_transposed_heads": ("if (mask) visible = mask[((b * H + h) * Lq + i) * Lkv + j] != 0;",
                                   "if (mask) visible = mask[((b * H + (H - 1 - h)) * Lq + i) * Lkv + j] != 0;"),
    "sdpa_exp_sign": ("s[j] = exp(s[j] - mx);", "s[j] = exp(mx - s[j]);"),
    "sdpa_no_scale": ("s[j] = scale * t;", "s[j] = t;"),
    "sdpa_normaliser": ("r += p * fabs(vb[j * D + d]);", "r += fabs(vb[j * D + d]);"),
    "qlinear_field_order": ("const uint32_t q = (word >> (bits * (k % f))) & fmask;",
                            "const uint32_t q = (word >> (bits * (f - 1 - k % f))) & fmask;"),
    "qlinear_group_index": ("wrow[k] = scales[n * ldsb + k / gs] * (double)q",
                            "wrow[k] = scales[n * ldsb + (k % gs) % ldsb] * (double)q"),
    "qlinear_scale_bias_swapped": (
        "scales[n * ldsb + k / gs] * (double)q + biases[n * ldsb + k / gs]",
        "biases[n * ldsb + k / gs] * (double)q + scales[n * ldsb + k / gs]"),
    "qlinear_signed_fields": ("* (double)q + biases", "* ((double)q - (double)(fmask >> 1)) + biases"),
    "qlinear_drops_bias": ("acc += bias[n];", ";"),
    "rmsnorm_sum_not_mean": ("sqrt(ss / (double)N + eps)", "sqrt(ss + eps)"),
    "rope_sign": ("yi[i] = xi[i] * c - xi[i + half] * s;", "yi[i] = xi[i] * c + xi[i + half] * s;"),
    "rope_pairing": ("double th = (double)pos[t] * inv_freq;", "double th = (double)pos[t] * inv_freq * 2.0;"),
    "swiglu_exp_sign": ("g / (1.0 + exp(-g)) * u", "g / (1.0 + exp(g)) * u"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, "mutation anchor must occur once: %s" % name
    path = tmp_path / ("oracle_%s.c" % name)
    path.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(path), str(tmp_path / ("lib_%s.so" % name)))
    O = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(O)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "mutation %s was not caught by any pin" % name
