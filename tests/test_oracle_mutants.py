"""Planted mistakes in the oracle must each fail at least one pin.

Each mutant is the oracle's C source with one plausible slip (a dropped term,
a wrong sign, a wrong or transposed index), compiled into a temporary
directory on the CPU and run through every check of tests/pins.py.  This is
what shows that the pins tie the oracle down, rather than restating it.
"""
import os

import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ccc_oracle.c")

MUTANTS = {
    "fwd_taps_reversed": [("z += wk[k] * bf16_to_f64(hist_bits(init, W - 1, x, x_stride, s, c, j + k));",
                           "z += wk[k] * bf16_to_f64(hist_bits(init, W - 1, x, x_stride, s, c, j + W - 1 - k));")],
    "fwd_tap_dropped": [("for (int k = 0; k < W; ++k) z += wk[k] * bf16_to_f64(hist_bits(",
                         "for (int k = 0; k < W - 1; ++k) z += wk[k] * bf16_to_f64(hist_bits(")],
    "fwd_bias_dropped": [("double z = b;\n    for (int k = 0; k < W; ++k) z += wk[k] * bf16_to_f64(hist_bits(",
                          "double z = 0.0;\n    for (int k = 0; k < W; ++k) z += wk[k] * bf16_to_f64(hist_bits(")],
    "fwd_silu_sign": [("return act ? z / (1.0 + exp(-z)) : z;", "return act ? z / (1.0 + exp(z)) : z;")],
    "activation_none_ignored": [("return act ? z / (1.0 + exp(-z)) : z;", "return z / (1.0 + exp(-z));")],
    "bwd_dz_sign": [("return g * sg * (1.0 + z * (1.0 - sg));", "return g * sg * (1.0 - z * (1.0 - sg));")],
    "bwd_grad_ignores_activation": [("if (!act) return g;", "if (0) return g;")],
    "bwd_bias_sign": [("const double zz = pre_activation(b,", "const double zz = pre_activation(-b,")],
    "bwd_dfinal_positions_reversed": [("d_final[((int64_t)n * H + (i - len)) * C + c]",
                                       "d_final[((int64_t)n * H + (H - 1 - (i - len))) * C + c]")],
    "bwd_dx_tap_dropped": [("for (int k = 0; k < W; ++k) {\n                        const int64_t j = i - k;",
                            "for (int k = 0; k < W - 1; ++k) {\n                        const int64_t j = i - k;")],
    "bwd_dweight_transposed": [("const double t = dz[j] * bf16_to_f64(hist_bits(init, H, x, x_stride, s, c, j + k));",
                                "const double t = dz[j] * bf16_to_f64(hist_bits(init, H, x, x_stride, s, c, j + H - k));")],
    "state_write_off_by_one": [("fin[i] = hist_bits(init, H, x, x_stride, s, c, len + i);",
                                "fin[i] = hist_bits(init, H, x, x_stride, s, c, len + i - 1);")],
    "state_read_reversed": [("init[i] = state[((int64_t)q * C + c) * L + i];",
                             "init[i] = state[((int64_t)q * C + c) * L + (H - 1 - i)];")],
    "empty_sequence_writes_state": [("if (state && len > 0) {", "if (state && len >= 0) {")],
    "bwd_history_ignored": [("if (hist)\n                    for (int i = 0; i < H; ++i) init[i] = hist",
                             "if (0)\n                    for (int i = 0; i < H; ++i) init[i] = hist")],
    "update_read_ignores_accepted": [("h[i] = slot[a - 1 + i];", "h[i] = slot[i];")],
    "update_write_unshifted": [("slot[p] = h[p + 1];", "slot[p] = h[p];")],
    "update_write_short": [("p < len + H - 1 && p < L", "p < len + H - 2 && p < L")],
    "update_empty_writes_state": [("if (len == 0) continue;", "if (len < 0) continue;")],
    "update_minus_one_negative_zero": [("out[(s + j) * out_stride + c] = 0.0;\n                    continue;",
                                        "out[(s + j) * out_stride + c] = -0.0;\n                    continue;")],
    "minus_one_needs_a_pool": [("const int32_t q = cache ? cache[n] : 0;\n            if (cache && q == -1) {",
                                "const int32_t q = state ? cache[n] : 0;\n            if (state && q == -1) {")],
    "bwd_dfinal_dropped": [("if (i >= len && d_final) acc = d_final", "if (0) acc = d_final")],
    "update_taps_reversed": [("for (int k = 0; k < W; ++k) z += wk[k] * bf16_to_f64(h[j + k]);",
                              "for (int k = 0; k < W; ++k) z += wk[k] * bf16_to_f64(h[j + W - 1 - k]);")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / f"{name}.c"
    path.write_text(src)
    so = oracle.compile_oracle(str(path), str(tmp_path / f"lib{name}.so"))
    mutant = oracle.Oracle(so)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(mutant)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
