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
    "fwd_taps_reversed": [("z += w0 * h0;", "z += w0 * h3;"), ("z += w3 * h3;", "z += w3 * h0;")],
    "fwd_bias_dropped": [("double z = b;", "double z = 0.0;")],
    "fwd_silu_sign": [("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));")],
    "bwd_dz_sign": [("(1.0 + zz * (1.0 - sg))", "(1.0 - zz * (1.0 - sg))")],
    "bwd_bias_sign": [("double zz = b;", "double zz = -b;")],
    "bwd_dfinal_positions_reversed": [("d_final[((int64_t)n * 3 + (i - len)) * C + c]",
                                       "d_final[((int64_t)n * 3 + (2 - (i - len))) * C + c]")],
    "bwd_dx_tap_dropped": [("for (int k = 0; k < 4; ++k) {\n                        const int64_t j = i - k;",
                            "for (int k = 0; k < 3; ++k) {\n                        const int64_t j = i - k;")],
    "bwd_dweight_transposed": [("const double t = dz[j] * bf16_to_f64(hist_bits(init3, x, x_stride, s, c, j + k));",
                                "const double t = dz[j] * bf16_to_f64(hist_bits(init3, x, x_stride, s, c, j + 3 - k));")],
    "state_write_off_by_one": [("fin[i] = hist_bits(init3, x, x_stride, s, c, len + i);",
                                "fin[i] = hist_bits(init3, x, x_stride, s, c, len + i - 1);")],
    "state_read_reversed": [("init3[i] = state[((int64_t)q * C + c) * L + i];",
                             "init3[i] = state[((int64_t)q * C + c) * L + (2 - i)];")],
    "empty_sequence_writes_state": [("if (state && len > 0) {", "if (state && len >= 0) {")],
    "bwd_history_ignored": [("if (hist)\n                    for (int i = 0; i < 3; ++i) init3[i] = hist",
                             "if (0)\n                    for (int i = 0; i < 3; ++i) init3[i] = hist")],
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
