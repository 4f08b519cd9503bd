"""The float64 oracle against library routines, closed forms and the pages'
contract (see tests/pins.py for what each pin checks and why)."""
import pytest

import oracle
from tests import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    check(orc)


def test_forward_conv1d_bf16_bias_no_state(orc):
    wl = pins.small_case(seed=21, lengths=(9, 3, 0, 4), n_minus_one=0,
                         b_dtype=__import__("torch").bfloat16)
    wl.conv_state = wl.cache_indices = wl.has_initial_state = None
    pins.check_forward_matches_conv1d(orc, wl)
    pins.check_backward_matches_autograd(orc, wl, with_d_final=False)


def test_backward_without_d_final(orc):
    pins.check_backward_matches_autograd(orc, pins.small_case(seed=4), with_d_final=False)


def test_all_slots_and_slot_zero(orc):
    # slot 0 is a valid slot; every request live
    wl = pins.small_case(seed=8, lengths=(4, 6, 3), n_minus_one=0, slots=3, has_init_p=1.0)
    pins.check_forward_matches_conv1d(orc, wl)
    pins.check_backward_matches_autograd(orc, wl)
