"""The oracle's restatement of the caller-owned metadata constraints
(FlashInfer causal_conv1d_fn, Parameters: offsets from 0, nondecreasing, at
most rows; cache indices -1 or a unique slot in [0, slots); the decode
step's accepted counts in [1, L - W + 2]), pinned by planted violations:
each breaks exactly one rule, so a check that confuses two rules, misses a
boundary or flags a valid value fails here."""
import numpy as np
import pytest

import oracle
from oracle import ACCEPTED, CU_ORDER, CU_RANGE, CU_START, SLOT_DUP, SLOT_RANGE

VALID = dict(rows=12, cu=[0, 3, 3, 9, 12], cache=[4, -1, 0, 7], n_slots=8, acc=[1, 3, 2, 1], max_acc=3)


def bits(rows=None, cu=None, cache="v", n_slots=None, acc="v", max_acc=None):
    v = VALID
    return oracle.check_metadata(v["rows"] if rows is None else rows,
                                 np.asarray(v["cu"] if cu is None else cu, dtype=np.int32),
                                 None if cache is None else np.asarray(v["cache"] if cache == "v" else cache, np.int32),
                                 v["n_slots"] if n_slots is None else n_slots,
                                 None if acc is None else np.asarray(v["acc"] if acc == "v" else acc, np.int32),
                                 v["max_acc"] if max_acc is None else max_acc)


def test_valid_metadata_is_clean():
    assert bits() == 0
    assert bits(cache=None, acc=None) == 0
    assert oracle.check_metadata(0, np.zeros(1, np.int32)) == 0            # N = 0, no rows
    assert bits(cu=[0, 0, 0, 0, 0]) == 0                                   # every sequence empty
    assert bits(cu=[0, 3, 3, 9, 10]) == 0                                  # padding rows after the last offset
    assert bits(cache=[-1, -1, -1, -1]) == 0                               # -1 may repeat
    assert bits(cache=[7, 0, 1, 2]) == 0                                   # both ends of [0, slots)
    assert bits(acc=[1, 3, 3, 1]) == 0                                     # both ends of [1, max]


@pytest.mark.parametrize("case,expected", [
    (dict(cu=[1, 3, 3, 9, 12]), CU_START),
    (dict(cu=[0, 3, 2, 9, 12]), CU_ORDER),
    (dict(cu=[0, 3, 3, 9, 13]), CU_RANGE),
    (dict(rows=11), CU_RANGE),
    (dict(cu=[0, -1, 3, 9, 12]), CU_ORDER | CU_RANGE),
    (dict(cache=[4, -1, 0, 8]), SLOT_RANGE),
    (dict(cache=[4, -2, 0, 7]), SLOT_RANGE),
    (dict(n_slots=7), SLOT_RANGE),
    (dict(cache=[4, -1, 4, 7]), SLOT_DUP),
    (dict(cache=[0, 0, -1, 0]), SLOT_DUP),
    (dict(acc=[0, 3, 2, 1]), ACCEPTED),
    (dict(acc=[1, 4, 2, 1]), ACCEPTED),
    (dict(max_acc=2), ACCEPTED),
    (dict(cu=[2, 1, 3, 9, 40], cache=[9, 9, 9, 9], acc=[5, 1, 1, 1]),
     CU_START | CU_ORDER | CU_RANGE | SLOT_RANGE | ACCEPTED),
])
def test_each_violation_sets_its_bit(case, expected):
    assert bits(**case) == expected


def test_unchecked_arrays_are_ignored():
    assert bits(cache=None, acc=[0, 9, 9, 9]) == ACCEPTED
    assert bits(cache=[9, 9, 9, 9], acc=None) == SLOT_RANGE
