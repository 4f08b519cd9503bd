"""ccc_check on the GPU against the oracle's restatement of the caller-owned
metadata constraints (FlashInfer causal_conv1d_fn, Parameters and Notes):
the status bits must be identical, for the workloads' own metadata (all
valid) and for random metadata with planted violations, including slot
bitmaps that span many words and duplicates that meet in different CTAs."""
import numpy as np
import pytest
import torch

import oracle
import ssm_depthwise_causal_gb300 as ccc
from ssm_depthwise_causal_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "decode", "spec_decode", "packed_small", "dense"])
def test_workload_metadata_is_valid(cuda_device, name):
    wl = workloads.WORKLOADS[name](device=cuda_device)
    n_slots = 0 if wl.conv_state is None else wl.conv_state.shape[0]
    max_acc = 0
    if wl.num_accepted is not None:
        max_acc = wl.conv_state.shape[2] - wl.width + 2
    got = ccc.check_metadata(wl.rows, wl.cu_seqlens, wl.cache_indices, n_slots, wl.num_accepted, max_acc)
    assert got == 0


def _random_case(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(0, 3000))
    rows = int(rng.integers(0, 50000))
    cut = np.sort(rng.integers(0, rows + 1, N))
    cu = np.concatenate([[0], cut]).astype(np.int64)
    n_slots = int(rng.integers(1, 100000))
    cache = rng.permutation(max(n_slots, N))[:N]
    cache = np.where(cache < n_slots, cache, -1)
    cache[rng.random(N) < 0.1] = -1
    max_acc = int(rng.integers(1, 8))
    acc = rng.integers(1, max_acc + 1, N)
    kind = seed % 7
    if N > 0:
        i = int(rng.integers(0, N + 1))
        j = int(rng.integers(0, N))
        if kind == 1:
            cu[0] = int(rng.integers(1, 5))
        elif kind == 2 and N >= 2:
            k = int(rng.integers(1, N + 1))
            cu[k] = cu[k - 1] - int(rng.integers(1, 4))
        elif kind == 3:
            cu[i] = rows + int(rng.integers(1, 5)) if rng.random() < 0.5 else -int(rng.integers(1, 5))
        elif kind == 4:
            cache[j] = n_slots + int(rng.integers(0, 3)) if rng.random() < 0.5 else -int(rng.integers(2, 9))
        elif kind == 5 and N >= 2:
            a, b = rng.choice(N, 2, replace=False)   # far apart: different CTAs when N > 256
            cache[a] = cache[b] = int(rng.integers(0, n_slots))
        elif kind == 6:
            acc[j] = 0 if rng.random() < 0.5 else max_acc + 1
    return rows, cu.astype(np.int32), cache.astype(np.int32), n_slots, acc.astype(np.int32), max_acc


@pytest.mark.parametrize("seed", range(40))
def test_random_metadata_matches_oracle(cuda_device, seed):
    rows, cu, cache, n_slots, acc, max_acc = _random_case(seed)
    expected = oracle.check_metadata(rows, cu, cache, n_slots, acc, max_acc)
    d = lambda a: torch.from_numpy(a).to(cuda_device)  # noqa: E731
    got = ccc.check_metadata(rows, d(cu), d(cache), n_slots, d(acc), max_acc)
    assert got == expected, (seed, got, expected)
    # without the optional arrays only the offsets are checked
    assert ccc.check_metadata(rows, d(cu)) == oracle.check_metadata(rows, cu)


def test_status_array_is_cleared_every_call(cuda_device):
    d = lambda a: torch.tensor(a, dtype=torch.int32, device=cuda_device)  # noqa: E731
    st = torch.full((ccc._lib.lib().ccc_check_status_words(64),), -1, dtype=torch.int32, device=cuda_device)
    ccc.ccc_check(10, d([0, 5, 10]), d([3, 3]), 64, status=st)
    assert int(st[0]) == ccc.CHECK_SLOT_DUP
    ccc.ccc_check(10, d([0, 5, 10]), d([3, 4]), 64, status=st)
    assert int(st[0]) == 0
