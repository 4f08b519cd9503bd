"""Randomized packed batches through the C ABI against the float64 oracle.

Each case draws its own mix -- the number of sequences (1 to 120, so both
depths of the kernels' search for a run's first sequence), lengths from
empty through a few rows to hundreds (so run boundaries land in every
position of a sequence, including its first W-1 rows), channels that leave a
partial slab, width, activation, dtypes, -1 requests, flags and padding rows
-- and compares forward, state, saved history and backward on every channel
with the tolerances of tests/gpu_helpers.py.
"""
import numpy as np
import pytest
import torch

from ssm_depthwise_causal_gb300 import workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    N = int(rng.integers(1, 121))
    kind = rng.integers(0, 3)
    if kind == 0:
        lengths = rng.integers(0, 6, N)
    elif kind == 1:
        lengths = rng.integers(0, 300, N)
    else:
        lengths = np.where(rng.random(N) < 0.25, 0, rng.integers(1, 90, N))
    C = int(rng.integers(1, 76)) * 8
    width = int(rng.integers(2, 5))
    act = "silu" if rng.random() < 0.6 else None
    kw = dict(
        n_minus_one=int(rng.integers(0, max(1, N // 5) + 1)),
        has_init_p=float(rng.random()),
        w_dtype=torch.bfloat16 if rng.random() < 0.5 else torch.float32,
        b_dtype=[None, torch.float32, torch.bfloat16][int(rng.integers(0, 3))],
        state_len=width - 1 + int(rng.integers(0, 3)),
    )
    rows = int(lengths.sum()) + int(rng.integers(0, 9))
    return lengths, C, rows, width, act, kw


@pytest.mark.parametrize("seed", range(48))
def test_random_batch(cuda_device, seed):
    lengths, C, rows, width, act, kw = _case(seed)
    wl = workloads.make_custom(lengths, C, rows=rows, seed=seed, device=cuda_device, width=width,
                               activation=act, **kw)
    g = torch.Generator(device=cuda_device).manual_seed(seed)
    d_final = torch.randn((wl.n_seqs, width - 1, C), generator=g, device=cuda_device)
    res = H.run_gpu(wl, d_final=d_final)
    sub = H.subset(wl, list(range(C)))
    ref = H.run_oracle(sub, d_final=d_final.double().cpu())
    H.compare(sub, ref, H.gpu_numpy(res), chans=list(range(C)))


@pytest.mark.parametrize("seed", range(8))
def test_random_batch_wide(cuda_device, seed):
    """Wider channel counts (many slabs, a ragged last one) on short batches:
    the backward's runs are then capped by the width (1216 / slabs), not by
    the rows, and its CTAs switch between one and eight warps."""
    rng = np.random.default_rng(5000 + seed)
    N = int(rng.integers(1, 40))
    lengths = np.where(rng.random(N) < 0.15, 0, rng.integers(1, 400, N))
    C = int(rng.integers(120, 520)) * 8
    width = int(rng.integers(2, 5))
    act = "silu" if rng.random() < 0.7 else None
    wl = workloads.make_custom(lengths, C, rows=int(lengths.sum()) + int(rng.integers(0, 9)), seed=seed,
                               device=cuda_device, width=width, activation=act,
                               n_minus_one=int(rng.integers(0, max(1, N // 5) + 1)),
                               has_init_p=float(rng.random()),
                               w_dtype=torch.bfloat16 if rng.random() < 0.5 else torch.float32,
                               b_dtype=[None, torch.float32, torch.bfloat16][int(rng.integers(0, 3))])
    g = torch.Generator(device=cuda_device).manual_seed(seed)
    d_final = torch.randn((wl.n_seqs, width - 1, C), generator=g, device=cuda_device)
    res = H.run_gpu(wl, d_final=d_final)
    sub = H.subset(wl, list(range(C)))
    ref = H.run_oracle(sub, d_final=d_final.double().cpu())
    H.compare(sub, ref, H.gpu_numpy(res), chans=list(range(C)))
