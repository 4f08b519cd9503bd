"""The worked example (tests/golden/make_golden.py) through the CUDA path,
checked against closed forms directly rather than against the oracle.

Inputs: C = 8, one sequence of 6 tokens with x[t, 0] = (t + 1) / 8 and zeros
elsewhere, taps (1/2, -1/4, 1/8, 1) on every channel (tap 3 on the current
token: FlashInfer causal_conv1d_fn, weight), bias 1/16, and slot 1 of a
two-slot pool holding (1, -1, 1/2, 7) on channel 0 as the initial state
(causal_conv1d_fn, conv_state / has_initial_state).  Every input is a dyadic
rational, so each pre-activation is exact in FP32: token 0 of channel 0 has
z = 1 exactly and every token of the zero channels has z = 1/16.  The BF16
outputs are the round-to-nearest-even of SiLU(z) (neither value lies near a
rounding midpoint, so the approximate exponential cannot flip them), the
state is the last three raw inputs with position 3 untouched, and the
backward with dy = 1 gives dbias = sum_j SiLU'(z_j) and dweight[k] =
sum_j SiLU'(z_j) h[j + k].
"""
import math

import numpy as np
import pytest
import torch

import ssm_depthwise_causal_gb300 as ccc

pytestmark = pytest.mark.gpu


def _silu(z):
    return z / (1.0 + math.exp(-z))


def _dsilu(z):
    s = 1.0 / (1.0 + math.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def _bf16(v):
    return torch.tensor([v], dtype=torch.float64).to(torch.bfloat16).item()


def test_worked_example_closed_forms(cuda_device):
    dev = cuda_device
    C, L = 8, 6
    x = torch.zeros((L, C), dtype=torch.bfloat16, device=dev)
    x[:, 0] = (torch.arange(L, device=dev, dtype=torch.float32) + 1) / 8
    w = torch.tensor([0.5, -0.25, 0.125, 1.0], device=dev).repeat(C, 1).contiguous()
    b = torch.full((C,), 1.0 / 16, device=dev)
    pool = torch.zeros((2, C, 4), dtype=torch.bfloat16, device=dev)
    pool[1, 0] = torch.tensor([1.0, -1.0, 0.5, 7.0])
    cu = torch.tensor([0, L], dtype=torch.int32, device=dev)
    cache = torch.tensor([1], dtype=torch.int32, device=dev)
    has_init = torch.tensor([1], dtype=torch.uint8, device=dev)
    out = torch.empty_like(x)
    hist = torch.empty((1, 3, C), dtype=torch.bfloat16, device=dev)
    ccc.ccc_fwd(x, w, b, pool, cu, cache, has_init, out, hist)
    dy = torch.ones_like(x)
    dx = torch.empty_like(x)
    dw = torch.empty((C, 4), device=dev)
    db = torch.empty((C,), device=dev)
    di = torch.empty((1, 3, C), device=dev)
    ws = torch.empty(ccc.ccc_workspace_size(L, 1, C, True), dtype=torch.uint8, device=dev)
    ccc.ccc_bwd(x, w, b, hist, cu, cache, has_init, dy, None, dx, dw, db, di, ws)
    torch.cuda.synchronize()

    hist0 = [1.0, -1.0, 0.5] + [(t + 1) / 8.0 for t in range(L)]
    taps = [0.5, -0.25, 0.125, 1.0]
    zs = [1.0 / 16 + sum(taps[k] * hist0[j + k] for k in range(4)) for j in range(L)]
    assert zs[0] == 1.0
    # forward: BF16 outputs bit for bit
    for j in range(L):
        assert out[j, 0].item() == _bf16(_silu(zs[j])), f"token {j}"
    assert all(v == _bf16(_silu(1.0 / 16)) for v in out[:, 1:].flatten().tolist())
    # state: the last three raw inputs at positions 0..2, position 3 and slot 0 untouched
    assert pool[1, 0].tolist() == [0.5, 0.625, 0.75, 7.0]
    assert pool[1, 1:, :3].abs().sum().item() == 0.0 and pool[0].abs().sum().item() == 0.0
    # backward with dy = 1
    dz = [_dsilu(z) for z in zs]
    assert math.isclose(db[0].item(), sum(dz), rel_tol=1e-5)
    for k in range(4):
        assert math.isclose(dw[0, k].item(), sum(dz[j] * hist0[j + k] for j in range(L)), rel_tol=1e-5,
                            abs_tol=1e-6), f"dweight[0][{k}]"
    dz1 = _dsilu(1.0 / 16)
    assert math.isclose(db[1].item(), L * dz1, rel_tol=1e-5)
    # d_init_state: history index i < 3 feeds token j = i - k through tap k
    for i in range(3):
        want = sum(taps[k] * dz[i - k] for k in range(4) if 0 <= i - k < L)
        assert math.isclose(di[0, i, 0].item(), want, rel_tol=1e-5, abs_tol=1e-6), f"d_init[{i}]"
