"""Full-size exact checks of the forward and backward work split.

With the taps one-hot at k, no bias and no activation, the method reduces
to data movement (FlashInfer causal_conv1d_fn, Parameters: bias first, then
the FMAs, tap W-1 on the current token; the backward's dH[i] = sum over k of
w_k dz[i-k]): token j of a sequence outputs history value h[j + k] (h = the
W-1 initial values, then the sequence's rows), and dx of row j is dy of row
j + W-1-k when that row is in the sequence, else 0.  So every output row
must equal an input row bit for bit -- a check of every run boundary, walk
and sequence edge of the kernels' split on the full packed and serving
workloads, where the oracle can only sample.  Expected rows are plain
slices of the inputs (no arithmetic)."""
import numpy as np
import pytest
import torch

import ssm_depthwise_causal_gb300 as ccc
from ssm_depthwise_causal_gb300 import workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _eq(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.fixture(scope="module")
def packed(cuda_device):
    return workloads.packed(device=cuda_device)


@pytest.mark.parametrize("W", [4, 3, 2])
def test_packed_fwd_bwd_one_hot(cuda_device, packed, W):
    dev = cuda_device
    wl = packed
    C, N, rows = wl.C, wl.n_seqs, wl.rows
    Hh = W - 1
    cu = wl.cu_seqlens.cpu().numpy()
    T = int(cu[-1])
    hist = torch.empty((N, Hh, C), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((C, W), device=dev)
    ws = torch.empty(ccc.ccc_workspace_size(rows, N, C, True), dtype=torch.uint8, device=dev)
    zero = torch.zeros((1, C), dtype=torch.bfloat16, device=dev)
    for k in range(W):
        w = torch.zeros((C, W), dtype=torch.float32, device=dev)
        w[:, k] = 1.0
        out = H.fill_sentinel(torch.empty_like(wl.x))
        dx = H.fill_sentinel(torch.empty_like(wl.x))
        ccc.ccc_fwd(wl.x, w, None, None, wl.cu_seqlens, None, None, out, hist, activation=None)
        ccc.ccc_bwd(wl.x, w, None, hist, wl.cu_seqlens, None, None, wl.dy, None, dx, dw, None, None, ws,
                    activation=None)
        torch.cuda.synchronize()
        sh = Hh - k  # out row j = x row j - sh; dx row j = dy row j + sh
        exp_out = torch.zeros_like(wl.x[:T])
        exp_dx = torch.zeros_like(wl.x[:T])
        for n in range(N):
            s, e = int(cu[n]), int(cu[n + 1])
            if e - s > sh:
                exp_out[s + sh:e] = wl.x[s:e - sh]
                exp_dx[s:e - sh] = wl.dy[s + sh:e]
        assert _eq(out[:T], exp_out), f"k={k}: out is not x shifted by {sh} rows within each sequence"
        assert _eq(dx[:T], exp_dx), f"k={k}: dx is not dy shifted by {sh} rows within each sequence"
        assert np.all(H.bits(out[T:]) == H.SENTINEL), "padding rows of out were written"
        assert np.all(H.bits(dx[T:]) == H.SENTINEL), "padding rows of dx were written"
        ne = torch.from_numpy(np.diff(cu) > 0).to(dev)
        assert torch.all(hist[ne].view(torch.int16) == 0), "no pool: the saved history is zeros"


def test_serving_fwd_one_hot_with_state(cuda_device):
    """The serving batch (a pool, has_initial_state, -1 requests): the first
    W-1-k outputs of a sequence come from its slot's positions (or zeros),
    then x shifted; -1 requests output zeros; the pool ends holding each live
    sequence's last three history values."""
    dev = cuda_device
    wl = workloads.serving(device=dev)
    C, N, W = wl.C, wl.n_seqs, 4
    Hh = W - 1
    cu = wl.cu_seqlens.cpu().numpy()
    cache = wl.cache_indices.cpu().numpy()
    hi = wl.has_initial_state.cpu().numpy()
    for k in (0, Hh):
        w = torch.zeros((C, W), dtype=torch.float32, device=dev)
        w[:, k] = 1.0
        pool = wl.conv_state.clone()
        out = H.fill_sentinel(torch.empty_like(wl.x))
        ccc.ccc_fwd(wl.x, w, None, pool, wl.cu_seqlens, wl.cache_indices, wl.has_initial_state, out,
                    activation=None)
        torch.cuda.synchronize()
        sh = Hh - k
        for n in range(N):
            s, e = int(cu[n]), int(cu[n + 1])
            if e == s:
                continue
            q = int(cache[n])
            if q == -1:
                assert torch.all(out[s:e].view(torch.int16) == 0), f"seq {n}: -1 output must be +0"
                continue
            init = wl.conv_state[q, :, :Hh].t() if hi[n] else torch.zeros((Hh, C), dtype=torch.bfloat16,
                                                                          device=dev)
            hseq = torch.cat([init, wl.x[s:e]], 0)  # history values of the sequence
            assert _eq(out[s:e], hseq[k:k + (e - s)]), f"k={k} seq {n}"
            assert _eq(pool[q, :, :Hh].t().contiguous(), hseq[-Hh:].contiguous()), f"k={k} seq {n}: state"
