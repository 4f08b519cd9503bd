"""The autograd wrapper and the checkpoint recompute (GPU).

* recompute_fwd re-runs a forward from the history it saved and must give
  the original output bit for bit, although the pool was overwritten in place
  meanwhile (cake_causal_conv1d_kcp, recompute_handle: y and the gradients of
  a recompute are bitwise those without one).
* causal_conv1d (CausalConv1dFn) gives the same gradients as ccc_bwd and, on
  CPU-checked values, as the float64 oracle.
"""
import numpy as np
import pytest
import torch

import ssm_depthwise_causal_gb300 as ccc
from ssm_depthwise_causal_gb300 import workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def test_recompute_is_bitwise(cuda_device):
    wl = workloads.make_custom((70, 0, 5, 130, 2), 264, rows=215, seed=6, device=cuda_device,
                               n_minus_one=1, has_init_p=0.7)
    pool = wl.conv_state.clone()
    hist = torch.empty((wl.n_seqs, 3, wl.C), dtype=torch.bfloat16, device=cuda_device)
    out1 = H.fill_sentinel(torch.empty_like(wl.x))
    ccc.causal_conv1d_fn(wl.x, wl.weight, pool, wl.cu_seqlens, wl.cache_indices,
                         wl.has_initial_state, bias=wl.bias, out=out1, saved_hist=hist)
    hist_before = hist.clone()
    out2 = H.fill_sentinel(torch.empty_like(wl.x))
    ccc.recompute_fwd(wl.x, wl.weight, hist, wl.cu_seqlens, wl.cache_indices, bias=wl.bias, out=out2)
    torch.cuda.synchronize()
    T = wl.valid_tokens
    assert torch.equal(out1[:T].view(torch.int16), out2[:T].view(torch.int16))
    assert torch.equal(hist.view(torch.int16), hist_before.view(torch.int16)), "saved history modified"


def test_autograd_matches_ccc_bwd_and_oracle(cuda_device):
    wl = workloads.make_custom((90, 33, 0, 140), 128, rows=270, seed=8, device=cuda_device,
                               with_state=False)
    x = wl.x.clone().requires_grad_(True)
    w = wl.weight.clone().requires_grad_(True)
    b = wl.bias.clone().requires_grad_(True)
    y = ccc.causal_conv1d(x, w, b, wl.cu_seqlens)
    y.backward(wl.dy)
    torch.cuda.synchronize()
    # same as a direct ccc_bwd
    res = H.run_gpu(wl)
    T = wl.valid_tokens
    assert torch.equal(x.grad[:T].view(torch.int16), res.dx[:T].view(torch.int16))
    assert torch.all(x.grad[T:] == 0)
    assert torch.equal(w.grad.view(torch.int32), res.dweight.view(torch.int32))
    assert torch.equal(b.grad.view(torch.int32), res.dbias.view(torch.int32))
    # and the oracle
    sub = H.subset(wl, list(range(wl.C)))
    ref = H.run_oracle(sub)
    H.assert_bf16_close(H.bits(y.detach()[:T]), ref["out"][:T], "out")
    H.assert_bf16_close(H.bits(x.grad[:T]), ref["dx"][:T], "dx")
    H.assert_reduction_close(w.grad.cpu().numpy(), ref["dweight"], ref["abs_dweight"], "dweight")
