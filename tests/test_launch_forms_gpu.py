"""Every launch form of the same random batch gives the same bits as the
plain ccc_fwd + ccc_bwd call: CCC_OPT_OVERLAP_PROLOGUE, strided rows (x, dy,
out and dx as column slices of wider buffers) and the channel-contiguous
pool (the allocation-free backward has its own file, collected last).  None of them changes what a warp computes
or the order in which it adds, so the comparison is bit for bit."""
import pytest
import torch

import ssm_depthwise_causal_gb300 as ccc
from ssm_depthwise_causal_gb300 import workloads
from tests import gpu_helpers as H
from tests import test_random_batches_gpu as R

pytestmark = pytest.mark.gpu


def _run(wl, d_final, overlap=False, pad=0, layout="history"):
    dev = wl.x.device
    x = H._wide(wl.x, pad) if pad else wl.x
    dy = H._wide(wl.dy, pad) if pad else wl.dy
    st = None
    if wl.conv_state is not None:
        st = wl.conv_state.clone() if layout == "history" else H.channel_contiguous_pool(wl.conv_state)
    h = wl.width - 1
    out = torch.zeros((wl.rows, wl.C + pad), dtype=torch.bfloat16, device=dev)[:, :wl.C]
    hist = torch.zeros((wl.n_seqs, h, wl.C), dtype=torch.bfloat16, device=dev)
    ccc.ccc_fwd(x, wl.weight, wl.bias, st, wl.cu_seqlens, wl.cache_indices, wl.has_initial_state, out, hist,
                activation=wl.activation, overlap=overlap)
    dx = torch.zeros((wl.rows, wl.C + pad), dtype=torch.bfloat16, device=dev)[:, :wl.C]
    dw = torch.zeros((wl.C, wl.width), device=dev)
    db = torch.zeros((wl.C,), device=dev) if wl.bias is not None else None
    di = torch.zeros((wl.n_seqs, h, wl.C), device=dev)
    args = (x, wl.weight, wl.bias, hist, wl.cu_seqlens, wl.cache_indices, wl.has_initial_state, dy, d_final,
            dx, dw, db, di)
    ws = torch.empty(ccc.ccc_workspace_size(wl.rows, wl.n_seqs, wl.C, True), dtype=torch.uint8, device=dev)
    ccc.ccc_bwd(*args, ws, activation=wl.activation, overlap=overlap)
    torch.cuda.synchronize()
    res = {"out": out.contiguous(), "hist": hist, "dx": dx.contiguous(), "dweight": dw, "d_init": di}
    if db is not None:
        res["dbias"] = db
    if st is not None:
        res["state"] = st.contiguous()
    return res


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("seed", range(16))
def test_launch_forms_bitwise(cuda_device, seed):
    lengths, C, rows, width, act, kw = R._case(seed)
    wl = workloads.make_custom(lengths, C, rows=rows, seed=seed, device=cuda_device, width=width,
                               activation=act, **kw)
    g = torch.Generator(device=cuda_device).manual_seed(seed)
    d_final = torch.randn((wl.n_seqs, width - 1, C), generator=g, device=cuda_device)
    base = _run(wl, d_final)
    for name, form in (("overlap", dict(overlap=True)), ("strided rows", dict(pad=24)),
                       ("channel-contiguous pool", dict(layout="channel"))):
        other = _run(wl, d_final, **form)
        for k, v in base.items():
            assert torch.equal(_bits(v), _bits(other[k])), f"{name}: {k}"
