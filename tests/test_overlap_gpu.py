"""CCC_OPT_OVERLAP_PROLOGUE (ccc_fwd_ex, ccc_bwd_ex, ccc_update_ex): the
kernels launched as programmatic dependents of the previous kernel give the
same bits as ordinary launches -- eagerly, and as back-to-back training or
decode steps captured in one CUDA graph (each kernel then a dependent of the
one before)."""
import pytest
import torch

import ssm_depthwise_causal_gb300 as ccc
from ssm_depthwise_causal_gb300 import workloads

pytestmark = pytest.mark.gpu


def _buffers(wl):
    """Output buffers, zero-filled (rows the method leaves alone -- padding,
    the saved history of empty sequences -- then compare equal too)."""
    dev = wl.x.device
    return dict(out=torch.zeros_like(wl.x), dx=torch.zeros_like(wl.x),
                hist=torch.zeros((wl.n_seqs, wl.width - 1, wl.C), dtype=torch.bfloat16, device=dev),
                dw=torch.empty((wl.C, wl.width), device=dev),
                db=None if wl.bias is None else torch.empty((wl.C,), device=dev),
                di=torch.empty((wl.n_seqs, wl.width - 1, wl.C), device=dev),
                ws=torch.empty(ccc.ccc_workspace_size(wl.rows, wl.n_seqs, wl.C, True), dtype=torch.uint8,
                               device=dev),
                state=None if wl.conv_state is None else wl.conv_state.clone())


def _step(wl, b, overlap, stream=None):
    ccc.ccc_fwd(wl.x, wl.weight, wl.bias, b["state"], wl.cu_seqlens, wl.cache_indices, wl.has_initial_state,
                b["out"], b["hist"], stream=stream, activation=wl.activation, overlap=overlap)
    ccc.ccc_bwd(wl.x, wl.weight, wl.bias, b["hist"], wl.cu_seqlens, wl.cache_indices, wl.has_initial_state,
                wl.dy, None, b["dx"], b["dw"], b["db"], b["di"], b["ws"], stream=stream,
                activation=wl.activation, overlap=overlap)


def _same(a, b):
    assert torch.equal(a["out"].view(torch.int16), b["out"].view(torch.int16))
    assert torch.equal(a["dx"].view(torch.int16), b["dx"].view(torch.int16))
    assert torch.equal(a["hist"].view(torch.int16), b["hist"].view(torch.int16))
    assert torch.equal(a["dw"].view(torch.int32), b["dw"].view(torch.int32))
    assert torch.equal(a["di"].view(torch.int32), b["di"].view(torch.int32))
    if a["db"] is not None:
        assert torch.equal(a["db"].view(torch.int32), b["db"].view(torch.int32))
    if a["state"] is not None:
        assert torch.equal(a["state"].view(torch.int16), b["state"].view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "packed_small"])
def test_overlap_eager_equals_plain(cuda_device, name):
    wl = workloads.WORKLOADS[name](device=cuda_device)
    plain, over = _buffers(wl), _buffers(wl)
    _step(wl, plain, False)
    _step(wl, over, True)
    torch.cuda.synchronize()
    _same(plain, over)


def test_overlap_steps_in_one_graph(cuda_device):
    """Five forward + backward steps in one CUDA graph with the option on (the
    forward of step k+1 a dependent of step k's reduce), replayed: every
    step leaves the same bits as one plain eager step (the workload has no
    pool, so the steps are identical)."""
    wl = workloads.make_custom(workloads.packed_lengths(seed=5, N=60, rows=8192), 1024, rows=8192, seed=5,
                               device=cuda_device, with_state=False)
    plain = _buffers(wl)
    _step(wl, plain, False)
    torch.cuda.synchronize()
    over = _buffers(wl)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _step(wl, over, True, stream=s)  # outside the capture first
    torch.cuda.synchronize()
    for t in ("out", "dx", "dw"):
        over[t].zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(5):
            _step(wl, over, True, stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    _same(plain, over)


@pytest.mark.parametrize("name", ["decode", "spec_decode"])
def test_overlap_update_steps_equal_plain(cuda_device, name):
    """ccc_update_ex with the option: three decode steps eagerly, then three
    more captured in one CUDA graph (each a dependent of the step before, on
    the pool it wrote), leave the same outputs and pool bits as six plain
    steps."""
    wl = workloads.WORKLOADS[name](device=cuda_device)
    acc = wl.num_accepted if wl.lengths.max() > 1 else None

    def run(pool, out, overlap, stream=None):
        ccc.ccc_update(wl.x, wl.weight, wl.bias, pool, wl.cu_seqlens, wl.cache_indices, acc, out,
                       stream=stream, overlap=overlap)

    pool_p, out_p = wl.conv_state.clone(), torch.zeros_like(wl.x)
    pool_o, out_o = wl.conv_state.clone(), torch.zeros_like(wl.x)
    for _ in range(3):
        run(pool_p, out_p, False)
        run(pool_o, out_o, True)
    torch.cuda.synchronize()
    assert torch.equal(out_p.view(torch.int16), out_o.view(torch.int16))
    assert torch.equal(pool_p.view(torch.int16), pool_o.view(torch.int16))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            run(pool_o, out_o, True, stream=s)
    g.replay()
    for _ in range(3):
        run(pool_p, out_p, False)
    torch.cuda.synchronize()
    assert torch.equal(out_p.view(torch.int16), out_o.view(torch.int16))
    assert torch.equal(pool_p.view(torch.int16), pool_o.view(torch.int16))
