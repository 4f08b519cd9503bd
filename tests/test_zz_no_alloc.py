"""ccc_bwd_noalloc: the backward for callers that cannot allocate device
memory (it runs on a fixed scratch array inside the library instead of a
caller-supplied workspace).

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.  Each case makes two calls in a row
-- the scratch array keeps the previous call's contents -- and compares them
with the ordinary ccc_bwd on the same inputs.  Both run the same kernels over
the same grid of partial sums, so every output must match bit for bit (a
leftover of an earlier call in the shared array would show up here).
"""
import numpy as np
import pytest
import torch

import ssm_depthwise_causal_gb300 as ccc
from ssm_depthwise_causal_gb300 import _lib, workloads
from tests import gpu_helpers as H


def _forward(wl):
    out = torch.empty_like(wl.x)
    hist = torch.empty((wl.n_seqs, 3, wl.C), dtype=torch.bfloat16, device=wl.x.device)
    ccc.causal_conv1d_fn(wl.x, wl.weight, wl.conv_state, wl.cu_seqlens, wl.cache_indices,
                         wl.has_initial_state, bias=wl.bias, out=out, saved_hist=hist)
    return hist


def _grads(wl, hist, noalloc):
    dev = wl.x.device
    dx = H.fill_sentinel(torch.empty_like(wl.x))
    dw = torch.full((wl.C, 4), float("nan"), device=dev)
    db = torch.full((wl.C,), float("nan"), device=dev) if wl.bias is not None else None
    di = torch.full((wl.n_seqs, 3, wl.C), float("nan"), device=dev)
    args = (wl.x, wl.weight, wl.bias, hist, wl.cu_seqlens, wl.cache_indices, wl.has_initial_state,
            wl.dy, None, dx, dw, db, di)
    if noalloc:
        ccc.ccc_bwd_noalloc(*args)
    else:
        ws = torch.empty(ccc.ccc_workspace_size(wl.rows, wl.n_seqs, wl.C, True), dtype=torch.uint8,
                         device=dev)
        ccc.ccc_bwd(*args, ws)
    torch.cuda.synchronize()
    return dx, dw, db, di


def _check_same(wl, got, want):
    T = wl.valid_tokens
    gdx, gdw, gdb, gdi = got
    wdx, wdw, wdb, wdi = want
    assert torch.equal(gdx[:T].view(torch.int16), wdx[:T].view(torch.int16)), "dx (noalloc vs workspace)"
    assert np.all(H.bits(gdx[T:]) == H.SENTINEL), "padding rows of dx were written"
    for g, w, what in ((gdw, wdw, "dweight"), (gdb, wdb, "dbias"), (gdi, wdi, "d_init_state")):
        if w is None:
            continue
        assert torch.equal(g.view(torch.int32), w.view(torch.int32)), f"{what} (noalloc vs workspace)"


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_two_calls(cuda_device):
    # call 1: 200 packed sequences (the 32-way search for each run's first
    # sequence); call 2: 4 sequences with a pool (all offsets in one warp
    # load) -- the second call runs on whatever the first left in the shared
    # scratch
    first = workloads.make_custom(workloads.packed_lengths(seed=3, N=200, rows=16384), 1024,
                                  rows=16384, seed=3, device=cuda_device, with_state=False)
    second = workloads.make_custom((300, 0, 17, 1200), 512, rows=1600, seed=4, device=cuda_device,
                                   n_minus_one=1)
    for wl in (first, second):
        need = ccc.ccc_workspace_size(wl.rows, wl.n_seqs, wl.C, True)
        assert 0 < need <= _lib.NOALLOC_SCRATCH_BYTES
        hist = _forward(wl)
        want = _grads(wl, hist, noalloc=False)
        got = _grads(wl, hist, noalloc=True)
        _check_same(wl, got, want)


@pytest.mark.gpu
def test_noalloc_largest_scratch_shape(cuda_device):
    # The backward's scratch is R x 5 x C floats with R x ceil(C / 256) <= 1216:
    # about 6.2 MB at most for the widths used here (C a multiple of 256),
    # far inside the fixed array; run the C = 7168 packed shape, the largest
    # of the benchmarks.
    wl = workloads.packed_small(device=cuda_device)
    need = ccc.ccc_workspace_size(wl.rows, wl.n_seqs, wl.C, True)
    assert 6_000_000 < need <= _lib.NOALLOC_SCRATCH_BYTES
    hist = _forward(wl)
    want = _grads(wl, hist, noalloc=False)
    got = _grads(wl, hist, noalloc=True)
    _check_same(wl, got, want)


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(8))
def test_noalloc_random_batches(cuda_device, seed):
    # random packed batches (widths 2-4, with and without SiLU, -1 requests,
    # flags, dtypes; the draw of tests/test_random_batches_gpu.py), each
    # backward run twice in a row on the shared scratch
    from tests import test_random_batches_gpu as R
    lengths, C, rows, width, act, kw = R._case(seed)
    wl = workloads.make_custom(lengths, C, rows=rows, seed=seed, device=cuda_device, width=width,
                               activation=act, **kw)
    hist = torch.zeros((wl.n_seqs, width - 1, C), dtype=torch.bfloat16, device=cuda_device)
    ccc.ccc_fwd(wl.x, wl.weight, wl.bias, wl.conv_state.clone(), wl.cu_seqlens, wl.cache_indices,
                wl.has_initial_state, torch.empty_like(wl.x), hist, activation=act)
    outs = []
    for noalloc in (False, True, True):
        dx = torch.zeros_like(wl.x)
        dw = torch.zeros((C, width), device=cuda_device)
        db = torch.zeros((C,), device=cuda_device) if wl.bias is not None else None
        di = torch.zeros((wl.n_seqs, width - 1, C), device=cuda_device)
        args = (wl.x, wl.weight, wl.bias, hist, wl.cu_seqlens, wl.cache_indices, wl.has_initial_state,
                wl.dy, None, dx, dw, db, di)
        if noalloc:
            ccc.ccc_bwd_noalloc(*args, activation=act)
        else:
            ws = torch.empty(ccc.ccc_workspace_size(wl.rows, wl.n_seqs, C, True), dtype=torch.uint8,
                             device=cuda_device)
            ccc.ccc_bwd(*args, ws, activation=act)
        torch.cuda.synchronize()
        outs.append((dx, dw, db, di))
    for got in outs[1:]:
        for g, w in zip(got, outs[0]):
            if w is not None:
                assert torch.equal(g.view(torch.int16) if g.dtype == torch.bfloat16 else g.view(torch.int32),
                                   w.view(torch.int16) if w.dtype == torch.bfloat16 else w.view(torch.int32))
