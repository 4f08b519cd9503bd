"""CUDA graph capture and replay (FlashInfer flashinfer.mamba.causal_conv1d_fn,
Notes: a replayed graph may see new offsets and slot values written into the
same device buffers, with sizes unchanged; the output and scratch buffers
are handed over before capture).

The library reads no device value on the host, never synchronizes and
allocates nothing, so a forward + backward (and a decode step) captured once
must replay correctly after the offsets, slots, flags, accepted counts and
activations are rewritten in place: every replay is compared bit for bit with
an eager call on the same new inputs.
"""
import numpy as np
import pytest
import torch

import ssm_depthwise_causal_gb300 as ccc
from ssm_depthwise_causal_gb300 import workloads

pytestmark = pytest.mark.gpu


def _lengths(rng, N, rows):
    cut = np.sort(rng.integers(0, rows + 1, N - 1))
    return np.diff(np.concatenate([[0], cut, [rows - int(rng.integers(0, 5))]])).clip(min=0)


def _eq(a, b):
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("width,act", [(4, "silu"), (3, None)])
def test_fwd_bwd_graph_replay_with_new_metadata(cuda_device, width, act):
    dev = cuda_device
    rng = np.random.default_rng(3)
    N, C, rows, slots = 40, 264, 3000, 64
    H = width - 1
    base = workloads.make_custom(_lengths(rng, N, rows - 8), C, rows=rows, seed=5, device=dev, slots=slots,
                                 n_minus_one=4, width=width, activation=act)
    # static buffers the graph captures
    x, dy, w, b = base.x.clone(), base.dy.clone(), base.weight, base.bias
    cu, cache, hi = base.cu_seqlens.clone(), base.cache_indices.clone(), base.has_initial_state.clone()
    pool = base.conv_state.clone()
    out = torch.empty_like(x)
    hist = torch.empty((N, H, C), dtype=torch.bfloat16, device=dev)
    dx = torch.empty_like(x)
    dw = torch.empty((C, width), device=dev)
    db = torch.empty((C,), device=dev)
    di = torch.empty((N, H, C), device=dev)
    wsb = torch.empty(ccc.ccc_workspace_size(rows, N, C, True), dtype=torch.uint8, device=dev)
    kw = dict(activation=act)

    def step():
        ccc.ccc_fwd(x, w, b, pool, cu, cache, hi, out, hist, None, **kw)
        ccc.ccc_bwd(x, w, b, hist, cu, cache, hi, dy, None, dx, dw, db, di, wsb, **kw)

    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside capture (one-time attribute set-up)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()

    for trial in range(3):
        # rewrite the device metadata and the data in place
        lens = _lengths(rng, N, rows - 8)
        cu.copy_(workloads.cu_from_lengths(lens).to(dev))
        perm = torch.from_numpy(rng.permutation(slots)[:N].astype(np.int32))
        perm[rng.choice(N, 5, replace=False)] = -1
        cache.copy_(perm.to(dev))
        hi.copy_(torch.from_numpy(rng.random(N) < 0.5).to(dev))
        g_in = torch.Generator(device=dev).manual_seed(100 + trial)
        x.copy_(workloads.normal_bf16((rows, C), g_in, dev))
        dy.copy_(workloads.normal_bf16((rows, C), g_in, dev))
        pool_before = pool.clone()
        g.replay()
        torch.cuda.synchronize()
        # eager reference on fresh buffers with the same inputs
        pool_e = pool_before.clone()
        out_e, dx_e = torch.empty_like(x), torch.empty_like(x)
        hist_e = torch.empty_like(hist)
        dw_e, db_e, di_e = torch.empty_like(dw), torch.empty_like(db), torch.empty_like(di)
        ws_e = torch.empty_like(wsb)
        ccc.ccc_fwd(x, w, b, pool_e, cu, cache, hi, out_e, hist_e, None, **kw)
        ccc.ccc_bwd(x, w, b, hist_e, cu, cache, hi, dy, None, dx_e, dw_e, db_e, di_e, ws_e, **kw)
        torch.cuda.synchronize()
        T = int(lens.sum())
        assert _eq(out[:T], out_e[:T]), f"trial {trial}: out"
        assert _eq(pool, pool_e), f"trial {trial}: conv_state"
        assert _eq(dx[:T], dx_e[:T]), f"trial {trial}: dx"
        assert _eq(dw, dw_e) and _eq(db, db_e), f"trial {trial}: dweight / dbias"
        ne = torch.from_numpy(lens > 0).to(dev)
        assert _eq(hist[ne], hist_e[ne]) and _eq(di, di_e), f"trial {trial}: saved_hist / d_init_state"


def test_decode_step_graph_replay(cuda_device):
    dev = cuda_device
    rng = np.random.default_rng(8)
    N, C, slots, L, k = 48, 520, 96, 6, 4
    g0 = workloads._gen(8, dev)
    pool = workloads.normal_bf16((slots, C, L), g0, dev)
    w = workloads.uniform((C, 4), g0, dev, -0.5, 0.5, torch.float32)
    b = (torch.randn((C,), generator=g0, device=dev) * 0.1)
    rows = N * k
    x = torch.empty((rows, C), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(x)
    cu = torch.zeros(N + 1, dtype=torch.int32, device=dev)
    cache = torch.zeros(N, dtype=torch.int32, device=dev)
    acc = torch.ones(N, dtype=torch.int32, device=dev)

    def fill(trial):
        lens = rng.integers(0, k + 1, N)
        cu.copy_(workloads.cu_from_lengths(lens).to(dev))
        perm = torch.from_numpy(rng.permutation(slots)[:N].astype(np.int32))
        perm[rng.choice(N, 3, replace=False)] = -1
        cache.copy_(perm.to(dev))
        acc.copy_(torch.from_numpy(rng.integers(1, L - 1, N).astype(np.int32)).to(dev))
        x.copy_(workloads.normal_bf16((rows, C), torch.Generator(device=dev).manual_seed(trial), dev))
        return int(lens.sum())

    fill(0)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ccc.ccc_update(x, w, b, pool.clone(), cu, cache, acc, out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ccc.ccc_update(x, w, b, pool, cu, cache, acc, out)
    for trial in range(1, 4):
        T = fill(trial)
        pool_e = pool.clone()
        g.replay()
        out_e = torch.empty_like(out)
        ccc.ccc_update(x, w, b, pool_e, cu, cache, acc, out_e)
        torch.cuda.synchronize()
        assert _eq(out[:T], out_e[:T]) and _eq(pool, pool_e), f"trial {trial}"
