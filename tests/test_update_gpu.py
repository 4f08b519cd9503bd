"""The speculative / single-token decode step (ccc_update) against the
float64 oracle, through the C ABI.

Reading under test (FlashInfer causal_conv1d_fn, Notes: the speculative step
right after a prefill is given an accepted count of one): the step reads the W-1
values at positions a-1 .. of the slot and leaves history value h[p+1] at
position p for p < len + W-2.  The oracle's pins tie that rule to torch
conv1d over the kept token stream; here the GPU follows the oracle step by
step on its own state, for the three pool layouts the kernels handle
differently (dense history-contiguous: a lane's whole block in registers;
channel-contiguous: 16-byte vectors; any other strides: element by element).
"""
import numpy as np
import pytest
import torch

import oracle
import ssm_depthwise_causal_gb300 as ccc
from ssm_depthwise_causal_gb300 import workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _pool(slots, C, L, layout, g, dev):
    """A [slots, C, L] BF16 pool in the given storage layout (same values for
    every layout: drawn in logical order)."""
    vals = workloads.normal_bf16((slots, C, L), g, dev)
    if layout == "dense":
        return vals.clone()
    if layout == "channel":
        return vals.transpose(1, 2).contiguous().transpose(1, 2)
    if layout == "padded":   # history axis contiguous, channel stride L + 3
        buf = torch.zeros((slots, C, L + 3), dtype=torch.bfloat16, device=dev)
        buf[:, :, :L] = vals
        return buf[:, :, :L]
    raise ValueError(layout)


def _bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _step_inputs(rng, N, C, k_of, dev, g):
    lengths = np.asarray(k_of, dtype=np.int64)
    rows = int(lengths.sum()) + 2                      # two padding rows
    x = workloads.normal_bf16((rows, C), g, dev)
    cu = workloads.cu_from_lengths(lengths).to(dev)
    return x, cu, lengths, rows


def _compare_step(out_gpu, ref_out, lengths, cache, what):
    cu = np.concatenate([[0], np.cumsum(lengths)])
    o = _bits(out_gpu)
    for n, q in enumerate(cache):
        s, e = cu[n], cu[n + 1]
        if e == s:
            continue
        if q == -1:
            assert np.all(o[s:e] == 0), f"{what}: -1 rows must be +0"
        else:
            H.assert_bf16_close(o[s:e], ref_out[s:e], f"{what} seq {n}")
    assert np.all(o[cu[-1]:] == H.SENTINEL), f"{what}: padding rows were written"


def _run_chain(dev, *, width, act, layout, C, N, L, kmax, steps, seed, w_dtype=torch.float32,
               b_dtype=torch.float32):
    """Prefill with ccc_fwd, then `steps` speculative steps with random draft
    counts (0..kmax) and accepted counts; GPU and oracle each carry their own
    pool, compared bit for bit after every call."""
    rng = np.random.default_rng(seed)
    g = workloads._gen(seed, dev)
    slots = N + 3
    pool = _pool(slots, C, L, layout, g, dev)
    pool_ref = pool.detach().cpu().contiguous()
    cache_np = rng.permutation(slots)[:N].astype(np.int32)
    cache_np[1] = -1
    cache = torch.from_numpy(cache_np).to(dev)
    weight = workloads.uniform((C, width), g, dev, -0.5, 0.5, w_dtype)
    bias = None if b_dtype is None else (torch.randn((C,), generator=g, device=dev) * 0.1).to(b_dtype)
    kw = dict(activation=act)
    # prefill
    pre = rng.integers(0, 6, N)
    x, cu, lengths, rows = _step_inputs(rng, N, C, pre, dev, g)
    hi = torch.from_numpy(rng.random(N) < 0.7).to(dev)
    out = H.fill_sentinel(torch.empty((rows, C), dtype=torch.bfloat16, device=dev))
    ws = torch.empty(max(1, ccc.ccc_workspace_size(rows, N, C, False)), dtype=torch.uint8, device=dev)
    ccc.ccc_fwd(x, weight, bias, pool, cu, cache, hi, out, None, ws, **kw)
    ref_out, pool_ref_np, _ = oracle.fwd(x, weight, bias, cu, pool_ref, cache, hi, **kw)
    torch.cuda.synchronize()
    _compare_step(out, ref_out, lengths, cache_np, "prefill")
    np.testing.assert_array_equal(_bits(pool), pool_ref_np, err_msg="pool after prefill")
    pool_ref = torch.from_numpy(pool_ref_np.view(np.int16)).view(torch.bfloat16)
    acc = np.ones(N, dtype=np.int32)        # after a prefill the accepted count is 1
    max_a = L - (width - 1) + 1
    seen_a = set()
    for step in range(steps):
        k = rng.integers(0, kmax + 1, N)
        k[0] = max(k[0], 1)
        x, cu, lengths, rows = _step_inputs(rng, N, C, k, dev, g)
        acc_t = torch.from_numpy(acc.copy()).to(dev)
        out = H.fill_sentinel(torch.empty((rows, C), dtype=torch.bfloat16, device=dev))
        ccc.ccc_update(x, weight, bias, pool, cu, cache, acc_t, out, **kw)
        ref_out, pool_ref_np = oracle.update(x, weight, bias, cu, pool_ref, cache, acc_t, **kw)
        torch.cuda.synchronize()
        what = f"step {step}"
        _compare_step(out, ref_out, lengths, cache_np, what)
        np.testing.assert_array_equal(_bits(pool), pool_ref_np, err_msg=f"pool after {what}")
        pool_ref = torch.from_numpy(pool_ref_np.view(np.int16)).view(torch.bfloat16)
        seen_a |= set(acc.tolist())
        # next accepted count: 1..len of this step (unchanged after an empty step)
        for n in range(N):
            if k[n] > 0:
                acc[n] = min(int(rng.integers(1, k[n] + 1)), max_a)
    return seen_a


@pytest.mark.parametrize("layout", ["dense", "channel", "padded"])
def test_decode_chain_layouts(cuda_device, layout):
    seen = _run_chain(cuda_device, width=4, act="silu", layout=layout, C=264, N=9, L=7, kmax=5,
                      steps=8, seed=1)
    assert max(seen) > 1


@pytest.mark.parametrize("width,act", [(2, "silu"), (3, None), (3, "silu"), (4, None), (2, None)])
def test_decode_chain_variants(cuda_device, width, act):
    _run_chain(cuda_device, width=width, act=act, layout="dense", C=520, N=7, L=width + 3, kmax=4,
               steps=6, seed=10 + width, w_dtype=torch.bfloat16, b_dtype=torch.bfloat16)
    _run_chain(cuda_device, width=width, act=act, layout="channel", C=136, N=5, L=width + 3, kmax=4,
               steps=4, seed=20 + width, b_dtype=None)


@pytest.mark.parametrize("width,L", [(w, L) for w in (2, 3, 4) for L in range(w - 1, 9)])
def test_dense_pool_every_length(cuda_device, width, L):
    """The dense history-contiguous pool at every length the register-block
    kernel is compiled for (L = W-1 .. 8), with drafts up to two tokens
    longer than the L - W + 2 the slot can keep: every position is written,
    every accepted offset is read, and the tokens past the slot's capacity
    take the kernel's one-token-at-a-time tail."""
    _run_chain(cuda_device, width=width, act="silu" if L % 2 else None, layout="dense", C=264, N=11, L=L,
               kmax=L - width + 4, steps=6, seed=60 + 10 * width + L)


def test_plain_decode_one_token(cuda_device):
    """k = 1 every step, accepted count omitted (= 1): the ordinary decode
    shift; the pool is exactly L = W-1 long."""
    dev = cuda_device
    g = workloads._gen(3, dev)
    N, C, L = 33, 1024, 3
    pool = workloads.normal_bf16((40, C, L), g, dev)
    cache = torch.randperm(40, generator=torch.Generator().manual_seed(3))[:N].to(torch.int32).to(dev)
    weight = workloads.uniform((C, 4), g, dev, -0.5, 0.5, torch.float32)
    bias = (torch.randn((C,), generator=g, device=dev) * 0.1)
    cu = torch.arange(N + 1, dtype=torch.int32, device=dev)
    pool_ref = pool.cpu()
    for step in range(5):
        x = workloads.normal_bf16((N, C), g, dev)
        out = torch.empty_like(x)
        ccc.ccc_update(x, weight, bias, pool, cu, cache, None, out)
        ref_out, st = oracle.update(x, weight, bias, cu, pool_ref, cache, None)
        torch.cuda.synchronize()
        H.assert_bf16_close(_bits(out), ref_out, f"step {step}")
        np.testing.assert_array_equal(_bits(pool), st)
        pool_ref = torch.from_numpy(st.view(np.int16)).view(torch.bfloat16)
    assert ccc.last_launch_count() == 1


def test_serving_decode_full_size(cuda_device):
    """The serving pool at full size (N = 256, C = 8192, pool [512, 8192, 6]),
    4-token speculative steps: every channel's pool update checked bit for bit
    against the write rule, outputs against the oracle on a spread of
    channels."""
    dev = cuda_device
    rng = np.random.default_rng(5)
    g = workloads._gen(5, dev)
    N, C, L, slots, k = 256, 8192, 6, 512, 4
    pool = workloads.normal_bf16((slots, C, L), g, dev)
    cache_np = rng.permutation(slots)[:N].astype(np.int32)
    cache_np[rng.choice(N, 13, replace=False)] = -1
    cache = torch.from_numpy(cache_np).to(dev)
    weight = workloads.uniform((C, 4), g, dev, -0.5, 0.5, torch.float32)
    bias = (torch.randn((C,), generator=g, device=dev) * 0.1).to(torch.bfloat16)
    lengths = rng.integers(1, k + 1, N)
    cu = workloads.cu_from_lengths(lengths).to(dev)
    x = workloads.normal_bf16((int(lengths.sum()), C), g, dev)
    acc = torch.from_numpy(rng.integers(1, 4, N).astype(np.int32)).to(dev)
    before = pool.clone()
    out = torch.empty_like(x)
    ccc.ccc_update(x, weight, bias, pool, cu, cache, acc, out)
    torch.cuda.synchronize()
    # every channel: the write rule, bit for bit
    pb, bb, xb = _bits(pool), _bits(before), _bits(x)
    cu_np = np.concatenate([[0], np.cumsum(lengths)])
    for n in range(N):
        q = cache_np[n]
        if q == -1:
            continue
        a = int(acc[n])
        hist = np.concatenate([bb[q, :, a - 1:a + 2].T, xb[cu_np[n]:cu_np[n + 1]]], 0)   # [3+len, C]
        n_w = min(int(lengths[n]) + 2, L)
        np.testing.assert_array_equal(pb[q, :, :n_w].T, hist[1:1 + n_w], err_msg=f"seq {n}")
        np.testing.assert_array_equal(pb[q, :, n_w:], bb[q, :, n_w:])
    live = set(int(q) for q in cache_np if q != -1)
    for q in range(slots):
        if q not in live:
            np.testing.assert_array_equal(pb[q], bb[q])
    # outputs on a spread of channels against the oracle
    chans = sorted(set(range(0, 8)) | set(range(C - 8, C)) | set(np.linspace(0, C - 1, 40).astype(int).tolist())
                   | {255, 256, 511, 512})
    idx = torch.as_tensor(chans, device=dev)
    ref_out, _ = oracle.update(x.index_select(1, idx).cpu(), weight.index_select(0, idx).cpu(),
                               bias.index_select(0, idx).cpu(), cu.cpu(),
                               before.index_select(1, idx).cpu(), cache.cpu(), acc.cpu())
    o = _bits(out.index_select(1, idx))
    for n in range(N):
        s, e = cu_np[n], cu_np[n + 1]
        if cache_np[n] == -1:
            assert np.all(o[s:e] == 0)
        else:
            H.assert_bf16_close(o[s:e], ref_out[s:e], f"seq {n}")


def test_btd_helpers(cuda_device):
    """[B, T, D] (non-packed) input of the conveniences equals the packed
    call with cu_seqlens = arange(B+1) * T; [B, D] / [B, k, D] decode input
    equals the packed update."""
    dev = cuda_device
    g = workloads._gen(8, dev)
    B, T, D = 3, 37, 264
    x = workloads.normal_bf16((B, T, D), g, dev)
    w = workloads.uniform((D, 3), g, dev, -0.5, 0.5, torch.float32)
    y = ccc.causal_conv1d_fn(x, w, activation=None)
    cu = torch.arange(B + 1, dtype=torch.int32, device=dev) * T
    y2 = ccc.causal_conv1d_fn(x.view(B * T, D), w, cu_seqlens=cu, activation=None)
    assert torch.equal(y.view(B * T, D).view(torch.int16), y2.view(torch.int16))
    dy = workloads.normal_bf16((B, T, D), g, dev)
    dx, dw, db, _ = ccc.causal_conv1d_bwd(x, w, dy, activation=None)
    dx2, dw2, _, _ = ccc.causal_conv1d_bwd(x.view(B * T, D), w, dy.view(B * T, D), cu, activation=None)
    assert dx.shape == (B, T, D) and torch.equal(dx.reshape(B * T, D).view(torch.int16), dx2.view(torch.int16))
    assert torch.equal(dw, dw2)
    # autograd on [B, T, D] input
    xg = x.clone().requires_grad_(True)
    wg = w.clone().requires_grad_(True)
    yg = ccc.causal_conv1d(xg, wg)
    (yg.float() * dy.float()).sum().backward()
    dx3, dw3, _, _ = ccc.causal_conv1d_bwd(x, w, dy)
    assert torch.equal(xg.grad.view(torch.int16), dx3.view(torch.int16))
    assert torch.equal(wg.grad, dw3)
    # decode: [B, D] and [B, k, D]
    pool = workloads.normal_bf16((B + 2, D, 5), g, dev)
    pool2 = pool.clone()
    cache = torch.tensor([4, 0, 2], dtype=torch.int32, device=dev)
    xt = workloads.normal_bf16((B, D), g, dev)
    yt = ccc.causal_conv1d_update(xt, w, pool, cache)
    yt2 = torch.empty_like(xt)
    ccc.ccc_update(xt, w, None, pool2, torch.arange(B + 1, dtype=torch.int32, device=dev), cache, None, yt2)
    assert yt.shape == (B, D) and torch.equal(yt.view(torch.int16), yt2.view(torch.int16))
    assert torch.equal(pool.view(torch.int16), pool2.view(torch.int16))
    xk = workloads.normal_bf16((B, 2, D), g, dev)
    acc = torch.tensor([1, 1, 1], dtype=torch.int32, device=dev)
    yk = ccc.causal_conv1d_update(xk, w, pool, cache, num_accepted=acc)
    yk2 = torch.empty((B * 2, D), dtype=torch.bfloat16, device=dev)
    ccc.ccc_update(xk.view(B * 2, D), w, None, pool2, torch.arange(B + 1, dtype=torch.int32, device=dev) * 2,
                   cache, acc, yk2)
    assert torch.equal(yk.view(B * 2, D).view(torch.int16), yk2.view(torch.int16))
    assert torch.equal(pool.view(torch.int16), pool2.view(torch.int16))


@pytest.mark.parametrize("layout", ["dense", "channel", "padded"])
def test_strided_token_rows(cuda_device, layout):
    """x a column slice of a wider matrix (row stride C + 64) and out with a
    padded row stride (C + 8), for every pool layout: the outputs equal a
    contiguous call bit for bit, the padding columns of out are untouched,
    and the pools end identical."""
    dev = cuda_device
    rng = np.random.default_rng(31)
    g = workloads._gen(31, dev)
    N, C, L, slots = 21, 264, 7, 30
    lengths = rng.integers(0, 6, N)
    rows = int(lengths.sum()) + 2
    cu = workloads.cu_from_lengths(lengths).to(dev)
    cache_np = rng.permutation(slots)[:N].astype(np.int32)
    cache_np[3] = -1
    cache = torch.from_numpy(cache_np).to(dev)
    acc = torch.from_numpy(rng.integers(1, L - 2, N).astype(np.int32)).to(dev)
    weight = workloads.uniform((C, 4), g, dev, -0.5, 0.5, torch.float32)
    bias = (torch.randn((C,), generator=g, device=dev) * 0.1).to(torch.bfloat16)
    wide = workloads.normal_bf16((rows, C + 64), g, dev)
    x_strided = wide[:, 32:32 + C]
    x = x_strided.contiguous()
    pool_a = _pool(slots, C, L, layout, g, dev)
    pool_b = _pool(slots, C, L, layout, workloads._gen(99, dev), dev)  # same layout, then the same values
    pool_b.copy_(pool_a)
    out_pad = H.fill_sentinel(torch.empty((rows, C + 8), dtype=torch.bfloat16, device=dev))
    out = H.fill_sentinel(torch.empty((rows, C), dtype=torch.bfloat16, device=dev))
    ccc.ccc_update(x_strided, weight, bias, pool_a, cu, cache, acc, out_pad[:, :C])
    ccc.ccc_update(x, weight, bias, pool_b, cu, cache, acc, out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(out_pad[:, :C]), _bits(out))
    assert np.all(_bits(out_pad[:, C:]) == H.SENTINEL), "padding columns of out were written"
    np.testing.assert_array_equal(_bits(pool_a), _bits(pool_b))


@pytest.mark.parametrize("width", [2, 3, 4])
def test_one_hot_taps_read_offsets(cuda_device, width):
    """With the taps one-hot at k, no bias and no activation, token j of a
    request with accepted count a must output the history value h[j + k]
    (the slot's positions a-1 .. a+W-3, then the request's tokens) bit for
    bit: an exact check of the kernels' offset selection and tap order, for
    every dense pool length the register-block kernel is compiled for, every
    accepted count, and the channel-contiguous pool."""
    dev = cuda_device
    rng = np.random.default_rng(80 + width)
    H = width - 1
    for L in list(range(H, 9)) + ["channel"]:
        layout = "channel" if L == "channel" else "dense"
        Lr = 7 if L == "channel" else L
        N, C, slots = 13, 264, 16
        g = workloads._gen(80 + width, dev)
        pool = _pool(slots, C, Lr, layout, g, dev)
        lengths = rng.integers(0, 6, N)
        x, cu, lengths, rows = _step_inputs(rng, N, C, lengths, dev, g)
        cache = torch.from_numpy(rng.permutation(slots)[:N].astype(np.int32)).to(dev)
        acc = torch.from_numpy((1 + np.arange(N) % (Lr - width + 2)).astype(np.int32)).to(dev)
        before = _bits(pool).astype(np.uint16)
        xb = _bits(x)
        cu_np = np.concatenate([[0], np.cumsum(lengths)])
        for k in range(width):
            w = torch.zeros((C, width), dtype=torch.float32, device=dev)
            w[:, k] = 1.0
            p = pool.clone() if layout == "dense" else _pool(slots, C, Lr, layout, g, dev)
            p.copy_(pool)
            out = H_fill(rows, C, dev)
            ccc.ccc_update(x, w, None, p, cu, cache, acc, out, activation=None)
            torch.cuda.synchronize()
            o = _bits(out)
            for n, q in enumerate(cache.tolist()):
                s, e = cu_np[n], cu_np[n + 1]
                a = int(acc[n])
                h = np.concatenate([before[q, :, a - 1:a - 1 + H].T, xb[s:e]], 0)
                np.testing.assert_array_equal(o[s:e], h[k:k + (e - s)], err_msg=f"L={L} k={k} seq {n}")


def H_fill(rows, C, dev):
    return H.fill_sentinel(torch.empty((rows, C), dtype=torch.bfloat16, device=dev))


@pytest.mark.parametrize("seed", range(16))
def test_random_decode_chains(cuda_device, seed):
    """Random prefill + speculative chains: width, activation, pool layout and
    length, channel count (partial slabs), batch size, draft counts, dtypes."""
    rng = np.random.default_rng(7000 + seed)
    width = int(rng.integers(2, 5))
    L = int(rng.integers(width - 1, 9))
    _run_chain(cuda_device, width=width, act="silu" if rng.random() < 0.6 else None,
               layout=["dense", "channel", "padded"][int(rng.integers(0, 3))],
               C=8 * int(rng.integers(1, 80)), N=int(rng.integers(2, 40)), L=L,
               kmax=int(rng.integers(1, 6)), steps=4, seed=seed,
               w_dtype=torch.bfloat16 if rng.random() < 0.5 else torch.float32,
               b_dtype=[None, torch.float32, torch.bfloat16][int(rng.integers(0, 3))])
