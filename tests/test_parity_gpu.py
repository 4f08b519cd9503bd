"""GPU path (through the C ABI) against the float64 oracle.

Small cases are compared element by element on every channel; the five
workloads run at full size and are compared on every channel (tiny, dense,
packed) or on every 8th / 32nd channel plus both sides of every slab edge
(serving, the one-million-token document) -- exact for those channels,
since channels never interact -- plus full-size properties (state bits,
untouched slots, -1 rows, padding, determinism, split = unsplit).
"""
import numpy as np
import pytest
import torch

from ssm_depthwise_causal_gb300 import workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def spread_channels(C, n=48):
    picks = set(range(0, min(C, 8))) | set(range(max(0, C - 8), C))
    for b in (127, 128, 255, 256, 511, 512, 1023, 1024):
        if b < C:
            picks.add(b)
    picks |= set(np.linspace(0, C - 1, n).round().astype(int).tolist())
    return sorted(picks)


def every_kth_channel(C, k):
    """Every k-th channel, plus both sides of every 256-channel slab edge
    (the backward's slab width) and of every 128-channel edge, and the last
    channels."""
    picks = set(range(0, C, k)) | set(range(max(0, C - 8), C))
    for e in range(128, C, 128):
        picks |= {e - 1, e}
    return sorted(picks)


def check(wl_gpu, res, *, chans=None, backward=True, d_final=None):
    chans = list(range(wl_gpu.C)) if chans is None else chans
    sub = H.subset(wl_gpu, chans)
    df = None if d_final is None else d_final[:, :, chans].double().cpu()
    ref = H.run_oracle(sub, backward=backward, d_final=df)
    return H.compare(sub, ref, H.gpu_numpy(res, chans), backward=backward, chans=chans)


def report(name, stats):
    """Print how the reduction outputs passed (visible with pytest -s / -rP)
    and bound them.  An element passes through the floor only when its sum
    cancels to below 1 % of the size of its terms (|err| > 1e-4 |ref| and
    |err| <= 1e-6 sum|terms| imply |ref| < 1e-2 sum|terms|), so how many do
    is a property of the data -- a few percent for sums of a million random
    terms; what bounds the arithmetic is the error against the terms' scale,
    held here to 1e-7 (ten times tighter than the floor)."""
    for what, st in stats.items():
        print(f"[reduction] {name} {what}: {st['n']} elements, {st['floor_only']} within the floor "
              f"1e-6*sum|terms| only, max |err|/|ref| {st['max_rel']:.3g}, "
              f"max |err|/sum|terms| {st['max_err_terms']:.3g}")
        assert st["max_err_terms"] <= 1e-7, f"{name} {what}: error above 1e-7 of the terms' scale"
        assert st["floor_only"] <= max(2, st["n"] // 20), f"{name} {what}: too many elements need the floor"


def test_tiny(cuda_device):
    wl = workloads.tiny(device=cuda_device)
    check(wl, H.run_gpu(wl))


@pytest.mark.parametrize("layout", ["history", "channel"])
@pytest.mark.parametrize("pad", [0, 24])
def test_tiny_layouts_and_strides(cuda_device, layout, pad):
    wl = workloads.tiny(seed=3, device=cuda_device)
    res = H.run_gpu(wl, pool_layout=layout, x_pad_cols=pad)
    if layout == "channel":  # compare in the logical [slots, C, L] view
        res.state = res.state.contiguous()
    check(wl, res)


EDGE = {
    # lengths, C, kwargs
    "short_and_empty": ((1, 2, 3, 4, 0, 5), 8, dict(n_minus_one=1)),
    "chunk_boundaries": ((63, 64, 65, 127, 128, 129, 0, 1), 24, dict(n_minus_one=1)),
    "n32_inline": (tuple(range(0, 64, 2)), 264, dict(n_minus_one=3)),
    "n33_map": (tuple(range(0, 66, 2)), 136, dict(n_minus_one=3)),
    "n100_short_all_init": (tuple(int(v) for v in np.random.default_rng(5).integers(0, 50, 100)),
                            40, dict(n_minus_one=10, has_init_p=1.0)),
    "single_long_no_state": ((1000,), 520, dict(with_state=False)),
    "bf16_w_bf16_b": ((33, 7, 90), 64, dict(w_dtype=torch.bfloat16, b_dtype=torch.bfloat16)),
    "no_bias": ((33, 7, 90), 64, dict(b_dtype=None)),
    "no_init": ((17, 3, 40), 32, dict(has_init_p=0.0)),
    "all_minus_one": ((5, 9), 16, dict(n_minus_one=2)),
    "all_empty": ((0, 0, 0), 16, dict()),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(cuda_device, name):
    lengths, C, kw = EDGE[name]
    T = sum(lengths)
    wl = workloads.make_custom(lengths, C, rows=T + 5, seed=11, device=cuda_device, **kw)
    check(wl, H.run_gpu(wl))


def test_d_final_carry(cuda_device):
    wl = workloads.make_custom((40, 2, 0, 70), 64, rows=120, seed=2, device=cuda_device,
                               n_minus_one=0, has_init_p=0.5)
    g = torch.Generator(device=cuda_device).manual_seed(9)
    d_final = torch.randn((wl.n_seqs, 3, wl.C), generator=g, device=cuda_device)
    check(wl, H.run_gpu(wl, d_final=d_final), d_final=d_final)


@pytest.mark.parametrize("width,act", [(4, "silu"), (3, None), (2, "silu")])
def test_no_pool_minus_one(cuda_device, width, act):
    """cache_indices without a pool (FlashInfer causal_conv1d_fn,
    cache_indices: -1 gives a zero output without touching state): the -1
    requests output +0 and have zero gradient, the others run from zero
    history; forward and backward (with and without d_final_state) against
    the oracle on every channel."""
    import dataclasses
    wl = workloads.make_custom((12, 30, 5, 0, 77, 1, 64), 136, rows=200, seed=4, device=cuda_device,
                               n_minus_one=2, width=width, activation=act)
    wl = dataclasses.replace(wl, conv_state=None, has_initial_state=None)
    assert int((wl.cache_indices == -1).sum()) == 2
    check(wl, H.run_gpu(wl))
    g = torch.Generator(device=cuda_device).manual_seed(6)
    d_final = torch.randn((wl.n_seqs, width - 1, wl.C), generator=g, device=cuda_device)
    check(wl, H.run_gpu(wl, d_final=d_final), d_final=d_final)


def _full_size(wl, backward=True, chans=None):
    res = H.run_gpu(wl, backward=backward)
    stats = check(wl, res, chans=spread_channels(wl.C) if chans is None else chans, backward=backward)
    report(wl.name, stats)
    return res


def test_dense_full(cuda_device):
    """The dense training batch (16384 rows, C 4096) on every channel."""
    wl = workloads.dense(device=cuda_device)
    _full_size(wl, chans=list(range(wl.C)))


def test_packed_full_and_deterministic(cuda_device):
    """The packed batch (65536 rows, C 7168, 200 sequences) on every
    channel, then ten repeats bitwise."""
    wl = workloads.packed(device=cuda_device)
    res = _full_size(wl, chans=list(range(wl.C)))
    # ten more backward runs: dweight / dbias / dx bitwise identical
    import ssm_depthwise_causal_gb300 as ccc
    ws = torch.empty(ccc.ccc_workspace_size(wl.rows, wl.n_seqs, wl.C, True), dtype=torch.uint8,
                     device=cuda_device)
    dx = torch.empty_like(wl.x)
    dw = torch.empty((wl.C, 4), device=cuda_device)
    db = torch.empty((wl.C,), device=cuda_device)
    T = wl.valid_tokens
    for _ in range(10):
        ccc.ccc_bwd(wl.x, wl.weight, wl.bias, res.hist, wl.cu_seqlens, None, None, wl.dy, None,
                    dx, dw, db, None, ws)
        torch.cuda.synchronize()
        assert torch.equal(dw.view(torch.int32), res.dweight.view(torch.int32))
        assert torch.equal(db.view(torch.int32), res.dbias.view(torch.int32))
        assert torch.equal(dx[:T].view(torch.int16), res.dx[:T].view(torch.int16))


def test_serving_full(cuda_device):
    """The serving prefill (273 403 rows, C 8192, 256 sequences, pool) on every
    8th channel and both sides of every slab edge, then the pool rule on
    every channel."""
    wl = workloads.serving(device=cuda_device)
    before = wl.conv_state.clone()
    res = _full_size(wl, backward=False, chans=every_kth_channel(wl.C, 8))
    # full-size state properties (every channel)
    cu = wl.cu_seqlens.cpu().tolist()
    ci = wl.cache_indices.cpu().tolist()
    live = set()
    for n in range(wl.n_seqs):
        q, s, e = ci[n], cu[n], cu[n + 1]
        if q == -1 or e == s:
            continue
        live.add(q)
        assert e - s >= 1
        if e - s >= 3:
            assert torch.equal(res.state[q, :, 0:3].view(torch.int16),
                               wl.x[e - 3:e].t().contiguous().view(torch.int16)), n
        assert torch.equal(res.state[q, :, 3:].view(torch.int16), before[q, :, 3:].view(torch.int16))
    for q in range(wl.conv_state.shape[0]):
        if q not in live:
            assert torch.equal(res.state[q].view(torch.int16), before[q].view(torch.int16)), q


def test_long_context_split_equals_unsplit(cuda_device):
    import ssm_depthwise_causal_gb300 as ccc
    wl = workloads.long_context(device=cuda_device)
    dev = cuda_device
    T, C, F = wl.rows, wl.C, wl.fragments
    L = T // F
    # unsplit, one call each way
    out_u = torch.empty_like(wl.x)
    ccc.ccc_fwd(wl.x, wl.weight, None, None, wl.cu_seqlens, None, None, out_u)
    dx_u = torch.empty_like(wl.x)
    dw_u = torch.empty((C, 4), device=dev)
    ws = torch.empty(ccc.ccc_workspace_size(T, 1, C, True), dtype=torch.uint8, device=dev)
    ccc.ccc_bwd(wl.x, wl.weight, None, None, wl.cu_seqlens, None, None, wl.dy, None, dx_u, dw_u,
                None, None, ws)
    # split: fragments chained through a one-slot pool, backward in reverse
    pool = torch.zeros((1, C, 4), dtype=torch.bfloat16, device=dev)
    cache = torch.zeros(1, dtype=torch.int32, device=dev)
    cu_f = torch.tensor([0, L], dtype=torch.int32, device=dev)
    out_s = torch.empty_like(wl.x)
    hists = []
    for k in range(F):
        hist = torch.empty((1, 3, C), dtype=torch.bfloat16, device=dev)
        hi = torch.tensor([k > 0], device=dev)
        ccc.ccc_fwd(wl.x[k * L:(k + 1) * L], wl.weight, None, pool, cu_f, cache, hi,
                    out_s[k * L:(k + 1) * L], hist)
        hists.append((hist, hi))
    dx_s = torch.empty_like(wl.x)
    wsf = torch.empty(ccc.ccc_workspace_size(L, 1, C, True), dtype=torch.uint8, device=dev)
    d_carry = None
    dw_s = torch.zeros((C, 4), dtype=torch.float64, device=dev)
    for k in reversed(range(F)):
        hist, hi = hists[k]
        dwk = torch.empty((C, 4), device=dev)
        d_init = torch.empty((1, 3, C), device=dev)
        ccc.ccc_bwd(wl.x[k * L:(k + 1) * L], wl.weight, None, hist, cu_f, cache, hi,
                    wl.dy[k * L:(k + 1) * L], d_carry, dx_s[k * L:(k + 1) * L], dwk, None, d_init,
                    wsf)
        dw_s += dwk.double()
        d_carry = d_init
    torch.cuda.synchronize()
    assert torch.equal(out_s.view(torch.int16), out_u.view(torch.int16)), "split fwd != unsplit"
    assert torch.equal(dx_s.view(torch.int16), dx_u.view(torch.int16)), "split dx != unsplit"
    assert torch.equal(pool[0, :, 0:3].view(torch.int16), wl.x[T - 3:T].t().contiguous().view(torch.int16))
    assert torch.all(d_carry == 0), "the first fragment read no state: d_init must be 0"
    # unsplit vs the oracle on every 32nd channel and both sides of every slab edge
    chans = every_kth_channel(C, 32)
    sub = H.subset(wl, chans)
    ref = H.run_oracle(sub)
    res = H.GpuResult(out=out_u, state=None, hist=H.fill_sentinel(torch.empty((1, 3, C), dtype=torch.bfloat16, device=dev)),
                      dx=dx_u, dweight=dw_u, dbias=None, d_init=None)
    g = H.gpu_numpy(res, chans)
    g["hist"] = ref["hist"]  # no history was saved in the unsplit call
    report(wl.name + " (unsplit)", H.compare(sub, ref, g))
    # fragment-summed dweight within the reduction tolerance of the oracle
    report(wl.name + " (8 fragments, summed)",
           {"dweight": H.assert_reduction_close(dw_s[chans].cpu().numpy(), ref["dweight"], ref["abs_dweight"],
                                                "split dweight")})


# ------------------------------------------------ widths 2, 3 / no activation --
# Megatron-Core core.ssm.causal_conv1d (causal_conv1d_cp: weight [D, W],
# optional activation): the same kernels instantiated for W = 2, 3 and for
# the identity activation, against the oracle at the same width.

VARIANTS = [(2, "silu"), (2, None), (3, "silu"), (3, None), (4, None)]

VARIANT_SHAPES = {
    # lengths, C, kwargs
    "short_and_empty": ((1, 2, 3, 4, 0, 5, 2), 264, dict(n_minus_one=1)),
    "chunk_boundaries": ((63, 64, 65, 127, 129, 0, 1), 40, dict(n_minus_one=1, has_init_p=1.0)),
    "n40_map": (tuple(int(v) for v in np.random.default_rng(7).integers(0, 90, 40)), 72,
                dict(n_minus_one=4)),
    "bf16_w_no_bias": ((33, 7, 90), 64, dict(w_dtype=torch.bfloat16, b_dtype=None)),
}


@pytest.mark.parametrize("shape", sorted(VARIANT_SHAPES))
@pytest.mark.parametrize("width,act", VARIANTS)
def test_width_activation_variants(cuda_device, width, act, shape):
    lengths, C, kw = VARIANT_SHAPES[shape]
    wl = workloads.make_custom(lengths, C, rows=sum(lengths) + 5, seed=17 + width, device=cuda_device,
                               width=width, activation=act, **kw)
    check(wl, H.run_gpu(wl))


@pytest.mark.parametrize("width,act", VARIANTS)
def test_variant_d_final_and_channel_pool(cuda_device, width, act):
    wl = workloads.make_custom((40, 2, 0, 70, 1), 136, rows=120, seed=5, device=cuda_device,
                               n_minus_one=1, has_init_p=0.6, width=width, activation=act)
    g = torch.Generator(device=cuda_device).manual_seed(3)
    d_final = torch.randn((wl.n_seqs, width - 1, wl.C), generator=g, device=cuda_device)
    check(wl, H.run_gpu(wl, d_final=d_final), d_final=d_final)
    res = H.run_gpu(wl, pool_layout="channel", x_pad_cols=8)
    res.state = res.state.contiguous()
    check(wl, res)


@pytest.mark.parametrize("width,act", VARIANTS)
def test_variant_split_equals_unsplit(cuda_device, width, act):
    """A 24 576-token document in 4 fragments chained through a one-slot pool
    (and d_init -> d_final backwards) equals the unsplit call bit for bit."""
    import ssm_depthwise_causal_gb300 as ccc
    dev = cuda_device
    T, C, F = 24576, 520, 4
    L = T // F
    wl = workloads.make_custom((T,), C, seed=23, device=dev, with_state=False, width=width,
                               activation=act)
    Hh = width - 1
    kw = dict(activation=act)
    out_u = torch.empty_like(wl.x)
    ccc.ccc_fwd(wl.x, wl.weight, wl.bias, None, wl.cu_seqlens, None, None, out_u, **kw)
    dx_u = torch.empty_like(wl.x)
    dw_u = torch.empty((C, width), device=dev)
    db_u = torch.empty((C,), device=dev)
    ws = torch.empty(ccc.ccc_workspace_size(T, 1, C, True), dtype=torch.uint8, device=dev)
    ccc.ccc_bwd(wl.x, wl.weight, wl.bias, None, wl.cu_seqlens, None, None, wl.dy, None, dx_u, dw_u,
                db_u, None, ws, **kw)
    pool = torch.zeros((1, C, Hh), dtype=torch.bfloat16, device=dev)
    cache = torch.zeros(1, dtype=torch.int32, device=dev)
    cu_f = torch.tensor([0, L], dtype=torch.int32, device=dev)
    out_s = torch.empty_like(wl.x)
    hists = []
    for k in range(F):
        hist = torch.empty((1, Hh, C), dtype=torch.bfloat16, device=dev)
        hi = torch.tensor([k > 0], device=dev)
        ccc.ccc_fwd(wl.x[k * L:(k + 1) * L], wl.weight, wl.bias, pool, cu_f, cache, hi,
                    out_s[k * L:(k + 1) * L], hist, **kw)
        hists.append((hist, hi))
    dx_s = torch.empty_like(wl.x)
    wsf = torch.empty(ccc.ccc_workspace_size(L, 1, C, True), dtype=torch.uint8, device=dev)
    d_carry = None
    for k in reversed(range(F)):
        hist, hi = hists[k]
        dwk = torch.empty((C, width), device=dev)
        dbk = torch.empty((C,), device=dev)
        d_init = torch.empty((1, Hh, C), device=dev)
        ccc.ccc_bwd(wl.x[k * L:(k + 1) * L], wl.weight, wl.bias, hist, cu_f, cache, hi,
                    wl.dy[k * L:(k + 1) * L], d_carry, dx_s[k * L:(k + 1) * L], dwk, dbk, d_init, wsf, **kw)
        d_carry = d_init
    torch.cuda.synchronize()
    assert torch.equal(out_s.view(torch.int16), out_u.view(torch.int16)), "split fwd != unsplit"
    assert torch.equal(dx_s.view(torch.int16), dx_u.view(torch.int16)), "split dx != unsplit"
    assert torch.equal(pool[0].view(torch.int16), wl.x[T - Hh:T].t().contiguous().view(torch.int16))
    # the unsplit call against the oracle on a channel subset
    chans = spread_channels(C, n=16)
    sub = H.subset(wl, chans)
    ref = H.run_oracle(sub)
    res = H.GpuResult(out=out_u, state=None,
                      hist=H.fill_sentinel(torch.empty((1, Hh, C), dtype=torch.bfloat16, device=dev)),
                      dx=dx_u, dweight=dw_u, dbias=db_u, d_init=None)
    got = H.gpu_numpy(res, chans)
    got["hist"] = ref["hist"]  # no history was saved in the unsplit call
    H.compare(sub, ref, got)


@pytest.mark.parametrize("width,act", [(4, "silu"), (3, None), (2, "silu")])
def test_all_row_strides(cuda_device, width, act):
    """x, dy, out and dx as column slices of wider buffers (row strides C + 24
    and C + 40: GDP feeds the conv a slice of the in_proj output,
    gdp_context_parallel), with N > 32 and a partial slab."""
    lengths = tuple(int(v) for v in np.random.default_rng(9).integers(0, 70, 45))
    wl = workloads.make_custom(lengths, 264, rows=sum(lengths) + 3, seed=31, device=cuda_device,
                               n_minus_one=3, width=width, activation=act)
    check(wl, H.run_gpu(wl, x_pad_cols=24, out_pad_cols=40))


# ------------------------------------------- metadata staging boundaries --
# The kernels stage a batch's offsets, slots and flags in shared memory for up
# to 1024 sequences (forward) and 256 (backward) and read them from global
# memory beyond that: both sides of both limits, with -1 requests, empty
# sequences, a pool and d_final_state, on every channel.

@pytest.mark.parametrize("N,width,act", [(256, 4, "silu"), (257, 4, "silu"), (1024, 4, "silu"),
                                         (1025, 4, "silu"), (2000, 4, "silu"), (300, 2, "silu"),
                                         (1100, 3, None)])
def test_many_sequences_staged_and_global_metadata(cuda_device, N, width, act):
    rng = np.random.default_rng(N)
    lengths = tuple(int(v) for v in rng.integers(0, 12, N))
    wl = workloads.make_custom(lengths, 264, rows=sum(lengths) + 7, seed=N, device=cuda_device,
                               n_minus_one=N // 20, has_init_p=0.5, slots=2 * N + 3, width=width,
                               activation=act)
    g = torch.Generator(device=cuda_device).manual_seed(N)
    d_final = torch.randn((wl.n_seqs, width - 1, wl.C), generator=g, device=cuda_device)
    check(wl, H.run_gpu(wl, d_final=d_final), d_final=d_final)


# --------------------------------------------- taps not 16-byte aligned --
# Aligned taps and bias go through shared memory; taps or a bias that are
# only element-aligned (a view one element into a buffer) take the per-lane
# path.  Both must give the oracle's results.

def _offset_view(t: torch.Tensor) -> torch.Tensor:
    """The same values one element into a larger buffer (not 16-byte aligned)."""
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    v = flat[1:].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 16 != 0
    return v


UNALIGNED = [(W, wd, bd, which) for W, wd, bd in ((4, torch.float32, torch.float32), (4, torch.bfloat16, torch.float32),
                                                  (3, torch.float32, torch.bfloat16))
             for which in ("weight", "bias", "both")] + [(2, torch.bfloat16, None, "weight")]


@pytest.mark.parametrize("width,w_dtype,b_dtype,which", UNALIGNED)
def test_unaligned_taps(cuda_device, width, w_dtype, b_dtype, which):
    import dataclasses
    wl = workloads.make_custom((40, 0, 7, 130, 2, 64), 264, rows=250, seed=41, device=cuda_device,
                               n_minus_one=1, width=width, w_dtype=w_dtype, b_dtype=b_dtype)
    w = _offset_view(wl.weight) if which in ("weight", "both") else wl.weight
    b = _offset_view(wl.bias) if which in ("bias", "both") and wl.bias is not None else wl.bias
    wl = dataclasses.replace(wl, weight=w, bias=b)
    check(wl, H.run_gpu(wl))


# ------------------------------------- backward CTA size at its threshold --
# The backward runs its tasks (slabs x runs) as one-warp CTAs when they would
# give every SM at most 7, else as 8-warp CTAs.  Both sides of that switch,
# at C = 256 (1 slab) and 512 (2 slabs), against the oracle on every channel.

@pytest.mark.parametrize("slabs", [1, 2])
@pytest.mark.parametrize("side", [0, 1])
def test_backward_cta_size_threshold(cuda_device, slabs, side):
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    runs = 7 * sms // slabs + side           # tasks = slabs * runs: <= 7 * sms, then just above
    rows = 16 * runs                          # runs = ceil(rows / 16) (below the width cap)
    assert runs <= 1216 // slabs
    rng = np.random.default_rng(runs)
    lengths = [int(v) for v in rng.integers(1, 400, 200)]
    while sum(lengths) > rows - 5:
        lengths.pop()
    wl = workloads.make_custom(tuple(lengths), 256 * slabs, rows=rows, seed=runs, device=cuda_device,
                               n_minus_one=3, has_init_p=0.5)
    g = torch.Generator(device=cuda_device).manual_seed(runs)
    d_final = torch.randn((wl.n_seqs, 3, wl.C), generator=g, device=cuda_device)
    check(wl, H.run_gpu(wl, d_final=d_final), d_final=d_final)


# ------------------------------------------------------- an empty batch --
# rows == 0 (every sequence empty; the row tensors have no storage): the
# forward touches nothing, the backward's gradients are all zero -- dweight,
# dbias and the initial-state gradient of every (empty) sequence.

def test_all_empty_batch(cuda_device):
    import ssm_depthwise_causal_gb300 as ccc
    dev, C, N = cuda_device, 264, 3
    x = torch.empty((0, C), dtype=torch.bfloat16, device=dev)
    w = torch.randn((C, 4), device=dev)
    b = torch.randn((C,), device=dev)
    pool = torch.randn((5, C, 4), device=dev).to(torch.bfloat16)
    before = pool.clone()
    cu = torch.zeros(N + 1, dtype=torch.int32, device=dev)
    cache = torch.tensor([0, -1, 3], dtype=torch.int32, device=dev)
    hi = torch.ones(N, dtype=torch.uint8, device=dev)
    hist = torch.full((N, 3, C), float("nan"), device=dev).to(torch.bfloat16)
    ccc.ccc_fwd(x, w, b, pool, cu, cache, hi, torch.empty_like(x), hist)
    dw = torch.full((C, 4), float("nan"), device=dev)
    db = torch.full((C,), float("nan"), device=dev)
    di = torch.full((N, 3, C), float("nan"), device=dev)
    ccc.ccc_bwd(x, w, b, hist, cu, cache, hi, torch.empty_like(x), None, torch.empty_like(x), dw, db, di, None)
    torch.cuda.synchronize()
    assert torch.equal(pool.view(torch.int16), before.view(torch.int16))
    assert torch.isnan(hist.float()).all()
    assert (dw == 0).all() and (db == 0).all() and (di == 0).all()
