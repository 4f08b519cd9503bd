"""Pins that tie the float64 oracle to something other than itself.

Each ``check_*`` takes a loaded oracle (``oracle.Oracle``) and raises
``AssertionError`` when the oracle disagrees with:

* a library routine: ``torch.nn.functional.conv1d`` (depthwise, groups=C)
  followed by ``torch.nn.functional.silu`` in float64 for the forward, and
  torch autograd of that same composition for every gradient;
* finite differences of the oracle's own forward for dweight / dbias;
* closed forms: the impulse response of each tap and the zero-weight case;
* the contract of FlashInfer ``flashinfer.mamba.causal_conv1d_fn``
  (Parameters): the -1 sentinel, padding rows, the state positions written,
  empty sequences, has_initial_state omitted;
* the invariant of ``cake_causal_conv1d_kcp`` (description) that a fragment
  continuing a document from the previous fragment's tail reproduces the
  unsplit result.

``tests/test_oracle_pins.py`` runs them on the oracle, and
``tests/test_oracle_mutants.py`` on deliberately broken copies of it, to show
that a dropped term, a wrong sign, a wrong index or a transposed operand is
caught.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

from ssm_depthwise_causal_gb300 import workloads

F64 = torch.float64


def _bf16(values) -> torch.Tensor:
    return torch.as_tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)


def small_case(seed=1, C=8, lengths=(5, 0, 7, 2, 1, 9), rows=None, n_minus_one=1,
               has_init_p=0.5, slots=None, b_dtype=torch.float32):
    """A tiny packed batch with a pool, a -1 request, an empty sequence,
    short (<3) sequences and padding rows."""
    lengths = np.asarray(lengths)
    rows = int(lengths.sum()) + 3 if rows is None else rows
    return workloads.make_custom(lengths, C, rows=rows, seed=seed, slots=slots,
                                 n_minus_one=n_minus_one, has_init_p=has_init_p,
                                 b_dtype=b_dtype)


def _history(wl, n):
    """(init [3, C] float64, x_seq [len, C] float64, read_state) for sequence n."""
    cu = wl.cu_seqlens.tolist()
    s, e = cu[n], cu[n + 1]
    x_seq = wl.x[s:e].to(F64)
    read = bool(wl.has_initial_state[n]) if wl.has_initial_state is not None else False
    if wl.conv_state is not None and read:
        q = int(wl.cache_indices[n])
        init = wl.conv_state[q, :, 0:3].to(F64).t().contiguous()   # [3, C], pos 0 oldest
    else:
        init = torch.zeros(3, wl.C, dtype=F64)
    return init, x_seq, read


def _torch_forward(init, x_seq, w, b):
    """Library composition: depthwise conv1d over [init; x] then SiLU."""
    h = torch.cat([init, x_seq], 0).t().unsqueeze(0)            # [1, C, len+3]
    z = F.conv1d(h, w.unsqueeze(1), b, groups=w.shape[0])        # [1, C, len]
    return F.silu(z)[0].t()                                      # [len, C]


def _live(wl, n):
    return wl.cache_indices is None or int(wl.cache_indices[n]) != -1


def check_forward_matches_conv1d(orc, wl=None):
    wl = wl or small_case()
    out, _, _ = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                        wl.cache_indices, wl.has_initial_state)
    w = wl.weight.to(F64)
    b = None if wl.bias is None else wl.bias.to(F64)
    cu = wl.cu_seqlens.tolist()
    for n in range(wl.n_seqs):
        s, e = cu[n], cu[n + 1]
        if e == s:
            continue
        if not _live(wl, n):
            got = out[s:e]
            assert np.all(got == 0.0) and not np.any(np.signbit(got)), "-1 output must be +0"
            continue
        init, x_seq, _ = _history(wl, n)
        ref = _torch_forward(init, x_seq, w, b).numpy()
        np.testing.assert_allclose(out[s:e], ref, rtol=1e-12, atol=1e-14)
    assert np.all(np.isnan(out[cu[-1]:])), "padding rows must not be written"


def check_backward_matches_autograd(orc, wl=None, with_d_final=True):
    wl = wl or small_case()
    out, _, hist = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                           wl.cache_indices, wl.has_initial_state)
    gen = torch.Generator().manual_seed(7)
    d_final = torch.randn(wl.n_seqs, 3, wl.C, generator=gen, dtype=F64) if with_d_final else None
    hist_arg = hist if wl.conv_state is not None else None
    got = orc.bwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.dy, hist_arg,
                  wl.cache_indices, wl.has_initial_state, d_final)
    w = wl.weight.to(F64).clone().requires_grad_(True)
    b = None if wl.bias is None else wl.bias.to(F64).clone().requires_grad_(True)
    cu = wl.cu_seqlens.tolist()
    loss = torch.zeros((), dtype=F64)
    grads_x, grads_init = {}, {}
    for n in range(wl.n_seqs):
        s, e = cu[n], cu[n + 1]
        if e == s or not _live(wl, n):
            continue
        init, x_seq, read = _history(wl, n)
        x_seq = x_seq.clone().requires_grad_(True)
        init = init.clone().requires_grad_(read)
        y = _torch_forward(init, x_seq, w, b)
        loss = loss + (y * wl.dy[s:e].to(F64)).sum()
        if d_final is not None:
            final = torch.cat([init, x_seq], 0)[e - s:e - s + 3]     # [3, C]
            loss = loss + (final * d_final[n]).sum()
        grads_x[n] = x_seq
        grads_init[n] = (init, read)
    loss.backward()
    for n in range(wl.n_seqs):
        s, e = cu[n], cu[n + 1]
        if e == s or not _live(wl, n):
            assert np.all(got["dx"][s:e] == 0.0), "dx of a -1 request must be 0"
            assert np.all(got["d_init"][n] == 0.0), "d_init of an empty/-1 sequence must be 0"
            continue
        np.testing.assert_allclose(got["dx"][s:e], grads_x[n].grad.numpy(), rtol=1e-11, atol=1e-13)
        init, read = grads_init[n]
        ref_di = init.grad.numpy() if read else np.zeros((3, wl.C))
        np.testing.assert_allclose(got["d_init"][n], ref_di, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(got["dweight"], w.grad.numpy(), rtol=1e-11, atol=1e-12)
    if b is not None:
        np.testing.assert_allclose(got["dbias"], b.grad.numpy(), rtol=1e-11, atol=1e-12)
    assert np.all(np.isnan(got["dx"][cu[-1]:])), "dx padding rows must not be written"


def check_weight_grad_finite_difference(orc):
    """dweight/dbias from central differences of the oracle's own forward."""
    wl = small_case(seed=3, lengths=(6, 4, 8), n_minus_one=0, has_init_p=1.0)
    w = wl.weight.to(F64).numpy().copy()
    b = wl.bias.to(F64).numpy().copy()
    dy = wl.dy.to(F64).numpy()
    valid = slice(0, int(wl.cu_seqlens[-1]))

    def loss(wv, bv):
        out, _, _ = orc.fwd(wl.x, wv, bv, wl.cu_seqlens, wl.conv_state,
                            wl.cache_indices, wl.has_initial_state)
        return float((out[valid] * dy[valid]).sum())

    _, _, hist = orc.fwd(wl.x, w, b, wl.cu_seqlens, wl.conv_state, wl.cache_indices,
                         wl.has_initial_state)
    got = orc.bwd(wl.x, w, b, wl.cu_seqlens, wl.dy, hist, wl.cache_indices,
                  wl.has_initial_state, None)
    eps = 1e-6
    for c in (0, 3, 7):
        for k in range(4):
            wp, wm = w.copy(), w.copy()
            wp[c, k] += eps
            wm[c, k] -= eps
            fd = (loss(wp, b) - loss(wm, b)) / (2 * eps)
            assert abs(fd - got["dweight"][c, k]) <= 1e-6 * max(1.0, abs(fd)), (c, k, fd, got["dweight"][c, k])
        bp, bm = b.copy(), b.copy()
        bp[c] += eps
        bm[c] -= eps
        fd = (loss(w, bp) - loss(w, bm)) / (2 * eps)
        assert abs(fd - got["dbias"][c]) <= 1e-6 * max(1.0, abs(fd)), (c, fd, got["dbias"][c])


def check_impulse_response(orc):
    """x = unit impulse at row t0 of channel 3, w = e_k, no bias, no state:
    the only nonzero output is SiLU(1) at row t0 + 3 - k (tap 3 = current
    token, FlashInfer causal_conv1d_fn, weight)."""
    C, L, t0 = 8, 12, 4
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    for k in range(4):
        x = np.zeros((L, C), dtype=np.float32)
        x[t0, 3] = 1.0
        w = np.zeros((C, 4))
        w[:, k] = 1.0
        cu = torch.tensor([0, L], dtype=torch.int32)
        out, _, _ = orc.fwd(_bf16(x), w, None, cu)
        expect = np.zeros((L, C))
        expect[t0 + 3 - k, 3] = silu1
        np.testing.assert_allclose(out, expect, rtol=1e-15, atol=0.0)


def check_zero_weight(orc):
    """w = 0: every valid output is SiLU(bias) = b / (1 + e^-b); no bias: +0."""
    wl = small_case(seed=5)
    w = np.zeros((wl.C, 4))
    b = wl.bias.to(F64).numpy()
    out, _, _ = orc.fwd(wl.x, w, b, wl.cu_seqlens, wl.conv_state, wl.cache_indices,
                        wl.has_initial_state)
    cu = wl.cu_seqlens.tolist()
    expect = b / (1.0 + np.exp(-b))
    for n in range(wl.n_seqs):
        s, e = cu[n], cu[n + 1]
        ref = np.broadcast_to(expect, (e - s, wl.C)) if _live(wl, n) else np.zeros((e - s, wl.C))
        np.testing.assert_allclose(out[s:e], ref, rtol=1e-15, atol=0.0)
    out0, _, _ = orc.fwd(wl.x, w, None, wl.cu_seqlens)
    assert np.all(out0[: cu[-1]] == 0.0)


def check_state_rules(orc):
    """Bit-exact state contract of causal_conv1d_fn (conv_state, cu_seqlens,
    cache_indices, has_initial_state)."""
    wl = small_case(seed=11, lengths=(7, 0, 2, 1, 5, 3), n_minus_one=1, slots=10)
    before = wl.conv_state.view(torch.int16).numpy().view(np.uint16).copy()
    _, st, hist = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                          wl.cache_indices, wl.has_initial_state)
    xb = wl.x.view(torch.int16).numpy().view(np.uint16)
    cu = wl.cu_seqlens.tolist()
    cache = wl.cache_indices.tolist()
    hi = wl.has_initial_state.tolist()
    touched = set()
    for n in range(wl.n_seqs):
        s, e = cu[n], cu[n + 1]
        L = e - s
        q = cache[n]
        if q == -1 or L == 0:
            continue
        touched.add(q)
        init = before[q, :, 0:3].T if hi[n] else np.zeros((3, wl.C), np.uint16)   # [3, C]
        np.testing.assert_array_equal(hist[n], init)
        full = np.concatenate([init, xb[s:e]], 0)                 # [L+3, C]
        np.testing.assert_array_equal(st[q, :, 0:3].T, full[L:L + 3])
        if L >= 3:
            np.testing.assert_array_equal(st[q, :, 0:3].T, xb[e - 3:e])
        np.testing.assert_array_equal(st[q, :, 3:], before[q, :, 3:])
    for q in range(before.shape[0]):
        if q not in touched:
            np.testing.assert_array_equal(st[q], before[q])
    # has_initial_state omitted == all false
    o1, _, _ = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                       wl.cache_indices, None)
    o2, _, _ = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                       wl.cache_indices, torch.zeros(wl.n_seqs, dtype=torch.bool))
    np.testing.assert_array_equal(o1, o2)


def check_split_invariance(orc, cuts=(1, 2, 3, 5, 12), L=23, C=8):
    """A document processed as two fragments, the second starting from the
    first's written state (and the first's backward seeded with the second's
    d_init), reproduces the unsplit result (cake_causal_conv1d_kcp)."""
    wl = workloads.make_custom([L], C, seed=13, slots=1, has_init_p=1.0)
    cache = torch.tensor([0], dtype=torch.int32)
    yes = torch.tensor([True])
    gen = torch.Generator().manual_seed(2)
    d_last = torch.randn(1, 3, C, generator=gen, dtype=F64)
    out_u, st_u, hist_u = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                                  cache, yes)
    g_u = orc.bwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.dy, hist_u, cache, yes, d_last)
    for r in cuts:
        xa, xb = wl.x[:r], wl.x[r:]
        cua = torch.tensor([0, r], dtype=torch.int32)
        cub = torch.tensor([0, L - r], dtype=torch.int32)
        out_a, st_a, hist_a = orc.fwd(xa, wl.weight, wl.bias, cua, wl.conv_state, cache, yes)
        out_b, st_b, hist_b = orc.fwd(xb, wl.weight, wl.bias, cub,
                                      torch.from_numpy(st_a.view(np.int16)).view(torch.bfloat16),
                                      cache, yes)
        np.testing.assert_array_equal(np.concatenate([out_a, out_b]), out_u)
        np.testing.assert_array_equal(st_b, st_u)
        g_b = orc.bwd(xb, wl.weight, wl.bias, cub, wl.dy[r:], hist_b, cache, yes, d_last)
        g_a = orc.bwd(xa, wl.weight, wl.bias, cua, wl.dy[:r], hist_a, cache, yes,
                      g_b["d_init"])
        np.testing.assert_array_equal(np.concatenate([g_a["dx"], g_b["dx"]]), g_u["dx"])
        np.testing.assert_array_equal(g_a["d_init"], g_u["d_init"])
        np.testing.assert_allclose(g_a["dweight"] + g_b["dweight"], g_u["dweight"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(g_a["dbias"] + g_b["dbias"], g_u["dbias"], rtol=1e-12, atol=1e-14)


ALL_CHECKS = [
    check_forward_matches_conv1d,
    check_backward_matches_autograd,
    check_weight_grad_finite_difference,
    check_impulse_response,
    check_zero_weight,
    check_state_rules,
    check_split_invariance,
]
