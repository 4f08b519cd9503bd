"""Pins that tie the float64 oracle to something other than itself.

Each ``check_*`` takes a loaded oracle (``oracle.Oracle``) and raises
``AssertionError`` when the oracle disagrees with:

* a library routine: ``torch.nn.functional.conv1d`` (depthwise, groups=C)
  followed by ``torch.nn.functional.silu`` (or nothing, for the
  no-activation variant) in float64 for the forward, and torch autograd of
  that same composition for every gradient, at widths W = 2, 3, 4;
* finite differences of the oracle's own forward for dweight / dbias;
* closed forms: the impulse response of each tap and the zero-weight case;
* the contract of FlashInfer ``flashinfer.mamba.causal_conv1d_fn``
  (Parameters): the -1 sentinel, padding rows, the state positions written,
  empty sequences, has_initial_state omitted;
* the invariant of ``cake_causal_conv1d_kcp`` (description) that a fragment
  continuing a document from the previous fragment's tail reproduces the
  unsplit result;
* for the speculative state update: decoding a document token by token, or
  in speculative steps of which only a prefix is kept, gives for every kept
  token the output of torch conv1d over the whole kept stream.

``tests/test_oracle_pins.py`` runs them on the oracle, and
``tests/test_oracle_mutants.py`` on deliberately broken copies of it, to show
that a dropped term, a wrong sign, a wrong index or a transposed operand is
caught.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch
import torch.nn.functional as F

from ssm_depthwise_causal_gb300 import workloads

F64 = torch.float64


def _bf16(values) -> torch.Tensor:
    return torch.as_tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)


def _u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def small_case(seed=1, C=8, lengths=(5, 0, 7, 2, 1, 9), rows=None, n_minus_one=1,
               has_init_p=0.5, slots=None, b_dtype=torch.float32, width=4, activation="silu"):
    """A tiny packed batch with a pool, a -1 request, an empty sequence,
    short (< W-1) sequences and padding rows."""
    lengths = np.asarray(lengths)
    rows = int(lengths.sum()) + 3 if rows is None else rows
    return workloads.make_custom(lengths, C, rows=rows, seed=seed, slots=slots,
                                 n_minus_one=n_minus_one, has_init_p=has_init_p,
                                 b_dtype=b_dtype, width=width, activation=activation)


def _history(wl, n):
    """(init [H, C] float64, x_seq [len, C] float64, read_state) for sequence n."""
    H = wl.width - 1
    cu = wl.cu_seqlens.tolist()
    s, e = cu[n], cu[n + 1]
    x_seq = wl.x[s:e].to(F64)
    read = bool(wl.has_initial_state[n]) if wl.has_initial_state is not None else False
    if wl.conv_state is not None and read:
        q = int(wl.cache_indices[n])
        init = wl.conv_state[q, :, 0:H].to(F64).t().contiguous()   # [H, C], pos 0 oldest
    else:
        init = torch.zeros(H, wl.C, dtype=F64)
    return init, x_seq, read


def _torch_forward(init, x_seq, w, b, activation="silu"):
    """Library composition: depthwise conv1d over [init; x] then SiLU (or
    nothing)."""
    h = torch.cat([init, x_seq], 0).t().unsqueeze(0)            # [1, C, len+H]
    z = F.conv1d(h, w.unsqueeze(1), b, groups=w.shape[0])        # [1, C, len]
    y = F.silu(z) if activation else z
    return y[0].t()                                              # [len, C]


def _live(wl, n):
    return wl.cache_indices is None or int(wl.cache_indices[n]) != -1


def check_forward_matches_conv1d(orc, wl=None):
    wl = wl or small_case()
    out, _, _ = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                        wl.cache_indices, wl.has_initial_state, activation=wl.activation)
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
        ref = _torch_forward(init, x_seq, w, b, wl.activation).numpy()
        np.testing.assert_allclose(out[s:e], ref, rtol=1e-12, atol=1e-14)
    assert np.all(np.isnan(out[cu[-1]:])), "padding rows must not be written"


def check_backward_matches_autograd(orc, wl=None, with_d_final=True):
    wl = wl or small_case()
    H = wl.width - 1
    out, _, hist = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                           wl.cache_indices, wl.has_initial_state, activation=wl.activation)
    gen = torch.Generator().manual_seed(7)
    d_final = torch.randn(wl.n_seqs, H, wl.C, generator=gen, dtype=F64) if with_d_final else None
    hist_arg = hist if wl.conv_state is not None else None
    got = orc.bwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.dy, hist_arg,
                  wl.cache_indices, wl.has_initial_state, d_final, activation=wl.activation)
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
        y = _torch_forward(init, x_seq, w, b, wl.activation)
        loss = loss + (y * wl.dy[s:e].to(F64)).sum()
        if d_final is not None:
            final = torch.cat([init, x_seq], 0)[e - s:e - s + H]     # [H, C]
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
        ref_di = init.grad.numpy() if read else np.zeros((H, wl.C))
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
    the only nonzero output is SiLU(1) (or 1 without activation) at row
    t0 + W-1 - k (tap W-1 = current token, FlashInfer causal_conv1d_fn,
    weight), for every width W = 2, 3, 4."""
    C, L, t0 = 8, 12, 4
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    for W in (2, 3, 4):
        for act, peak in (("silu", silu1), (None, 1.0)):
            for k in range(W):
                x = np.zeros((L, C), dtype=np.float32)
                x[t0, 3] = 1.0
                w = np.zeros((C, W))
                w[:, k] = 1.0
                cu = torch.tensor([0, L], dtype=torch.int32)
                out, _, _ = orc.fwd(_bf16(x), w, None, cu, activation=act)
                expect = np.zeros((L, C))
                expect[t0 + W - 1 - k, 3] = peak
                np.testing.assert_allclose(out, expect, rtol=1e-15, atol=0.0, err_msg=f"W={W} k={k} {act}")


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


def check_state_rules(orc, width=4):
    """Bit-exact state contract of causal_conv1d_fn (conv_state, cu_seqlens,
    cache_indices, has_initial_state), with W-1 carried values."""
    H = width - 1
    wl = small_case(seed=11, lengths=(7, 0, 2, 1, 5, 3), n_minus_one=1, slots=10, width=width)
    before = _u16(wl.conv_state).copy()
    _, st, hist = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                          wl.cache_indices, wl.has_initial_state)
    xb = _u16(wl.x)
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
        init = before[q, :, 0:H].T if hi[n] else np.zeros((H, wl.C), np.uint16)   # [H, C]
        np.testing.assert_array_equal(hist[n], init)
        full = np.concatenate([init, xb[s:e]], 0)                 # [L+H, C]
        np.testing.assert_array_equal(st[q, :, 0:H].T, full[L:L + H])
        if L >= H:
            np.testing.assert_array_equal(st[q, :, 0:H].T, xb[e - H:e])
        np.testing.assert_array_equal(st[q, :, H:], before[q, :, H:])
    for q in range(before.shape[0]):
        if q not in touched:
            np.testing.assert_array_equal(st[q], before[q])
    # has_initial_state omitted == all false
    o1, _, _ = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                       wl.cache_indices, None)
    o2, _, _ = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                       wl.cache_indices, torch.zeros(wl.n_seqs, dtype=torch.bool))
    np.testing.assert_array_equal(o1, o2)


def check_split_invariance(orc, cuts=(1, 2, 3, 5, 12), L=23, C=8, width=4, activation="silu"):
    """A document processed as two fragments, the second starting from the
    first's written state (and the first's backward seeded with the second's
    d_init), reproduces the unsplit result (cake_causal_conv1d_kcp)."""
    H = width - 1
    wl = workloads.make_custom([L], C, seed=13, slots=1, has_init_p=1.0, width=width)
    cache = torch.tensor([0], dtype=torch.int32)
    yes = torch.tensor([True])
    gen = torch.Generator().manual_seed(2)
    d_last = torch.randn(1, H, C, generator=gen, dtype=F64)
    act = dict(activation=activation)
    out_u, st_u, hist_u = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                                  cache, yes, **act)
    g_u = orc.bwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.dy, hist_u, cache, yes, d_last, **act)
    for r in cuts:
        xa, xb = wl.x[:r], wl.x[r:]
        cua = torch.tensor([0, r], dtype=torch.int32)
        cub = torch.tensor([0, L - r], dtype=torch.int32)
        out_a, st_a, hist_a = orc.fwd(xa, wl.weight, wl.bias, cua, wl.conv_state, cache, yes, **act)
        out_b, st_b, hist_b = orc.fwd(xb, wl.weight, wl.bias, cub,
                                      torch.from_numpy(st_a.view(np.int16)).view(torch.bfloat16),
                                      cache, yes, **act)
        np.testing.assert_array_equal(np.concatenate([out_a, out_b]), out_u)
        np.testing.assert_array_equal(st_b, st_u)
        g_b = orc.bwd(xb, wl.weight, wl.bias, cub, wl.dy[r:], hist_b, cache, yes, d_last, **act)
        g_a = orc.bwd(xa, wl.weight, wl.bias, cua, wl.dy[:r], hist_a, cache, yes,
                      g_b["d_init"], **act)
        np.testing.assert_array_equal(np.concatenate([g_a["dx"], g_b["dx"]]), g_u["dx"])
        np.testing.assert_array_equal(g_a["d_init"], g_u["d_init"])
        np.testing.assert_allclose(g_a["dweight"] + g_b["dweight"], g_u["dweight"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(g_a["dbias"] + g_b["dbias"], g_u["dbias"], rtol=1e-12, atol=1e-14)


def check_variants_match_torch(orc):
    """Widths 2 and 3 and the no-activation variant (Megatron-Core
    causal_conv1d_cp: weight [D, W], activation optional) against torch
    conv1d / autograd, and their state and split rules."""
    for W in (2, 3, 4):
        for act in ("silu", None):
            if W == 4 and act == "silu":
                continue  # the main pins
            wl = small_case(seed=30 + W, lengths=(5, 0, 7, 1, 2, 9), width=W, activation=act)
            check_forward_matches_conv1d(orc, wl)
            check_backward_matches_autograd(orc, wl)
        check_state_rules(orc, width=W)
        check_split_invariance(orc, cuts=(1, 2, 7), L=17, width=W, activation=None if W == 3 else "silu")


# ----------------------------------------------------- speculative update --

def _stream_case(seed, C, n_live, T, width, slots, L):
    """True token streams [n_live][T, C] (BF16 values), the taps, a bias, an
    initial pool and distinct slots."""
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    streams = [_bf16(rng.standard_normal((T, C))) for _ in range(n_live)]
    w = (torch.rand((C, width), generator=g, dtype=F64) - 0.5)
    b = torch.randn(C, generator=g, dtype=F64) * 0.1
    pool = _bf16(rng.standard_normal((slots, C, L)))
    slot_ids = rng.permutation(slots)[:n_live + 1].astype(np.int32)
    return rng, streams, w, b, pool, slot_ids


def _pack(chunks, C):
    lengths = [c.shape[0] for c in chunks]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    x = torch.cat(chunks, 0) if sum(lengths) else torch.zeros((0, C), dtype=torch.bfloat16)
    return x, cu


def check_update_decode_chain(orc, width=4, activation="silu"):
    """Prefill a prefix of each stream, then decode the rest one token per
    step with accepted count 1 (causal_conv1d_fn, Notes): every output equals
    torch conv1d over the whole stream from the initial state, and the state
    ends as the last W-1 tokens."""
    H = width - 1
    C, T, L = 8, 12, H + 2
    rng, streams, w, b, pool, slot_ids = _stream_case(41, C, 3, T, width, 6, L)
    prefix = [4, 1, 0]
    cache = torch.tensor(slot_ids[:3])
    init = [pool[q, :, 0:H].to(F64).t() for q in slot_ids[:3]]
    refs = [_torch_forward(init[i], streams[i].to(F64), w, b, activation).numpy() for i in range(3)]
    before = _u16(pool).copy()
    x, cu = _pack([streams[i][:prefix[i]] for i in range(3)], C)
    out, st, _ = orc.fwd(x, w, b, cu, pool, cache, torch.tensor([True] * 3), activation=activation)
    for i in range(3):
        np.testing.assert_allclose(out[int(cu[i]):int(cu[i + 1])], refs[i][:prefix[i]], rtol=1e-12, atol=1e-14)
    state = torch.from_numpy(st.view(np.int16)).view(torch.bfloat16)
    for t in range(T):
        chunks = [streams[i][t:t + 1] if t >= prefix[i] else streams[i][:0] for i in range(3)]
        x, cu = _pack(chunks, C)
        out, st = orc.update(x, w, b, cu, state, cache, None, activation=activation)
        for i in range(3):
            if t >= prefix[i]:
                np.testing.assert_allclose(out[int(cu[i])], refs[i][t], rtol=1e-12, atol=1e-14,
                                           err_msg=f"stream {i} token {t}")
        state = torch.from_numpy(st.view(np.int16)).view(torch.bfloat16)
    final = _u16(state)
    for i, q in enumerate(slot_ids[:3]):
        np.testing.assert_array_equal(final[q, :, 0:H].T, _u16(streams[i])[T - H:T])
    for q in range(pool.shape[0]):
        if q not in slot_ids[:3]:
            np.testing.assert_array_equal(final[q], before[q])


def check_update_speculative_chain(orc, width=4, activation="silu"):
    """Speculative steps: each live sequence feeds k drafts whose first m are
    the stream's next tokens and the rest junk; the next step brings accepted
    count m.  Every kept output equals torch conv1d over the kept stream;
    a -1 request writes zeros and leaves its slot alone; a step with no token
    leaves the slot alone (and the accepted count stands); positions at and
    past k + W-2 are never written."""
    H = width - 1
    C, T, kmax = 8, 48, 5
    L = kmax + H + 1
    rng, streams, w, b, pool, slot_ids = _stream_case(43, C, 3, T, width, 8, L)
    cache = torch.tensor(slot_ids)          # 3 live slots, then a -1 request
    cache[3] = -1
    init = [pool[q, :, 0:H].to(F64).t() for q in slot_ids[:3]]
    refs = [_torch_forward(init[i], streams[i].to(F64), w, b, activation).numpy() for i in range(3)]
    state = pool.clone()
    pos = [0, 0, 0]
    acc = [1, 1, 1, 1]
    saw_full = saw_partial = saw_empty = False
    for step in range(14):
        chunks, keep = [], []
        for i in range(3):
            k = int(rng.integers(0 if i == 2 else 1, kmax + 1))
            k = min(k, T - pos[i])
            m = int(rng.integers(1, k + 1)) if k > 0 else 0
            junk = _bf16(rng.standard_normal((k - m, C)) * 3.0)
            chunks.append(torch.cat([streams[i][pos[i]:pos[i] + m], junk], 0))
            keep.append((k, m))
            saw_full |= k > 0 and m == k
            saw_partial |= 0 < m < k
            saw_empty |= k == 0
        chunks.append(_bf16(rng.standard_normal((int(rng.integers(0, 3)), C))))
        x, cu = _pack(chunks, C)
        before = _u16(state).copy()
        out, st = orc.update(x, w, b, cu, state, cache, torch.tensor(acc, dtype=torch.int32),
                             activation=activation)
        for i in range(3):
            k, m = keep[i]
            s = int(cu[i])
            q = slot_ids[i]
            if k == 0:
                np.testing.assert_array_equal(st[q], before[q])
                continue
            np.testing.assert_allclose(out[s:s + m], refs[i][pos[i]:pos[i] + m], rtol=1e-12, atol=1e-14,
                                       err_msg=f"step {step} stream {i}")
            np.testing.assert_array_equal(st[q, :, k + H - 1:], before[q, :, k + H - 1:])
            pos[i] += m
            acc[i] = m
        s3, e3 = int(cu[3]), int(cu[4])
        assert np.all(out[s3:e3] == 0.0) and not np.any(np.signbit(out[s3:e3]))
        untouched = [q for q in range(pool.shape[0]) if q not in slot_ids[:3]]
        np.testing.assert_array_equal(st[untouched], before[untouched])
        state = torch.from_numpy(st.view(np.int16)).view(torch.bfloat16)
    assert saw_full and saw_partial and saw_empty


def check_update_special_cases(orc):
    """One token with accepted count 1 is a one-token prefill from the state
    (same output, same positions 0:W-1); more tokens leave h[p+1] at position
    p for p < len + W-2."""
    for W in (2, 3, 4):
        H = W - 1
        wl = small_case(seed=50 + W, lengths=(1, 1, 4, 2), n_minus_one=0, slots=6, has_init_p=1.0,
                        width=W)
        wl = dataclasses.replace(wl, conv_state=_bf16(np.random.default_rng(W).standard_normal((6, wl.C, 8))))
        cu = wl.cu_seqlens
        one = torch.tensor([0, 1, 2], dtype=torch.int32)
        out_p, st_p, _ = orc.fwd(wl.x[:2], wl.weight, wl.bias, one, wl.conv_state, wl.cache_indices[:2],
                                 torch.tensor([True, True]))
        out_u, st_u = orc.update(wl.x[:2], wl.weight, wl.bias, one, wl.conv_state, wl.cache_indices[:2])
        np.testing.assert_array_equal(out_u, out_p)
        for q in wl.cache_indices[:2].tolist():
            np.testing.assert_array_equal(st_u[q, :, 0:H], st_p[q, :, 0:H])
        # the write rule on longer steps, with accepted counts > 1
        before = _u16(wl.conv_state)
        accepted = torch.tensor([1, 2, 3, 2], dtype=torch.int32)
        _, st = orc.update(wl.x, wl.weight, wl.bias, cu, wl.conv_state, wl.cache_indices, accepted)
        xb = _u16(wl.x)
        for n, q in enumerate(wl.cache_indices.tolist()):
            s, e = int(cu[n]), int(cu[n + 1])
            a = int(accepted[n])
            h = np.concatenate([before[q, :, a - 1:a - 1 + H].T, xb[s:e]], 0)     # [H+len, C]
            n_w = (e - s) + H - 1
            np.testing.assert_array_equal(st[q, :, :n_w].T, h[1:1 + n_w])
            np.testing.assert_array_equal(st[q, :, n_w:], before[q, :, n_w:])


def check_update_impulse(orc):
    """Closed form of the decode step's read offset and tap order: with the
    taps one-hot at k (no bias, no activation), token j of a request with
    accepted count a outputs history value h[j + k] exactly, where h is the
    slot's positions a-1 .. a+W-3 followed by the request's tokens -- so a
    wrong read offset, a reversed tap order or a dropped chaining of the
    step's own tokens changes the output."""
    L = 8
    for W in (2, 3, 4):
        H = W - 1
        wl = small_case(seed=70 + W, lengths=(1, 3, 4, 2, 0, 5), n_minus_one=0, slots=9, has_init_p=1.0,
                        width=W)
        pool = _bf16(np.random.default_rng(70 + W).standard_normal((9, wl.C, L)))
        cu = wl.cu_seqlens
        N = len(cu) - 1
        accepted = torch.tensor([1 + (n % (L - W + 2)) for n in range(N)], dtype=torch.int32)
        xb = oracle_values(wl.x)
        pv = oracle_values(pool)
        for k in range(W):
            w = torch.zeros((wl.C, W), dtype=torch.float32)
            w[:, k] = 1.0
            out, _ = orc.update(wl.x, w, None, cu, pool, wl.cache_indices, accepted, activation=None)
            for n, q in enumerate(wl.cache_indices.tolist()):
                s, e = int(cu[n]), int(cu[n + 1])
                a = int(accepted[n])
                h = np.concatenate([pv[q, :, a - 1:a - 1 + H].T, xb[s:e]], 0)
                for j in range(e - s):
                    np.testing.assert_array_equal(out[s + j], h[j + k], err_msg=f"W={W} k={k} seq {n} token {j}")


def oracle_values(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a BF16 tensor (the top 16 bits of an FP32)."""
    u = _u16(t).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def check_update_variants(orc):
    """The decode and speculative chains at widths 2 and 3 and without
    activation."""
    for W, act in ((2, "silu"), (3, None), (4, None)):
        check_update_decode_chain(orc, width=W, activation=act)
        check_update_speculative_chain(orc, width=W, activation=act)



# ------------------------------------------------ -1 without a pool --

def check_minus_one_without_pool(orc):
    """cache_indices given without a pool (FlashInfer causal_conv1d_fn,
    cache_indices: the -1 sentinel gives a zero output and touches no state):
    the -1 requests output +0 and contribute nothing to dx, dweight or dbias;
    every other request is conv1d from zero history (no pool to read)."""
    for W, act in ((4, "silu"), (3, None), (2, "silu")):
        wl = small_case(seed=60 + W, lengths=(6, 4, 0, 9, 3, 2), n_minus_one=2, width=W, activation=act)
        wl = dataclasses.replace(wl, conv_state=None, has_initial_state=None)
        assert (wl.cache_indices == -1).sum() == 2
        check_forward_matches_conv1d(orc, wl)
        check_backward_matches_autograd(orc, wl)


# ------------------------------------------------------- brute force --

def _silu(z):
    """SiLU(z) = z * sigma(z), sigma(z) = 1 / (1 + e^-z)."""
    return z * (1.0 / (1.0 + math.exp(-z)))


def _silu_grad(z):
    """d/dz [z * sigma(z)] = sigma(z) * (1 + z * (1 - sigma(z)))."""
    sg = 1.0 / (1.0 + math.exp(-z))
    return sg * (1.0 + z * (1.0 - sg))


def brute_force(x, w, b, cu, pool=None, cache=None, has_init=None, dy=None, d_final=None,
                activation="silu"):
    """The method written out as Python float loops (no numpy or torch
    arithmetic), one sequence and one channel at a time, straight from the
    definition (FlashInfer causal_conv1d_fn, Parameters; cake_causal_conv1d_kcp,
    Returns):

    * the history is a Python list: W-1 initial values (pool positions
      0..W-2 of the request's slot when has_init, zeros otherwise), then the
      sequence's inputs;
    * z_j = b + w_0 h[j] + ... + w_{W-1} h[j+W-1] (bias first), y_j = SiLU(z_j);
    * the pool slot receives the history list's last W-1 entries;
    * dH = dL/dh by the chain rule, scattered from every token: z_j adds
      w_k dz_j to dH[j+k], and the final-state gradient d_final[p] lands on
      h[len+p] (the value written to position p);
    * dx = dH[W-1:], d_init = dH[:W-1] when the state was read (else 0),
      dweight[c][k] = sum dz_j h[j+k], dbias[c] = sum dz_j.

    Inputs are nested Python lists of floats (x [rows][C], w [C][W], b [C] or
    None, pool [slots][C][L], dy [rows][C], d_final [N][W-1][C]).  Returns a
    dict of nested lists, plus for every floating output the sum of the
    absolute values of the terms that formed it ("*_mag"), the scale of its
    rounding error."""
    rows, C = len(x), len(x[0])
    W = len(w[0])
    H = W - 1
    N = len(cu) - 1
    act = activation is not None
    out = [[None] * C for _ in range(rows)]
    out_mag = [[None] * C for _ in range(rows)]
    new_pool = None if pool is None else [[list(p) for p in slot] for slot in pool]
    hist = [[[None] * C for _ in range(H)] for _ in range(N)]
    res = dict(out=out, out_mag=out_mag, pool=new_pool, hist=hist)
    if dy is not None:
        dx = [[None] * C for _ in range(rows)]
        dx_mag = [[None] * C for _ in range(rows)]
        d_init = [[[0.0] * C for _ in range(H)] for _ in range(N)]
        d_init_mag = [[[0.0] * C for _ in range(H)] for _ in range(N)]
        dweight = [[0.0] * W for _ in range(C)]
        dweight_mag = [[0.0] * W for _ in range(C)]
        dbias = [0.0] * C
        dbias_mag = [0.0] * C
        res.update(dx=dx, dx_mag=dx_mag, d_init=d_init, d_init_mag=d_init_mag, dweight=dweight,
                   dweight_mag=dweight_mag, dbias=dbias, dbias_mag=dbias_mag)
    for n in range(N):
        s, e = cu[n], cu[n + 1]
        L = e - s
        q = None if cache is None else cache[n]
        if q == -1:                      # zero output, no state access, zero gradient
            for j in range(L):
                for c in range(C):
                    out[s + j][c] = 0.0
                    out_mag[s + j][c] = 0.0
                    if dy is not None:
                        dx[s + j][c] = 0.0
                        dx_mag[s + j][c] = 0.0
            if L > 0:
                for i in range(H):
                    hist[n][i] = [0.0] * C
            continue
        read = pool is not None and has_init is not None and bool(has_init[n])
        for c in range(C):
            init = [pool[q][c][i] for i in range(H)] if read else [0.0] * H
            h = init + [x[s + j][c] for j in range(L)]
            if L > 0:
                for i in range(H):
                    hist[n][i][c] = h[i]
            bias = 0.0 if b is None else b[c]
            z = []
            for j in range(L):
                acc, mag = bias, abs(bias)
                for k in range(W):
                    acc += w[c][k] * h[j + k]
                    mag += abs(w[c][k] * h[j + k])
                z.append(acc)
                out[s + j][c] = _silu(acc) if act else acc
                out_mag[s + j][c] = mag
            if new_pool is not None and L > 0:
                new_pool[q][c][0:H] = h[L:L + H]
            if dy is None:
                continue
            dz = [(_silu_grad(z[j]) if act else 1.0) * dy[s + j][c] for j in range(L)]
            dH = [0.0] * (L + H)
            dH_mag = [0.0] * (L + H)
            if d_final is not None:
                for p in range(H):
                    dH[L + p] += d_final[n][p][c]
                    dH_mag[L + p] += abs(d_final[n][p][c])
            for j in range(L):
                for k in range(W):
                    dH[j + k] += w[c][k] * dz[j]
                    dH_mag[j + k] += abs(w[c][k] * dz[j])
            for i in range(L + H):
                if i >= H:
                    dx[s + i - H][c] = dH[i]
                    dx_mag[s + i - H][c] = dH_mag[i]
                elif read and L > 0:
                    d_init[n][i][c] = dH[i]
                    d_init_mag[n][i][c] = dH_mag[i]
            for j in range(L):
                for k in range(W):
                    dweight[c][k] += dz[j] * h[j + k]
                    dweight_mag[c][k] += abs(dz[j] * h[j + k])
                dbias[c] += dz[j]
                dbias_mag[c] += abs(dz[j])
    return res


def _close_to_brute(got, want, mag, what, rel=1e-15):
    """|oracle - brute force| <= rel * (sum of |terms|), element by element,
    over the elements the brute force defines (None = not written)."""
    got = np.asarray(got, dtype=np.float64)
    for idx in np.ndindex(*got.shape):
        wv = want
        mv = mag
        for i in idx:
            wv = wv[i]
            mv = mv[i]
        if wv is None:
            assert np.isnan(got[idx]), f"{what}{idx}: written, but the method leaves it alone"
            continue
        assert abs(got[idx] - wv) <= rel * mv, f"{what}{idx}: oracle {got[idx]!r} brute force {wv!r}"
        if wv == 0.0 and mv == 0.0:
            assert not math.copysign(1.0, got[idx]) < 0, f"{what}{idx}: -0 where +0 is due"


def check_brute_force_direct_summation(orc):
    """The oracle against the brute force above on tiny batches (up to 4
    sequences of 0 to 6 tokens, C = 8) at every width, with and without
    SiLU, with a pool, a -1 request, has_initial_state flags and a
    final-state gradient, and without a pool (-1 requests still zero):
    values within 1e-15 of the scale of their terms, the pool and the
    saved history bit for bit."""
    cases = [
        # lengths, width, activation, with pool, -1 requests
        ((5, 0, 6, 2), 4, "silu", True, 1),
        ((1, 3, 6, 4), 4, None, True, 1),
        ((6, 2, 0, 5), 3, "silu", True, 1),
        ((4, 6, 1), 3, None, True, 0),
        ((2, 5, 6, 0), 2, "silu", True, 1),
        ((6, 1, 3), 2, None, True, 1),
        ((3, 6, 0, 4), 4, "silu", False, 1),
        ((6, 5), 3, "silu", False, 0),
    ]
    for t, (lengths, W, act, with_pool, m1) in enumerate(cases):
        wl = small_case(seed=90 + t, C=8, lengths=lengths, n_minus_one=m1, has_init_p=0.6, width=W,
                        activation=act, slots=6)
        if not with_pool:
            wl = dataclasses.replace(wl, conv_state=None, has_initial_state=None)
        H = W - 1
        gen = torch.Generator().manual_seed(100 + t)
        d_final = torch.randn(wl.n_seqs, H, wl.C, generator=gen, dtype=F64)
        vals = lambda a: None if a is None else oracle_values(a).tolist()  # noqa: E731
        ci = None if wl.cache_indices is None else [int(v) for v in wl.cache_indices]
        hi = None if wl.has_initial_state is None else [bool(v) for v in wl.has_initial_state]
        bf = brute_force(vals(wl.x), wl.weight.double().tolist(),
                         None if wl.bias is None else wl.bias.double().tolist(),
                         [int(v) for v in wl.cu_seqlens], vals(wl.conv_state), ci, hi,
                         vals(wl.dy), d_final.tolist(), act)
        out, st, hist = orc.fwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.conv_state,
                                wl.cache_indices, wl.has_initial_state, activation=act)
        tag = f"case {t} (W={W}, {act}, pool={with_pool}): "
        _close_to_brute(out, bf["out"], bf["out_mag"], tag + "out")
        if with_pool:
            np.testing.assert_array_equal(oracle_values_bits(st), np.asarray(bf["pool"]), err_msg=tag + "pool")
        lens = np.diff(wl.cu_seqlens.numpy())
        for n in range(wl.n_seqs):
            if lens[n] > 0:
                np.testing.assert_array_equal(oracle_values_bits(hist[n]), np.asarray(bf["hist"][n]),
                                              err_msg=tag + f"saved history {n}")
        g = orc.bwd(wl.x, wl.weight, wl.bias, wl.cu_seqlens, wl.dy, hist if with_pool else None,
                    wl.cache_indices, wl.has_initial_state, d_final, activation=act)
        _close_to_brute(g["dx"], bf["dx"], bf["dx_mag"], tag + "dx")
        _close_to_brute(g["d_init"], bf["d_init"], bf["d_init_mag"], tag + "d_init")
        _close_to_brute(g["dweight"], bf["dweight"], bf["dweight_mag"], tag + "dweight")
        if wl.bias is not None:
            _close_to_brute(g["dbias"], bf["dbias"], bf["dbias_mag"], tag + "dbias")


def oracle_values_bits(bits: np.ndarray) -> np.ndarray:
    """Exact float64 values of BF16 bit patterns (uint16 arrays)."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


ALL_CHECKS = [
    check_forward_matches_conv1d,
    check_backward_matches_autograd,
    check_weight_grad_finite_difference,
    check_impulse_response,
    check_zero_weight,
    check_state_rules,
    check_split_invariance,
    check_variants_match_torch,
    check_update_decode_chain,
    check_update_speculative_chain,
    check_update_special_cases,
    check_update_impulse,
    check_update_variants,
    check_minus_one_without_pool,
    check_brute_force_direct_summation,
]
