"""GB300-native packed depthwise causal Conv1d (+ SiLU): width 4 (and 2, 3).

This package is a thin binding over ``libccc.so`` (C ABI in ``include/ccc.h``):
every function marshals torch tensors into pointers, sizes and strides and
calls the library on the current CUDA stream.  All arithmetic runs in the
library's CUDA kernels; there is no Python or CPU fallback, and importing the
package fails loudly when the library has not been built
(``python -c "import __graft_entry__ as g; g.build()"``).

Entry points (same names as the C ABI):

* ``ccc_workspace_size(rows, n_seqs, channels, for_bwd)``
* ``ccc_fwd(...)``  -- forward + in-place conv_state update
  (FlashInfer ``flashinfer.mamba.causal_conv1d_fn``)
* ``ccc_bwd(...)``  -- one-pass dx, with FP32 dweight/dbias summed in a fixed order
  (``cake_causal_conv1d_kcp``, Returns)
* ``ccc_update(...)`` -- speculative / single-token decode step on the pool
* ``ccc_bwd_noalloc(...)`` -- ``ccc_bwd`` on the library's own scratch

``ccc_fwd``, ``ccc_bwd`` and ``ccc_update`` take ``overlap=True`` to call
``ccc_fwd_ex`` / ``ccc_bwd_ex`` / ``ccc_update_ex`` with
``CCC_OPT_OVERLAP_PROLOGUE`` (the kernel's prologue may overlap the kernel
before it; the contract is in ``include/ccc.h``).

The width W is the second dimension of ``weight`` ([C, W], W in 2..4) and
``activation`` is ``"silu"`` (default) or ``None`` (Megatron-Core
``core.ssm.causal_conv1d``, causal_conv1d_cp).  On top: the allocating
conveniences ``causal_conv1d_fn`` / ``causal_conv1d_bwd`` /
``causal_conv1d_update``, which create outputs and the workspace when they
are not given and accept ``[B, T, D]`` (non-packed) input as well as packed
``[rows, C]``; ``recompute_fwd`` (bitwise re-run of a forward from its saved
history) and the autograd wrapper ``causal_conv1d`` / ``CausalConv1dFn``.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib

CCC_F32, CCC_BF16, CCC_NONE = 0, 1, -1
CCC_ACT_NONE, CCC_ACT_SILU = 0, 1
# Status bits of ccc_check (include/ccc.h).
CHECK_CU_START, CHECK_CU_ORDER, CHECK_CU_RANGE = 1, 2, 4
CHECK_SLOT_RANGE, CHECK_SLOT_DUP, CHECK_ACCEPTED = 8, 16, 32

__all__ = ["ccc_workspace_size", "ccc_fwd", "ccc_bwd", "ccc_bwd_noalloc", "ccc_update",
           "causal_conv1d_fn", "causal_conv1d_bwd", "causal_conv1d_update", "recompute_fwd",
           "CausalConv1dFn", "causal_conv1d", "CCCError", "library_path", "last_launch_count",
           "ccc_check", "check_metadata"]


class CCCError(RuntimeError):
    """A nonzero ccc_status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib.status_string(status)} ({status})")


def library_path() -> str:
    return _lib.path()


def last_launch_count() -> int:
    """Kernels the last ccc_fwd / ccc_bwd / ccc_update on this thread launched."""
    return _lib.lib().ccc_last_launch_count()


def _ptr(t: Optional[torch.Tensor]):
    # a plain int: the entry points declare their pointers c_void_p, which
    # takes one directly (cheaper than building a c_void_p per argument)
    return None if t is None else t.data_ptr()


def _dtype_code(t: Optional[torch.Tensor]) -> int:
    if t is None:
        return CCC_NONE
    if t.dtype == torch.float32:
        return CCC_F32
    if t.dtype == torch.bfloat16:
        return CCC_BF16
    raise TypeError(f"weight/bias must be float32 or bfloat16, got {t.dtype}")


def _act_code(activation) -> int:
    if activation is None:
        return CCC_ACT_NONE
    if activation in ("silu", "swish"):
        return CCC_ACT_SILU
    raise ValueError(f"activation must be 'silu', 'swish' or None, got {activation!r}")


def _width(weight: torch.Tensor) -> int:
    if weight.dim() != 2:
        raise ValueError("weight must be [C, W]")
    return int(weight.shape[1])


def _on_current_device(*tensors) -> None:
    """Every given tensor must be a CUDA tensor on the current device: the
    library launches on the current device, so a tensor elsewhere would be
    read through a peer mapping or fault."""
    cur = None
    for t in tensors:
        if t is None:
            continue
        d = t.get_device()  # -1 for a CPU tensor
        if d < 0:
            raise ValueError(f"expected CUDA tensors, got one on {t.device}")
        if cur is None:
            cur = torch.cuda.current_device()
        if d != cur:
            raise ValueError(f"a tensor is on cuda:{d} but the current device is cuda:{cur}; "
                             f"call inside torch.cuda.device({d})")


# The current stream's raw handle without building a torch.cuda.Stream
# object (a few microseconds per call); the public route where absent.
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    if stream is None:
        if _raw_current_stream is not None:
            return _raw_current_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _rows_view(t: torch.Tensor, name: str):
    if t.dim() == 3 and t.shape[0] == 1:
        t = t[0]
    if t.dim() != 2 or t.dtype != torch.bfloat16 or t.stride(1) != 1:
        raise ValueError(f"{name} must be BF16 [rows, C] with contiguous channels")
    return t, t.shape[0], t.shape[1], t.stride(0)


def _pool_args(conv_state, C):
    if conv_state is None:
        return 0, 0, (0, 0, 0)
    n_slots, sC, L = conv_state.shape
    if sC != C or conv_state.dtype != torch.bfloat16:
        raise ValueError("conv_state must be BF16 [slots, C, L]")
    return n_slots, L, conv_state.stride()


def ccc_workspace_size(rows: int, n_seqs: int, channels: int, for_bwd: bool) -> int:
    return int(_lib.lib().ccc_workspace_size(rows, n_seqs, channels, int(bool(for_bwd))))


def ccc_fwd(x, weight, bias, conv_state, cu_seqlens, cache_indices, has_initial_state, out,
            saved_hist=None, workspace=None, stream=None, activation="silu", overlap=False) -> None:
    """Forward through the C ABI.  Tensors are CUDA tensors laid out as in
    include/ccc.h; ``conv_state`` is updated in place.  ``overlap=True``
    sets CCC_OPT_OVERLAP_PROLOGUE (ccc_fwd_ex): only when the kernel enqueued
    just before on the stream writes none of cu_seqlens, cache_indices,
    has_initial_state, weight and bias."""
    x2, rows, C, xs = _rows_view(x, "x")
    o2, orows, oC, os_ = _rows_view(out, "out")
    if (orows, oC) != (rows, C):
        raise ValueError("out must match x")
    N = cu_seqlens.numel() - 1
    n_slots, L, st = _pool_args(conv_state, C)
    _on_current_device(x2, weight, bias, conv_state, cu_seqlens, cache_indices, has_initial_state, o2,
                       saved_hist, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _lib.lib().ccc_fwd_ex(
        _ptr(x2), rows, C, xs, _ptr(weight), _dtype_code(weight), _width(weight),
        _ptr(bias), _dtype_code(bias), _act_code(activation),
        _ptr(conv_state), n_slots, L, st[0], st[1], st[2],
        _ptr(cu_seqlens), N, _ptr(cache_indices), _ptr(has_initial_state),
        _ptr(o2), os_, _ptr(saved_hist), _ptr(workspace), ws_bytes,
        _lib.OPT_OVERLAP_PROLOGUE if overlap else 0, _stream(stream))
    if rc != 0:
        raise CCCError(rc, "ccc_fwd")


def ccc_bwd(x, weight, bias, saved_hist, cu_seqlens, cache_indices, has_initial_state, dy,
            d_final_state, dx, dweight, dbias, d_init_state, workspace=None, stream=None,
            activation="silu", overlap=False) -> None:
    """Backward through the C ABI (see include/ccc.h for every argument);
    ``overlap`` as in ccc_fwd (ccc_bwd_ex)."""
    x2, rows, C, xs = _rows_view(x, "x")
    g2, grows, gC, gs = _rows_view(dy, "dy")
    d2, drows, dC, ds = _rows_view(dx, "dx")
    if (grows, gC) != (rows, C) or (drows, dC) != (rows, C):
        raise ValueError("dy and dx must match x")
    N = cu_seqlens.numel() - 1
    _on_current_device(x2, weight, bias, saved_hist, cu_seqlens, cache_indices, has_initial_state, g2,
                       d_final_state, d2, dweight, dbias, d_init_state, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _lib.lib().ccc_bwd_ex(
        _ptr(x2), rows, C, xs, _ptr(weight), _dtype_code(weight), _width(weight),
        _ptr(bias), _dtype_code(bias), _act_code(activation),
        _ptr(saved_hist), _ptr(cu_seqlens), N, _ptr(cache_indices), _ptr(has_initial_state),
        _ptr(g2), gs, _ptr(d_final_state), _ptr(d2), ds, _ptr(dweight), _ptr(dbias),
        _ptr(d_init_state), _ptr(workspace), ws_bytes, _lib.OPT_OVERLAP_PROLOGUE if overlap else 0,
        _stream(stream))
    if rc != 0:
        raise CCCError(rc, "ccc_bwd")


def ccc_bwd_noalloc(x, weight, bias, saved_hist, cu_seqlens, cache_indices, has_initial_state, dy,
                    d_final_state, dx, dweight, dbias, d_init_state, stream=None,
                    activation="silu") -> None:
    """ccc_bwd for callers that cannot allocate device memory: the library
    uses its own fixed scratch array (``_lib.NOALLOC_SCRATCH_BYTES``) instead
    of a workspace.  Shapes needing more scratch raise CCCError
    (CCC_ERR_WORKSPACE).  Calls share that array: serialize calls whose GPU
    work could overlap."""
    x2, rows, C, xs = _rows_view(x, "x")
    g2, grows, gC, gs = _rows_view(dy, "dy")
    d2, drows, dC, ds = _rows_view(dx, "dx")
    if (grows, gC) != (rows, C) or (drows, dC) != (rows, C):
        raise ValueError("dy and dx must match x")
    N = cu_seqlens.numel() - 1
    _on_current_device(x2, weight, bias, saved_hist, cu_seqlens, cache_indices, has_initial_state, g2,
                       d_final_state, d2, dweight, dbias, d_init_state)
    rc = _lib.lib().ccc_bwd_noalloc(
        _ptr(x2), rows, C, xs, _ptr(weight), _dtype_code(weight), _width(weight),
        _ptr(bias), _dtype_code(bias), _act_code(activation),
        _ptr(saved_hist), _ptr(cu_seqlens), N, _ptr(cache_indices), _ptr(has_initial_state),
        _ptr(g2), gs, _ptr(d_final_state), _ptr(d2), ds, _ptr(dweight), _ptr(dbias),
        _ptr(d_init_state), _stream(stream))
    if rc != 0:
        raise CCCError(rc, "ccc_bwd_noalloc")


def ccc_update(x, weight, bias, conv_state, cu_seqlens, cache_indices, num_accepted, out,
               stream=None, activation="silu", overlap=False) -> None:
    """Speculative / single-token decode step through the C ABI: the new
    tokens' outputs from the history in ``conv_state`` (read at positions
    num_accepted-1 ..), and the pool update for the next step (include/ccc.h,
    ccc_update)."""
    x2, rows, C, xs = _rows_view(x, "x")
    o2, orows, oC, os_ = _rows_view(out, "out")
    if (orows, oC) != (rows, C):
        raise ValueError("out must match x")
    N = cu_seqlens.numel() - 1
    n_slots, L, st = _pool_args(conv_state, C)
    _on_current_device(x2, weight, bias, conv_state, cu_seqlens, cache_indices, num_accepted, o2)
    rc = _lib.lib().ccc_update_ex(
        _ptr(x2), rows, C, xs, _ptr(weight), _dtype_code(weight), _width(weight),
        _ptr(bias), _dtype_code(bias), _act_code(activation),
        _ptr(conv_state), n_slots, L, st[0], st[1], st[2],
        _ptr(cu_seqlens), N, _ptr(cache_indices), _ptr(num_accepted),
        _ptr(o2), os_, _lib.OPT_OVERLAP_PROLOGUE if overlap else 0, _stream(stream))
    if rc != 0:
        raise CCCError(rc, "ccc_update")


def ccc_check(rows, cu_seqlens, cache_indices=None, n_slots=0, num_accepted=None, max_accepted=0,
              status=None, stream=None) -> torch.Tensor:
    """Device-side check of the metadata (include/ccc.h, ccc_check): returns
    the int32-viewed status array whose word 0 receives the CCC_CHECK_* bits
    once the stream gets there (no synchronization here)."""
    N = cu_seqlens.numel() - 1
    words = int(_lib.lib().ccc_check_status_words(int(n_slots))) if cache_indices is not None else 1
    if status is None:
        status = torch.empty(words, dtype=torch.int32, device=cu_seqlens.device)
    if status.dtype != torch.int32 or not status.is_contiguous():
        raise ValueError("status must be a contiguous int32 tensor")
    _on_current_device(cu_seqlens, cache_indices, num_accepted, status)
    rc = _lib.lib().ccc_check(int(rows), _ptr(cu_seqlens), N, _ptr(cache_indices), int(n_slots),
                              _ptr(num_accepted), int(max_accepted), _ptr(status), status.numel(),
                              _stream(stream))
    if rc != 0:
        raise CCCError(rc, "ccc_check")
    return status


def check_metadata(rows, cu_seqlens, cache_indices=None, n_slots=0, num_accepted=None,
                   max_accepted=0) -> int:
    """ccc_check, then a host read of the result (synchronizes the current
    stream): 0 when every value is valid, else the OR of CHECK_* bits."""
    st = ccc_check(rows, cu_seqlens, cache_indices, n_slots, num_accepted, max_accepted)
    return int(st[0].item()) & 0xffffffff


def _workspace(rows, N, C, for_bwd, device, given):
    need = ccc_workspace_size(rows, N, C, for_bwd)
    if given is not None or need == 0:
        return given
    return torch.empty(need, dtype=torch.uint8, device=device)


def _packed(x, cu_seqlens):
    """(x as [rows, C], cu_seqlens, unpack) for packed [rows, C] / [1, rows, C]
    input or non-packed [B, T, D] input (B sequences of T tokens: Megatron-Core
    causal_conv1d_cp, x; each batch row is its own sequence)."""
    if x.dim() == 3 and x.shape[0] > 1:
        if cu_seqlens is not None:
            raise ValueError("cu_seqlens is for packed [rows, C] input, not [B, T, D]")
        B, T, D = x.shape
        if x.stride(2) != 1 or x.stride(0) != T * x.stride(1):
            x = x.contiguous()
        flat = x.view(B * T, D) if x.is_contiguous() else x.as_strided((B * T, D), (x.stride(1), 1))
        cu = torch.arange(B + 1, dtype=torch.int32, device=x.device) * T
        return flat, cu, (lambda t: t.view(B, T, D))
    x2, rows, _, _ = _rows_view(x, "x")
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, rows], dtype=torch.int32, device=x.device)
    return x2, cu_seqlens, (lambda t: t.view(x.shape) if x.dim() == 3 else t)


def causal_conv1d_fn(x, weight, conv_state=None, cu_seqlens=None, cache_indices=None,
                     has_initial_state=None, *, bias=None, activation="silu", out=None,
                     workspace=None, saved_hist=None, stream=None) -> torch.Tensor:
    """Allocating forward: ``out`` and the workspace are created when omitted
    (rows past cu_seqlens[-1] of an ``out`` made here hold whatever the
    allocator left).  ``x`` is
    packed ``[rows, C]`` with ``cu_seqlens``, or ``[B, T, D]``."""
    x2, cu, unpack = _packed(x, cu_seqlens)
    rows, C = x2.shape
    N = cu.numel() - 1
    o2 = torch.empty_like(x2) if out is None else out.reshape(rows, C)
    workspace = _workspace(rows, N, C, False, x.device, workspace)
    ccc_fwd(x2, weight, bias, conv_state, cu, cache_indices, has_initial_state, o2,
            saved_hist, workspace, stream, activation)
    return unpack(o2) if out is None else out


def causal_conv1d_bwd(x, weight, dy, cu_seqlens=None, *, bias=None, activation="silu",
                      saved_hist=None, cache_indices=None, has_initial_state=None,
                      d_final_state=None, dx=None, want_d_init=False, workspace=None, stream=None):
    """Allocating backward: returns ``(dx, dweight, dbias, d_init_state)``
    (dweight FP32 [C, W]; dbias None without a bias, d_init_state
    [N, W-1, C] only when requested)."""
    x2, cu, unpack = _packed(x, cu_seqlens)
    g2, _, _ = _packed(dy, cu_seqlens)
    rows, C = x2.shape
    N = cu.numel() - 1
    W = _width(weight)
    dev = x.device
    d2 = torch.empty_like(x2) if dx is None else dx.reshape(rows, C)
    dweight = torch.empty((C, W), dtype=torch.float32, device=dev)
    dbias = torch.empty((C,), dtype=torch.float32, device=dev) if bias is not None else None
    d_init = torch.empty((N, W - 1, C), dtype=torch.float32, device=dev) if want_d_init else None
    workspace = _workspace(rows, N, C, True, dev, workspace)
    ccc_bwd(x2, weight, bias, saved_hist, cu, cache_indices, has_initial_state, g2,
            d_final_state, d2, dweight, dbias, d_init, workspace, stream, activation)
    return (unpack(d2) if dx is None else dx), dweight, dbias, d_init


def causal_conv1d_update(x, weight, conv_state, cache_indices, *, cu_seqlens=None,
                         num_accepted=None, bias=None, activation="silu", out=None,
                         stream=None) -> torch.Tensor:
    """Allocating decode step: ``x`` is ``[B, k, D]`` (k new tokens for each
    of B sequences; [B, D] means k = 1) or packed ``[rows, C]`` with
    ``cu_seqlens``; ``conv_state`` is updated in place (ccc_update)."""
    squeeze = x.dim() == 2 and cu_seqlens is None
    if squeeze:
        x = x.unsqueeze(1)   # [B, D]: one token per sequence
    x2, cu, unpack = _packed(x, cu_seqlens)
    o2 = torch.empty_like(x2)
    ccc_update(x2, weight, bias, conv_state, cu, cache_indices, num_accepted, o2, stream, activation)
    y = unpack(o2)
    if squeeze:
        y = y.reshape(y.shape[0], y.shape[-1])
    if out is not None:
        out.copy_(y)
        return out
    return y


def recompute_fwd(x, weight, saved_hist, cu_seqlens, cache_indices=None, *, bias=None,
                  activation="silu", out=None, workspace=None, stream=None) -> torch.Tensor:
    """Re-run the forward from the history a previous ccc_fwd saved.

    ``saved_hist`` [N, W-1, C] is read as a pool of N slots (slot n =
    sequence n, positions along dim 1), so the recomputed output is bit for
    bit the original one even though the real conv_state was updated in place
    since (the checkpoint recompute of ``cake_causal_conv1d_kcp``,
    recompute_handle).  ``saved_hist`` itself is not modified: the final state
    is written into a scratch copy."""
    N = cu_seqlens.numel() - 1
    pool = saved_hist.clone().transpose(1, 2)     # [N, C, W-1] view, channel axis contiguous
    slots = torch.arange(N, dtype=torch.int32, device=x.device)
    if cache_indices is not None:  # -1 requests stay -1 (zero output)
        slots = torch.where(cache_indices == -1, cache_indices, slots)
    every = torch.ones(N, dtype=torch.bool, device=x.device)
    return causal_conv1d_fn(x, weight, pool, cu_seqlens, slots, every, bias=bias, activation=activation,
                            out=out, workspace=workspace, stream=stream)


class CausalConv1dFn(torch.autograd.Function):
    """Autograd wrapper: forward = ccc_fwd (saving the initial history),
    backward = ccc_bwd.  The backward recomputes the pre-activations from x
    and the saved history, so nothing of the forward output is kept.

    Gradients flow to x, weight and bias; conv_state is an in-place
    serving buffer and gets none (use ccc_bwd's d_init_state /
    d_final_state directly to chain fragments)."""

    @staticmethod
    def forward(ctx, x, weight, bias, cu_seqlens, conv_state, cache_indices, has_initial_state,
                activation="silu"):
        x2, cu, unpack = _packed(x, cu_seqlens)
        rows, C = x2.shape
        N = cu.numel() - 1
        hist = torch.empty((N, _width(weight) - 1, C), dtype=torch.bfloat16, device=x.device)
        out = causal_conv1d_fn(x2, weight, conv_state, cu, cache_indices, has_initial_state,
                               bias=bias, activation=activation, saved_hist=hist)
        empty = torch.empty(0, device=x.device)
        ctx.save_for_backward(x2, weight, bias if bias is not None else empty, cu, hist,
                              cache_indices if cache_indices is not None else empty,
                              has_initial_state if has_initial_state is not None else empty)
        ctx.has_bias = bias is not None
        ctx.has_cache = cache_indices is not None
        ctx.has_init = has_initial_state is not None
        ctx.activation = activation
        ctx.x_shape = x.shape
        return unpack(out)

    @staticmethod
    def backward(ctx, dout):
        x2, weight, bias, cu, hist, cache, has_init = ctx.saved_tensors
        bias = bias if ctx.has_bias else None
        cache = cache if ctx.has_cache else None
        has_init = has_init if ctx.has_init else None
        g2 = dout.reshape(x2.shape)
        if g2.stride(-1) != 1:
            g2 = g2.contiguous()
        # rows past cu_seqlens[-1] are not written by the kernel: start from 0
        dx = torch.zeros_like(x2)
        dx, dw, db, _ = causal_conv1d_bwd(x2, weight, g2, cu, bias=bias, activation=ctx.activation,
                                          saved_hist=hist, cache_indices=cache,
                                          has_initial_state=has_init, dx=dx)
        dw = dw.to(weight.dtype)
        db = None if db is None else db.to(bias.dtype)
        return dx.view(ctx.x_shape), dw, db, None, None, None, None, None


def causal_conv1d(x, weight, bias=None, cu_seqlens=None, conv_state=None, cache_indices=None,
                  has_initial_state=None, activation="silu") -> torch.Tensor:
    """Differentiable causal Conv1d (+ SiLU) of packed ``[rows, C]`` input
    with ``cu_seqlens`` or ``[B, T, D]`` input (see CausalConv1dFn)."""
    return CausalConv1dFn.apply(x, weight, bias, cu_seqlens, conv_state, cache_indices,
                                has_initial_state, activation)
