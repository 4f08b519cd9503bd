"""GB300-native packed, width-4, depthwise causal Conv1d + SiLU.

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
* ``ccc_bwd(...)``  -- fused dx + deterministic FP32 dweight/dbias
  (``cake_causal_conv1d_kcp``, Returns)

the allocating conveniences ``causal_conv1d_fn`` / ``causal_conv1d_bwd``,
which create ``out`` / ``dx`` / the workspace when they are not given,
``recompute_fwd`` (bitwise re-run of a forward from its saved history) and the
autograd wrapper ``causal_conv1d`` / ``CausalConv1dFn``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _lib

CCC_F32, CCC_BF16, CCC_NONE = 0, 1, -1

__all__ = ["ccc_workspace_size", "ccc_fwd", "ccc_bwd", "ccc_bwd_noalloc", "causal_conv1d_fn",
           "causal_conv1d_bwd", "recompute_fwd", "CausalConv1dFn", "causal_conv1d",
           "CCCError", "library_path", "last_launch_count"]


class CCCError(RuntimeError):
    """A nonzero ccc_status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib.status_string(status)} ({status})")


def library_path() -> str:
    return _lib.path()


def last_launch_count() -> int:
    """Kernels the last ccc_fwd / ccc_bwd on this thread launched."""
    return _lib.lib().ccc_last_launch_count()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: Optional[torch.Tensor]) -> int:
    if t is None:
        return CCC_NONE
    if t.dtype == torch.float32:
        return CCC_F32
    if t.dtype == torch.bfloat16:
        return CCC_BF16
    raise TypeError(f"weight/bias must be float32 or bfloat16, got {t.dtype}")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


def _rows_view(t: torch.Tensor, name: str):
    if t.dim() == 3 and t.shape[0] == 1:
        t = t[0]
    if t.dim() != 2 or t.dtype != torch.bfloat16 or t.stride(1) != 1:
        raise ValueError(f"{name} must be BF16 [rows, C] with contiguous channels")
    return t, t.shape[0], t.shape[1], t.stride(0)


def ccc_workspace_size(rows: int, n_seqs: int, channels: int, for_bwd: bool) -> int:
    return int(_lib.lib().ccc_workspace_size(rows, n_seqs, channels, int(bool(for_bwd))))


def ccc_fwd(x, weight, bias, conv_state, cu_seqlens, cache_indices, has_initial_state, out,
            saved_hist=None, workspace=None, stream=None) -> None:
    """Forward through the C ABI.  Tensors are CUDA tensors laid out as in
    include/ccc.h; ``conv_state`` is updated in place."""
    x2, rows, C, xs = _rows_view(x, "x")
    o2, orows, oC, os_ = _rows_view(out, "out")
    if (orows, oC) != (rows, C):
        raise ValueError("out must match x")
    N = cu_seqlens.numel() - 1
    if conv_state is not None:
        n_slots, sC, L = conv_state.shape
        if sC != C or conv_state.dtype != torch.bfloat16:
            raise ValueError("conv_state must be BF16 [slots, C, L]")
        st = conv_state.stride()
    else:
        n_slots, L, st = 0, 0, (0, 0, 0)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _lib.lib().ccc_fwd(
        _ptr(x2), rows, C, xs, _ptr(weight), _dtype_code(weight), _ptr(bias), _dtype_code(bias),
        _ptr(conv_state), n_slots, L, st[0], st[1], st[2],
        _ptr(cu_seqlens), N, _ptr(cache_indices), _ptr(has_initial_state),
        _ptr(o2), os_, _ptr(saved_hist), _ptr(workspace), ws_bytes, _stream(stream))
    if rc != 0:
        raise CCCError(rc, "ccc_fwd")


def ccc_bwd(x, weight, bias, saved_hist, cu_seqlens, cache_indices, has_initial_state, dy,
            d_final_state, dx, dweight, dbias, d_init_state, workspace=None, stream=None) -> None:
    """Backward through the C ABI (see include/ccc.h for every argument)."""
    x2, rows, C, xs = _rows_view(x, "x")
    g2, grows, gC, gs = _rows_view(dy, "dy")
    d2, drows, dC, ds = _rows_view(dx, "dx")
    if (grows, gC) != (rows, C) or (drows, dC) != (rows, C):
        raise ValueError("dy and dx must match x")
    N = cu_seqlens.numel() - 1
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _lib.lib().ccc_bwd(
        _ptr(x2), rows, C, xs, _ptr(weight), _dtype_code(weight), _ptr(bias), _dtype_code(bias),
        _ptr(saved_hist), _ptr(cu_seqlens), N, _ptr(cache_indices), _ptr(has_initial_state),
        _ptr(g2), gs, _ptr(d_final_state), _ptr(d2), ds, _ptr(dweight), _ptr(dbias),
        _ptr(d_init_state), _ptr(workspace), ws_bytes, _stream(stream))
    if rc != 0:
        raise CCCError(rc, "ccc_bwd")


def ccc_bwd_noalloc(x, weight, bias, saved_hist, cu_seqlens, cache_indices, has_initial_state, dy,
                    d_final_state, dx, dweight, dbias, d_init_state, stream=None) -> None:
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
    rc = _lib.lib().ccc_bwd_noalloc(
        _ptr(x2), rows, C, xs, _ptr(weight), _dtype_code(weight), _ptr(bias), _dtype_code(bias),
        _ptr(saved_hist), _ptr(cu_seqlens), N, _ptr(cache_indices), _ptr(has_initial_state),
        _ptr(g2), gs, _ptr(d_final_state), _ptr(d2), ds, _ptr(dweight), _ptr(dbias),
        _ptr(d_init_state), _stream(stream))
    if rc != 0:
        raise CCCError(rc, "ccc_bwd_noalloc")


def _workspace(rows, N, C, for_bwd, device, given):
    need = ccc_workspace_size(rows, N, C, for_bwd)
    if given is not None or need == 0:
        return given
    return torch.empty(need, dtype=torch.uint8, device=device)


def causal_conv1d_fn(x, weight, conv_state=None, cu_seqlens=None, cache_indices=None,
                     has_initial_state=None, *, bias=None, out=None, workspace=None,
                     saved_hist=None, stream=None) -> torch.Tensor:
    """Allocating forward: ``out`` and the workspace are created when omitted
    (unused trailing rows of an allocated ``out`` are unspecified)."""
    x2, rows, C, _ = _rows_view(x, "x")
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, rows], dtype=torch.int32, device=x.device)
    N = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty_like(x)
    workspace = _workspace(rows, N, C, False, x.device, workspace)
    ccc_fwd(x, weight, bias, conv_state, cu_seqlens, cache_indices, has_initial_state, out,
            saved_hist, workspace, stream)
    return out


def causal_conv1d_bwd(x, weight, dy, cu_seqlens, *, bias=None, saved_hist=None,
                      cache_indices=None, has_initial_state=None, d_final_state=None,
                      dx=None, want_d_init=False, workspace=None, stream=None):
    """Allocating backward: returns ``(dx, dweight, dbias, d_init_state)``
    (dbias None without a bias, d_init_state None unless requested)."""
    x2, rows, C, _ = _rows_view(x, "x")
    N = cu_seqlens.numel() - 1
    dev = x.device
    if dx is None:
        dx = torch.empty_like(x)
    dweight = torch.empty((C, 4), dtype=torch.float32, device=dev)
    dbias = torch.empty((C,), dtype=torch.float32, device=dev) if bias is not None else None
    d_init = torch.empty((N, 3, C), dtype=torch.float32, device=dev) if want_d_init else None
    workspace = _workspace(rows, N, C, True, dev, workspace)
    ccc_bwd(x, weight, bias, saved_hist, cu_seqlens, cache_indices, has_initial_state, dy,
            d_final_state, dx, dweight, dbias, d_init, workspace, stream)
    return dx, dweight, dbias, d_init


def recompute_fwd(x, weight, saved_hist, cu_seqlens, cache_indices=None, *, bias=None, out=None,
                  workspace=None, stream=None) -> torch.Tensor:
    """Re-run the forward from the history a previous ccc_fwd saved.

    ``saved_hist`` [N, 3, C] is read as a pool of N slots (slot n = sequence
    n, positions along dim 1), so the recomputed output is bit for bit the
    original one even though the real conv_state was updated in place since
    (the checkpoint recompute of ``cake_causal_conv1d_kcp``, recompute_handle).
    ``saved_hist`` itself is not modified: the final state is written into a
    scratch copy."""
    x2, rows, C, _ = _rows_view(x, "x")
    N = cu_seqlens.numel() - 1
    pool = saved_hist.clone().transpose(1, 2)     # [N, C, 3] view, channel axis contiguous
    slots = torch.arange(N, dtype=torch.int32, device=x.device)
    if cache_indices is not None:  # -1 requests stay -1 (zero output)
        slots = torch.where(cache_indices == -1, cache_indices, slots)
    every = torch.ones(N, dtype=torch.bool, device=x.device)
    return causal_conv1d_fn(x, weight, pool, cu_seqlens, slots, every, bias=bias, out=out,
                            workspace=workspace, stream=stream)


class CausalConv1dFn(torch.autograd.Function):
    """Autograd wrapper: forward = ccc_fwd (saving the initial history),
    backward = ccc_bwd.  The backward recomputes the pre-activations from x
    and the saved history, so nothing of the forward output is kept.

    Gradients flow to x, weight and bias; conv_state is an in-place
    serving buffer and gets none (use ccc_bwd's d_init_state /
    d_final_state directly to chain fragments)."""

    @staticmethod
    def forward(ctx, x, weight, bias, cu_seqlens, conv_state, cache_indices, has_initial_state):
        x2, rows, C, _ = _rows_view(x, "x")
        N = cu_seqlens.numel() - 1
        hist = torch.empty((N, 3, C), dtype=torch.bfloat16, device=x.device)
        out = causal_conv1d_fn(x, weight, conv_state, cu_seqlens, cache_indices, has_initial_state,
                               bias=bias, saved_hist=hist)
        ctx.save_for_backward(x, weight, bias if bias is not None else torch.empty(0, device=x.device),
                              cu_seqlens, hist,
                              cache_indices if cache_indices is not None else torch.empty(0, device=x.device),
                              has_initial_state if has_initial_state is not None else
                              torch.empty(0, device=x.device))
        ctx.has_bias = bias is not None
        ctx.has_cache = cache_indices is not None
        ctx.has_init = has_initial_state is not None
        return out

    @staticmethod
    def backward(ctx, dout):
        x, weight, bias, cu_seqlens, hist, cache, has_init = ctx.saved_tensors
        bias = bias if ctx.has_bias else None
        cache = cache if ctx.has_cache else None
        has_init = has_init if ctx.has_init else None
        dout = dout.contiguous() if dout.stride(-1) != 1 else dout
        # rows past cu_seqlens[-1] are not written by the kernel: start from 0
        dx = torch.zeros_like(x)
        dx, dw, db, _ = causal_conv1d_bwd(x, weight, dout, cu_seqlens, bias=bias, saved_hist=hist,
                                          cache_indices=cache, has_initial_state=has_init, dx=dx)
        dw = dw.to(weight.dtype)
        db = None if db is None else db.to(bias.dtype)
        return dx, dw, db, None, None, None, None


def causal_conv1d(x, weight, bias=None, cu_seqlens=None, conv_state=None, cache_indices=None,
                  has_initial_state=None) -> torch.Tensor:
    """Differentiable packed causal Conv1d + SiLU (see CausalConv1dFn)."""
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, x.shape[-2]], dtype=torch.int32, device=x.device)
    return CausalConv1dFn.apply(x, weight, bias, cu_seqlens, conv_state, cache_indices,
                                has_initial_state)
