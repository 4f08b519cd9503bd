"""float64 CPU oracle of the packed depthwise causal Conv1d (+ SiLU).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the CUDA library and its binding) never does, and this package never touches
the CUDA library: the two share nothing but the seeded input generators.

The arithmetic lives in ``ccc_oracle.c`` (plain C, float64, one loop per
formula); this module only marshals numpy arrays.  ``build()`` compiles it with
gcc; it is also built on first use when the shared object is missing.

Every function here follows FlashInfer ``flashinfer.mamba.causal_conv1d_fn``
(Parameters: x, weight, conv_state, cu_seqlens, cache_indices,
has_initial_state, bias) for the forward and state update, and the fused
``dx`` + FP32 ``dweight`` backward of ``cake_causal_conv1d_kcp`` (Returns) with
the ordered, deterministic reduction of Megatron-Core ``core.ssm.causal_conv1d``
(``assert_causal_conv1d_deterministic``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ccc_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None


def compile_oracle(src: str, out: str) -> str:
    """gcc the oracle source ``src`` into the shared object ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                    "-Wall", "-Wextra", src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no GPU needed)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_oracle(_SRC, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i64, i32 = ctypes.c_int64, ctypes.c_int32
    lib.oracle_fwd.argtypes = [P, i64, i32, i64, P, i32, P, i32, P, i32, i32, P, i32, P, P, P, i64, P]
    lib.oracle_fwd.restype = ctypes.c_int
    lib.oracle_bwd.argtypes = [P, i64, i32, i64, P, i32, P, i32, P, P, i32, P, P, P, i64,
                               P, P, i64, P, P, P, P, P]
    lib.oracle_bwd.restype = ctypes.c_int
    lib.oracle_update.argtypes = [P, i64, i32, i64, P, i32, P, i32, P, i32, i32, P, i32, P, P, P, i64]
    lib.oracle_update.restype = ctypes.c_int
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a) -> np.ndarray:
    """BF16 data as a C-contiguous uint16 array (accepts torch bf16 tensors)."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        import torch
        a = a.detach().cpu().contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(a).view(np.uint16)


def _f64(a) -> np.ndarray:
    """Exact widening of FP32/BF16 values (torch tensor or array) to float64."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _u8(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.uint8)


class Oracle:
    """One loaded copy of the oracle library (the default one, or a mutant a
    test compiled on purpose to show that the pins catch it)."""

    def __init__(self, path: str):
        self.path = path
        self.lib = _bind(path)

    def fwd(self, x, weight, bias, cu_seqlens, conv_state=None, cache_indices=None,
            has_initial_state=None, activation="silu"):
        return _fwd(self.lib, x, weight, bias, cu_seqlens, conv_state, cache_indices,
                    has_initial_state, activation)

    def bwd(self, x, weight, bias, cu_seqlens, dy, hist=None, cache_indices=None,
            has_initial_state=None, d_final_state=None, want_d_init=True, activation="silu"):
        return _bwd(self.lib, x, weight, bias, cu_seqlens, dy, hist, cache_indices,
                    has_initial_state, d_final_state, want_d_init, activation)

    def update(self, x, weight, bias, cu_seqlens, conv_state, cache_indices, accepted=None,
               activation="silu"):
        return _update(self.lib, x, weight, bias, cu_seqlens, conv_state, cache_indices, accepted,
                       activation)


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def fwd(x, weight, bias, cu_seqlens, conv_state=None, cache_indices=None,
        has_initial_state=None, activation="silu"):
    """See ``_fwd``."""
    return default().fwd(x, weight, bias, cu_seqlens, conv_state, cache_indices,
                         has_initial_state, activation)


def bwd(x, weight, bias, cu_seqlens, dy, hist=None, cache_indices=None,
        has_initial_state=None, d_final_state=None, want_d_init=True, activation="silu"):
    """See ``_bwd``."""
    return default().bwd(x, weight, bias, cu_seqlens, dy, hist, cache_indices,
                         has_initial_state, d_final_state, want_d_init, activation)


def _act(activation) -> int:
    """1 for SiLU (Megatron-Core causal_conv1d_cp, activation: "silu" or
    "swish"), 0 for none."""
    if activation is None:
        return 0
    if activation in ("silu", "swish"):
        return 1
    raise ValueError(f"unsupported activation {activation!r}")


def _taps(weight):
    """Weights as float64 [C, W] and the width W."""
    w = _f64(weight)
    if w.ndim != 2:
        raise ValueError("weight must be [C, W]")
    return np.ascontiguousarray(w), int(w.shape[1])


def update(x, weight, bias, cu_seqlens, conv_state, cache_indices, accepted=None,
           activation="silu"):
    """See ``_update``."""
    return default().update(x, weight, bias, cu_seqlens, conv_state, cache_indices, accepted,
                            activation)


def _fwd(lib, x, weight, bias, cu_seqlens, conv_state, cache_indices, has_initial_state,
         activation):
    """Forward of the oracle (width W = weight.shape[1]).

    Returns ``(out, state, hist)``: ``out`` float64 ``[rows, C]`` with NaN in
    every row the method does not write; ``state`` the updated pool (a copy,
    uint16 bits ``[slots, C, L]``) or None; ``hist`` uint16 ``[N, W-1, C]``,
    the initial history each nonempty sequence used (rows of empty sequences
    are left as 0xFFFF)."""
    xb = _bits(x)
    rows, C = xb.shape
    w, W = _taps(weight)
    b = _f64(bias)
    cu = _i32(cu_seqlens)
    N = cu.shape[0] - 1
    st = None if conv_state is None else _bits(conv_state).copy()
    slots, L = (0, 0) if st is None else (st.shape[0], st.shape[2])
    cache = _i32(cache_indices)
    hi = _u8(has_initial_state)
    out = np.full((rows, C), np.nan)
    hist = np.full((N, W - 1, C), 0xFFFF, dtype=np.uint16)
    rc = lib.oracle_fwd(_ptr(xb), rows, C, C, _ptr(w), W, _ptr(b), _act(activation), _ptr(st),
                        slots, L, _ptr(cu), N, _ptr(cache), _ptr(hi), _ptr(out), C, _ptr(hist))
    if rc != 0:
        raise ValueError(f"oracle_fwd rejected its arguments ({rc})")
    return out, st, hist


def _bwd(lib, x, weight, bias, cu_seqlens, dy, hist, cache_indices,
         has_initial_state, d_final_state, want_d_init, activation):
    """Backward of the oracle (width W = weight.shape[1]).

    ``hist`` is the ``[N, W-1, C]`` BF16 initial history (None: zeros).
    Returns a dict with ``dx`` (float64 ``[rows, C]``, NaN in rows not
    written), ``dweight`` ``[C, W]``, ``dbias`` ``[C]``, ``d_init``
    ``[N, W-1, C]`` (or None), and ``abs_dweight`` / ``abs_dbias``, the sums
    of the absolute values of the reduced terms."""
    xb = _bits(x)
    rows, C = xb.shape
    w, W = _taps(weight)
    b = _f64(bias)
    cu = _i32(cu_seqlens)
    N = cu.shape[0] - 1
    h = _bits(hist)
    cache = _i32(cache_indices)
    hi = _u8(has_initial_state)
    dyb = _bits(dy)
    dfin = _f64(d_final_state)
    dx = np.full((rows, C), np.nan)
    dweight = np.zeros((C, W))
    dbias = np.zeros(C)
    d_init = np.full((N, W - 1, C), np.nan) if want_d_init else None
    adw = np.zeros((C, W))
    adb = np.zeros(C)
    rc = lib.oracle_bwd(_ptr(xb), rows, C, C, _ptr(w), W, _ptr(b), _act(activation), _ptr(h),
                        _ptr(cu), N, _ptr(cache), _ptr(hi), _ptr(dyb), C, _ptr(dfin), _ptr(dx), C,
                        _ptr(dweight), _ptr(dbias), _ptr(d_init), _ptr(adw), _ptr(adb))
    if rc != 0:
        raise ValueError(f"oracle_bwd rejected its arguments or could not allocate ({rc})")
    return dict(dx=dx, dweight=dweight, dbias=dbias, d_init=d_init,
                abs_dweight=adw, abs_dbias=adb)


def _update(lib, x, weight, bias, cu_seqlens, conv_state, cache_indices, accepted, activation):
    """Speculative / single-token state update of the oracle (width W =
    weight.shape[1]).

    Returns ``(out, state)``: ``out`` float64 ``[rows, C]`` with NaN in every
    row not written, ``state`` the updated pool (a copy, uint16 bits
    ``[slots, C, L]``).  ``accepted`` None means 1 for every sequence."""
    xb = _bits(x)
    rows, C = xb.shape
    w, W = _taps(weight)
    b = _f64(bias)
    cu = _i32(cu_seqlens)
    N = cu.shape[0] - 1
    st = _bits(conv_state).copy()
    slots, L = st.shape[0], st.shape[2]
    cache = _i32(cache_indices)
    acc = _i32(accepted)
    out = np.full((rows, C), np.nan)
    rc = lib.oracle_update(_ptr(xb), rows, C, C, _ptr(w), W, _ptr(b), _act(activation), _ptr(st),
                           slots, L, _ptr(cu), N, _ptr(cache), _ptr(acc), _ptr(out), C)
    if rc != 0:
        raise ValueError(f"oracle_update rejected its arguments ({rc})")
    return out, st


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of BF16 bit patterns (for comparisons in tests)."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def threads() -> int:
    """Threads the oracle's OpenMP loops use in this process."""
    n = os.environ.get("OMP_NUM_THREADS")
    if n:
        return int(n)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# Violation bits of the metadata check (the same values as the library's
# CCC_CHECK_* status bits, restated here so the oracle imports nothing from it).
CU_START, CU_ORDER, CU_RANGE, SLOT_RANGE, SLOT_DUP, ACCEPTED = 1, 2, 4, 8, 16, 32


def check_metadata(rows, cu_seqlens, cache_indices=None, n_slots=0, accepted=None, max_accepted=0) -> int:
    """The caller-owned constraints of FlashInfer causal_conv1d_fn
    (Parameters: the offsets begin at 0, never decrease and end at or before
    row `rows`, so each lies in [0, rows]; a cache index is -1 or a slot in
    [0, n_slots), and no slot serves two sequences), and the accepted count
    of the decode step in [1, max_accepted]: the OR of one bit per kind of
    violation, 0 when all hold.  Plain loops over the values."""
    cu = [int(v) for v in np.asarray(_host(cu_seqlens)).reshape(-1)]
    bits = 0
    if cu and cu[0] != 0:
        bits |= CU_START
    for i, v in enumerate(cu):
        if v < 0 or v > rows:
            bits |= CU_RANGE
        if i > 0 and v < cu[i - 1]:
            bits |= CU_ORDER
    if cache_indices is not None:
        seen = set()
        for q in (int(v) for v in np.asarray(_host(cache_indices)).reshape(-1)):
            if q == -1:
                continue
            if q < 0 or q >= n_slots:
                bits |= SLOT_RANGE
            elif q in seen:
                bits |= SLOT_DUP
            else:
                seen.add(q)
    if accepted is not None:
        for a in (int(v) for v in np.asarray(_host(accepted)).reshape(-1)):
            if a < 1 or a > max_accepted:
                bits |= ACCEPTED
    return bits


def _host(a):
    """numpy view of a CPU or CUDA tensor (or array-like)."""
    if hasattr(a, "detach"):
        return a.detach().cpu().numpy()
    return a
