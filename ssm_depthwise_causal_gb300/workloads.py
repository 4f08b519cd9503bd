"""Seeded synthetic inputs for the packed causal Conv1d workloads.

This module only draws numbers: sequence lengths, slot IDs, flags and the
BF16/FP32 tensors.  It holds none of the convolution's arithmetic, so both
the CUDA path and the float64 oracle can be fed from it without sharing any
of the method.

Layout of every workload (FlashInfer ``flashinfer.mamba.causal_conv1d_fn``,
Parameters):

* ``x``            BF16 ``[rows, C]``, channels contiguous; rows past
                   ``cu_seqlens[-1]`` are padding.
* ``weight``       FP32 or BF16 ``[C, 4]`` (tap 3 on the current token).
* ``bias``         FP32 or BF16 ``[C]`` or ``None``.
* ``conv_state``   BF16 pool ``[slots, C, L]`` or ``None``.
* ``cu_seqlens``   int32 ``[N + 1]``.
* ``cache_indices``int32 ``[N]`` (``-1`` = padded request) or ``None``.
* ``has_initial_state`` bool ``[N]`` or ``None``.
* ``dy``           BF16 ``[rows, C]`` upstream gradient (training workloads).

Structure (lengths, slots, flags) is drawn with numpy's PCG64 so it is the
same on every machine.  Dense tensors are drawn with a seeded
``torch.Generator`` on the requested device (the CPU and CUDA generators give
different streams, so a test always draws both sides' bytes once and hands the
same bytes to both).  FP32 draws are rounded to BF16 by torch's
round-to-nearest-even conversion.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass
class Workload:
    name: str
    rows: int
    C: int
    lengths: np.ndarray            # int64 [N]
    cu_seqlens: torch.Tensor       # int32 [N+1]
    x: torch.Tensor                # bf16 [rows, C]
    weight: torch.Tensor           # fp32 / bf16 [C, W] (W = 4 unless stated)
    bias: Optional[torch.Tensor]   # fp32 / bf16 [C] or None
    conv_state: Optional[torch.Tensor] = None      # bf16 [slots, C, L]
    cache_indices: Optional[torch.Tensor] = None   # int32 [N]
    has_initial_state: Optional[torch.Tensor] = None  # bool [N]
    dy: Optional[torch.Tensor] = None              # bf16 [rows, C]
    fragments: int = 1             # >1: process as consecutive fragments
    training: bool = True          # forward + backward
    activation: Optional[str] = "silu"  # "silu" or None
    num_accepted: Optional[torch.Tensor] = None    # int32 [N], decode steps only

    @property
    def width(self) -> int:
        return int(self.weight.shape[1])

    @property
    def n_seqs(self) -> int:
        return int(self.lengths.shape[0])

    @property
    def valid_tokens(self) -> int:
        return int(self.lengths.sum())

    def to(self, device) -> "Workload":
        def mv(t):
            return None if t is None else t.to(device)
        return dataclasses.replace(
            self, cu_seqlens=mv(self.cu_seqlens), x=mv(self.x),
            weight=mv(self.weight), bias=mv(self.bias),
            conv_state=mv(self.conv_state), cache_indices=mv(self.cache_indices),
            has_initial_state=mv(self.has_initial_state), dy=mv(self.dy))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, g: torch.Generator, device, std: float = 1.0,
                chunk_rows: int = 1 << 16) -> torch.Tensor:
    """N(0, std^2) drawn in FP32 and rounded to BF16 (RNE), in row chunks so
    that multi-GB tensors never need an FP32 copy of the whole thing."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if out.numel() == 0:  # an empty batch: nothing to draw
        return out
    flat = out.view(shape[0], -1) if len(shape) > 1 else out.view(-1, 1)
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(flat.shape[0], r0 + chunk_rows)
        blk = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device,
                          dtype=torch.float32)
        if std != 1.0:
            blk.mul_(std)
        flat[r0:r1].copy_(blk)
    return out


def uniform(shape, g, device, lo, hi, dtype) -> torch.Tensor:
    t = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    t = t * (hi - lo) + lo
    return t.to(dtype)


def cu_from_lengths(lengths: np.ndarray) -> torch.Tensor:
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=cu[1:])
    return torch.from_numpy(cu.astype(np.int32))


def make_custom(lengths, C, rows=None, *, seed=0, device="cpu",
                w_dtype=torch.float32, b_dtype=torch.float32,
                slots=None, state_len=4, n_minus_one=0, has_init_p=0.5,
                with_state=True, training=True, x_std=1.0, width=4,
                activation="silu") -> Workload:
    """A general packed workload: given lengths, draw slots, flags and tensors.

    Draw order: slots, flags, x, weight, bias, state, dy (lengths are given).
    ``b_dtype=None`` gives no bias; ``with_state=False`` gives no pool;
    ``width`` is the number of taps W (weight [C, W])."""
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    N = len(lengths)
    T = int(lengths.sum())
    rows = T if rows is None else rows
    assert rows >= T
    cache = has_init = None
    if with_state:
        slots = max(N, 1) * 2 if slots is None else slots
        cache_np = rng.permutation(slots)[:N].astype(np.int32)
        if n_minus_one:
            idx = rng.choice(N, size=n_minus_one, replace=False)
            cache_np[idx] = -1
        hi_np = rng.random(N) < has_init_p
        cache = torch.from_numpy(cache_np)
        has_init = torch.from_numpy(hi_np)
    g = _gen(seed, device)
    x = normal_bf16((rows, C), g, device, std=x_std)
    weight = uniform((C, width), g, device, -0.5, 0.5, w_dtype)
    bias = None
    if b_dtype is not None:
        bias = (torch.randn((C,), generator=g, device=device) * 0.1).to(b_dtype)
    state = None
    if with_state:
        state = normal_bf16((slots, C, state_len), g, device)
    dy = normal_bf16((rows, C), g, device) if training else None
    return Workload(
        name=f"custom(N={N},C={C},rows={rows})", rows=rows, C=C, lengths=lengths,
        cu_seqlens=cu_from_lengths(lengths).to(device), x=x, weight=weight,
        bias=bias, conv_state=state,
        cache_indices=None if cache is None else cache.to(device),
        has_initial_state=None if has_init is None else has_init.to(device),
        dy=dy, training=training, activation=activation)


# --------------------------------------------------------------------------
# The five workloads.  Shapes follow the pages' workloads: the GDP conv
# channel layout [V(d_inner*M), K(ngroups*d_state*M), Q(ngroups*d_state)]
# (core.ssm.gdp_context_parallel, module description) for C=7168, the serving
# pool of causal_conv1d_fn for the prefill case, and one long document split
# into context-parallel fragments (cake_causal_conv1d_kcp) for the last.
# --------------------------------------------------------------------------

def tiny(seed=0, device="cpu") -> Workload:
    """rows 1040, C 256, lengths {100, 300, 24, 600} + 16 padding rows, pool
    [8, 256, 4], slots = first 4 of a permutation of 0..7 with sequence 2
    (0-based) set to -1, has_initial_state ~ Bernoulli(0.5)."""
    rng = np.random.default_rng(seed)
    lengths = np.array([100, 300, 24, 600], dtype=np.int64)
    C, rows, slots = 256, 1040, 8
    cache_np = rng.permutation(slots)[:4].astype(np.int32)
    cache_np[2] = -1
    hi_np = rng.random(4) < 0.5
    g = _gen(seed, device)
    x = normal_bf16((rows, C), g, device)
    weight = uniform((C, 4), g, device, -0.5, 0.5, torch.float32)
    bias = (torch.randn((C,), generator=g, device=device) * 0.1).float()
    state = normal_bf16((slots, C, 4), g, device)
    dy = normal_bf16((rows, C), g, device)
    return Workload("tiny rows=1040 C=256 N=4", rows, C, lengths,
                    cu_from_lengths(lengths).to(device), x, weight, bias,
                    state, torch.from_numpy(cache_np).to(device),
                    torch.from_numpy(hi_np).to(device), dy)


def dense(seed=0, device="cpu", C=4096, seqs=4, seqlen=4096) -> Workload:
    """4 x 4096 tokens packed as rows 16384, C 4096, no state."""
    lengths = np.full(seqs, seqlen, dtype=np.int64)
    rows = int(lengths.sum())
    g = _gen(seed, device)
    x = normal_bf16((rows, C), g, device)
    weight = uniform((C, 4), g, device, -0.5, 0.5, torch.float32)
    bias = (torch.randn((C,), generator=g, device=device) * 0.1).float()
    dy = normal_bf16((rows, C), g, device)
    return Workload(f"dense rows={rows} C={C} N={seqs}", rows, C, lengths,
                    cu_from_lengths(lengths).to(device), x, weight, bias, dy=dy)


def packed_lengths(seed=0, N=200, rows=65536, mean=320.0, sigma=1.0,
                   n_empty=6, max_len=8192) -> np.ndarray:
    """Lognormal lengths with the given mean, clipped to [0, max_len],
    exactly n_empty forced to zero, scaled down (floor) if they overflow."""
    rng = np.random.default_rng(seed)
    mu = math.log(mean) - sigma * sigma / 2.0
    lengths = np.rint(rng.lognormal(mu, sigma, N)).astype(np.int64)
    lengths = np.clip(lengths, 0, max_len)
    lengths[rng.choice(N, size=n_empty, replace=False)] = 0
    tot = int(lengths.sum())
    if tot > rows:
        lengths = np.floor(lengths * (rows / tot)).astype(np.int64)
    return lengths


def packed(seed=0, device="cpu", C=7168, rows=65536, N=200) -> Workload:
    """GDP conv channels C = 7168 = V 2048*2 + K 8*128*2 + Q 1024; rows 65536
    holding 200 lognormal-length sequences (mean ~320, ~3 % empty), the rest
    padding; weight BF16, bias FP32, no state."""
    lengths = packed_lengths(seed, N=N, rows=rows)
    g = _gen(seed, device)
    x = normal_bf16((rows, C), g, device)
    weight = uniform((C, 4), g, device, -0.5, 0.5, torch.bfloat16)
    bias = (torch.randn((C,), generator=g, device=device) * 0.1).float()
    dy = normal_bf16((rows, C), g, device)
    return Workload(f"packed rows={rows} C={C} N={N}", rows, C, lengths,
                    cu_from_lengths(lengths).to(device), x, weight, bias, dy=dy)


def serving(seed=0, device="cpu", C=8192, N=256, slots=512, max_len=2048,
            n_minus_one=13) -> Workload:
    """N 256 prefill requests, lengths U{1..2048}, C 8192, pool
    [512, 8192, 4], distinct random slots with 13 (5 %) set to -1,
    has_initial_state ~ Bernoulli(0.5), weight FP32, bias BF16; forward only."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(1, max_len + 1, size=N).astype(np.int64)
    cache_np = rng.choice(slots, size=N, replace=False).astype(np.int32)
    cache_np[rng.choice(N, size=n_minus_one, replace=False)] = -1
    hi_np = rng.random(N) < 0.5
    rows = int(lengths.sum())
    g = _gen(seed, device)
    x = normal_bf16((rows, C), g, device)
    weight = uniform((C, 4), g, device, -0.5, 0.5, torch.float32)
    bias = (torch.randn((C,), generator=g, device=device) * 0.1).to(torch.bfloat16)
    state = normal_bf16((slots, C, 4), g, device)
    return Workload(f"serving rows={rows} C={C} N={N}", rows, C, lengths,
                    cu_from_lengths(lengths).to(device), x, weight, bias,
                    state, torch.from_numpy(cache_np).to(device),
                    torch.from_numpy(hi_np).to(device), None, training=False)


def long_context(seed=0, device="cpu", C=4096, T=1 << 20, fragments=8) -> Workload:
    """One T-token document, C 4096, weight FP32, no bias, processed as
    `fragments` consecutive fragments chained through a one-slot pool."""
    lengths = np.array([T], dtype=np.int64)
    g = _gen(seed, device)
    x = normal_bf16((T, C), g, device)
    weight = uniform((C, 4), g, device, -0.5, 0.5, torch.float32)
    dy = normal_bf16((T, C), g, device)
    return Workload(f"long T={T} C={C} fragments={fragments}", T, C, lengths,
                    cu_from_lengths(lengths).to(device), x, weight, None,
                    dy=dy, fragments=fragments)


def decode(seed=0, device="cpu", C=8192, N=256, slots=512, draft=1, state_len=4,
           n_minus_one=13) -> Workload:
    """One decode step of the serving batch after its prefill: N 256
    requests, `draft` new tokens each (1: plain decode; more: speculative
    drafts), C 8192, pool [512, 8192, state_len] (history axis contiguous),
    distinct random slots with 13 (5 %) set to -1, weight FP32, bias BF16;
    accepted counts U{1..draft} from the previous step (all 1 for a plain
    decode: the first step after a prefill)."""
    rng = np.random.default_rng(seed)
    lengths = np.full(N, draft, dtype=np.int64)
    cache_np = rng.choice(slots, size=N, replace=False).astype(np.int32)
    cache_np[rng.choice(N, size=n_minus_one, replace=False)] = -1
    acc_np = rng.integers(1, draft + 1, size=N).astype(np.int32)
    rows = int(lengths.sum())
    g = _gen(seed, device)
    x = normal_bf16((rows, C), g, device)
    weight = uniform((C, 4), g, device, -0.5, 0.5, torch.float32)
    bias = (torch.randn((C,), generator=g, device=device) * 0.1).to(torch.bfloat16)
    state = normal_bf16((slots, C, state_len), g, device)
    return Workload(f"decode N={N} draft={draft} C={C} pool=[{slots},{C},{state_len}]", rows, C, lengths,
                    cu_from_lengths(lengths).to(device), x, weight, bias,
                    state, torch.from_numpy(cache_np).to(device), None, None, training=False,
                    num_accepted=torch.from_numpy(acc_np).to(device))


def spec_decode(seed=0, device="cpu") -> Workload:
    """A speculative decode step of the serving batch: 4 draft tokens per
    request, pool [512, 8192, 6] (room for 4 + W - 2 values)."""
    return decode(seed, device, draft=4, state_len=6)


def packed_small(seed=0, device="cpu") -> Workload:
    """The packed workload at a quarter of the rows (16384 rows, 50
    sequences): each tensor is 235 MB, still larger than L2, for profiler
    captures that replay the kernel many times."""
    return packed(seed, device, rows=16384, N=50)


WORKLOADS = {
    "tiny": tiny,
    "decode": decode,
    "spec_decode": spec_decode,
    "dense": dense,
    "packed": packed,
    "packed_small": packed_small,
    "serving": serving,
    "long": long_context,
}
