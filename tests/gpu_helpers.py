"""Shared plumbing of the GPU parity tests: run a workload through the C ABI
on the GPU, run the float64 oracle on the same bytes (optionally on a subset
of channels -- channels are independent, so the oracle's answer for a subset
is exactly its answer for those channels of the full problem), and compare
with the tolerances the method's contract sets:

* conv_state, saved history, -1 rows and padding rows: bit-exact;
* BF16 out / dx: |gpu - ref32| <= 2^-7 |ref32| + 1e-3, ref32 = FP32 rounding
  of the oracle's float64 value (one BF16 ulp plus an absolute floor);
* FP32 dweight / dbias: |err| <= 1e-4 |ref| or |err| <= 1e-6 sum|terms| (the
  conditioning floor for sums that cancel to near zero);
* FP32 d_init_state (four products and a carry): |err| <= 1e-4 |ref| + 1e-5.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
import ssm_depthwise_causal_gb300 as ccc
from ssm_depthwise_causal_gb300 import workloads

SENTINEL = 0x7FC1  # a NaN bit pattern the kernels never produce


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def fill_sentinel(t: torch.Tensor) -> torch.Tensor:
    t.view(torch.int16).fill_(SENTINEL - 0x10000 if SENTINEL > 0x7FFF else SENTINEL)
    return t


@dataclasses.dataclass
class GpuResult:
    out: torch.Tensor
    state: torch.Tensor | None
    hist: torch.Tensor
    dx: torch.Tensor | None = None
    dweight: torch.Tensor | None = None
    dbias: torch.Tensor | None = None
    d_init: torch.Tensor | None = None


def channel_contiguous_pool(pool: torch.Tensor) -> torch.Tensor:
    """Same logical [slots, C, L] pool stored channel-contiguous."""
    return pool.transpose(1, 2).contiguous().transpose(1, 2)


def _wide(t: torch.Tensor, pad: int) -> torch.Tensor:
    """`t` [rows, C] as a column slice of a wider buffer (row stride C + pad)."""
    wide = torch.zeros((t.shape[0], t.shape[1] + pad), dtype=t.dtype, device=t.device)
    wide[:, :t.shape[1]] = t
    return wide[:, :t.shape[1]]


def run_gpu(wl: workloads.Workload, *, backward=True, d_final=None, want_d_init=True,
            pool_layout="history", x_pad_cols=0, out_pad_cols=0) -> GpuResult:
    """One forward (+ backward) of a device-resident workload through the C ABI.
    `x_pad_cols` / `out_pad_cols` give x and dy / out and dx row strides
    larger than C."""
    dev = wl.x.device
    x = _wide(wl.x, x_pad_cols) if x_pad_cols else wl.x
    state = None
    if wl.conv_state is not None:
        state = wl.conv_state.clone() if pool_layout == "history" else channel_contiguous_pool(wl.conv_state)
    H = wl.width - 1
    out = fill_sentinel(torch.empty((wl.rows, wl.C + out_pad_cols), dtype=torch.bfloat16, device=dev))
    out = out[:, :wl.C]
    hist = fill_sentinel(torch.empty((wl.n_seqs, H, wl.C), dtype=torch.bfloat16, device=dev))
    ws = torch.empty(max(1, ccc.ccc_workspace_size(wl.rows, wl.n_seqs, wl.C, False)),
                     dtype=torch.uint8, device=dev)
    ccc.ccc_fwd(x, wl.weight, wl.bias, state, wl.cu_seqlens, wl.cache_indices,
                wl.has_initial_state, out, hist, ws, activation=wl.activation)
    res = GpuResult(out=out, state=state, hist=hist)
    if backward:
        dx = fill_sentinel(torch.empty((wl.rows, wl.C + out_pad_cols), dtype=torch.bfloat16, device=dev))
        dx = dx[:, :wl.C]
        dy = _wide(wl.dy, x_pad_cols) if x_pad_cols else wl.dy
        dw = torch.full((wl.C, wl.width), float("nan"), device=dev)
        db = torch.full((wl.C,), float("nan"), device=dev) if wl.bias is not None else None
        di = torch.full((wl.n_seqs, H, wl.C), float("nan"), device=dev) if want_d_init else None
        wsb = torch.empty(ccc.ccc_workspace_size(wl.rows, wl.n_seqs, wl.C, True), dtype=torch.uint8,
                          device=dev)
        ccc.ccc_bwd(x, wl.weight, wl.bias, hist, wl.cu_seqlens, wl.cache_indices,
                    wl.has_initial_state, dy, d_final, dx, dw, db, di, wsb, activation=wl.activation)
        res.dx, res.dweight, res.dbias, res.d_init = dx, dw, db, di
    torch.cuda.synchronize()
    return res


def subset(wl: workloads.Workload, chans) -> workloads.Workload:
    """CPU copy of the workload restricted to channels `chans`."""
    idx = torch.as_tensor(chans, dtype=torch.long, device=wl.x.device)

    def pick(t, dim):
        return None if t is None else t.index_select(dim, idx).cpu()

    return dataclasses.replace(
        wl, C=len(chans), x=pick(wl.x, 1), weight=pick(wl.weight, 0), bias=pick(wl.bias, 0),
        conv_state=pick(wl.conv_state, 1), dy=pick(wl.dy, 1),
        cu_seqlens=wl.cu_seqlens.cpu(),
        cache_indices=None if wl.cache_indices is None else wl.cache_indices.cpu(),
        has_initial_state=None if wl.has_initial_state is None else wl.has_initial_state.cpu())


def run_oracle(wl_cpu: workloads.Workload, *, backward=True, d_final=None):
    out, state, hist = oracle.fwd(wl_cpu.x, wl_cpu.weight, wl_cpu.bias, wl_cpu.cu_seqlens,
                                  wl_cpu.conv_state, wl_cpu.cache_indices, wl_cpu.has_initial_state,
                                  activation=wl_cpu.activation)
    res = dict(out=out, state=state, hist=hist)
    if backward:
        h = hist if wl_cpu.conv_state is not None else None
        res.update(oracle.bwd(wl_cpu.x, wl_cpu.weight, wl_cpu.bias, wl_cpu.cu_seqlens, wl_cpu.dy,
                              h, wl_cpu.cache_indices, wl_cpu.has_initial_state, d_final,
                              activation=wl_cpu.activation))
    return res


def live_rows(wl) -> np.ndarray:
    """Boolean [rows]: row belongs to a live (non -1) sequence."""
    m = np.zeros(wl.rows, dtype=bool)
    cu = wl.cu_seqlens.cpu().numpy()
    ci = None if wl.cache_indices is None else wl.cache_indices.cpu().numpy()
    for n in range(wl.n_seqs):
        if ci is None or ci[n] != -1:
            m[cu[n]:cu[n + 1]] = True
    return m


def minus_one_rows(wl) -> np.ndarray:
    m = np.zeros(wl.rows, dtype=bool)
    if wl.cache_indices is None:
        return m
    cu = wl.cu_seqlens.cpu().numpy()
    ci = wl.cache_indices.cpu().numpy()
    for n in range(wl.n_seqs):
        if ci[n] == -1:
            m[cu[n]:cu[n + 1]] = True
    return m


def assert_bf16_close(gpu_bits: np.ndarray, ref64: np.ndarray, what: str, rows=None, chans=None):
    """`rows` / `chans` (optional) map array indices back to absolute row and
    channel numbers for the failure message."""
    got = (gpu_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r32 = ref64.astype(np.float32).astype(np.float64)
    err = np.abs(got - r32)
    tol = 2.0 ** -7 * np.abs(r32) + 1e-3
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        where = i
        if rows is not None and len(i) == 2:
            where = (int(rows[i[0]]), int(chans[i[1]]) if chans is not None else int(i[1]))
        bad_rows = np.unique(idx[:, 0])
        abs_rows = rows[bad_rows] if rows is not None else bad_rows
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance in {len(bad_rows)} rows "
            f"(rows {abs_rows[:8].tolist()}...); first at row/channel {where}: gpu {got[i]!r} "
            f"(bits {int(gpu_bits[i]):#06x}) ref {r32[i]!r}")


def assert_reduction_close(gpu: np.ndarray, ref: np.ndarray, abs_terms: np.ndarray, what: str) -> dict:
    """The FP32 reduction tolerance.  Returns how the elements passed:
    ``n`` elements, ``floor_only`` of them within 1e-6 sum|terms| but not
    within 1e-4 |ref| (sums that cancel to near zero), ``max_rel`` the
    largest |err| / |ref| and ``max_err_terms`` the largest
    |err| / sum|terms|."""
    err = np.abs(gpu.astype(np.float64) - ref)
    rel_ok = err <= 1e-4 * np.abs(ref)
    floor_ok = err <= 1e-6 * abs_terms
    ok = rel_ok | floor_ok
    if not ok.all():
        i = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {int((~ok).sum())} elements out of tolerance; first at "
                             f"{tuple(i)}: gpu {gpu[tuple(i)]!r} ref {ref[tuple(i)]!r} "
                             f"sum|terms| {abs_terms[tuple(i)]!r}")
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(ref != 0, err / np.abs(ref), np.where(err == 0, 0.0, np.inf))
        per_terms = np.where(abs_terms > 0, err / abs_terms, 0.0)
    return dict(n=int(err.size), floor_only=int((~rel_ok).sum()), max_rel=float(rel.max(initial=0.0)),
                max_err_terms=float(per_terms.max(initial=0.0)))


def compare(wl_cpu, ref, gpu: dict, *, backward=True, rows_checked=None, chans=None) -> dict:
    """Compare GPU results (numpy, same channel subset) against the oracle.
    Returns the reduction statistics of dweight (and dbias) for the
    backward (see assert_reduction_close)."""
    T = int(wl_cpu.cu_seqlens[-1])
    live = live_rows(wl_cpu)
    m1 = minus_one_rows(wl_cpu)
    rows = np.arange(wl_cpu.rows) if rows_checked is None else rows_checked
    lv = rows[live[rows]]
    assert_bf16_close(gpu["out"][lv], ref["out"][lv], "out", lv, chans)
    mo = rows[m1[rows]]
    assert np.all(gpu["out"][mo] == 0), "-1 rows of out must be +0"
    pad = rows[rows >= T]
    assert np.all(gpu["out"][pad] == SENTINEL), "padding rows of out were written"
    if ref.get("state") is not None:
        np.testing.assert_array_equal(gpu["state"], ref["state"], err_msg="conv_state")
    lens = np.diff(wl_cpu.cu_seqlens.cpu().numpy())
    ne = lens > 0
    np.testing.assert_array_equal(gpu["hist"][ne], ref["hist"][ne], err_msg="saved_hist")
    assert np.all(gpu["hist"][~ne] == SENTINEL), "saved_hist rows of empty sequences were written"
    if not backward:
        return {}
    assert_bf16_close(gpu["dx"][lv], ref["dx"][lv], "dx", lv, chans)
    assert np.all(gpu["dx"][mo] == 0), "-1 rows of dx must be +0"
    assert np.all(gpu["dx"][pad] == SENTINEL), "padding rows of dx were written"
    stats = {"dweight": assert_reduction_close(gpu["dweight"], ref["dweight"], ref["abs_dweight"], "dweight")}
    if gpu.get("dbias") is not None:
        stats["dbias"] = assert_reduction_close(gpu["dbias"], ref["dbias"], ref["abs_dbias"], "dbias")
    if gpu.get("d_init") is not None:
        di, rdi = gpu["d_init"].astype(np.float64), ref["d_init"]
        ok = np.abs(di - rdi) <= 1e-4 * np.abs(rdi) + 1e-5
        assert ok.all(), f"d_init_state: {int((~ok).sum())} elements out of tolerance"
    return stats


def gpu_numpy(res: GpuResult, chans=None) -> dict:
    def sel(t, dim):
        if t is None:
            return None
        if chans is not None:
            t = t.index_select(dim, torch.as_tensor(chans, dtype=torch.long, device=t.device))
        return t

    d = dict(out=bits(sel(res.out, 1)), hist=bits(sel(res.hist, 2)))
    if res.state is not None:
        d["state"] = bits(sel(res.state, 1))
    if res.dx is not None:
        d["dx"] = bits(sel(res.dx, 1))
        d["dweight"] = sel(res.dweight, 0).cpu().numpy()
        d["dbias"] = None if res.dbias is None else sel(res.dbias, 0).cpu().numpy()
        d["d_init"] = None if res.d_init is None else sel(res.d_init, 2).cpu().numpy()
    return d
