#!/usr/bin/env python3
"""Throughput benchmark: one step = forward + backward of the packed width-4
causal depthwise Conv1d + SiLU on the GDP conv-channel workload
(C = 7168 = V 2048*2 + K 8*128*2 + Q 1024, rows 65536 holding 200
lognormal-length sequences, weight BF16, bias FP32), through the C ABI.

Prints one JSON line (rank 0).  ``value`` is valid tokens per second of the
whole job (all ranks; each rank is an independent replica on its own GPU),
timed with CUDA events on the launch stream over K steps after W warm-up
steps, inputs resident in HBM; each step replays the ccc_fwd and ccc_bwd
calls, each captured once as a CUDA graph.  ``e2e`` is the same metric with the inputs
copied from pinned host memory and the results copied back inside every
step.  ``roofline`` is for the backward call (the dominant kernel),
``cpu_baseline`` times the float64 oracle on a bounded sample of the same
workload on this host's cores.  ``configs`` (one GPU) holds the forward and
forward + backward throughput of every workload (tiny, dense, packed,
serving, long, and long as chained fragments), device-timed the same way.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "fwd+bwd tokens/s and effective HBM GB/s (% of ~8 TB/s) at C=7168 packed"
UNIT = "tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ setup --

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
        return dist
    return None


def job_max(value: float, dist, device) -> float:
    """Max of a per-rank number over all ranks (the job's time is its slowest
    rank's); identity on one process."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world_size: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank is a replica processing its own batch."""
    return world_size * tokens_per_rank / (ms_per_step / 1e3)


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(wl):
    """Bytes the method must move (no halo re-reads or partials).

    Forward: x read + out written for valid tokens of live sequences (-1
    sequences write zeros and read nothing), weights, bias, and 3 state rows
    read / written per sequence with a pool.  Backward: x, dy read and dx
    written per valid token, weights, bias, dweight and dbias written.  The
    saved history (3 rows per sequence, written by the forward and read by
    the backward) is not counted, so the figures err low."""
    T, C = wl.valid_tokens, wl.C
    wsz = wl.weight.element_size()
    bsz = 0 if wl.bias is None else wl.bias.element_size()
    lens = wl.lengths
    if wl.cache_indices is not None:
        live = wl.cache_indices.cpu().numpy() != -1
    else:
        live = np.ones(len(lens), dtype=bool)
    T_live = int(lens[live].sum())
    fwd = T_live * C * 2 + T * C * 2 + C * 4 * wsz + C * bsz
    if wl.conv_state is not None:
        hi = wl.has_initial_state.cpu().numpy() if wl.has_initial_state is not None else np.zeros(len(lens), bool)
        fwd += int((live & hi & (lens > 0)).sum()) * 3 * C * 2 + int((live & (lens > 0)).sum()) * 3 * C * 2
    bwd = T_live * C * 4 + T * C * 2 + C * 4 * wsz + C * bsz + C * 5 * 4
    return fwd, bwd


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"ccc_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- traffic --

# The sources that decide what the backward launch does (kernel, helpers,
# launch configuration) and the build script (compiler flags): a change to
# any of them, or extra compiler flags in the environment, makes recorded
# counters stale.
BWD_SOURCES = ("ssm_depthwise_causal_gb300/csrc/ccc_bwd.cu", "ssm_depthwise_causal_gb300/csrc/ccc_device.cuh",
               "ssm_depthwise_causal_gb300/csrc/ccc_internal.h", "ssm_depthwise_causal_gb300/csrc/ccc_api.cu",
               "ssm_depthwise_causal_gb300/_build.py")


def kernel_source_hash():
    h = hashlib.sha256()
    for f in BWD_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    h.update(os.environ.get("CCC_EXTRA_NVCC_FLAGS", "").strip().encode())
    return h.hexdigest()


def recorded_traffic():
    """DRAM bytes per backward launch from the committed ncu summary, or None
    when the kernel sources changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "bwd_packed_traffic.json")
    try:
        rec = json.load(open(p))
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------- cpu oracle --

def oracle_sample(wl, chans):
    x = wl.x[:, :chans].contiguous().cpu()
    dy = wl.dy[:, :chans].contiguous().cpu()
    w = wl.weight[:chans].cpu()
    b = None if wl.bias is None else wl.bias[:chans].cpu()
    return x, dy, w, b, wl.cu_seqlens.cpu()


def time_oracle(wl, target_s=12.0):
    """Time the float64 oracle (as it stands) on a bounded sample of the
    workload: all rows and sequences, the first `chans` channels, repeated
    `reps` times, sized to about `target_s` seconds of CPU work.  Returns
    (tokens/s scaled to the full channel count, threads, sample text, s)."""
    import oracle
    oracle.build()
    C = wl.C
    chans = min(C, 64)
    x, dy, w, b, cu = oracle_sample(wl, chans)
    t0 = time.perf_counter()
    _, _, hist = oracle.fwd(x, w, b, cu)
    oracle.bwd(x, w, b, cu, dy, hist)
    probe = max(time.perf_counter() - t0, 1e-3)
    per_chan = probe / chans
    chans = int(min(C, max(8, target_s / per_chan)))
    chans = max(8, chans - chans % 8)
    reps = max(1, int(round(target_s / (per_chan * chans))))
    x, dy, w, b, cu = oracle_sample(wl, chans)
    t0 = time.perf_counter()
    for _ in range(reps):
        _, _, hist = oracle.fwd(x, w, b, cu)
        oracle.bwd(x, w, b, cu, dy, hist)
    dt = time.perf_counter() - t0
    tok_s = reps * wl.valid_tokens * (chans / C) / dt
    sample = (f"{reps} x fwd+bwd over all {wl.valid_tokens} valid tokens, first {chans} of {C} "
              f"channels ({dt:.1f} s); tokens/s scaled by {chans}/{C}")
    return tok_s, oracle.threads(), sample, dt


# ------------------------------------------------------------------ runs --

def headline_config(wl, ws):
    """The `config` object of the headline line (the same for both arms)."""
    return {"workload": "packed C=7168 rows=65536 N=200 lognormal lengths, fwd+bwd",
            "rows": wl.rows, "C": wl.C, "n_seqs": wl.n_seqs, "valid_tokens": wl.valid_tokens,
            "weight": "bf16", "bias": "f32", "state": "none",
            "l2": "inputs larger than L2 (x, dy, out, dx 939 MB each)",
            "parallelism": f"replicas x{ws}"}


def capture(call, stream, reps=1):
    """`reps` back-to-back calls of `call` (which enqueues library calls on
    `stream` and returns how many kernels they launched) captured as one
    CUDA graph, after one eager call outside the capture; returns the graph
    and the kernel launches one replay makes."""
    stream.wait_stream(torch.cuda.current_stream())  # inputs made on the default stream
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        launches = sum(call() for _ in range(reps))
    torch.cuda.synchronize()
    return g, launches


def time_graph(g, stream):
    """Milliseconds of one replay of graph `g` on `stream`, between two CUDA
    events."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def time_flushed(call, flush, stream, K, W):
    """Per-call time of `call` (a one-launch-per-call L2-resident step) with
    L2 flushed before every call: K (flush, call) pairs captured as one CUDA
    graph, minus K flushes alone (also one graph), divided by K -- no event or
    launch gap between calls.  Also returns the per-call time with each call
    between its own two events after a flush (that includes the launch
    latency), and the kernel launches of the K calls."""
    def pair():
        flush.zero_()
        return call()

    def flush_only():
        flush.zero_()
        return 0

    g_w, _ = capture(pair, stream, reps=W)
    g_pair, n = capture(pair, stream, reps=K)
    g_flush, _ = capture(flush_only, stream, reps=K)
    time_graph(g_w, stream)
    time_graph(g_flush, stream)
    ms = (time_graph(g_pair, stream) - time_graph(g_flush, stream)) / K
    g_one, _ = capture(call, stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            g_one.replay()
            b.record(stream)
    torch.cuda.synchronize()
    return ms, statistics.mean(a.elapsed_time(b) for a, b in ev), n


def time_calls(call, stream, K, W):
    """Milliseconds per call of K back-to-back calls of `call`, captured as
    one CUDA graph and replayed once, after W warm-up calls (their own
    graph); returns (ms per call, kernel launches in the timed region)."""
    g_w, _ = capture(call, stream, reps=W)
    g_k, n = capture(call, stream, reps=K)
    time_graph(g_w, stream)
    return time_graph(g_k, stream) / K, n


def run_reference(args, ws, rank):
    from ssm_depthwise_causal_gb300 import workloads
    if rank != 0:
        return
    wl = workloads.packed(device="cpu")
    vals = []
    threads, sample = 0, ""
    # each step a bounded sample: at most --ref-seconds, and about 100 s of
    # planned work for all K steps together (the all-channel samples run ~1.4x
    # the plan), so the whole run ends within a few minutes
    target = max(2.0, min(args.ref_seconds, 100.0 / max(1, args.steps)))
    for _ in range(args.warmup):
        time_oracle(wl, target_s=min(2.0, target))
    for _ in range(args.steps):
        v, threads, sample, _ = time_oracle(wl, target_s=target)
        vals.append(v)
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wl.valid_tokens / v,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": headline_config(wl, args.gpus),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, ws, rank, local):
    import ssm_depthwise_causal_gb300 as ccc
    from ssm_depthwise_causal_gb300 import workloads

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(ws, "nccl")
    ccc._lib.lib()  # fail loudly if the library is missing

    wl = workloads.packed(device=dev)
    T, C, N, rows = wl.valid_tokens, wl.C, wl.n_seqs, wl.rows
    config = headline_config(wl, ws)
    out = torch.empty_like(wl.x)
    dx = torch.empty_like(wl.x)
    hist = torch.empty((N, 3, C), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((C, 4), dtype=torch.float32, device=dev)
    db = torch.empty((C,), dtype=torch.float32, device=dev)
    ws_f = torch.empty(max(1, ccc.ccc_workspace_size(rows, N, C, False)), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(ccc.ccc_workspace_size(rows, N, C, True), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    # The step's calls with CCC_OPT_OVERLAP_PROLOGUE: each kernel's prologue
    # may overlap the kernel before it.  The contract holds here: a forward
    # follows the previous step's reduce (which writes dweight / dbias), a
    # backward follows its forward; neither writes the offsets or the taps.
    def fwd_call(overlap=True):
        ccc.ccc_fwd(wl.x, wl.weight, wl.bias, None, wl.cu_seqlens, None, None, out, hist, ws_f, stream=stream,
                    overlap=overlap)
        return ccc.last_launch_count()

    def bwd_call(overlap=True):
        ccc.ccc_bwd(wl.x, wl.weight, wl.bias, hist, wl.cu_seqlens, None, None, wl.dy, None, dx, dw, db, None,
                    ws_b, stream=stream, overlap=overlap)
        return ccc.last_launch_count()

    def step_call():
        return fwd_call() + bwd_call()

    def plain_step_call():
        return fwd_call(False) + bwd_call(False)

    # K steps (ccc_fwd then ccc_bwd) captured as one CUDA graph -- the
    # library neither allocates nor synchronizes, so its calls capture -- and
    # replayed once between two events, after W warm-up steps (their own
    # graph); then K of each call alone (forward / backward split and the
    # backward's roofline).
    K = args.steps
    g_warm, _ = capture(step_call, stream, reps=args.warmup)
    g_step, gpu_launches = capture(step_call, stream, reps=K)
    time_graph(g_warm, stream)
    clocks = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    elapsed_ms = time_graph(g_step, stream)
    fwd_ms, _ = time_calls(fwd_call, stream, K, args.warmup)
    bwd_ms, _ = time_calls(bwd_call, stream, K, args.warmup)
    plain_ms, _ = time_calls(plain_step_call, stream, K, args.warmup)
    clk = clocks.stop()
    if dist:
        dist.barrier()
    elapsed_ms = job_max(elapsed_ms, dist, dev)
    ms_step = elapsed_ms / K
    value = job_throughput(ws, T, ms_step)
    fb, bb = algorithmic_bytes(wl)
    peak, peak_kind = measured_peak()
    eff_gbs = (fb + bb) / (ms_step / 1e3) / 1e9
    bwd_gbs = bb / (bwd_ms / 1e3) / 1e9

    # ---- end to end: every step copies its inputs in from pinned host memory
    # and its results out, through the public API.  Steps are pipelined the
    # way a caller would run them: two device buffer sets, one stream per
    # direction of copy and one for compute, so step k+1's inputs travel in
    # while step k computes and step k-1's results travel out.
    hx = torch.empty(wl.x.shape, dtype=wl.x.dtype, pin_memory=True)
    hdy = torch.empty(wl.dy.shape, dtype=wl.dy.dtype, pin_memory=True)
    hx.copy_(wl.x)
    hdy.copy_(wl.dy)
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    hdx = torch.empty(dx.shape, dtype=dx.dtype, pin_memory=True)
    hdw = torch.empty(dw.shape, dtype=dw.dtype, pin_memory=True)
    hdb = torch.empty(db.shape, dtype=db.dtype, pin_memory=True)
    sets = []
    for _ in range(2):
        sets.append(dict(x=torch.empty_like(wl.x), dy=torch.empty_like(wl.dy), out=torch.empty_like(wl.x),
                         dx=torch.empty_like(wl.x), hist=torch.empty_like(hist), dw=torch.empty_like(dw),
                         db=torch.empty_like(db)))
    h2d = hx.numel() * 2 + hdy.numel() * 2
    d2h = hout.numel() * 2 + hdx.numel() * 2 + hdw.numel() * 4 + hdb.numel() * 4
    e2e_steps = max(4, K)  # the same number of steps as the device-timed region
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_free = [None, None]   # compute of the step two back is done with set b's inputs
    out_free = [None, None]  # results of the step two back have left set b

    def e2e_step(k):
        b = k % 2
        d = sets[b]
        with torch.cuda.stream(s_in):
            if in_free[b] is not None:
                s_in.wait_event(in_free[b])
            d["x"].copy_(hx, non_blocking=True)
            d["dy"].copy_(hdy, non_blocking=True)
            in_ready = ev()
            in_ready.record(s_in)
        with torch.cuda.stream(stream):
            stream.wait_event(in_ready)
            if out_free[b] is not None:
                stream.wait_event(out_free[b])
            ccc.ccc_fwd(d["x"], wl.weight, wl.bias, None, wl.cu_seqlens, None, None, d["out"], d["hist"], ws_f,
                        stream=stream)
            fwd_done = ev()
            fwd_done.record(stream)
            ccc.ccc_bwd(d["x"], wl.weight, wl.bias, d["hist"], wl.cu_seqlens, None, None, d["dy"], None, d["dx"],
                        d["dw"], d["db"], None, ws_b, stream=stream)
            bwd_done = ev()
            bwd_done.record(stream)
            in_free[b] = bwd_done
        with torch.cuda.stream(s_out):
            s_out.wait_event(fwd_done)
            hout.copy_(d["out"], non_blocking=True)
            s_out.wait_event(bwd_done)
            hdx.copy_(d["dx"], non_blocking=True)
            hdw.copy_(d["dw"], non_blocking=True)
            hdb.copy_(d["db"], non_blocking=True)
            done = ev()
            done.record(s_out)
            out_free[b] = done

    for k in range(2):  # warm the pipeline's buffers and streams
        e2e_step(k)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    in_free[:] = [None, None]
    out_free[:] = [None, None]
    e0.record(s_in)
    s_out.wait_stream(s_in)
    stream.wait_stream(s_in)
    for k in range(e2e_steps):
        e2e_step(k)
    s_out.wait_stream(stream)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = job_max(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    e2e_val = job_throughput(ws, T, e2e_ms)
    link = measure_link([(sets[0]["x"], hx), (sets[0]["dy"], hdy)],
                        [(hout, sets[0]["out"]), (hdx, sets[0]["dx"])], s_in, s_out)
    link["e2e_copy_gbs"] = (h2d + d2h) / (e2e_ms / 1e3) / 1e9
    link["frac"] = link["e2e_copy_gbs"] / link["both_gbs"]

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        tok_s, threads, sample, _ = time_oracle(wl, target_s=args.ref_seconds)
        cpu = {"value": tok_s, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample}

    # ---- every workload's forward and forward + backward (one GPU)
    configs = None
    if ws == 1 and not args.no_configs:
        wl = out = dx = hist = sets = hx = hdy = hout = hdx = None  # the headline's buffers are done
        torch.cuda.empty_cache()
        cclk = ClockSampler(local)
        cclk.start()
        rows_c, launches_c = time_configs(dev, K, args.warmup)
        configs = {"unit_gbs": "GB/s (algorithmic bytes / CUDA-event time)", "peak": peak,
                   "peak_kind": peak_kind, "steps": K, "warmup": args.warmup, "workloads": rows_c,
                   "gpu_launches": launches_c, "clocks": cclk.stop()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage_dtype": "bf16",
            "data": "synthetic",
            "config": config,
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "launch": "calls with CCC_OPT_OVERLAP_PROLOGUE (ccc_fwd_ex / ccc_bwd_ex), K steps in one CUDA graph",
            "ms_per_step_plain_launch": plain_ms,
            "fwd_tokens_per_s": ws * T / (fwd_ms / 1e3),
            "effective_gbs": eff_gbs, "frac_of_nominal_8tbs": eff_gbs / NOMINAL_HBM_GBS,
            "frac_of_measured_hbm": eff_gbs / peak,
            "roofline": {"kernel": "ccc_bwd call (fused backward + ordered reduce)",
                         "bound": "hbm", "achieved": bwd_gbs, "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": bwd_gbs / peak, "traffic": recorded_traffic(),
                         "algorithmic_bytes_per_launch": bb},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "steps": e2e_steps,
                    "how": "pinned host x, dy in and out, dx, dweight, dbias back every step; steps pipelined "
                           "over two device buffer sets with separate copy-in, compute and copy-out streams",
                    "link": link},
            "gpu_launches": gpu_launches,
            "clocks": clk,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def measure_link(h2d_pairs, d2h_pairs, s_in, s_out, reps=3):
    """The host link's ceiling on the e2e step's own pinned buffers: the
    step's input copies alone, its result copies alone, and both at once on
    separate streams (which the pipelined step overlaps).  GB/s, best of
    `reps`; pairs are (dst, src)."""
    def run(pairs_in, pairs_out):
        best = None
        nbytes = sum(d.numel() * d.element_size() for d, _ in pairs_in + pairs_out)
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            with torch.cuda.stream(s_in):
                for d, h in pairs_in:
                    d.copy_(h, non_blocking=True)
            with torch.cuda.stream(s_out):
                for h, d in pairs_out:
                    h.copy_(d, non_blocking=True)
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        return nbytes / best / 1e9
    return {"h2d_gbs": run(h2d_pairs, []), "d2h_gbs": run([], d2h_pairs), "both_gbs": run(h2d_pairs, d2h_pairs),
            "how": "pinned-host copies of the step's x, dy in and out, dx back, on separate copy streams"}


UPDATE_METRIC = "decode-step tokens/s and effective HBM GB/s of ccc_update (serving pool, C=8192)"


def update_algorithmic_bytes(wl):
    """Bytes a decode step must move: x read and out written for the new
    tokens of live requests (-1 requests write zeros only), W-1 state values
    read and min(len + W-2, L) written per live channel, weights and bias.
    Also returns the state bytes a dense history-contiguous pool moves at
    sector granularity (each live slot's [C, L] block read and written)."""
    C, W = wl.C, wl.width
    H = W - 1
    L = wl.conv_state.shape[2]
    lens = wl.lengths
    live = wl.cache_indices.cpu().numpy() != -1
    ne = lens > 0
    n_w = np.minimum(lens + H - 1, L)
    b = int((lens[live] * 4).sum()) * C + int((lens[~live] * 2).sum()) * C
    b += int((live & ne).sum()) * C * 2 * H + int((n_w[live & ne] * 2).sum()) * C
    b += C * W * wl.weight.element_size() + (0 if wl.bias is None else C * wl.bias.element_size())
    block = int((lens[live] * 4).sum()) * C + int((lens[~live] * 2).sum()) * C + int((live & ne).sum()) * C * 4 * L
    return b, block


def run_update(args, ws, rank, local):
    """Decode-step timing of ccc_update: K steps, each after an L2 flush (the
    whole step's working set fits in L2), timed alone with CUDA events."""
    import ssm_depthwise_causal_gb300 as ccc
    from ssm_depthwise_causal_gb300 import workloads

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(ws, "nccl")
    ccc._lib.lib()
    wl = workloads.WORKLOADS[args.workload](device=dev)
    if wl.num_accepted is None:
        raise SystemExit("--op update needs a decode workload (decode, spec_decode)")
    T, C, N = wl.valid_tokens, wl.C, wl.n_seqs
    pool = wl.conv_state
    out = torch.empty_like(wl.x)
    acc = wl.num_accepted if wl.lengths.max() > 1 else None
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    # With CCC_OPT_OVERLAP_PROLOGUE the step's first round trip (offsets,
    # slots, accepted counts, taps) overlaps the kernel before it.  The
    # contract holds: the kernel before each step is the L2 flush (or the
    # previous step), which writes none of those.
    def call(x, s, overlap=True):
        ccc.ccc_update(x, wl.weight, wl.bias, pool, wl.cu_seqlens, wl.cache_indices, acc, out, stream=s,
                       overlap=overlap)

    K = args.steps
    step = lambda: (call(wl.x, stream), ccc.last_launch_count())[1]  # noqa: E731
    plain_step = lambda: (call(wl.x, stream, False), ccc.last_launch_count())[1]  # noqa: E731
    clocks = ClockSampler(local)
    if dist:
        dist.barrier()
    clocks.start()
    time.sleep(0.3)
    ms, ms_events, launches = time_flushed(step, flush, stream, K, args.warmup)
    ms_plain, _, _ = time_flushed(plain_step, flush, stream, K, args.warmup)
    clk = clocks.stop()
    ms = job_max(ms, dist, dev)
    value = job_throughput(ws, T, ms)
    alg, block = update_algorithmic_bytes(wl)
    peak, peak_kind = measured_peak()
    gbs = alg / (ms / 1e3) / 1e9

    # end to end: the new tokens from pinned host memory, outputs back
    hx = torch.empty(wl.x.shape, dtype=wl.x.dtype, pin_memory=True)
    hx.copy_(wl.x)
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    xin = torch.empty_like(wl.x)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(K):
            xin.copy_(hx, non_blocking=True)
            call(xin, stream)
            hout.copy_(out, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = job_max(e0.elapsed_time(e1) / K, dist, dev)
    if rank == 0:
        line = {
            "metric": UPDATE_METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "storage_dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "n_seqs": N, "tokens": T, "C": C,
                       "pool": list(pool.shape), "l2": "flushed before every timed step (working set < L2)",
                       "parallelism": f"replicas x{ws}"},
            "effective_gbs": gbs,
            "timing": "K (L2 flush, step) pairs in one CUDA graph minus K flushes alone, per step; "
                      "ms_per_step_events: each step between its own events after a flush",
            "launch": "CCC_OPT_OVERLAP_PROLOGUE (the step's metadata and tap loads overlap the kernel "
                      "before it); ms_per_step_plain_launch: the same without the option",
            "ms_per_step_events": ms_events,
            "ms_per_step_plain_launch": job_max(ms_plain, dist, dev),
            "roofline": {"kernel": "update_block_kernel (one launch per step)", "bound": "hbm", "achieved": gbs,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": None, "algorithmic_bytes_per_launch": alg,
                         "state_block_bytes_per_launch": block},
            "e2e": {"value": job_throughput(ws, T, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": hout.numel() * 2,
                    "ms_per_step": e2e_ms},
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def run_profile(args, local):
    """W warm-up steps then one step of the same calls, nothing else: the
    command the ncu captures run."""
    import ssm_depthwise_causal_gb300 as ccc
    from ssm_depthwise_causal_gb300 import workloads
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = workloads.WORKLOADS[args.workload](device=dev)
    T, C, N, rows = wl.valid_tokens, wl.C, wl.n_seqs, wl.rows
    out = torch.empty_like(wl.x)
    if wl.num_accepted is not None:  # a decode step: ccc_update only
        acc = wl.num_accepted if wl.lengths.max() > 1 else None
        for _ in range(args.warmup + 1):
            ccc.ccc_update(wl.x, wl.weight, wl.bias, wl.conv_state, wl.cu_seqlens, wl.cache_indices, acc, out)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": wl.name, "valid_tokens": T}), flush=True)
        return
    hist = torch.empty((N, 3, C), dtype=torch.bfloat16, device=dev)
    ws_f = torch.empty(max(1, ccc.ccc_workspace_size(rows, N, C, False)), dtype=torch.uint8, device=dev)
    state = None if wl.conv_state is None else wl.conv_state.clone()
    if wl.training:
        dx = torch.empty_like(wl.x)
        dw = torch.empty((C, 4), dtype=torch.float32, device=dev)
        db = None if wl.bias is None else torch.empty((C,), dtype=torch.float32, device=dev)
        ws_b = torch.empty(ccc.ccc_workspace_size(rows, N, C, True), dtype=torch.uint8, device=dev)
    for _ in range(args.warmup + 1):
        ccc.ccc_fwd(wl.x, wl.weight, wl.bias, state, wl.cu_seqlens, wl.cache_indices,
                    wl.has_initial_state, out, hist, ws_f)
        if wl.training:
            ccc.ccc_bwd(wl.x, wl.weight, wl.bias, hist, wl.cu_seqlens, wl.cache_indices,
                        wl.has_initial_state, wl.dy, None, dx, dw, db, None, ws_b)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": wl.name, "valid_tokens": T}), flush=True)


CONFIG_WORKLOADS = ("tiny", "dense", "packed", "serving", "long")


def working_set_bytes(wl):
    """Device bytes one step touches: x and out (and dy, dx when training),
    plus the pool."""
    n = wl.x.numel() * 2 * (4 if wl.training else 2)
    if wl.conv_state is not None:
        n += wl.conv_state.numel() * 2
    return n


def time_fragment_chain(ccc, wl, out, dx, stream, steps, warmup):
    """The long document as `fragments` consecutive calls chained through a
    one-slot pool (forward: fragment k reads the state fragment k-1 wrote;
    backward in reverse, d_init_state of fragment k as d_final_state of
    fragment k-1): device time of the forward chain and of the backward chain
    (the host-side sum of the per-fragment dweight is not included).  Steps
    run back to back: every tensor is far larger than L2."""
    dev = wl.x.device
    T, C, F = wl.rows, wl.C, wl.fragments
    Lf = T // F
    pool = torch.zeros((1, C, 4), dtype=torch.bfloat16, device=dev)
    cache = torch.zeros(1, dtype=torch.int32, device=dev)
    cu_f = torch.tensor([0, Lf], dtype=torch.int32, device=dev)
    flags = [torch.tensor([k > 0], device=dev) for k in range(F)]
    hists = [torch.empty((1, 3, C), dtype=torch.bfloat16, device=dev) for _ in range(F)]
    d_init = [torch.empty((1, 3, C), dtype=torch.float32, device=dev) for _ in range(F)]
    dws = [torch.empty((C, 4), dtype=torch.float32, device=dev) for _ in range(F)]
    ws_f = torch.empty(ccc.ccc_workspace_size(Lf, 1, C, True), dtype=torch.uint8, device=dev)
    part = lambda t, k: t[k * Lf:(k + 1) * Lf]  # noqa: E731

    def fwd_chain():
        n = 0
        for k in range(F):
            ccc.ccc_fwd(part(wl.x, k), wl.weight, wl.bias, pool, cu_f, cache, flags[k], part(out, k), hists[k],
                        None, stream=stream, overlap=True)
            n += ccc.last_launch_count()
        return n

    def bwd_chain():
        n, carry = 0, None
        for k in reversed(range(F)):
            ccc.ccc_bwd(part(wl.x, k), wl.weight, wl.bias, hists[k], cu_f, cache, flags[k], part(wl.dy, k), carry,
                        part(dx, k), dws[k], None, d_init[k], ws_f, stream=stream, overlap=True)
            n += ccc.last_launch_count()
            carry = d_init[k]
        return n

    s_ms, n = time_calls(lambda: fwd_chain() + bwd_chain(), stream, steps, warmup)
    f_ms, _ = time_calls(fwd_chain, stream, steps, warmup)
    b_ms, _ = time_calls(bwd_chain, stream, steps, warmup)
    return {"split_fragments": F, "split_fwd_ms": f_ms, "split_bwd_ms": b_ms, "split_step_ms": s_ms,
            "split_step_tokens_per_s": T / (s_ms / 1e3)}, n


def time_configs(dev, steps, warmup):
    """Forward and (for training workloads) forward + backward of every
    workload through the C ABI, each call captured once as a CUDA graph and
    replayed, device-timed with CUDA events on the launch stream: `steps`
    steps after `warmup` warm-up steps.  A workload whose
    step touches more than twice the L2 size runs its steps back to back
    (as the headline does); a smaller one (the tiny batch) is preceded by an
    L2 flush (a write of twice the L2 size) every step.  A forward with a
    pool updates it in place every step; the work per step does not depend on
    the values, so the pool is not restored between steps.  Returns (rows,
    kernel launches in the timed regions)."""
    import ssm_depthwise_causal_gb300 as ccc
    from ssm_depthwise_causal_gb300 import workloads

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = None
    peak, _ = measured_peak()
    stream = torch.cuda.Stream(device=dev)
    rows_out = []
    for name in CONFIG_WORKLOADS:
        wl = workloads.WORKLOADS[name](device=dev)
        T, C, N, rows = wl.valid_tokens, wl.C, wl.n_seqs, wl.rows
        flushed = working_set_bytes(wl) < 2 * l2
        if flushed and flush is None:
            flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
        out = torch.empty_like(wl.x)
        hist = torch.empty((N, 3, C), dtype=torch.bfloat16, device=dev)
        state = wl.conv_state
        dx = dw = db = ws_b = None
        if wl.training:
            dx = torch.empty_like(wl.x)
            dw = torch.empty((C, 4), dtype=torch.float32, device=dev)
            db = None if wl.bias is None else torch.empty((C,), dtype=torch.float32, device=dev)
            ws_b = torch.empty(ccc.ccc_workspace_size(rows, N, C, True), dtype=torch.uint8, device=dev)

        # with CCC_OPT_OVERLAP_PROLOGUE, as the headline (each call follows
        # this library's previous call or an L2 flush)
        def fwd():
            ccc.ccc_fwd(wl.x, wl.weight, wl.bias, state, wl.cu_seqlens, wl.cache_indices, wl.has_initial_state,
                        out, hist, None, stream=stream, overlap=True)
            return ccc.last_launch_count()

        def bwd():
            ccc.ccc_bwd(wl.x, wl.weight, wl.bias, hist, wl.cu_seqlens, wl.cache_indices, wl.has_initial_state,
                        wl.dy, None, dx, dw, db, None, ws_b, stream=stream, overlap=True)
            return ccc.last_launch_count()

        K = steps
        if flushed:  # L2 flushed before every call (see time_flushed)
            fwd_ms, _, n_f = time_flushed(fwd, flush, stream, K, warmup)
            bwd_ms = step_ms = None
            timed_launches = n_f
            if wl.training:
                bwd_ms, _, n_b = time_flushed(bwd, flush, stream, K, warmup)
                step_ms = fwd_ms + bwd_ms
                timed_launches += n_b
        else:  # back to back: K calls in one graph between two events (as the headline)
            fwd_ms, timed_launches = time_calls(fwd, stream, K, warmup)
            bwd_ms = step_ms = None
            if wl.training:
                bwd_ms, _ = time_calls(bwd, stream, K, warmup)
                step_ms, timed_launches = time_calls(lambda: fwd() + bwd(), stream, K, warmup)
        fb, bb = algorithmic_bytes(wl)
        row = {"workload": wl.name, "valid_tokens": T, "C": C, "n_seqs": N,
               "l2": ("flushed before every call: K (flush, call) pairs in one CUDA graph minus K flushes"
                      if flushed else "inputs larger than L2, K calls back to back in one CUDA graph between two events"),
               "fwd_ms": fwd_ms, "fwd_tokens_per_s": T / (fwd_ms / 1e3),
               "fwd_gbs": fb / (fwd_ms / 1e3) / 1e9, "fwd_frac": fb / (fwd_ms / 1e3) / 1e9 / peak,
               "fwd_algorithmic_bytes": fb}
        if wl.training:
            row.update({"bwd_ms": bwd_ms, "bwd_gbs": bb / (bwd_ms / 1e3) / 1e9,
                        "bwd_frac": bb / (bwd_ms / 1e3) / 1e9 / peak, "bwd_algorithmic_bytes": bb,
                        "step_ms": step_ms, "step_tokens_per_s": T / (step_ms / 1e3),
                        "step_gbs": (fb + bb) / (step_ms / 1e3) / 1e9,
                        "step_frac": (fb + bb) / (step_ms / 1e3) / 1e9 / peak})
        rows_out.append((row, timed_launches))
        if wl.training and getattr(wl, "fragments", 1) > 1:
            chain, n_chain = time_fragment_chain(ccc, wl, out, dx, stream, steps, warmup)
            row.update(chain)
            rows_out[-1] = (row, timed_launches + n_chain)
        wl = out = hist = state = dx = dw = db = ws_b = None  # free this workload's tensors
        torch.cuda.empty_cache()
    flush = None
    torch.cuda.empty_cache()
    return [r for r, _ in rows_out], sum(n for _, n in rows_out)


def run_configs(args, local):
    """--op configs: the per-workload table alone, one JSON line."""
    import ssm_depthwise_causal_gb300 as ccc

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    ccc._lib.lib()
    peak, peak_kind = measured_peak()
    clocks = ClockSampler(local)
    clocks.start()
    rows, launches = time_configs(dev, args.steps, args.warmup)
    clk = clocks.stop()
    print(json.dumps({"op": "configs", "steps": args.steps, "warmup": args.warmup, "peak": peak,
                      "peak_kind": peak_kind, "unit_gbs": "GB/s (algorithmic bytes / CUDA-event time)",
                      "data": "synthetic", "configs": rows, "gpu_launches": launches, "clocks": clk}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-seconds", type=float, default=12.0,
                    help="approximate CPU seconds of one oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload table (forward and forward+backward of every workload)")
    ap.add_argument("--profile", action="store_true",
                    help="run warm-up + one step of --workload only (for ncu captures)")
    ap.add_argument("--workload", default="packed",
                    choices=["tiny", "dense", "packed", "packed_small", "serving", "long", "decode", "spec_decode"])
    ap.add_argument("--op", default="fwdbwd", choices=["fwdbwd", "update", "configs"],
                    help="fwdbwd: the packed training step (the headline); update: one decode step "
                         "(ccc_update) of --workload decode / spec_decode; configs: forward and "
                         "forward+backward of every workload, device-timed")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    ws, rank, local = dist_env()
    if args.profile:
        run_profile(args, local)
    elif args.op == "configs":
        run_configs(args, local)
    elif args.op == "update":
        if args.workload not in ("decode", "spec_decode"):
            args.workload = "decode"
        run_update(args, ws, rank, local)
    elif args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
