"""The byte counts behind bench.py's effective-bandwidth and roofline
figures, checked by hand on small CPU workloads (no GPU needed)."""
import numpy as np
import torch

import bench
from ssm_depthwise_causal_gb300 import workloads


def test_fwdbwd_bytes_packed_without_state():
    wl = workloads.make_custom((5, 0, 7), 16, rows=15, seed=1, with_state=False,
                               w_dtype=torch.bfloat16)
    fwd, bwd = bench.algorithmic_bytes(wl)
    T, C = 12, 16
    assert fwd == T * C * 2 + T * C * 2 + C * 4 * 2 + C * 4
    assert bwd == T * C * 4 + T * C * 2 + C * 4 * 2 + C * 4 + C * 5 * 4


def test_update_bytes_by_hand():
    wl = workloads.decode(device="cpu", C=16, N=6, slots=12, draft=3, state_len=6, n_minus_one=2)
    alg, block = bench.update_algorithmic_bytes(wl)
    C, L, H = 16, 6, 3
    live = (wl.cache_indices.numpy() != -1)
    n_live, n_dead = int(live.sum()), int((~live).sum())
    per_live = 3 * 4 + 2 * H + 2 * min(3 + H - 1, L)          # x + out, state read, state write
    expect = C * (n_live * per_live + n_dead * 3 * 2) + C * 4 * 4 + C * 2
    assert alg == expect
    assert block == C * (n_live * (3 * 4 + 4 * L) + n_dead * 3 * 2)
    assert n_dead == 2 and np.all(wl.lengths == 3)


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the oracle timed on the host cores) runs
    without a GPU and prints the contract's JSON line."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--ref-seconds", "0.2"], capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["higher_is_better"] is True and line["vs_baseline"] is None
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["C"] == 7168 and line["config"]["rows"] == 65536


def test_reference_arm_line():
    """`bench.py --impl reference` (the float64 oracle on the host cores; no
    GPU) prints one JSON line with the keys the benchmark contract names."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--ref-seconds", "1"], capture_output=True, text=True, timeout=600,
                         cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0 and line["warmup"] >= 3
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert "workload" in line["config"]
