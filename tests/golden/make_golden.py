"""Writes tests/golden/worked_example.json from the float64 oracle alone.

The pages print no worked example, so this fixture is a frozen oracle run on
a hand-picked input whose outputs also have closed forms (checked by
tests/test_golden.py): one channel group of C = 8, a sequence of length 6 with
x[t, c] = (t + 1) / 8 for c = 0 and zeros elsewhere, taps w[c] = (1/2, -1/4,
1/8, 1) (tap 3 on the current token, FlashInfer causal_conv1d_fn, weight),
bias 1/16, and a three-value initial state (1, -1, 1/2) read from slot 1 of a
two-slot pool (causal_conv1d_fn, conv_state / has_initial_state).

Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def example():
    C, L = 8, 6
    x = np.zeros((L, C), np.float32)
    x[:, 0] = (np.arange(L) + 1) / 8.0
    w = np.tile(np.array([0.5, -0.25, 0.125, 1.0]), (C, 1))
    b = np.full(C, 1.0 / 16)
    state = np.zeros((2, C, 4), np.float32)
    state[1, 0, 0:3] = [1.0, -1.0, 0.5]
    state[1, 0, 3] = 7.0
    return dict(x=x, w=w, b=b, state=state, cu=[0, L], cache=[1], has_init=[True])


def run(ex):
    bf = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)
    out, st, hist = oracle.fwd(bf(ex["x"]), ex["w"], ex["b"], torch.tensor(ex["cu"], dtype=torch.int32),
                               bf(ex["state"]), torch.tensor(ex["cache"], dtype=torch.int32),
                               torch.tensor(ex["has_init"]))
    dy = np.ones_like(ex["x"])
    g = oracle.bwd(bf(ex["x"]), ex["w"], ex["b"], torch.tensor(ex["cu"], dtype=torch.int32), bf(dy),
                   hist, torch.tensor(ex["cache"], dtype=torch.int32), torch.tensor(ex["has_init"]))
    return dict(out_c0=out[:, 0].tolist(), out_c1=out[:, 1].tolist(),
                state_c0=oracle.bf16_bits_to_f64(st[1, 0]).tolist(),
                dx_c0=g["dx"][:, 0].tolist(), dweight_c0=g["dweight"][0].tolist(),
                dbias_c0=float(g["dbias"][0]), d_init_c0=g["d_init"][0, :, 0].tolist())


if __name__ == "__main__":
    ex = example()
    res = run(ex)
    doc = {"source": "frozen float64 oracle run (tests/golden/make_golden.py); inputs listed there",
           "results": res}
    with open(os.path.join(HERE, "worked_example.json"), "w") as f:
        json.dump(doc, f, indent=1)
    print("wrote worked_example.json")
