"""Writes tests/golden/tiny_fp32_oracle.json from the fp64 oracle alone.

The fixture is a drift guard: it records summary numbers of the oracle on the
tiny fp32 decoder-layer workload (batch 1, seq 32, hidden 64, 4 query / 2 KV
heads, head dim 16, SwiGLU intermediate 172, eps 1e-6, RoPE base 1e6, lm-head
vocab 256, seed 0). Any later change of the oracle's arithmetic shows up as a
change of this file. Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as O  # noqa: E402
from bwd_qwen3_layer_gb300 import synth  # noqa: E402

TINY = dict(B=1, S=32, H=64, Hq=4, Hkv=2, d=16, I=172, eps=1e-6, rope_base=1e6)
V = 256


def compute():
    cfg = O.LayerConfig(**TINY)
    w = synth.layer_weights(0, cfg.H, cfg.Hq, cfg.Hkv, cfg.d, cfg.I)
    inp = synth.layer_inputs(0, cfg.T, cfg.H)
    Y, s = O.layer_forward(cfg, w, inp["X"])
    dX, g, _ = O.layer_backward(cfg, w, s, inp["dY"])
    lm = synth.lmhead_inputs(0, cfg.T, cfg.H, V)
    r = O.lmhead_ce(lm["X"], lm["W"], lm["targets"])
    out = {
        "workload": TINY | {"V": V, "seed": 0},
        "Y_l2": float(np.linalg.norm(Y)),
        "Y_sum": float(Y.sum()),
        "dX_l2": float(np.linalg.norm(dX)),
        "grad_l2": {k: float(np.linalg.norm(v)) for k, v in g.items()},
        "lse_sum": float(s["lse"].sum()),
        "ce_loss": r["loss"],
        "ce_argmax": [int(a) for a in r["argmax"]],
        "ce_dX_l2": float(np.linalg.norm(r["dX"])),
        "ce_dW_l2": float(np.linalg.norm(r["dW"])),
    }
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_fp32_oracle.json"), "w") as f:
        json.dump(compute(), f, indent=1, sort_keys=True)
        f.write("\n")
