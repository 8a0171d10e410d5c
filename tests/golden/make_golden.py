"""Writes tiny_layer.json: the oracle's routing and a sample of its output on the tiny
workload (H=256, E=8, K=2, F=128, one shared expert, 16 tokens, seed 0).

Calls only ``oracle`` and the seeded input generator ``synth``.  The file is a
regression fixture for the oracle itself (its pins live in test_oracle_pins.py);
rerun this script only when a change to the oracle is justified by the pages.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402


def main():
    wl = synth.WORKLOADS["tiny"]
    cfg = oracle.config_of(wl)
    x = synth.gen_x(wl, 16)
    wr, bias = synth.gen_router(wl)
    out = oracle.layer_forward(cfg, x, wr, bias, synth.gen_experts(wl),
                               synth.gen_experts(wl, shared=True))
    doc = {
        "about": "oracle output on the tiny workload, seed 0 (regression fixture written by make_golden.py)",
        "ids": out["ids"].tolist(),
        "keff": out["keff"].tolist(),
        "w": [[float(v) for v in row] for row in out["w"]],
        "y_first8": [[float(v) for v in row[:8]] for row in out["y"]],
        "y_rms": float(np.sqrt((out["y"] ** 2).mean())),
    }
    with open(os.path.join(HERE, "tiny_layer.json"), "w") as f:
        json.dump(doc, f, indent=0)


if __name__ == "__main__":
    main()
