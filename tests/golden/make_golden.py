"""Writes the oracle regression fixtures in this folder.

Calls only ``oracle`` (and the seeded input generators). The fixture records
sampled outputs and state entries of the fp64 oracle on the tiny GDA workload
(1 sequence, H=4, D_k=D_v=64, T=32, fp32 inputs, K=1, zero state, seed 0), so
that a later change to the oracle's arithmetic shows up as a diff here.
Run: python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gated_delta_net_02_gb300 import inputs  # noqa: E402

SAMPLES = [(0, 0, 0), (5, 1, 17), (31, 3, 63), (16, 2, 40), (31, 0, 1)]
STATE_SAMPLES = [(0, 0, 0), (1, 5, 9), (3, 63, 63), (2, 30, 31)]


def compute():
    b = inputs.tiny_gda(0)
    out, S, slots = oracle.forward(
        inputs.to_f64(b.q), inputs.to_f64(b.k), inputs.to_f64(b.v),
        inputs.to_f64(b.g), inputs.to_f64(b.beta), inputs.to_f64(b.state),
        mode="gda", scale=b.scale, n_slots=1)
    lines = []
    for (t, h, j) in SAMPLES:
        lines.append(f"out {t} {h} {j} {float(out[t, h, j])!r}")
    for (h, i, j) in STATE_SAMPLES:
        lines.append(f"state {h} {i} {j} {float(S[0, h, i, j])!r}")
    lines.append(f"out_l2 {float(np.linalg.norm(out))!r}")
    lines.append(f"state_l2 {float(np.linalg.norm(S))!r}")
    return lines


if __name__ == "__main__":
    path = os.path.join(HERE, "tiny_gda_oracle.txt")
    with open(path, "w") as f:
        f.write("# fp64 oracle on the tiny GDA workload (seed 0); written by "
                "make_golden.py from oracle/ only\n")
        f.write("\n".join(compute()) + "\n")
    print(path)
