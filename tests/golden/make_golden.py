"""Writes the stored expected values under tests/golden/ from the oracle (and the seeded generator) only.

Run from the repository root: python tests/golden/make_golden.py
"""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402


def main():
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w, seed=0)
    du = inp["d_u"].copy()
    oracle.run_steps(du, inp["x"], inp["d_dv"], w.P)
    words = du.reshape(-1).view(np.uint32)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_seed0_after_4_steps.txt")
    with open(path, "w") as f:
        f.write("# d_u bits (hex, row-major [8, 16, 32]) after steps ti = 0..3 of the tiny workload\n")
        f.write("# (T=4, P=2, C=16, hd=32, all N(0,1), seed 0); written by tests/golden/make_golden.py from the oracle\n")
        for k in range(0, words.size, 8):
            f.write(" ".join(f"{v:08x}" for v in words[k:k + 8]) + "\n")


if __name__ == "__main__":
    main()
