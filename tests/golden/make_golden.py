"""Writes tests/golden/tiny_oracle.txt: the oracle's output on the seeded 'tiny'
workload (M=1, K=1024, N=256).  Calls only the seeded generator and oracle/.

Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402


def main():
    w = synth.workload("tiny")
    bits, scales, signs, x = synth.make_inputs(w)
    y = oracle.forward(bits, scales, signs, w.perm, x)[0]
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.txt")
    with open(path, "w") as f:
        f.write("# oracle y[0][n] for the seeded tiny workload (M=1, K=1024, N=256, seed 0xB1711A01)\n")
        f.write("# written by tests/golden/make_golden.py (calls synth and oracle only)\n")
        for v in y:
            f.write(f"{v:.17g}\n")
    print("wrote", path, np.linalg.norm(y))


if __name__ == "__main__":
    main()
