"""Write tests/golden/tiny_fp32_fwd.txt from the fp64 oracle (and nothing else).

The pages print no worked numeric example of the scan, so this fixture is a
regression record of the oracle itself on the tiny fp32 workload (batch 1,
D=16, N=4, L=64, seed 0, A = -(n+1) without jitter, h0 = 0): any later change
to the oracle's arithmetic shows up as a diff here.  Run from the repo root:
    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from scan_inputs import WORKLOADS, make_inputs  # noqa: E402


def compute():
    w = dict(WORKLOADS["tiny_fp32"])
    x = make_inputs(w["Bt"], w["D"], w["N"], w["L"], seed=w["seed"], in_dtype="f32",
                    a_jitter=w["a_jitter"])
    return oracle.scan_fwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)


def main():
    y, hL = compute()
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_fp32_fwd.txt")
    with open(path, "w") as f:
        f.write("# oracle regression record: tiny fp32 forward (1,16,4,64), seed 0\n")
        f.write("# written by tests/golden/make_golden.py from oracle.scan_fwd only\n")
        f.write("# y: 16 rows x 64 values, then hL: 16 rows x 4 values\n")
        for row in y[0]:
            f.write(" ".join(repr(float(v)) for v in row) + "\n")
        for row in hL[0]:
            f.write(" ".join(repr(float(v)) for v in row) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
