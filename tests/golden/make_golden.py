"""Write tests/golden/oracle_c1_rows.txt from the oracle alone.

The fixture freezes the oracle's outputs on a few rows of the 2-head, S=256,
d128 Gaussian FP8 workload so that any later change to the oracle's arithmetic
shows up as a diff (and must then name the passage that justifies it).
Run:  python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from fp8_causal_prefill_flash_gb300 import workloads as wl  # noqa: E402

ROWS = [(0, h, i) for h in (0, 1) for i in (0, 1, 2, 63, 64, 65, 127, 128, 200, 255)]


def compute():
    c = wl.make_case("fp8_h2_s256_d128")
    rows = np.array(ROWS, dtype=np.int64)
    ref = oracle.ref_fp64(c.q, c.k, c.v, c.dq, c.dk, c.dv, rows=rows)
    lp, _ = oracle.emul_leanp(c.q, c.k, c.v, c.dq, c.dk, c.dv, rows=rows)
    ab, _ = oracle.emul_exact_fp8(c.q, c.k, c.v, c.dq, c.dk, c.dv, rows=rows)
    return rows, ref, lp, ab


def main():
    rows, ref, lp, ab = compute()
    path = os.path.join(HERE, "oracle_c1_rows.txt")
    with open(path, "w") as f:
        f.write("# oracle outputs, 2-head S=256 d128 Gaussian FP8 workload (seeds 0,1,2)\n")
        f.write("# written by tests/golden/make_golden.py from oracle/ only\n")
        f.write("# b h i path d0..d7 (%.17g)\n")
        for n, (b, h, i) in enumerate(rows):
            for name, arr in (("ref", ref), ("leanp", lp), ("ablation", ab)):
                vals = " ".join("%.17g" % x for x in arr[n, :8])
                f.write(f"{b} {h} {i} {name} {vals}\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
