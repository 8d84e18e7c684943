"""Regression pin: the oracle still reproduces its frozen outputs."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_golden_rows(oracle_mod):
    sys.path.insert(0, os.path.join(HERE, "golden"))
    import make_golden
    rows, ref, lp, ab = make_golden.compute()
    want = {}
    with open(os.path.join(HERE, "golden", "oracle_c1_rows.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            p = line.split()
            want[(int(p[0]), int(p[1]), int(p[2]), p[3])] = np.array([float(x) for x in p[4:]])
    for n, (b, h, i) in enumerate(rows):
        for name, arr in (("ref", ref), ("leanp", lp), ("ablation", ab)):
            assert np.allclose(arr[n, :8], want[(b, h, i, name)], rtol=1e-14, atol=1e-15)
