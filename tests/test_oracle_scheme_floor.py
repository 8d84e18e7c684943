"""The accuracy floor of the Lean-P code on diffuse rows (CPU only).

"Zyphra ZYFA: FP8 FlashAttention for AMD MI355X", "How accurate is ZYFA's FP8
attention?", reports relative RMS errors against fp64 attention; the target
for this build is 3e-2.  These pins show where the scheme itself sits, so
that a GPU result can be judged against the scheme and not only against the
target:

1. The Lean-P code floor(x + c) read as e4m3 approximates 2^((x-56)/8) with a
   log-ratio standard deviation of 3.151% whatever the offset c: the error is
   a periodic function of x (period one code) times the piecewise-linear
   mantissa of e4m3, and an offset only moves the period.  The closed form
   over one binade, with a_m = ln(1 + m/8) and g = ln(2)/8,
       E[f]   = 1/8 sum_m (a_m - g (m + 1/2))
       E[f^2] = 1/8 sum_m (a_m^2 - 2 a_m g (m + 1/2) + g^2 ((m+1)^3 - m^3)/3),
   must equal the oracle's value on a fine grid.  Rounding the exact value to
   the nearest e4m3 (the exact-softmax FP8 ablation) gives 2.65%.
2. On rows with many keys and diffuse weights the output's relative RMS
   error is the weights' own relative error: each output is a weighted mean
   of about n/e values, and independent per-key errors of size sigma move it
   by sigma times its own RMS.  On the headline workload's distribution
   (N(0,1) inputs, per-tensor e4m3, d = 128) rows with 16K and 24K keys
   therefore sit at about 3.1e-2 under both anchorings of the code grid
   (integer binades, the product's reading, and the running maximum, the
   second reading), above the 3e-2 target, and the ablation at about 2.6e-2.
   Neither anchoring can bring such rows under 3e-2.
3. The target applies to the whole output, and there the short rows weigh
   heavily: row i's output has a size of about |v| / sqrt(i), so the rows
   with fewer than 512 keys hold about half of the sum of squares at 32K,
   and their errors are smaller (few keys, dominant weights).  A uniform
   sample of a few hundred rows rarely contains them and lands near the
   long-row floor; the stratified sample of workloads.stratified_rows (all
   short rows, weighted long rows) estimates the whole output, and is pinned
   here against the exact value on a problem computed in full.
"""
import math

import numpy as np
import pytest

import oracle
from fp8_causal_prefill_flash_gb300 import workloads as wl

#: code-unit grid: 8 binades of normal e4m3 codes, 4096 points per code
X = np.linspace(40.0, 104.0, 64 * 4096, endpoint=False) + 0.5 / 4096
EXACT = 2.0 ** ((X - 56.0) / 8.0)  # e4m3 code of 2^y is 8y + 56


def floor_std_closed_form():
    g = math.log(2.0) / 8.0
    a = [math.log(1.0 + m / 8.0) for m in range(8)]
    ef = sum(a[m] - g * (m + 0.5) for m in range(8)) / 8.0
    ef2 = sum(a[m] ** 2 - 2 * a[m] * g * (m + 0.5) + g * g * ((m + 1) ** 3 - m ** 3) / 3.0
              for m in range(8)) / 8.0
    return math.sqrt(ef2 - ef * ef)


@pytest.mark.parametrize("offset", [0.0, 1.0 / 64, 0.25, 0.5, 0.75])
def test_code_error_std_is_the_same_for_every_offset(offset):
    codes = oracle.leanp_code(X + offset).astype(np.uint8)
    r = np.log(oracle.e4m3_decode(codes) / EXACT)
    assert r.std() == pytest.approx(floor_std_closed_form(), rel=2e-4)
    assert 0.0315 < r.std() < 0.0316


def test_nearest_e4m3_error_std():
    r = np.log(oracle.e4m3_round(EXACT) / EXACT)
    assert 0.0264 < r.std() < 0.0266


@pytest.fixture(scope="module")
def diffuse():
    """The headline distribution with two heads and 24576 keys; 96 rows near
    16K keys and 96 near 24K keys."""
    c = wl.make_case("fp8_h32_s32k_d128", Hq=2, Hkv=2, S=24576)
    rng = np.random.default_rng(11)
    sets = {}
    for lo in (16384, 24448):
        rows = np.stack([np.zeros(96, np.int64), rng.integers(0, 2, 96),
                         rng.integers(lo, lo + 128, 96)], 1)
        ref, _, _ = oracle.attention("ref", c.q, c.k, c.v, c.dq, c.dk, c.dv, rows=rows)
        sets[lo] = (rows, ref)
    return c, sets


def _rel(c, rows, ref, path):
    out, _, _ = oracle.attention(path, c.q, c.k, c.v, c.dq, c.dk, c.dv, rows=rows)
    return float(np.sqrt(np.mean((out - ref) ** 2)) / np.sqrt(np.mean(ref ** 2)))


@pytest.mark.parametrize("path", ["leanp", "leanp_a3"])
def test_long_diffuse_rows_sit_at_the_code_floor(diffuse, path):
    c, sets = diffuse
    for lo, (rows, ref) in sets.items():
        e = _rel(c, rows, ref, path)
        print(f"{path} rows near {lo} keys: rel-RMS {e:.4e}")
        # at the element floor (3.15%) within the sampling spread, and above 3e-2
        assert 3.0e-2 <= e <= 3.3e-2, (lo, e)


def test_long_diffuse_rows_ablation(diffuse):
    c, sets = diffuse
    for lo, (rows, ref) in sets.items():
        e = _rel(c, rows, ref, "exact_fp8")
        assert 2.45e-2 <= e <= 2.8e-2, (lo, e)


def test_stratified_sample_estimates_the_whole_output():
    """The GPU gates and the benchmark estimate the whole output's relative
    RMS error from workloads.stratified_rows (every row with fewer than 512
    keys, plus weighted rows beyond).  On a problem small enough to compute
    in full (2 heads, 2048 rows each) the estimate must equal the exact value,
    and the short rows must hold a large share of the output's sum of
    squares."""
    c = wl.make_case("fp8_h32_s32k_d128", Hq=2, Hkv=2, S=2048)
    B, Hq, Hkv, S, Dqk, Dv = c.shape
    ref, _, _ = oracle.attention("ref", c.q, c.k, c.v, c.dq, c.dk, c.dv)
    out, _, _ = oracle.attention("leanp", c.q, c.k, c.v, c.dq, c.dk, c.dv)
    exact = float(np.sqrt(np.sum((out - ref) ** 2) / np.sum(ref ** 2)))
    rows, w = wl.stratified_rows(B, Hq, S, short=512, n_long=768, seed=1)
    o = np.stack([out[b, i, h] for b, h, i in rows])
    r = np.stack([ref[b, i, h] for b, h, i in rows])
    est = float(np.sqrt(np.sum(w[:, None] * (o - r) ** 2) / np.sum(w[:, None] * r ** 2)))
    assert est == pytest.approx(exact, rel=0.03), (est, exact)
    assert w.sum() == B * Hq * S
    share = np.sum(ref[:, :512] ** 2) / np.sum(ref ** 2)
    assert share > 0.5, share
