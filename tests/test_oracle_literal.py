"""Hand-expanded Lean-P cases with literal codes and weights (CPU only).

Each expected value below was worked out by hand from the definitions, not
computed by the oracle.  The cases use Dqk = 2 and q = (1, 1), so the score of
key j is the sum of its two e4m3 values, and the softmax scale ln(2)/8 with
unit descales, so that lambda = log2(e)*scale = 1/8 and the code-unit score is
u_j = 8*lambda*s_j = s_j exactly.  All scores sit 0.5 or 0.25 away from the
integers (no rounding decision is ambiguous) except in the planted cases.

Lean-P ("Zyphra ZYFA: FP8 FlashAttention for AMD MI355X", "Lean P: one
multiply-add instead of an exponential" and "Per-block scaling and a rounded
row sum"), integer-binade anchoring: per 64-key block e = ceil(max u / 8),
code = clamp(floor(u - 8e + 112), 0, 126), weight = dec(code) * 2^(e - 7).

Row of 68 keys (u, code, dec(code), weight):
  block 0, e = ceil(20.5/8) = 3, x = u + 88, weight factor 2^-4
    key 0   20.5    108  96        6
    key 1    2.5     90  20        5/4
    key 2  -13.5     74   5        5/16
    key 3    7.5     95  30        15/8
    key 4  -83.5      4  2^-7      2^-11      (subnormal code)
    key 5  -78.5      9  9/512     9/8192
    keys 6..63 -448  0   0         0          (clamped)
  block 1, e = ceil(-30.5/8) = -3, x = u + 136, weight factor 2^-10
    key 64 -30.5    105  72        72/1024
    key 65 -40.25    95  30        30/1024
    key 66 -131.5     4  2^-7      2^-17      (subnormal code)
    key 67 -36.75    99  44        44/1024
Key 4 and key 66 pin the ceiling of the block exponent and the constants:
a floor or a rounded exponent, or T = 8 with C = 120, moves them out of the
subnormal range and changes their weights (normal codes are compensated).

Running-maximum anchoring (the second reading of the block scale, oracle path "leanp_a3"):
one 128-key tile, m = 20.5 for every row, k = floor((m - block max)/8),
code = clamp(floor(u - m + 8k + 112 + 1/64), 0, 126), weight relative to
2^(m/8) = dec(code) * 2^(-7-k):
  block 0, k = 0:  codes 112, 94, 78, 99, 8, 13, 0...  weights 1, 28/128,
                   7/128, 44/128, 2^-13, 13/65536, 0...
  block 1, k = floor(51/8) = 6: codes 109, 99, 8, 102; weights 104, 44,
                   2^-6, 56 times 2^-13.
"""
import math
from fractions import Fraction as Fr

import numpy as np
import pytest
import torch

import oracle

SCALE = math.log(2.0) / 8.0  # lambda = log2(e) * scale = 1/8 with unit descales

KEYS = ([(20, 0.5), (2.5, 0), (-13, -0.5), (7.5, 0), (-80, -3.5), (-80, 1.5)] +
        [(-448, 0)] * 58 + [(-32, 1.5), (-40, -0.25), (-128, -3.5), (-36, -0.75)])
VALUES = [1, -2, 4, 0.5, 448, -448] + [96] * 58 + [8, -8, 448, 2]

LEANP_W = ({0: Fr(6), 1: Fr(5, 4), 2: Fr(5, 16), 3: Fr(15, 8), 4: Fr(1, 2 ** 11),
            5: Fr(9, 8192)} | {j: Fr(0) for j in range(6, 64)} |
           {64: Fr(72, 1024), 65: Fr(30, 1024), 66: Fr(1, 2 ** 17), 67: Fr(44, 1024)})
A3_W = ({0: Fr(1), 1: Fr(28, 128), 2: Fr(7, 128), 3: Fr(44, 128), 4: Fr(1, 2 ** 13),
         5: Fr(13, 65536)} | {j: Fr(0) for j in range(6, 64)} |
        {64: Fr(104, 2 ** 13), 65: Fr(44, 2 ** 13), 66: Fr(1, 2 ** 19), 67: Fr(56, 2 ** 13)})
A3_M = 20.5  # running maximum of every row, in code units


def e4m3(vals, shape):
    """e4m3 codes of values that e4m3 represents exactly (torch's cast)."""
    t = torch.tensor(np.asarray(vals, dtype=np.float32).reshape(shape))
    codes = t.to(torch.float8_e4m3fn)
    assert torch.equal(codes.float(), t), "a literal is not an e4m3 value"
    return codes.view(torch.uint8).numpy()


def case(keys, values):
    S = len(keys)
    q = e4m3(np.ones((S, 2)), (1, S, 1, 2))
    k = e4m3(keys, (1, S, 1, 2))
    v = e4m3(values, (1, S, 1, 1))
    return q, k, v


def expected_rows(weights, values):
    """out_i = sum_{j<=i} w_j v_j / sum_{j<=i} w_j and ln sum_{j<=i} w_j."""
    out, lse = [], []
    num = den = Fr(0)
    for j in range(len(values)):
        num += weights[j] * Fr(values[j])
        den += weights[j]
        out.append(float(num / den))
        lse.append(math.log(den))
    return np.array(out), np.array(lse)


@pytest.mark.parametrize("path", ["leanp", "leanp_a3"])
def test_literal_codes_and_weights(path):
    q, k, v = case(KEYS, VALUES)
    out, amb, lse = oracle.attention(path, q, k, v, 1.0, 1.0, 1.0, scale=SCALE)
    weights = LEANP_W if path == "leanp" else A3_W
    exp_out, exp_lse = expected_rows(weights, VALUES)
    if path == "leanp_a3":
        exp_lse = exp_lse + A3_M / 8.0 * math.log(2.0)
    np.testing.assert_allclose(out[0, :, 0, 0], exp_out, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0, :], exp_lse, rtol=0, atol=1e-12)
    assert np.all(amb == 0.0), "no rounding decision of these rows is near a tie"


def test_literal_block_exponent_is_a_ceiling():
    """The same row with the block exponents one binade lower (the floor of
    max/8) gives key 4 the normal code 12 (weight 3/4096) instead of the
    subnormal 4 (2^-11): the oracle must hold the ceiling's value."""
    q, k, v = case(KEYS[:5], VALUES[:5])
    out, _, lse = oracle.attention("leanp", q, k, v, 1.0, 1.0, 1.0, scale=SCALE)
    floor_w = dict(LEANP_W)
    floor_w[4] = Fr(3, 4096)
    got = math.exp(lse[0, 0, 4])
    assert got == pytest.approx(float(sum(LEANP_W[j] for j in range(5))), rel=1e-14)
    assert got != pytest.approx(float(sum(floor_w[j] for j in range(5))), rel=1e-9)


def test_planted_code_tie():
    """Key 1 at u = 2 puts the floor argument exactly on the integer 90: the
    code may be 89 (dec 18) or 90 (dec 20), so the ambiguous mass of row 1 is
    (20 - 18)/16 over the row sum 6 + 20/16."""
    keys = [(20, 0.5), (2, 0)]
    q, k, v = case(keys, [1, -2])
    out, amb, lse = oracle.attention("leanp", q, k, v, 1.0, 1.0, 1.0, scale=SCALE)
    assert amb[0, 0, 0] == 0.0
    assert amb[0, 1, 0] == pytest.approx((2 / 16) / (6 + 20 / 16), rel=1e-14)
    # the weight itself is the floor's: code 90 (u + 88 = 90 exactly)
    assert math.exp(lse[0, 0, 1]) == pytest.approx(6 + 20 / 16, rel=1e-14)


def test_planted_block_exponent_tie():
    """u0 = 24 puts max/8 exactly on 3: e may be 3 or 4.  Key 0's weight is 8
    either way (code 112 with 2^-4, or code 104 with 2^-3), but key 1
    (u = -83.5) has the subnormal code 4 (weight 2^-11) with e = 3 and code 0
    with e = 4.  Key 0's floor argument 112 is also exactly an integer (code
    111, dec 120, or 112, dec 128).  Relative to 2^(e-7) = 2^-4 the row sums
    are 8 and 8 + 2^-11, so row 0 has ambiguous mass 0.5/8 and row 1
    (0.5 + 2^-11)/(8 + 2^-11)."""
    keys = [(24, 0), (-80, -3.5)]
    q, k, v = case(keys, [1, 2])
    out, amb, lse = oracle.attention("leanp", q, k, v, 1.0, 1.0, 1.0, scale=SCALE)
    assert amb[0, 0, 0] == pytest.approx(0.5 / 8, rel=1e-14)
    assert amb[0, 1, 0] == pytest.approx((0.5 + 2 ** -11) / (8 + 2 ** -11), rel=1e-14)
    assert out[0, 1, 0, 0] == pytest.approx((8 * 1 + 2 ** -11 * 2) / (8 + 2 ** -11), rel=1e-14)


def test_descales_must_be_positive_and_finite():
    """Descales are amax/448 of a tensor (or 1): every definition rejects zero,
    negative and non-finite values (the library states the same contract)."""
    q, k, v = case(KEYS[:3], VALUES[:3])
    for path in ("ref", "leanp", "leanp_a3", "exact_fp8", "variant_e"):
        for bad in (0.0, -1.0, float("inf"), float("nan")):
            for pos in range(3):
                d = [1.0, 1.0, 1.0]
                d[pos] = bad
                with pytest.raises(ValueError):
                    oracle.attention(path, q, k, v, *d, scale=SCALE)
