"""Pins for the oracle's number formats and the Lean-P code function.

Each check ties the oracle to something other than itself: a library routine
(torch's float8_e4m3fn / bfloat16 conversions), a fact the article prints, or
a closed form.
"""
import math

import numpy as np
import pytest
import torch


def torch_e4m3_values():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_torch(oracle_mod):
    """All 256 e4m3 codes decode like torch's float8_e4m3fn (NaN at 0x7F/0xFF)."""
    ours = oracle_mod.e4m3_decode(np.arange(256))
    theirs = torch_e4m3_values()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], theirs[~nan])
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF]


def test_e4m3_code_grows_by_8_per_doubling(oracle_mod):
    """[ART-MTP] "Lean P: one multiply-add instead of an exponential": the e4m3
    bit pattern, read as an integer, grows by 8 each time the value doubles."""
    dec = oracle_mod.e4m3_decode(np.arange(128))
    for c in range(8, 126 - 8 + 1):
        assert dec[c + 8] == 2.0 * dec[c], c
    # so the code of 2^x is 8x + 56 for every normal power of two
    for x in range(-6, 9):
        assert dec[8 * x + 56] == 2.0 ** x


def test_e4m3_round_matches_torch(oracle_mod):
    """RNE to e4m3 equals torch's conversion, including exact midpoints."""
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(2000) * 10.0,
        np.exp2(rng.uniform(-12, 8.5, 2000)),
        # exact midpoints between neighbouring codes (ties to even)
        (torch_e4m3_values()[1:126] + torch_e4m3_values()[2:127]) / 2.0,
        [0.0, 2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -9, 447.9, 448.0],
    ])
    vals = vals[np.abs(vals) <= 448.0]
    ours = oracle_mod.e4m3_round(vals)
    theirs = torch.from_numpy(vals).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64)
    # float64 -> float32 is exact for these values (<= 24 significant bits)
    assert np.array_equal(ours, theirs.numpy())


def test_e4m3_round_saturates(oracle_mod):
    assert oracle_mod.e4m3_round([500.0, -1e9])[0] == 448.0
    assert oracle_mod.e4m3_round([-1e9])[0] == -448.0


def test_bf16_roundtrip_matches_torch(oracle_mod):
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(3000) * 3.0, np.exp2(rng.uniform(-130, 100, 500))])
    x32 = x.astype(np.float32)
    bits = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle_mod.bf16_decode(bits), want)
    assert np.array_equal(oracle_mod.bf16_round(x32.astype(np.float64)), want)


def test_leanp_constants(oracle_mod):
    """C is the e4m3 code of 2^T."""
    T, C = oracle_mod.leanp_constants()
    assert oracle_mod.e4m3_decode([C])[0] == 2.0 ** T
    assert C + 8 <= 126  # one binade of headroom below the largest finite code


def test_leanp_code_closed_form(oracle_mod):
    """code(x) = clamp(floor(x), 0, 126)."""
    xs = np.array([-1e9, -3.5, -1e-12, 0.0, 0.999, 1.0, 55.99, 56.0, 111.2, 126.0, 126.9, 1e6])
    want = [0, 0, 0, 0, 0, 1, 55, 56, 111, 126, 126, 126]
    assert list(oracle_mod.leanp_code(xs)) == want


def test_leanp_element_band(oracle_mod):
    """Closed-form band of one Lean-P probability.

    For x in the normal code range, dec(floor(x)) / 2^(x/8 - 7) lies in
    (2^(-1/8), max_m (1+m/8)/2^(m/8)] = (0.917, 1.0607]: floor loses less than
    one code (1/8 of a binade) and the e4m3 grid is the chord of 2^t, which
    lies above the curve by at most 6.07% (at m = 4).
    """
    lo = 2.0 ** (-1.0 / 8.0)
    hi = max((1 + m / 8.0) / 2.0 ** (m / 8.0) for m in range(8))
    assert abs(hi - 1.5 / math.sqrt(2.0)) < 1e-15
    xs = np.concatenate([np.linspace(8.0, 125.999, 200001), np.arange(8.0, 126.0)])
    ratio = oracle_mod.e4m3_decode(oracle_mod.leanp_code(xs)) / np.exp2(xs / 8.0 - 7.0)
    assert ratio.min() > lo
    assert ratio.max() <= hi + 1e-15
    # both ends of the band are reached
    assert ratio.min() < lo + 1e-4
    assert ratio.max() > hi - 1e-12
