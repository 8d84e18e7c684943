"""Pins for the oracle's e4m3 quantiser of Q and K, with and without the
Hadamard rotation ([ART-MTP] "How accurate is ZYFA's FP8 attention?": most
FP8 error comes from quantising the inputs, and rotating Q and K roughly
halves it).

The rotation is checked against scipy's Sylvester Hadamard matrix; the codes
against torch's float8_e4m3fn cast; exact integer inputs pin the butterfly
arithmetic bit for bit.
"""
import numpy as np
import pytest
import scipy.linalg as sl
import torch


def torch_codes(x32):
    """torch's e4m3 (RNE) codes of fp32 values already inside +-448."""
    return torch.from_numpy(np.asarray(x32, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def rotation(D):
    """The orthonormal rotation the definition describes, from scipy."""
    hb = 64 if D == 192 else D
    Hb = sl.hadamard(hb).astype(np.float64) / np.sqrt(hb)
    return sl.block_diag(*([Hb] * (D // hb)))


@pytest.mark.parametrize("D", [128, 192])
def test_unrotated_codes_are_torch_cast(oracle_mod, D):
    x = np.random.default_rng(D).standard_normal((37, D)).astype(np.float32)
    codes, ds = oracle_mod.quantize_e4m3(x, False)
    amax = np.float32(np.max(np.abs(x)))
    sc = np.float32(448.0) / amax
    assert np.array_equal(codes, torch_codes(x * sc))
    assert ds == np.float32(amax / np.float32(448.0))


@pytest.mark.parametrize("D", [128, 192])
def test_rotation_matches_sylvester_hadamard(oracle_mod, D):
    """dec(code) * descale is the orthonormal rotation of x within e4m3's
    half-ulp (plus the subnormal floor), a wrong sign or index fails."""
    x = np.random.default_rng(7).standard_normal((25, D)).astype(np.float32)
    codes, ds = oracle_mod.quantize_e4m3(x, True)
    y = x.astype(np.float64) @ rotation(D).T
    got = oracle_mod.e4m3_decode(codes) * ds
    floor = 2.0 ** -10 * np.max(np.abs(y)) / 448.0 * 64
    assert np.all(np.abs(got - y) <= 2.0 ** -4 * np.abs(y) + floor)
    # a rotation with its rows permuted (a wrong index) is far off
    wrong = np.roll(rotation(D), 1, axis=0)
    assert np.max(np.abs(got - x.astype(np.float64) @ wrong.T)) > 0.5


@pytest.mark.parametrize("D", [128, 192])
def test_integer_inputs_are_exact(oracle_mod, D):
    """Small integers: the fp32 butterflies are exact, so the codes equal
    torch's cast of (H x) * 448/amax computed in fp32."""
    rng = np.random.default_rng(11)
    x = rng.integers(-8, 9, size=(9, D)).astype(np.float32)
    codes, ds = oracle_mod.quantize_e4m3(x, True)
    hb = 64 if D == 192 else D
    H = sl.block_diag(*([sl.hadamard(hb)] * (D // hb))).astype(np.float64)
    y = (x.astype(np.float64) @ H.T).astype(np.float32)  # exact integers
    amax = np.float32(np.max(np.abs(y)))
    assert np.array_equal(codes, torch_codes(y * (np.float32(448.0) / amax)))
    norm = np.float32(0.125) if D == 192 else np.float32(1.0 / np.sqrt(128.0))
    assert ds == np.float32(np.float32(amax / np.float32(448.0)) * norm)


def test_bf16_input_equals_f32_input(oracle_mod):
    x = np.random.default_rng(3).standard_normal((16, 128)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16
    xb = (bits.astype(np.uint32) << 16).view(np.float32)
    for rot in (False, True):
        c1, d1 = oracle_mod.quantize_e4m3(bits, rot)
        c2, d2 = oracle_mod.quantize_e4m3(xb, rot)
        assert np.array_equal(c1, c2) and d1 == d2


def test_zero_tensor(oracle_mod):
    codes, ds = oracle_mod.quantize_e4m3(np.zeros((3, 192), np.float32), True)
    assert not codes.any() and ds == np.float32(0.125)


def test_rotation_shrinks_qk_error_with_outliers(oracle_mod):
    """The articles' claim: rotating Q and K roughly halves the error of the
    quantised inputs.  With a few scaled channels (the outlier workloads), the
    error of Q K^T from the quantised inputs drops by at least half."""
    rng = np.random.default_rng(5)
    for D, nout, f in [(128, 1, 8.0), (192, 4, 20.0)]:
        q = rng.standard_normal((256, 2, D)).astype(np.float32)
        k = rng.standard_normal((256, 2, D)).astype(np.float32)
        ch = rng.choice(D, nout, replace=False)
        q[..., ch] *= f
        k[..., ch] *= f
        ref = np.einsum("shd,thd->hst", q.astype(np.float64), k.astype(np.float64))
        err = []
        for rot in (False, True):
            cq, dq = oracle_mod.quantize_e4m3(q, rot)
            ck, dk = oracle_mod.quantize_e4m3(k, rot)
            s = np.einsum("shd,thd->hst", oracle_mod.e4m3_decode(cq) * dq,
                          oracle_mod.e4m3_decode(ck) * dk)
            err.append(np.sqrt(np.mean((s - ref) ** 2)) / np.sqrt(np.mean(ref ** 2)))
        assert err[1] <= 0.5 * err[0], (D, err)
