"""GPU parity of Lean-P with the code grid anchored at the running row maximum
(ATTN_VARIANT_LEANP_A3) against the oracle's "leanp_a3" definition, through
the C ABI, and its exact invariants.

"Zyphra ZYFA: FP8 FlashAttention for AMD MI355X", "Lean P: one multiply-add
instead of an exponential" and "Per-block scaling and a rounded row sum"
leave open what the power of two of a 64-key block is relative to; this path
takes the running maximum, so the key holding it gets exactly the code of 2^T
and O is rescaled exactly whenever the maximum grows."""
import numpy as np
import pytest
import torch

import fp8_causal_prefill_flash_gb300 as fa
import oracle
from fp8_causal_prefill_flash_gb300 import workloads as wl

from gpu_helpers import FP8_RMS_TOL, check_rows, dev_fp8, rel_rms, run_fp8, vmax_fp8

pytestmark = pytest.mark.gpu

A3 = fa.ATTN_VARIANT_LEANP_A3


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


def _parity(case, scale=None):
    gpu = run_fp8(A3, case, scale=scale or 0.0)
    emul, amb, _ = oracle.attention("leanp_a3", case.q, case.k, case.v, case.dq, case.dk,
                                    case.dv, scale=scale)
    check_rows(gpu, emul, amb, vmax_fp8(case))
    return gpu


def test_h2_s256_d128_every_row():
    case = wl.make_case("fp8_h2_s256_d128")
    gpu = _parity(case)
    ref = oracle.ref_fp64(case.q, case.k, case.v, case.dq, case.dk, case.dv)
    assert rel_rms(gpu, ref) <= FP8_RMS_TOL


@pytest.mark.parametrize("S", [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 600, 1100])
def test_ragged_lengths(S):
    case = wl.fp8_gaussian_case(1, 2, 1, S, 128, 128, seeds=(700 + S, 800 + S, 900 + S))
    _parity(case)


def test_gqa_batch_outliers():
    case = wl.fp8_gaussian_case(2, 8, 2, 300, 128, 128, seeds=(21, 22, 23), outlier_seed=24,
                                outliers_qk=1, factor=8.0)
    _parity(case)


def test_mla_shape():
    case = wl.fp8_gaussian_case(1, 2, 2, 333, 192, 128, seeds=(31, 32, 33), outlier_seed=34,
                                outliers_qk=4, factor=20.0, outliers_v=False)
    gpu = _parity(case)
    ref = oracle.ref_fp64(case.q, case.k, case.v, case.dq, case.dk, case.dv)
    assert rel_rms(gpu, ref) <= FP8_RMS_TOL


def test_explicit_softmax_scale():
    case = wl.fp8_gaussian_case(1, 1, 1, 700, 128, 128, seeds=(41, 42, 43))
    _parity(case, scale=0.21)


def test_v_ones_gives_exactly_one():
    """V = 1 (code 0x38) and dv = 1: the rounded row sum is exactly the sum of
    the weights P.V saw, so every output is bf16 1.0 bit for bit."""
    case = wl.fp8_gaussian_case(1, 2, 2, 700, 128, 128, seeds=(51, 52, 53))
    q, k, _, d = dev_fp8(case)
    v = torch.full_like(q, 0x38)
    d[2] = torch.ones(1, dtype=torch.float32, device="cuda")
    out = fa.attn_fwd_ex(A3, q, k, v, *d, out_dtype=fa.ATTN_OUT_BF16)
    torch.cuda.synchronize()
    assert bool((out.float() == 1.0).all())


def test_q_zero_gives_prefix_mean():
    """Q = 0: every score is 0, every key gets the code of 2^T, so row i is the
    mean of v_0..v_i (fp32 output, within fp32 accumulation)."""
    case = wl.fp8_gaussian_case(1, 2, 2, 400, 128, 128, seeds=(54, 55, 56))
    q, k, v, d = dev_fp8(case)
    q.zero_()
    out = fa.attn_fwd_ex(A3, q, k, v, *d).cpu().numpy().astype(np.float64)
    vv = oracle.e4m3_decode(case.v) * case.dv
    mean = np.cumsum(vv, axis=1) / np.arange(1, 401)[None, :, None, None]
    assert np.max(np.abs(out - mean)) <= 1e-5 * np.max(np.abs(vv))


def test_running_maximum_key_is_exact():
    """One key per row dominates by more than the e4m3 range: the output is
    that key's value row (its code is exactly 2^T, every other key clamps to
    zero or lands in a block scaled far below)."""
    case = wl.fp8_gaussian_case(1, 1, 1, 300, 128, 128, seeds=(57, 58, 59))
    case.q[...] = 0
    case.q[0, :, 0, 0] = 0x7E            # 448
    case.k[0, :, 0, :] = 0
    case.k[0, 37, 0, 0] = 0x7E           # key 37 scores 448*448 against every row
    case.dq = case.dk = 1.0              # about 25,600 binades above every other key
    gpu = run_fp8(A3, case)
    vv = oracle.e4m3_decode(case.v)[0, :, 0, :] * case.dv
    np.testing.assert_allclose(gpu[0, 37:, 0, :], np.broadcast_to(vv[37], (263, 128)),
                               rtol=0, atol=1e-6 * np.max(np.abs(vv)))
