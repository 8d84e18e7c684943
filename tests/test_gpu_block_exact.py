"""GPU parity of the diagnostic block-exact variant (ATTN_VARIANT_BLOCK_EXACT)
against the oracle's variant E, through the C ABI.

The variant keeps Lean-P's 64-key power-of-two block scale and rounded row sum
and rounds the exact probability to the nearest e4m3 instead of taking the
Lean-P code ("Zyphra ZYFA: FP8 FlashAttention for AMD MI355X", "Lean P",
"Per-block scaling and a rounded row sum").  Rows are compared under the same
per-row gate as Lean-P: the oracle bounds the weight mass whose e4m3 rounding
an fp32 argument and the approximate exponential may flip.
"""
import numpy as np
import pytest
import torch

import fp8_causal_prefill_flash_gb300 as fa
import oracle
from fp8_causal_prefill_flash_gb300 import workloads as wl

from gpu_helpers import FP8_RMS_TOL, check_rows, dev_fp8, rel_rms, run_fp8, vmax_fp8

pytestmark = pytest.mark.gpu

E = fa.ATTN_VARIANT_BLOCK_EXACT


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


def _parity(case, causal=True, dq=None, dk=None, dv=None):
    dq, dk, dv = (case.dq if dq is None else dq, case.dk if dk is None else dk,
                  case.dv if dv is None else dv)
    q, k, v, _ = dev_fp8(case)
    d = [torch.from_numpy(np.asarray(x, np.float32).reshape(-1).copy()).cuda() for x in (dq, dk, dv)]
    out, lse = fa.attn_fwd_full(E, q, k, v, *d, out_dtype=fa.ATTN_OUT_F32, causal=causal,
                                return_lse=True)
    torch.cuda.synchronize()
    gpu = out.cpu().numpy().astype(np.float64)
    emul, amb, else_ = oracle.attention("variant_e", case.q, case.k, case.v, dq, dk, dv,
                                        causal=causal)
    vmax = float(np.max(np.abs(oracle.e4m3_decode(case.v)))) * float(np.max(dv))
    check_rows(gpu, emul, amb, vmax)
    a = np.minimum(amb.transpose(0, 2, 1), 0.5)
    glse = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(glse - else_) <= 2e-5 * (1 + np.abs(else_)) + 2.0 * a / (1.0 - a))
    return gpu


def test_h2_s256_d128():
    case = wl.make_case("fp8_h2_s256_d128")
    gpu = _parity(case)
    ref = oracle.ref_fp64(case.q, case.k, case.v, case.dq, case.dk, case.dv)
    assert rel_rms(gpu, ref) <= FP8_RMS_TOL


@pytest.mark.parametrize("S", [1, 63, 64, 65, 129, 257, 600])
def test_ragged_lengths(S):
    _parity(wl.fp8_gaussian_case(1, 2, 2, S, 128, 128, seeds=(130, 131, 132)))


def test_mla_shape_noncausal():
    case = wl.fp8_gaussian_case(1, 2, 2, 300, 192, 128, seeds=(133, 134, 135), outlier_seed=136,
                                outliers_qk=4, factor=20.0, outliers_v=False)
    _parity(case, causal=False)


def test_per_bkv_descales_and_gqa():
    B, Hkv = 2, 2
    case = wl.fp8_gaussian_case(B, 4, Hkv, 333, 128, 128, seeds=(137, 138, 139))
    rng = np.random.default_rng(140)
    dq, dk, dv = (x * rng.uniform(0.5, 2.0, (B, Hkv)) for x in (case.dq, case.dk, case.dv))
    _parity(case, dq=dq, dk=dk, dv=dv)


def test_v_ones_gives_exactly_one():
    """The rounded row sum makes the weights sum to one exactly."""
    case = wl.fp8_gaussian_case(1, 2, 2, 300, 128, 128, seeds=(141, 142, 143))
    case.v[:] = 0x38  # e4m3 1.0
    case.dv = 1.0
    gpu = run_fp8(E, case, out_f32=False)
    assert np.all(gpu == 1.0)


def test_sink_input_beats_the_ablation():
    """With an attention sink the block scale keeps the small probabilities,
    as for Lean-P: the error against fp64 is far below the ablation's."""
    case = wl.fp8_sink_case(1, 2, 2, 1024, 128, 128)
    ref = oracle.ref_fp64(case.q, case.k, case.v, case.dq, case.dk, case.dv)
    e = rel_rms(_parity(case), ref)
    a = rel_rms(run_fp8(fa.ATTN_VARIANT_EXACT_FP8, case), ref)
    assert e <= 0.3 * a, (e, a)
