"""GPU parity of the flash_attn_func-style options against the oracle, through
the C ABI (attn_fwd_full): non-causal attention, per-(batch, kv head)
descales and the per-row log-sum-exp, on every path."""
import math

import numpy as np
import pytest
import torch

import fp8_causal_prefill_flash_gb300 as fa
import oracle
from fp8_causal_prefill_flash_gb300 import workloads as wl

from gpu_helpers import EMUL_TOL, check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


def _fp8_dev(case, dq, dk, dv):
    q, k, v = (torch.from_numpy(a).cuda() for a in (case.q, case.k, case.v))
    d = [torch.from_numpy(np.asarray(x, np.float32).reshape(-1).copy()).cuda() for x in (dq, dk, dv)]
    return q, k, v, d


def _vmax(case, dv):
    return float(np.max(np.abs(oracle.e4m3_decode(case.v)))) * float(np.max(dv))


def _fp8_parity(variant, case, dq, dk, dv, causal):
    q, k, v, d = _fp8_dev(case, dq, dk, dv)
    out, lse = fa.attn_fwd_full(variant, q, k, v, *d, out_dtype=fa.ATTN_OUT_F32, causal=causal,
                                return_lse=True)
    torch.cuda.synchronize()
    gpu, glse = out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)
    path = {fa.ATTN_VARIANT_LEANP: "leanp", fa.ATTN_VARIANT_EXACT_FP8: "exact_fp8",
            fa.ATTN_VARIANT_LEANP_A3: "leanp_a3"}[variant]
    emul, amb, else_ = oracle.attention(path, case.q, case.k, case.v, dq, dk, dv, causal=causal)
    check_rows(gpu, emul, amb, _vmax(case, dv))
    # log-sum-exp: the row sums agree up to the weight mass near a rounding
    # decision (amb, relative) and fp32 accumulation
    a = np.minimum(amb.transpose(0, 2, 1), 0.5)
    assert np.all(np.abs(glse - else_) <= 2e-5 * (1 + np.abs(else_)) + 2.0 * a / (1.0 - a)), \
        float(np.max(np.abs(glse - else_)))
    return gpu, glse


@pytest.mark.parametrize("S", [1, 100, 257, 600])
@pytest.mark.parametrize("variant", [fa.ATTN_VARIANT_LEANP, fa.ATTN_VARIANT_EXACT_FP8,
                                     fa.ATTN_VARIANT_LEANP_A3])
def test_noncausal_fp8(S, variant):
    case = wl.fp8_gaussian_case(1, 4, 2, S, 128, 128, seeds=(101, 102, 103))
    _fp8_parity(variant, case, case.dq, case.dk, case.dv, causal=False)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("variant", [fa.ATTN_VARIANT_LEANP, fa.ATTN_VARIANT_EXACT_FP8,
                                     fa.ATTN_VARIANT_LEANP_A3])
def test_per_bkv_descales(causal, variant):
    B, Hq, Hkv = 2, 4, 2
    case = wl.fp8_gaussian_case(B, Hq, Hkv, 333, 128, 128, seeds=(104, 105, 106))
    rng = np.random.default_rng(107)
    dq, dk, dv = (x * rng.uniform(0.5, 2.0, (B, Hkv)) for x in (case.dq, case.dk, case.dv))
    _fp8_parity(variant, case, dq, dk, dv, causal)


def test_noncausal_mla_shape():
    case = wl.fp8_gaussian_case(1, 2, 2, 300, 192, 128, seeds=(108, 109, 110), outlier_seed=111,
                                outliers_qk=4, factor=20.0, outliers_v=False)
    _fp8_parity(fa.ATTN_VARIANT_LEANP, case, case.dq, case.dk, case.dv, causal=False)


@pytest.mark.parametrize("causal", [True, False])
def test_lse_against_fp64(causal):
    """Lean-P's log-sum-exp lies in the element band of the fp64 one; the
    exact ablation's equals it within fp32 accumulation."""
    case = wl.fp8_gaussian_case(1, 2, 2, 500, 128, 128, seeds=(112, 113, 114))
    _, _, ref = oracle.attention("ref", case.q, case.k, case.v, case.dq, case.dk, case.dv,
                                 causal=causal)
    _, lp = _fp8_parity(fa.ATTN_VARIANT_LEANP, case, case.dq, case.dk, case.dv, causal)
    d = lp - ref
    assert d.min() > math.log(2.0 ** (-1.0 / 8.0)) - 1e-4 and d.max() < math.log(1.0607) + 1e-4
    _, ex = _fp8_parity(fa.ATTN_VARIANT_EXACT_FP8, case, case.dq, case.dk, case.dv, causal)
    assert np.max(np.abs(ex - ref)) < 1e-4


@pytest.mark.parametrize("causal", [True, False])
def test_bf16_options(causal):
    b = wl.bf16_gaussian_case(1, 4, 2, 300, 128, 128)
    q, k, v = (torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16) for a in (b.q, b.k, b.v))
    out, lse = fa.attn_fwd_full(fa.ATTN_VARIANT_BF16, q, k, v, out_dtype=fa.ATTN_OUT_F32,
                                causal=causal, return_lse=True)
    torch.cuda.synchronize()
    emul, _, else_ = oracle.attention("bf16", b.q, b.k, b.v, causal=causal)
    vmax = float(np.max(np.abs(oracle.bf16_decode(b.v))))
    assert np.max(np.abs(out.cpu().numpy() - emul)) <= EMUL_TOL * vmax
    assert np.max(np.abs(lse.cpu().numpy() - else_)) < 1e-4
    _, _, ref = oracle.attention("ref_bf16", b.q, b.k, b.v, causal=causal)
    assert np.max(np.abs(lse.cpu().numpy() - ref)) < 1e-3


def test_flash_attn_style_wrappers():
    case = wl.fp8_gaussian_case(1, 4, 2, 200, 128, 128, seeds=(115, 116, 117))
    q, k, v, d = _fp8_dev(case, case.dq, case.dk, case.dv)
    o1, l1 = fa.flash_attn_fp8_func(q, k, v, *d, causal=False, return_softmax_lse=True)
    o2 = fa.attn_fwd_ex(fa.ATTN_VARIANT_LEANP, q, k, v, *d, out_dtype=fa.ATTN_OUT_BF16, causal=False)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and l1.shape == (1, 4, 200)
    b = wl.bf16_gaussian_case(1, 2, 2, 64, 128, 128)
    qb, kb, vb = (torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16) for a in (b.q, b.k, b.v))
    ob = fa.flash_attn_bf16_func(qb, kb, vb, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(ob, fa.attn_fwd_bf16(qb, kb, vb))


@pytest.mark.parametrize("S", [1, 129, 511])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("variant", [fa.ATTN_VARIANT_LEANP, fa.ATTN_VARIANT_EXACT_FP8,
                                     fa.ATTN_VARIANT_LEANP_A3])
def test_mla_gqa_batched_options(S, causal, variant):
    """The MLA shape (Dqk 192, Dv 128) with GQA, B = 2, descales per (batch,
    kv head) and the LSE, over ragged lengths, causal and not."""
    B, Hq, Hkv = 2, 4, 2
    case = wl.fp8_gaussian_case(B, Hq, Hkv, S, 192, 128, seeds=(118, 119, 120), outlier_seed=121,
                                outliers_qk=4, factor=20.0, outliers_v=False)
    rng = np.random.default_rng(122 + S)
    dq, dk, dv = (x * rng.uniform(0.5, 2.0, (B, Hkv)) for x in (case.dq, case.dk, case.dv))
    _fp8_parity(variant, case, dq, dk, dv, causal)


def test_float8_tensors_and_binding_errors():
    """torch float8_e4m3fn tensors give the same bits as their uint8 views;
    the binding refuses wrong dtypes, layouts and shapes before calling the
    library."""
    case = wl.fp8_gaussian_case(1, 4, 2, 200, 128, 128, seeds=(123, 124, 125))
    q, k, v, d = _fp8_dev(case, case.dq, case.dk, case.dv)
    a = fa.attn_fwd_fp8(q, k, v, *d)
    b = fa.attn_fwd_fp8(*(t.view(torch.float8_e4m3fn) for t in (q, k, v)), *d)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    with pytest.raises(TypeError):
        fa.attn_fwd_fp8(q.float(), k, v, *d)                        # not e4m3 codes
    with pytest.raises(ValueError):
        fa.attn_fwd_fp8(q.transpose(1, 2), k, v, *d)                # not contiguous BSHD
    with pytest.raises(TypeError):
        fa.attn_fwd_fp8(q.cpu(), k, v, *d)                          # not on the GPU
    with pytest.raises(fa.AttnError):
        fa.attn_fwd_fp8(q[:, :, :3].contiguous(), k, v, *d)         # Hq % Hkv != 0


def test_host_descales_are_checked():
    """The descale contract (finite and greater than zero) at the binding:
    host numbers are checked before any launch; device descales are the
    caller's (fp8attn.h).  A valid host descale gives the device tensor's
    result bit for bit."""
    case = wl.fp8_gaussian_case(1, 2, 2, 130, 128, 128, seeds=(126, 127, 128))
    q, k, v, d = _fp8_dev(case, case.dq, case.dk, case.dv)
    for bad in (0.0, -case.dq, float("inf"), float("nan")):
        with pytest.raises(ValueError):
            fa.flash_attn_fp8_func(q, k, v, bad, d[1], d[2])
    a = fa.flash_attn_fp8_func(q, k, v, float(d[0].item()), d[1], d[2])
    b = fa.flash_attn_fp8_func(q, k, v, *d)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
