"""GPU parity: the sm_103a kernels against the CPU oracle, through the C ABI.

Small and ragged shapes are compared on every row; the invariants of the
method (rounded row sum, causality, head mapping, determinism) are checked
bitwise where they are exact.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import fp8_causal_prefill_flash_gb300 as fa
import oracle
from fp8_causal_prefill_flash_gb300 import workloads as wl

from gpu_helpers import (BF16_RMS_TOL, EMUL_TOL, FP8_RMS_TOL, check_rows, dev_bf16, dev_fp8,
                         rel_rms, run_bf16, run_fp8, vmax_fp8)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


def _leanp_parity(case, scale=None):
    gpu = run_fp8(fa.ATTN_VARIANT_LEANP, case, scale=scale or 0.0)
    emul, amb = oracle.emul_leanp(case.q, case.k, case.v, case.dq, case.dk, case.dv, scale=scale)
    check_rows(gpu, emul, amb, vmax_fp8(case))
    return gpu


def test_leanp_h2_s256_d128():
    case = wl.make_case("fp8_h2_s256_d128")
    gpu = _leanp_parity(case)
    ref = oracle.ref_fp64(case.q, case.k, case.v, case.dq, case.dk, case.dv)
    assert rel_rms(gpu, ref) <= FP8_RMS_TOL
    # the bf16-output product entry point agrees with the fp32-output one
    q, k, v, d = dev_fp8(case)
    out = fa.attn_fwd_fp8(q, k, v, *d)
    torch.cuda.synchronize()
    assert np.max(np.abs(out.float().cpu().numpy() - gpu)) <= 2.0 ** -8 * np.max(np.abs(gpu)) + 1e-6


def test_exact_fp8_h2_s256_d128():
    case = wl.make_case("fp8_h2_s256_d128")
    gpu = run_fp8(fa.ATTN_VARIANT_EXACT_FP8, case)
    emul, amb = oracle.emul_exact_fp8(case.q, case.k, case.v, case.dq, case.dk, case.dv)
    check_rows(gpu, emul, amb, vmax_fp8(case))
    ref = oracle.ref_fp64(case.q, case.k, case.v, case.dq, case.dk, case.dv)
    assert rel_rms(gpu, ref) <= FP8_RMS_TOL


def test_bf16_h2_s256_d128():
    case = wl.bf16_gaussian_case(1, 2, 2, 256, 128, 128)
    gpu = run_bf16(case)
    ref = oracle.ref_fp64_bf16(case.q, case.k, case.v)
    assert rel_rms(gpu, ref) <= BF16_RMS_TOL
    emul = oracle.emul_bf16(case.q, case.k, case.v)
    vmax = float(np.max(np.abs(oracle.bf16_decode(case.v))))
    assert np.max(np.abs(gpu - emul)) <= EMUL_TOL * vmax


@pytest.mark.parametrize("S", [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 600])
def test_leanp_ragged_lengths(S):
    case = wl.fp8_gaussian_case(1, 2, 1, S, 128, 128, seeds=(100 + S, 200 + S, 300 + S))
    _leanp_parity(case)


@pytest.mark.parametrize("S", [1, 65, 200, 513])
def test_exact_fp8_ragged_lengths(S):
    case = wl.fp8_gaussian_case(1, 2, 1, S, 128, 128, seeds=(400 + S, 500 + S, 600 + S))
    gpu = run_fp8(fa.ATTN_VARIANT_EXACT_FP8, case)
    emul, amb = oracle.emul_exact_fp8(case.q, case.k, case.v, case.dq, case.dk, case.dv)
    check_rows(gpu, emul, amb, vmax_fp8(case))


@pytest.mark.parametrize("S", [1, 100, 300])
def test_bf16_ragged_lengths(S):
    case = wl.bf16_gaussian_case(1, 2, 1, S, 128, 128, seeds=(S, S + 1, S + 2))
    gpu = run_bf16(case)
    emul = oracle.emul_bf16(case.q, case.k, case.v)
    vmax = float(np.max(np.abs(oracle.bf16_decode(case.v))))
    assert np.max(np.abs(gpu - emul)) <= EMUL_TOL * vmax


def test_leanp_gqa_and_batch():
    case = wl.fp8_gaussian_case(2, 8, 2, 300, 128, 128, seeds=(21, 22, 23), outlier_seed=24,
                                outliers_qk=1, factor=8.0)
    _leanp_parity(case)


def test_leanp_mla_shape():
    case = wl.fp8_gaussian_case(1, 2, 2, 333, 192, 128, seeds=(31, 32, 33), outlier_seed=34,
                                outliers_qk=4, factor=20.0, outliers_v=False)
    gpu = _leanp_parity(case)
    ref = oracle.ref_fp64(case.q, case.k, case.v, case.dq, case.dk, case.dv)
    assert rel_rms(gpu, ref) <= FP8_RMS_TOL


def test_exact_fp8_mla_shape():
    case = wl.fp8_gaussian_case(1, 2, 2, 260, 192, 128, seeds=(35, 36, 37))
    gpu = run_fp8(fa.ATTN_VARIANT_EXACT_FP8, case)
    emul, amb = oracle.emul_exact_fp8(case.q, case.k, case.v, case.dq, case.dk, case.dv)
    check_rows(gpu, emul, amb, vmax_fp8(case))


def test_explicit_softmax_scale():
    case = wl.fp8_gaussian_case(1, 1, 1, 200, 128, 128, seeds=(41, 42, 43))
    _leanp_parity(case, scale=0.21)


# ------------------------------------------------------------------ invariants

def test_v_ones_gives_exactly_one():
    """Rounded row sum: with V = 1 every Lean-P output is exactly 1.0 in bf16."""
    case = wl.fp8_gaussian_case(1, 4, 2, 700, 128, 128, seeds=(51, 52, 53))
    q, k, v, d = dev_fp8(case)
    v = torch.full_like(v, 0x38)
    d[2] = torch.ones(1, dtype=torch.float32, device="cuda")
    out = fa.attn_fwd_fp8(q, k, v, *d)
    torch.cuda.synchronize()
    assert torch.all(out.float() == 1.0)


def test_q_zero_gives_prefix_mean():
    case = wl.fp8_gaussian_case(1, 2, 2, 300, 128, 128, seeds=(54, 55, 56))
    q, k, v, d = dev_fp8(case)
    q.zero_()
    out = fa.attn_fwd_ex(fa.ATTN_VARIANT_LEANP, q, k, v, *d).cpu().numpy()
    vf = oracle.e4m3_decode(case.v) * case.dv
    want = np.cumsum(vf, axis=1) / np.arange(1, 301)[None, :, None, None]
    assert np.max(np.abs(out - want)) <= 1e-5 * np.max(np.abs(vf))


def test_future_keys_do_not_change_earlier_rows():
    case = wl.fp8_gaussian_case(1, 2, 1, 512, 128, 128, seeds=(57, 58, 59))
    q, k, v, d = dev_fp8(case)
    a = fa.attn_fwd_fp8(q, k, v, *d).clone()
    i0 = 300
    k2, v2 = k.clone(), v.clone()
    k2[:, i0 + 1:] = torch.randint(0, 126, k2[:, i0 + 1:].shape, dtype=torch.uint8, device="cuda")
    v2[:, i0 + 1:] = torch.randint(0, 126, v2[:, i0 + 1:].shape, dtype=torch.uint8, device="cuda")
    b = fa.attn_fwd_fp8(q, k2, v2, *d)
    torch.cuda.synchronize()
    assert torch.equal(a[:, :i0 + 1], b[:, :i0 + 1])


def test_gqa_equals_repeated_heads():
    case = wl.fp8_gaussian_case(1, 6, 2, 260, 128, 128, seeds=(61, 62, 63))
    q, k, v, d = dev_fp8(case)
    a = fa.attn_fwd_fp8(q, k, v, *d)
    b = fa.attn_fwd_fp8(q, k.repeat_interleave(3, dim=2).contiguous(),
                        v.repeat_interleave(3, dim=2).contiguous(), *d)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_repeated_launches_are_bitwise_identical():
    case = wl.fp8_gaussian_case(1, 4, 4, 1024, 128, 128, seeds=(64, 65, 66))
    q, k, v, d = dev_fp8(case)
    first = fa.attn_fwd_fp8(q, k, v, *d).clone()
    for _ in range(50):
        again = fa.attn_fwd_fp8(q, k, v, *d)
        assert torch.equal(first, again)


def test_bitwise_identical_over_7200_launches():
    """The articles report bitwise-identical output over 7,200 launches
    ("Zyphra ZYFA: FP8 FlashAttention for AMD MI355X", "How accurate is
    ZYFA's FP8 attention?").  Here: 7,200 Lean-P launches of a 3.4-wave
    problem (B=1, 32 heads, S=4096), each compared with the first on the
    device."""
    case = wl.fp8_gaussian_case(1, 32, 32, 4096, 128, 128, seeds=(76, 77, 78))
    q, k, v, d = dev_fp8(case)
    first = fa.attn_fwd_fp8(q, k, v, *d).clone()
    out = torch.empty_like(first)
    diff = torch.zeros(1, dtype=torch.int64, device="cuda")
    for _ in range(7200):
        fa.attn_fwd_fp8(q, k, v, *d, out=out)
        diff += (out.view(torch.int16) != first.view(torch.int16)).sum()
    torch.cuda.synchronize()
    assert diff.item() == 0


@pytest.mark.parametrize("variant", [fa.ATTN_VARIANT_EXACT_FP8, fa.ATTN_VARIANT_BLOCK_EXACT,
                                     fa.ATTN_VARIANT_BF16, fa.ATTN_VARIANT_LEANP_A3])
@pytest.mark.parametrize("causal", [True, False])
def test_every_variant_is_deterministic(variant, causal):
    """Every path, causal or not, with fp32 output and the log-sum-exp: 20
    launches on a multi-wave grid give the same bits (no atomics, a fixed
    accumulation order), and no launch reports a status."""
    if variant == fa.ATTN_VARIANT_BF16:
        b = wl.bf16_gaussian_case(2, 16, 4, 3000, 128, 128)
        args = dev_bf16(b)
    else:
        c = wl.fp8_gaussian_case(2, 16, 4, 3000, 128, 128, seeds=(67, 68, 69))
        q, k, v, d = dev_fp8(c)
        args = (q, k, v, *d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = [t.clone() for t in fa.attn_fwd_full(variant, *args, out_dtype=fa.ATTN_OUT_F32,
                                                  causal=causal, return_lse=True,
                                                  dev_status=status)]
    for _ in range(20):
        again = fa.attn_fwd_full(variant, *args, out_dtype=fa.ATTN_OUT_F32, causal=causal,
                                 return_lse=True, dev_status=status)
        assert all(torch.equal(x, y) for x, y in zip(first, again))
    torch.cuda.synchronize()
    # a bounded wait that ran out would set ATTN_ERR_TIMEOUT and leave rows unwritten
    assert int(status.item()) == fa.ATTN_OK, fa.status_string(int(status.item()))


# ------------------------------------------------------------------ failure paths

def test_stalled_loads_report_timeout_and_context_survives():
    """Test hook: no copies are issued, every bounded wait expires, the kernel
    reports ATTN_ERR_TIMEOUT in the status word and the context stays usable."""
    case = wl.fp8_gaussian_case(1, 2, 2, 256, 128, 128, seeds=(1, 2, 3))
    q, k, v, d = dev_fp8(case)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fa.attn_fwd_ex(fa.ATTN_VARIANT_LEANP, q, k, v, *d, flags=fa.ATTN_FLAG_TEST_STALL_LOADS,
                   dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == fa.ATTN_ERR_TIMEOUT
    # the next normal call works and agrees with the oracle
    status.zero_()
    gpu = fa.attn_fwd_ex(fa.ATTN_VARIANT_LEANP, q, k, v, *d, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    emul, amb = oracle.emul_leanp(case.q, case.k, case.v, case.dq, case.dk, case.dv)
    check_rows(gpu.cpu().numpy().astype(np.float64), emul, amb, vmax_fp8(case))


def test_argument_errors_are_reported():
    case = wl.fp8_gaussian_case(1, 2, 2, 64, 128, 128)
    q, k, v, d = dev_fp8(case)
    v64 = torch.zeros((1, 64, 2, 64), dtype=torch.uint8, device="cuda")
    _, st = fa.attn_fwd_ex(fa.ATTN_VARIANT_LEANP, q, k, v64, *d, raise_on_error=False)
    assert st == fa.ATTN_ERR_UNSUPPORTED  # Dv = 64
    q3 = torch.zeros((1, 64, 3, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.AttnError) as e:
        fa.attn_fwd_fp8(q3, k, v, *d)
    assert e.value.status == fa.ATTN_ERR_INVALID_ARG
    q64 = torch.zeros((1, 64, 2, 64), dtype=torch.uint8, device="cuda")
    k64 = torch.zeros((1, 64, 2, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.AttnError) as e:
        fa.attn_fwd_fp8(q64, k64, v, *d)
    assert e.value.status == fa.ATTN_ERR_UNSUPPORTED


# ------------------------------------------------------------------ out-of-bounds writes

@pytest.mark.parametrize("variant", [fa.ATTN_VARIANT_LEANP, fa.ATTN_VARIANT_EXACT_FP8,
                                     fa.ATTN_VARIANT_BLOCK_EXACT, fa.ATTN_VARIANT_BF16,
                                     fa.ATTN_VARIANT_LEANP_A3])
@pytest.mark.parametrize("S,causal", [(1, True), (65, True), (300, False), (257, True)])
@pytest.mark.parametrize("out_dtype", [fa.ATTN_OUT_BF16, fa.ATTN_OUT_F32])
def test_no_write_outside_output_and_lse(variant, S, causal, out_dtype):
    """The output and log-sum-exp are views into larger buffers filled with a
    canary byte: every byte before and after the views must be untouched, and
    every element of the views must have been written (no canary left)."""
    B, Hq, Hkv = 1, 4, 2
    if variant == fa.ATTN_VARIANT_BF16:
        args = dev_bf16(wl.bf16_gaussian_case(B, Hq, Hkv, S, 128, 128))
    else:
        q, k, v, d = dev_fp8(wl.fp8_gaussian_case(B, Hq, Hkv, S, 128, 128, seeds=(70, 71, 72)))
        args = (q, k, v, *d)
    esz = 4 if out_dtype == fa.ATTN_OUT_F32 else 2
    n_out = B * S * Hq * 128 * esz
    pad = 4096
    raw = torch.full((pad + n_out + pad,), 0xA5, dtype=torch.uint8, device="cuda")
    dt = torch.float32 if out_dtype == fa.ATTN_OUT_F32 else torch.bfloat16
    out = raw[pad:pad + n_out].view(dt).view(B, S, Hq, 128)
    n_lse = B * Hq * S * 4
    raw_lse = torch.full((pad + n_lse + pad,), 0xA5, dtype=torch.uint8, device="cuda")
    lse_view = raw_lse[pad:pad + n_lse].view(torch.float32).view(B, Hq, S)
    lib = fa.load_library()
    ptrs = [ctypes.c_void_p(t.data_ptr()) for t in args]
    if variant == fa.ATTN_VARIANT_BF16:
        ptrs = ptrs + [None, None, None]
    st = lib.attn_fwd_full(int(variant), *ptrs, ctypes.c_void_p(out.data_ptr()), int(out_dtype),
                           ctypes.c_void_p(lse_view.data_ptr()), B, Hq, Hkv, S, 128, 128,
                           int(causal), ctypes.c_float(0.0), 0, None, None, 0,
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == fa.ATTN_OK, fa.status_string(st)
    torch.cuda.synchronize()
    for r in (raw, raw_lse):
        h = r.cpu().numpy()
        assert np.all(h[:pad] == 0xA5) and np.all(h[-pad:] == 0xA5)
    # every output element written: a canary float (0xA5A5A5A5 / 0xA5A5) would be
    # about -2.9e-16 / -2.9e-16 in bf16; finite outputs of attention on these
    # inputs never equal it
    body = raw[pad:pad + n_out].cpu().numpy()
    words = body.view(np.uint32 if esz == 4 else np.uint16)
    canary = 0xA5A5A5A5 if esz == 4 else 0xA5A5
    assert not np.any(words == canary)
    lse_words = raw_lse[pad:pad + n_lse].cpu().numpy().view(np.uint32)
    assert not np.any(lse_words == 0xA5A5A5A5)
    assert torch.isfinite(out.float()).all()


# ------------------------------------------------------------------ item order

@pytest.mark.parametrize("variant", [fa.ATTN_VARIANT_LEANP, fa.ATTN_VARIANT_EXACT_FP8,
                                     fa.ATTN_VARIANT_BLOCK_EXACT, fa.ATTN_VARIANT_BF16,
                                     fa.ATTN_VARIANT_LEANP_A3])
@pytest.mark.parametrize("causal", [True, False])
def test_chunked_item_order_gives_the_same_bits(variant, causal):
    """Work items chunked by (batch, kv head), the order used for problems
    whose K and V exceed L2, against the plain longest-first order: the same
    output and log-sum-exp bit for bit, on a multi-wave grid with B = 2 and
    GQA."""
    if variant == fa.ATTN_VARIANT_BF16:
        args = dev_bf16(wl.bf16_gaussian_case(2, 12, 3, 2100, 128, 128))
    else:
        q, k, v, d = dev_fp8(wl.fp8_gaussian_case(2, 12, 3, 2100, 128, 128, seeds=(73, 74, 75)))
        args = (q, k, v, *d)
    plain = fa.attn_fwd_full(variant, *args, out_dtype=fa.ATTN_OUT_F32, causal=causal,
                             return_lse=True, split=False)
    chunked = fa.attn_fwd_full(variant, *args, out_dtype=fa.ATTN_OUT_F32, causal=causal,
                               return_lse=True, flags=fa.ATTN_FLAG_TEST_CHUNK_UNITS, split=False)
    torch.cuda.synchronize()
    assert torch.equal(plain[0], chunked[0]) and torch.equal(plain[1], chunked[1])


# ------------------------------------------------------------------ extreme ranges

@pytest.mark.parametrize("spread", [50.0, 300.0])
@pytest.mark.parametrize("variant", [fa.ATTN_VARIANT_LEANP, fa.ATTN_VARIANT_EXACT_FP8,
                                     fa.ATTN_VARIANT_LEANP_A3])
def test_extreme_logit_ranges(spread, variant):
    """Descales that spread the logits over hundreds of nats: the lazy
    reference must move by exact powers of two, far-below blocks clamp their
    UE8M0 factor, and the ablation flushes tiny probabilities; the output still
    matches the oracle's emulation under the per-row gate and stays finite."""
    case = wl.fp8_gaussian_case(1, 2, 2, 700, 128, 128, seeds=(79, 80, 81))
    # logit standard deviation ~ spread nats: scale dq*dk accordingly
    q8 = oracle.e4m3_decode(case.q) * case.dq
    k8 = oracle.e4m3_decode(case.k) * case.dk
    s_std = float(np.std(np.einsum("bshd,bthd->bhst", q8[:, :64], k8[:, :64])))
    f = spread / (s_std / np.sqrt(128.0))
    dq, dk = case.dq * np.sqrt(f), case.dk * np.sqrt(f)
    q, k, v, _ = dev_fp8(case)
    d = [torch.tensor([x], dtype=torch.float32, device="cuda") for x in (dq, dk, case.dv)]
    out = fa.attn_fwd_ex(variant, q, k, v, *d)
    torch.cuda.synchronize()
    gpu = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(gpu).all()
    path = {fa.ATTN_VARIANT_LEANP: "leanp", fa.ATTN_VARIANT_EXACT_FP8: "exact_fp8",
            fa.ATTN_VARIANT_LEANP_A3: "leanp_a3"}[variant]
    emul, amb, _ = oracle.attention(path, case.q, case.k, case.v, dq, dk, case.dv)
    check_rows(gpu.reshape(-1, 128), emul.reshape(-1, 128), amb.reshape(-1), vmax_fp8(case))


def test_nan_key_codes_per_path():
    """A NaN code (0x7F) in a key row: Lean-P's saturating multiply-add turns
    the NaN score into code 0 and the block maximum skips it, so that key gets
    weight 0 and every output stays finite; the ablation's exponential
    propagates the NaN to the rows that see the key (behaviour stated in
    fp8attn.h)."""
    case = wl.fp8_gaussian_case(1, 2, 2, 300, 128, 128, seeds=(82, 83, 84))
    case.k[0, 100, :, 5] = 0x7F
    q, k, v, d = dev_fp8(case)
    lp = fa.attn_fwd_ex(fa.ATTN_VARIANT_LEANP, q, k, v, *d)
    ab = fa.attn_fwd_ex(fa.ATTN_VARIANT_EXACT_FP8, q, k, v, *d)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(lp).all())
    assert bool(torch.isfinite(ab[0, :100]).all()) and bool(torch.isnan(ab[0, 100:]).all())
