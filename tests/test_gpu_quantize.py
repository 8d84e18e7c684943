"""GPU parity of the e4m3 quantiser of Q and K (with and without the Hadamard
rotation) against the oracle, through the C ABI, and its end-to-end effect on
the attention error.

The codes are decided in fp32 on both sides in the same butterfly order, so
they are compared bit for bit, as is the descale.
"""
import numpy as np
import pytest
import torch

import fp8_causal_prefill_flash_gb300 as fa
import oracle
from fp8_causal_prefill_flash_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


def _input(shape, dtype, seed, outliers=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    if outliers:
        ch = rng.choice(shape[-1], outliers, replace=False)
        x[..., ch] *= 20.0
    if dtype == "bf16":
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)
        dev = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        return bits, dev
    return x, torch.from_numpy(x).cuda()


@pytest.mark.parametrize("shape", [(1, 1, 1, 128), (2, 37, 3, 128), (1, 300, 2, 192),
                                   (1, 5000, 8, 128), (3, 1111, 1, 192)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rotate", [False, True])
def test_codes_and_descale_bitwise(shape, dtype, rotate):
    host, dev = _input(shape, dtype, seed=sum(shape) + rotate, outliers=2)
    codes, ds = fa.attn_quantize_fp8(dev, hadamard=rotate)
    torch.cuda.synchronize()
    want_codes, want_ds = oracle.quantize_e4m3(host, rotate)
    got = codes.cpu().numpy()
    assert np.array_equal(got, want_codes), int((got != want_codes).sum())
    assert ds.item() == np.float32(want_ds)


def test_zero_input():
    x = torch.zeros((1, 4, 2, 192), dtype=torch.float32, device="cuda")
    codes, ds = fa.attn_quantize_fp8(x, hadamard=True)
    torch.cuda.synchronize()
    assert not codes.any().item() and ds.item() == 0.125


def test_rotation_lowers_attention_error_with_outliers():
    """Q and K with scaled channels (the outlier workloads), quantised with and
    without the rotation on the GPU, V unrotated; Lean-P attention against
    fp64 attention on the unquantised inputs."""
    B, S, H, D = 1, 512, 2, 128
    rng = np.random.default_rng(17)
    q = rng.standard_normal((B, S, H, D)).astype(np.float32)
    k = rng.standard_normal((B, S, H, D)).astype(np.float32)
    v = rng.standard_normal((B, S, H, D)).astype(np.float32)
    ch = rng.choice(D, 2, replace=False)
    q[..., ch] *= 8.0
    k[..., ch] *= 8.0
    qt, kt, vt = (torch.from_numpy(a).cuda() for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(a).double().permute(0, 2, 1, 3) for a in (q, k, v)),
        is_causal=True).permute(0, 2, 1, 3).numpy()
    err = []
    for rot in (False, True):
        cq, dq = fa.attn_quantize_fp8(qt, hadamard=rot)
        ck, dk = fa.attn_quantize_fp8(kt, hadamard=rot)
        cv, dv = fa.attn_quantize_fp8(vt, hadamard=False)
        out = fa.attn_fwd_ex(fa.ATTN_VARIANT_LEANP, cq, ck, cv, dq, dk, dv,
                             out_dtype=fa.ATTN_OUT_F32)
        torch.cuda.synchronize()
        o = out.cpu().numpy().astype(np.float64)
        err.append(float(np.sqrt(np.mean((o - ref) ** 2)) / np.sqrt(np.mean(ref ** 2))))
    print(f"Lean-P rel-RMS vs fp64 on unquantised inputs: plain {err[0]:.4f}, "
          f"rotated {err[1]:.4f}")
    assert err[1] < 0.8 * err[0], err


def test_quantised_inputs_run_the_headline_path():
    """The quantiser's codes and descales feed attn_fwd_fp8 unchanged: the
    result equals the oracle's emulation on those codes (rotated Q, K)."""
    case = wl.fp8_gaussian_case(1, 2, 2, 300, 128, 128, seeds=(61, 62, 63))
    rng = np.random.default_rng(64)
    q = torch.from_numpy(rng.standard_normal((1, 300, 2, 128)).astype(np.float32)).cuda()
    k = torch.from_numpy(rng.standard_normal((1, 300, 2, 128)).astype(np.float32)).cuda()
    cq, dq = fa.attn_quantize_fp8(q, hadamard=True)
    ck, dk = fa.attn_quantize_fp8(k, hadamard=True)
    cv = torch.from_numpy(case.v).cuda()
    dv = torch.tensor([case.dv], dtype=torch.float32, device="cuda")
    out = fa.attn_fwd_ex(fa.ATTN_VARIANT_LEANP, cq, ck, cv, dq, dk, dv, out_dtype=fa.ATTN_OUT_F32)
    torch.cuda.synchronize()
    qc, kc = cq.cpu().numpy(), ck.cpu().numpy()
    emul, amb = oracle.emul_leanp(qc, kc, case.v, dq.item(), dk.item(), case.dv)
    vmax = float(np.max(np.abs(oracle.e4m3_decode(case.v)))) * case.dv
    err = np.max(np.abs(out.cpu().numpy().astype(np.float64) - emul), axis=-1)
    a = np.minimum(amb, 0.5)
    assert np.all(err <= 2e-3 * vmax + 2.0 * a / (1.0 - a) * vmax)


def test_from_bf16_wrapper_equals_the_manual_composition():
    """flash_attn_fp8_from_bf16 is the four calls made by hand, bit for bit,
    and (with outlier channels) more accurate with the rotation than without."""
    rng = np.random.default_rng(30)
    x = [rng.standard_normal((1, 700, 4, 128)).astype(np.float32) for _ in range(3)]
    ch = rng.choice(128, 2, replace=False)
    x[0][..., ch] *= 8.0
    x[1][..., ch] *= 8.0
    q, k, v = (torch.from_numpy(a).cuda().to(torch.bfloat16) for a in x)
    got, lse = fa.flash_attn_fp8_from_bf16(q, k, v, hadamard=True, causal=False,
                                           return_softmax_lse=True)
    cq, dq = fa.attn_quantize_fp8(q, hadamard=True)
    ck, dk = fa.attn_quantize_fp8(k, hadamard=True)
    cv, dv = fa.attn_quantize_fp8(v, hadamard=False)
    want, lse_w = fa.flash_attn_fp8_func(cq, ck, cv, dq, dk, dv, causal=False,
                                         return_softmax_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(got, want) and torch.equal(lse, lse_w)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(t.double().permute(0, 2, 1, 3) for t in (q, k, v))).permute(0, 2, 1, 3)
    plain = fa.flash_attn_fp8_from_bf16(q, k, v, hadamard=False, causal=False)
    err = lambda o: float(((o.double() - ref) ** 2).mean().sqrt() / (ref ** 2).mean().sqrt())
    assert err(got) < err(plain), (err(got), err(plain))
