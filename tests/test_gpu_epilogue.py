"""The Lean-P path writes its bf16 output through TMA stores: each softmax warp
converts its 32 rows into a shared-memory slot and stores 64-column boxes with
cp.async.bulk.tensor; the tensor map clips rows past S, and a box that lies
wholly past S is not issued.  The fp32 output goes through direct stores of the
same values, so the bf16 output must equal the fp32 output rounded to bf16 bit
for bit, at ragged lengths (boxes partly and wholly past S), with B = 2, GQA,
causal or not."""
import numpy as np
import pytest
import torch

import fp8_causal_prefill_flash_gb300 as fa
from fp8_causal_prefill_flash_gb300 import workloads as wl

from gpu_helpers import dev_fp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("S", [1, 31, 32, 33, 100, 129, 200, 255, 257, 300, 513])
def test_bf16_output_is_the_fp32_output_rounded(S, causal):
    case = wl.fp8_gaussian_case(2, 8, 2, S, 128, 128, seeds=(900 + S, 901 + S, 902 + S))
    q, k, v, d = dev_fp8(case)
    # whole items (the split schedule's epilogue has its own test)
    f32 = fa.attn_fwd_full(fa.ATTN_VARIANT_LEANP, q, k, v, *d, out_dtype=fa.ATTN_OUT_F32,
                           causal=causal, split=False)
    bf = fa.attn_fwd_full(fa.ATTN_VARIANT_LEANP, q, k, v, *d, out_dtype=fa.ATTN_OUT_BF16,
                          causal=causal, split=False)
    prod = fa.attn_fwd_fp8(q, k, v, *d, causal=causal)
    torch.cuda.synchronize()
    want = f32.to(torch.bfloat16)
    assert torch.equal(bf.view(torch.int16), want.view(torch.int16))
    assert torch.equal(prod.view(torch.int16), want.view(torch.int16))


def test_bf16_output_in_a_larger_buffer_leaves_the_rest_untouched():
    """The output as a view at an offset of a canary-filled buffer: the TMA
    stores write exactly the view (the map's extent is the view's S)."""
    B, H, S = 1, 4, 200
    case = wl.fp8_gaussian_case(B, H, H, S, 128, 128, seeds=(950, 951, 952))
    q, k, v, d = dev_fp8(case)
    n = B * S * H * 128
    pad = 4096
    raw = torch.full((pad + n + pad,), -7.0, dtype=torch.bfloat16, device="cuda")
    out = raw[pad:pad + n].view(B, S, H, 128)
    fa.attn_fwd_fp8(q, k, v, *d, out=out)
    torch.cuda.synchronize()
    assert bool((raw[:pad] == -7.0).all()) and bool((raw[pad + n:] == -7.0).all())
    assert not bool((out == -7.0).any())
