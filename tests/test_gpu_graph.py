"""CUDA-graph capture of the C-ABI calls: the descales live in device memory
and the calls allocate nothing and never synchronise, so a captured
quantise + attention sequence replays on new data (new inputs and new
descales written into the same buffers) with the same bits as eager calls."""
import numpy as np
import pytest
import torch

import fp8_causal_prefill_flash_gb300 as fa
from fp8_causal_prefill_flash_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


def _fp8(case):
    q, k, v = (torch.from_numpy(a).cuda() for a in (case.q, case.k, case.v))
    d = [torch.tensor([x], dtype=torch.float32, device="cuda") for x in (case.dq, case.dk, case.dv)]
    return q, k, v, d


def test_attention_replays_on_new_inputs_and_descales():
    c0 = wl.fp8_gaussian_case(1, 4, 2, 700, 128, 128, seeds=(180, 181, 182))
    c1 = wl.fp8_gaussian_case(1, 4, 2, 700, 128, 128, seeds=(183, 184, 185))
    q, k, v, d = _fp8(c0)
    out = torch.empty((1, 700, 4, 128), dtype=torch.bfloat16, device="cuda")
    fa.attn_fwd_fp8(q, k, v, *d, out=out)  # first call outside capture (per-device setup)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.attn_fwd_fp8(q, k, v, *d, out=out)
    # new data and new descales in the same buffers, then replay
    q1, k1, v1, d1 = _fp8(c1)
    for dst, src in zip((q, k, v, *d), (q1, k1, v1, *d1)):
        dst.copy_(src)
    g.replay()
    torch.cuda.synchronize()
    want = fa.attn_fwd_fp8(q1, k1, v1, *d1)
    torch.cuda.synchronize()
    assert torch.equal(out, want)


def test_quantise_and_attention_in_one_graph():
    """Rotate-and-quantise Q and K, quantise V, attend: one graph, replayed on
    fresh bf16 activations, equals the same calls made eagerly."""
    B, S, H, D = 1, 520, 2, 128
    gen = torch.Generator(device="cuda")
    gen.manual_seed(190)
    xs = [torch.randn((B, S, H, D), generator=gen, device="cuda").to(torch.bfloat16)
          for _ in range(3)]
    codes = [torch.empty((B, S, H, D), dtype=torch.uint8, device="cuda") for _ in range(3)]
    ds = [torch.empty(1, dtype=torch.float32, device="cuda") for _ in range(3)]
    out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")

    def seq():
        for i, rot in enumerate((True, True, False)):
            fa.attn_quantize_fp8(xs[i], hadamard=rot, codes=codes[i], descale=ds[i])
        fa.attn_fwd_fp8(*codes, *ds, out=out)

    seq()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        seq()
    fresh = [torch.randn((B, S, H, D), generator=gen, device="cuda").to(torch.bfloat16)
             for _ in range(3)]
    for dst, src in zip(xs, fresh):
        dst.copy_(src)
    g.replay()
    torch.cuda.synchronize()
    got = out.clone()
    seq()  # eager, same buffers
    torch.cuda.synchronize()
    assert torch.equal(got, out)
    assert not torch.equal(got, torch.zeros_like(got))
