"""Many short work items per CTA, on every path: S of one to three key tiles
with 8 batches and 32 query heads, so that each persistent CTA runs several
items of one to five key tiles back to back (at S = 100 query tile 1 of every
item lies wholly beyond the sequence).  This exercises the phase bookkeeping
of every mbarrier across item boundaries, where the softmax writes P_t(0)
without waiting for a P.V product and the issuing warps run furthest ahead.

Checks: the device status word stays 0 (a bounded wait that ran out would set
ATTN_ERR_TIMEOUT and leave rows unwritten), sampled rows match the oracle's
definition of the same path, and three launches give the same bits."""
import numpy as np
import pytest
import torch

import fp8_causal_prefill_flash_gb300 as fa
import oracle
from fp8_causal_prefill_flash_gb300 import workloads as wl

from gpu_helpers import EMUL_TOL, check_rows, dev_bf16, dev_fp8

pytestmark = pytest.mark.gpu

B, HQ, HKV = 8, 32, 8
PATHS = {fa.ATTN_VARIANT_LEANP: "leanp", fa.ATTN_VARIANT_EXACT_FP8: "exact_fp8",
         fa.ATTN_VARIANT_BLOCK_EXACT: "variant_e", fa.ATTN_VARIANT_BF16: "bf16",
         fa.ATTN_VARIANT_LEANP_A3: "leanp_a3"}


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("S", [100, 300])
@pytest.mark.parametrize("variant", list(PATHS))
def test_many_short_items_per_cta(variant, S, causal):
    seeds = (400 + S, 401 + S, 402 + S)
    if variant == fa.ATTN_VARIANT_BF16:
        case = wl.bf16_gaussian_case(B, HQ, HKV, S, 128, 128, seeds=seeds)
        args = dev_bf16(case)
        dq = dk = dv = 1.0
        vmax = float(np.max(np.abs(oracle.bf16_decode(case.v))))
    else:
        case = wl.fp8_gaussian_case(B, HQ, HKV, S, 128, 128, seeds=seeds)
        q, k, v, d = dev_fp8(case)
        args = (q, k, v, *d)
        dq, dk, dv = case.dq, case.dk, case.dv
        vmax = float(np.max(np.abs(oracle.e4m3_decode(case.v)))) * dv
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(3):
        out, _ = fa.attn_fwd_full(variant, *args, out_dtype=fa.ATTN_OUT_F32, causal=causal,
                                  return_lse=True, dev_status=status)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(status.item()) == fa.ATTN_OK, fa.status_string(int(status.item()))
    assert all(torch.equal(outs[0], o) for o in outs[1:])

    rng = np.random.default_rng(403 + S)
    n = 1200
    rows = np.stack([rng.integers(0, B, n), rng.integers(0, HQ, n), rng.integers(0, S, n)],
                    axis=1).astype(np.int64)
    want, amb, _ = oracle.attention(PATHS[variant], case.q, case.k, case.v, dq, dk, dv,
                                    rows=rows, causal=causal)
    gpu = outs[0].cpu().numpy().astype(np.float64)
    got = np.stack([gpu[b, i, h] for b, h, i in rows])
    check_rows(got, want, np.zeros(n) if amb is None else amb, vmax, tol=EMUL_TOL)
