"""The debug library's clock64 role timeline (attn_debug_timeline): one
Lean-P call, then the stamps of CTA 0's first work item must be present and
ordered as the pipeline's dependencies require."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_causal_prefill_flash_gb300 as fa
from fp8_causal_prefill_flash_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_role_timeline_respects_the_hand_overs():
    lib = fa.load_timeline_library()
    B, H, S = 1, 4, 4096
    c = wl.fp8_gaussian_case(B, H, H, S, 128, 128, seeds=(200, 201, 202))
    q, k, v = (torch.from_numpy(a).cuda() for a in (c.q, c.k, c.v))
    d = [torch.tensor([x], dtype=torch.float32, device="cuda") for x in (c.dq, c.dk, c.dv)]
    out = torch.empty((B, S, H, 128), dtype=torch.float32, device="cuda")
    fa.debug_timeline(lib, reset=True)  # start from zeros
    st = lib.attn_fwd_ex(fa.ATTN_VARIANT_LEANP, *(ctypes.c_void_p(t.data_ptr()) for t in (q, k, v, *d)),
                         ctypes.c_void_p(out.data_ptr()), fa.ATTN_OUT_F32, B, H, H, S, 128, 128, 1,
                         0.0, 0, None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == fa.ATTN_OK
    torch.cuda.synchronize()
    tl = fa.debug_timeline(lib, reset=True).astype(np.int64)
    # CTA 0 takes the longest item first: query block 15, 31 and 32 key tiles
    nk = (31, 32)
    for t in (0, 1):
        for j in range(nk[t]):
            s = tl[t, j, :5]
            assert np.all(s > 0) and np.all(np.diff(s) >= 0), (t, j, s)
            pv = tl[2 + t, j, :3]
            assert np.all(pv > 0) and np.all(np.diff(pv) >= 0), (t, j, pv)
            assert pv[2] >= s[4]            # P.V issued after P was stored
    for j in range(nk[0]):
        assert tl[3, j, 5] >= tl[0, j, 2]   # S1(j) issued after S0(j) was drained
        assert tl[1, j, 1] >= tl[3, j, 5]   # softmax 1 sees S1(j) after its issue
        if j + 1 < nk[0]:
            assert tl[2, j + 1, 5] >= tl[1, j, 2]  # S0(j+1) issued after S1(j) was drained
    # one key tile of the pipeline, in clocks (printed for the record)
    period = np.median(np.diff(tl[0, 4:nk[0], 1]))
    print(f"median period per key tile (softmax 0, S ready to S ready): {period:.0f} clk")
