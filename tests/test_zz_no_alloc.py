"""attn_fwd_fp8_noalloc, called through the C ABI (GPU).

This entry point is for callers that may not allocate device memory, such as
a runtime that owns every allocation or a serving loop that allows none after
start-up.  It runs Lean-P with the split schedule, and it takes the scratch
that the schedule needs from a fixed array inside the library instead of a
caller's workspace.

The tests check four things:
- Its output equals attn_fwd_full with a workspace, which is the same
  schedule on the same kernel.
- Its output is within bf16 rounding of attn_fwd_fp8, which runs whole items.
- Both hold on two calls in a row, for a problem that splits and for one that
  does not, and when two problems alternate on the shared array.
- A problem whose schedule needs more scratch than the array holds is
  rejected before anything runs.

This file is named to run last: pytest collects test files in order, so a
run that stops at its first failure has already run every other test.  It
also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp8_causal_prefill_flash_gb300 as fa
import oracle
from fp8_causal_prefill_flash_gb300 import workloads as wl

from gpu_helpers import check_rows

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024  # ATTN_NOALLOC_SCRATCH_BYTES of include/fp8attn.h


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    lib = fa.load_library()
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.attn_fwd_fp8_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
    lib.attn_fwd_fp8_noalloc.restype = i
    return lib


def inputs(B, Hq, Hkv, S, seed):
    case = wl.fp8_gaussian_case(B, Hq, Hkv, S, 128, 128, seeds=(seed, seed + 1, seed + 2))
    q, k, v = (torch.from_numpy(a).cuda() for a in (case.q, case.k, case.v))
    d = [torch.tensor([x], dtype=torch.float32, device="cuda") for x in (case.dq, case.dk, case.dv)]
    return case, q, k, v, d


def noalloc(lib, q, k, v, d, out=None):
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty((B, S, Hq, 128), dtype=torch.bfloat16, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.attn_fwd_fp8_noalloc(P(q), P(k), P(v), *(P(x) for x in d), P(out), B, Hq, Hkv, S,
                                  D, 128, 1, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


def check_against_existing(case, q, k, v, d, got):
    """got (bf16) against attn_fwd_full with a workspace (same schedule: the
    same bits), attn_fwd_fp8 (whole items: within one bf16 rounding step) and
    the oracle's emulation on sampled rows (the per-row gate)."""
    same = fa.attn_fwd_full(fa.ATTN_VARIANT_LEANP, q, k, v, *d)
    whole = fa.attn_fwd_fp8(q, k, v, *d)
    torch.cuda.synchronize()
    assert torch.equal(got, same)
    g, w = got.float(), whole.float()
    assert float((g - w).abs().max()) <= float(w.abs().max()) * 2.0 ** -7
    B, Hq, Hkv, S, _, _ = case.shape
    rng = np.random.default_rng(S + Hq)
    rows = np.stack([rng.integers(0, B, 300), rng.integers(0, Hq, 300), rng.integers(0, S, 300)],
                    axis=1).astype(np.int64)
    want, amb, _ = oracle.attention("leanp", case.q, case.k, case.v, case.dq, case.dk, case.dv,
                                    rows=rows)
    gg = g.cpu().numpy().astype(np.float64)
    vmax = float(np.max(np.abs(oracle.e4m3_decode(case.v)))) * case.dv
    # bf16 output: the emulation gate plus half a bf16 step of the row's values
    check_rows(np.stack([gg[b, i, h] for b, h, i in rows]), want, amb, vmax, tol=2e-3 + 2.0 ** -9)


@pytest.mark.parametrize("shape", [(1, 8, 8, 2048), (2, 4, 2, 2000), (1, 32, 32, 2048)],
                         ids=["splits", "splits_gqa_ragged", "whole_items"])
def test_two_calls_in_a_row_match_the_existing_entry_points(lib, shape):
    B, Hq, Hkv, S = shape
    case, q, k, v, d = inputs(B, Hq, Hkv, S, 600)
    need = fa.workspace_size(fa.ATTN_VARIANT_LEANP, B, Hq, Hkv, S, 128, 128, True)
    assert (need > 0) == (Hq != 32) and need <= SCRATCH_BYTES
    for _ in range(2):
        st, got = noalloc(lib, q, k, v, d)
        assert st == fa.ATTN_OK, fa.status_string(st)
        check_against_existing(case, q, k, v, d, got)


def test_two_problems_alternate_on_the_shared_scratch(lib):
    a = inputs(1, 8, 8, 2048, 610)
    b = inputs(1, 2, 2, 4096, 620)
    outs = []
    for _ in range(2):
        for case, q, k, v, d in (a, b):
            st, out = noalloc(lib, q, k, v, d)
            assert st == fa.ATTN_OK, fa.status_string(st)
            outs.append(out)
    torch.cuda.synchronize()
    for i, (case, q, k, v, d) in enumerate((a, b, a, b)):
        check_against_existing(case, q, k, v, d, outs[i])


def test_problem_needing_more_scratch_is_rejected(lib):
    """One head of 24K keys: its split schedule needs more than 32 MiB."""
    case, q, k, v, d = inputs(1, 1, 1, 24576, 630)
    need = fa.workspace_size(fa.ATTN_VARIANT_LEANP, 1, 1, 1, 24576, 128, 128, True)
    assert need > SCRATCH_BYTES
    out = torch.full((1, 24576, 1, 128), -7.0, dtype=torch.bfloat16, device="cuda")
    st, _ = noalloc(lib, q, k, v, d, out=out)
    torch.cuda.synchronize()
    assert st == fa.ATTN_ERR_UNSUPPORTED
    assert bool((out == -7.0).all()), "nothing may run for a rejected call"
