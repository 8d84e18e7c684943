"""Shared helpers for the GPU parity tests: move seeded cases to the device,
call the library through its C ABI and compare with the oracle."""
from __future__ import annotations

import inspect
import os

import numpy as np
import torch

import fp8_causal_prefill_flash_gb300 as fa
import oracle

#: max-abs gate against the CPU emulation of the identical scheme, relative
#: to max|v~| (the specification's 2e-3).
EMUL_TOL = 2e-3
#: relative-RMS gates against fp64 attention.
FP8_RMS_TOL = 3e-2
BF16_RMS_TOL = 5e-3


def dev_fp8(case):
    q = torch.from_numpy(case.q).cuda()
    k = torch.from_numpy(case.k).cuda()
    v = torch.from_numpy(case.v).cuda()
    d = [torch.tensor([x], dtype=torch.float32, device="cuda") for x in (case.dq, case.dk, case.dv)]
    return q, k, v, d


def dev_bf16(case):
    return tuple(torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
                 for a in (case.q, case.k, case.v))


def run_fp8(variant, case, out_f32=True, scale=0.0):
    q, k, v, d = dev_fp8(case)
    out = fa.attn_fwd_ex(variant, q, k, v, *d,
                         out_dtype=fa.ATTN_OUT_F32 if out_f32 else fa.ATTN_OUT_BF16,
                         softmax_scale=scale)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def run_bf16(case, out_f32=True):
    q, k, v = dev_bf16(case)
    out = fa.attn_fwd_ex(fa.ATTN_VARIANT_BF16, q, k, v,
                         out_dtype=fa.ATTN_OUT_F32 if out_f32 else fa.ATTN_OUT_BF16)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def vmax_fp8(case):
    return float(np.max(np.abs(oracle.e4m3_decode(case.v)))) * case.dv


def rel_rms(x, ref):
    return float(np.sqrt(np.mean((x - ref) ** 2)) / np.sqrt(np.mean(ref ** 2)))


#: every check_rows call of the session: (test, rows, rows that needed the
#: ambiguity term, largest amb of those rows, largest amb of all rows)
AMB_LOG: list[tuple[str, int, int, float, float]] = []

#: at most this fraction of a call's rows (and at least one row) may need the
#: ambiguity term; a larger count means the GPU decides roundings differently
#: from the oracle more often than the fp32 band explains
AMB_ROWS_FRAC = 0.01


def check_rows(gpu, emul, amb, vmax, tol=EMUL_TOL, amb_rows_frac=AMB_ROWS_FRAC):
    """Per row: |gpu - emul|_max <= tol*vmax + 2*amb/(1-amb)*vmax.

    `amb` is the oracle's bound on the weight mass an fp32 evaluation may move
    across a rounding decision; rows without such mass get the plain gate.
    Rows whose error exceeds the plain gate (and so use the term) must be few:
    at most ``amb_rows_frac`` of the rows, and at least one row is allowed.
    Returns (number of rows, number of rows that needed the ambiguity term).
    """
    err = np.max(np.abs(gpu - emul), axis=-1)
    amb = np.asarray(amb, dtype=np.float64).reshape(err.shape)
    a = np.minimum(amb, 0.5)
    plain = tol * vmax
    bound = plain + 2.0 * a / (1.0 - a) * vmax
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{int(bad.sum())} rows out of bound; first {idx.tolist()}: err "
            f"{err[bad][:5]} bound {bound[bad][:5]} amb {amb[bad][:5]}")
    needed = err > plain
    n_needed = int(needed.sum())
    amb_used = float(amb[needed].max()) if n_needed else 0.0
    caller = inspect.stack()[1]
    label = f"{os.path.basename(caller.filename)}:{caller.lineno}"
    AMB_LOG.append((label, int(err.size), n_needed, amb_used, float(amb.max()) if amb.size else 0.0))
    allowed = max(1, int(amb_rows_frac * err.size))
    assert n_needed <= allowed, (
        f"{n_needed} of {err.size} rows needed the ambiguity term (allowed {allowed}); "
        f"largest amb among them {amb_used:.3e}")
    return int(err.size), n_needed
