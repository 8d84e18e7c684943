"""Randomised properties of the oracle (CPU only): shapes, head groupings,
head dims, causality and descales drawn from a seeded generator (a fixed list
of cases, so that every run checks the same inputs and nothing depends on an
optional package), with checks that hold for any input.  A wrong index in the oracle (a head mapping, a batch or
row offset, a transposed operand) fails one of them.

- Every path's output row is a convex combination of the V rows it sees
  (softmax weights are positive and normalised): per column it lies between
  the minimum and the maximum of those V values.  The exact-FP8 ablation
  divides its e4m3-rounded weights by the unrounded sum, so its weights sum
  to 1 only within the rounding: each weight p moves by at most 2^-4 p (normal
  range) or 2^-10 (subnormal), with sum p >= 1 (the maximum has p = 1).
- Causal rows do not change when later keys and values change.
- Grouped-query attention equals attention on kv heads repeated per group.
- Rows computed alone equal the same rows of a full call.
- The unrotated quantiser reproduces its input within half an e4m3 step.
"""
import numpy as np
import pytest

import oracle

PATHS = ("ref", "leanp", "leanp_a3", "exact_fp8", "variant_e")


def _codes(rng, shape):
    x = rng.standard_normal(shape).astype(np.float32)
    x *= np.float32(448.0) / np.float32(np.max(np.abs(x)))
    import torch
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def draw_shapes(n, seed):
    """n cases (B, (Hq, Hkv), S, Dqk, causal, seed), drawn from one seed."""
    rng = np.random.default_rng(seed)
    heads = [(1, 1), (2, 1), (4, 2), (3, 3)]
    return [(int(rng.integers(1, 3)), heads[int(rng.integers(0, 4))], int(rng.integers(1, 201)),
             int(rng.choice([128, 192])), bool(rng.integers(0, 2)), int(rng.integers(0, 2**31)))
            for _ in range(n)]


@pytest.mark.parametrize("args", draw_shapes(25, 101))
def test_output_is_a_convex_combination_of_the_values_seen(args):
    B, (Hq, Hkv), S, Dqk, causal, seed = args
    rng = np.random.default_rng(seed)
    q, k, v = _codes(rng, (B, S, Hq, Dqk)), _codes(rng, (B, S, Hkv, Dqk)), _codes(rng, (B, S, Hkv, 128))
    dq, dk, dv = rng.uniform(0.002, 0.05), rng.uniform(0.002, 0.05), rng.uniform(0.1, 2.0)
    vv = oracle.e4m3_decode(v) * dv
    for path in PATHS:
        out, _, lse = oracle.attention(path, q, k, v, dq, dk, dv, causal=causal)
        assert np.isfinite(out).all() and np.isfinite(lse).all()
        for b in range(B):
            for h in range(Hq):
                g = h * Hkv // Hq
                for i in range(S):
                    seen = vv[b, :i + 1 if causal else S, g, :]
                    lo, hi = seen.min(axis=0), seen.max(axis=0)
                    tol = 1e-9 * (1 + np.abs(seen).max())
                    if path == "exact_fp8":
                        tol += (2.0 ** -4 + len(seen) * 2.0 ** -10) * np.abs(seen).max()
                    assert np.all(out[b, i, h] >= lo - tol) and np.all(out[b, i, h] <= hi + tol), \
                        (path, b, h, i)


@pytest.mark.parametrize("args", draw_shapes(20, 202))
def test_future_keys_and_row_subsets(args):
    B, (Hq, Hkv), S, Dqk, _, seed = args
    rng = np.random.default_rng(seed)
    q, k, v = _codes(rng, (B, S, Hq, Dqk)), _codes(rng, (B, S, Hkv, Dqk)), _codes(rng, (B, S, Hkv, 128))
    cut = int(rng.integers(0, S))
    k2, v2 = k.copy(), v.copy()
    k2[:, cut + 1:] = _codes(rng, k2[:, cut + 1:].shape) if cut + 1 < S else k2[:, cut + 1:]
    v2[:, cut + 1:] = _codes(rng, v2[:, cut + 1:].shape) if cut + 1 < S else v2[:, cut + 1:]
    rows = np.array([(int(rng.integers(0, B)), int(rng.integers(0, Hq)), int(rng.integers(0, S)))
                     for _ in range(6)], dtype=np.int64)
    for path in PATHS:
        full, _, _ = oracle.attention(path, q, k, v, 0.01, 0.01, 0.5)
        again, _, _ = oracle.attention(path, q, k2, v2, 0.01, 0.01, 0.5)
        assert np.array_equal(full[:, :cut + 1], again[:, :cut + 1]), path
        some, _, _ = oracle.attention(path, q, k, v, 0.01, 0.01, 0.5, rows=rows)
        assert np.array_equal(some, np.stack([full[b, i, h] for b, h, i in rows])), path


def draw_gqa(n, seed):
    rng = np.random.default_rng(seed)
    heads = [(4, 2), (6, 3), (4, 1)]
    return [(int(rng.integers(1, 151)), heads[int(rng.integers(0, 3))], bool(rng.integers(0, 2)),
             int(rng.integers(0, 2**31))) for _ in range(n)]


@pytest.mark.parametrize("S,heads,causal,seed", draw_gqa(20, 303))
def test_gqa_equals_repeated_kv_heads(S, heads, causal, seed):
    Hq, Hkv = heads
    rng = np.random.default_rng(seed)
    q, k, v = _codes(rng, (1, S, Hq, 128)), _codes(rng, (1, S, Hkv, 128)), _codes(rng, (1, S, Hkv, 128))
    rep = Hq // Hkv
    kr, vr = np.repeat(k, rep, axis=2), np.repeat(v, rep, axis=2)
    for path in PATHS:
        a, _, la = oracle.attention(path, q, k, v, 0.01, 0.01, 0.5, causal=causal)
        b, _, lb = oracle.attention(path, q, kr, vr, 0.01, 0.01, 0.5, causal=causal)
        assert np.array_equal(a, b) and np.array_equal(la, lb), path


def draw_quant(n, seed):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(1, 41)), int(rng.choice([128, 192])),
             float(10.0 ** rng.uniform(-3, 3)), int(rng.integers(0, 2**31))) for _ in range(n)]


@pytest.mark.parametrize("n,D,scale,seed", draw_quant(30, 404))
def test_unrotated_quantiser_reproduces_its_input(n, D, scale, seed):
    x = (np.random.default_rng(seed).standard_normal((n, D)) * scale).astype(np.float32)
    codes, ds = oracle.quantize_e4m3(x, False)
    back = oracle.e4m3_decode(codes) * np.float64(ds)
    # e4m3 keeps 3 mantissa bits: half a step is 2^-4 relative (normal range)
    # plus the subnormal step 2^-9 in units of the descale
    assert np.all(np.abs(back - x) <= 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * ds + 1e-30)
