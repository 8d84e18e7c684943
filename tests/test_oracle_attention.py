"""Pins for the oracle's attention definitions.

The oracle is checked against a library routine (torch's scaled dot product
attention in fp64), closed forms, invariants the articles state or imply, and
brute-force bounds, so that a dropped term, a wrong sign or index or a
transposed operand fails at least one check.
"""
import math

import numpy as np
import pytest
import torch

from fp8_causal_prefill_flash_gb300 import workloads as wl

LN2 = math.log(2.0)


def codes_of(x):
    """e4m3 codes of values that are exactly representable."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32))
    c = t.to(torch.float8_e4m3fn)
    assert torch.equal(c.to(torch.float32), t), "value not representable in e4m3"
    return c.view(torch.uint8).numpy().copy()


def rel_rms(x, ref):
    return float(np.sqrt(np.mean((x - ref) ** 2)) / np.sqrt(np.mean(ref ** 2)))


@pytest.fixture(scope="module")
def small_case():
    return wl.fp8_gaussian_case(1, 4, 2, 150, 16, 16, seeds=(3, 4, 5))


def test_ref_fp64_matches_torch_sdpa(oracle_mod, small_case):
    """ref_fp64 equals torch SDPA (fp64, is_causal, GQA by repeat) on dequantized inputs."""
    c = small_case
    B, Hq, Hkv, S, Dqk, Dv = c.shape
    for scale in (None, 0.37):
        ours = oracle_mod.ref_fp64(c.q, c.k, c.v, c.dq, c.dk, c.dv, scale=scale)
        dec = torch.from_numpy(oracle_mod.e4m3_decode(np.arange(256)))
        qf = dec[torch.from_numpy(c.q).long()] * c.dq
        kf = dec[torch.from_numpy(c.k).long()] * c.dk
        vf = dec[torch.from_numpy(c.v).long()] * c.dv
        rep = Hq // Hkv
        qf, kf, vf = (t.permute(0, 2, 1, 3) for t in (qf, kf, vf))
        kf = kf.repeat_interleave(rep, dim=1)
        vf = vf.repeat_interleave(rep, dim=1)
        want = torch.nn.functional.scaled_dot_product_attention(
            qf, kf, vf, is_causal=True, scale=(1 / math.sqrt(Dqk) if scale is None else scale))
        want = want.permute(0, 2, 1, 3).numpy()
        assert np.allclose(ours, want, rtol=1e-12, atol=1e-12)


def test_ref_bf16_matches_torch_sdpa(oracle_mod):
    c = wl.bf16_gaussian_case(1, 2, 1, 70, 8, 8, seeds=(1, 2, 3))
    ours = oracle_mod.ref_fp64_bf16(c.q, c.k, c.v)
    dec = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    qf, kf, vf = (dec(a).permute(0, 2, 1, 3) for a in (c.q, c.k, c.v))
    kf, vf = kf.repeat_interleave(2, dim=1), vf.repeat_interleave(2, dim=1)
    want = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, is_causal=True)
    assert np.allclose(ours, want.permute(0, 2, 1, 3).numpy(), rtol=1e-12, atol=1e-12)


def test_row_sampling_matches_full(oracle_mod, small_case):
    c = small_case
    full_ref = oracle_mod.ref_fp64(c.q, c.k, c.v, c.dq, c.dk, c.dv)
    full_lp, full_amb = oracle_mod.emul_leanp(c.q, c.k, c.v, c.dq, c.dk, c.dv)
    rows = np.array([[0, 3, 149], [0, 0, 0], [0, 1, 64], [0, 2, 63]])
    r = oracle_mod.ref_fp64(c.q, c.k, c.v, c.dq, c.dk, c.dv, rows=rows)
    lp, amb = oracle_mod.emul_leanp(c.q, c.k, c.v, c.dq, c.dk, c.dv, rows=rows)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(r[n], full_ref[b, i, h])
        assert np.array_equal(lp[n], full_lp[b, i, h])
        assert amb[n] == full_amb[b, i, h]


def _all_paths(oracle_mod, q, k, v, dq=1.0, dk=1.0, dv=1.0, scale=None):
    ref = oracle_mod.ref_fp64(q, k, v, dq, dk, dv, scale=scale)
    lp, _ = oracle_mod.emul_leanp(q, k, v, dq, dk, dv, scale=scale)
    ab, _ = oracle_mod.emul_exact_fp8(q, k, v, dq, dk, dv, scale=scale)
    return ref, lp, ab


def test_q_zero_gives_prefix_mean(oracle_mod):
    """Q = 0: every logit is 0, so every path returns the causal prefix mean of V.
    (Lean-P: every code is C, every block scale equal; ablation: every p = 1.)"""
    S, D = 200, 8
    v = wl.fp8_gaussian_case(1, 2, 2, S, D, D, seeds=(1, 2, 3))
    q = np.zeros_like(v.q)
    ref, lp, ab = _all_paths(oracle_mod, q, v.k, v.v, 1.0, v.dk, v.dv)
    vf = oracle_mod.e4m3_decode(v.v) * v.dv
    want = np.cumsum(vf, axis=1) / np.arange(1, S + 1)[None, :, None, None]
    for got in (ref, lp, ab):
        assert np.allclose(got, want, rtol=1e-13, atol=1e-13)
    bq = np.zeros((1, S, 2, D), np.uint16)
    bv = wl.bf16_gaussian_case(1, 2, 2, S, D, D)
    bf = oracle_mod.emul_bf16(bq, bv.k, bv.v)
    wantb = np.cumsum(oracle_mod.bf16_decode(bv.v), axis=1) / np.arange(1, S + 1)[None, :, None, None]
    assert np.allclose(bf, wantb, rtol=1e-13, atol=1e-13)


def test_v_ones_rounded_row_sum_is_exact(oracle_mod):
    """V = 1: dividing by the sum of the ROUNDED probabilities ([ART-MTP] "Per-block
    scaling and a rounded row sum") makes every Lean-P output exactly dv; the
    ablation, whose row sum is unrounded, does not."""
    c = wl.fp8_gaussian_case(1, 2, 2, 300, 32, 32, seeds=(6, 7, 8))
    ones = np.full_like(c.v, codes_of([1.0])[0])
    ref, lp, ab = _all_paths(oracle_mod, c.q, c.k, ones, c.dq, c.dk, 0.75)
    assert np.all(lp == 0.75)
    assert np.allclose(ref, 0.75, rtol=1e-13)
    assert np.max(np.abs(ab - 0.75)) > 1e-4


def test_one_hot_dominant_key(oracle_mod):
    """A key whose logit exceeds every other by >= 40 binades returns its V row."""
    S, D = 130, 4
    q = np.zeros((1, S, 1, D), np.float32)
    q[..., 0] = 1.0
    k = np.zeros((1, S, 1, D), np.float32)
    star = 70
    k[0, star, 0, 0] = 64.0  # u = 8*lambda*64 with lambda = 1 -> 512 code units = 64 binades
    v = wl.gaussian((1, S, 1, D), 9).astype(np.float32)
    vc, dv = wl.quantize_e4m3(v)
    scale = LN2  # lambda = log2(e) * scale = 1
    ref, lp, ab = _all_paths(oracle_mod, codes_of(q), codes_of(k), vc, 1.0, 1.0, dv, scale=scale)
    vrow = oracle_mod.e4m3_decode(vc[0, star, 0]) * dv
    for got in (ref, lp, ab):
        assert np.allclose(got[0, star:, 0], vrow[None, :], rtol=0, atol=1e-12)


def test_causal_future_keys_do_not_matter(oracle_mod):
    c = wl.fp8_gaussian_case(1, 2, 1, 200, 16, 16, seeds=(11, 12, 13))
    i0 = 120
    k2, v2 = c.k.copy(), c.v.copy()
    rng = np.random.default_rng(0)
    k2[:, i0 + 1:] = rng.integers(0, 126, size=k2[:, i0 + 1:].shape, dtype=np.uint8)
    v2[:, i0 + 1:] = rng.integers(0, 126, size=v2[:, i0 + 1:].shape, dtype=np.uint8)
    a = _all_paths(oracle_mod, c.q, c.k, c.v, c.dq, c.dk, c.dv)
    b = _all_paths(oracle_mod, c.q, k2, v2, c.dq, c.dk, c.dv)
    for x, y in zip(a, b):
        assert np.array_equal(x[:, :i0 + 1], y[:, :i0 + 1])
        assert not np.array_equal(x[:, i0 + 1:], y[:, i0 + 1:])


def test_gqa_equals_repeated_kv(oracle_mod):
    """Query head h reads kv head floor(h*Hkv/Hq): GQA equals explicit repetition."""
    c = wl.fp8_gaussian_case(1, 6, 2, 90, 16, 16, seeds=(14, 15, 16))
    k_rep = np.repeat(c.k, 3, axis=2)
    v_rep = np.repeat(c.v, 3, axis=2)
    a = _all_paths(oracle_mod, c.q, c.k, c.v, c.dq, c.dk, c.dv)
    b = _all_paths(oracle_mod, c.q, k_rep, v_rep, c.dq, c.dk, c.dv)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_power_of_two_descale_equivariance(oracle_mod):
    c = wl.fp8_gaussian_case(1, 2, 2, 140, 16, 16, seeds=(17, 18, 19))
    a = _all_paths(oracle_mod, c.q, c.k, c.v, c.dq, c.dk, c.dv)
    b = _all_paths(oracle_mod, c.q, c.k, c.v, c.dq * 2, c.dk / 2, c.dv)
    d = _all_paths(oracle_mod, c.q, c.k, c.v, c.dq, c.dk, c.dv * 4)
    for x, y, z in zip(a, b, d):
        assert np.array_equal(x, y)
        assert np.array_equal(4 * x, z)


def test_leanp_two_key_band(oracle_mod):
    """Row 1 with V = (0, 1): out = w1/(w0+w1).  Each Lean-P weight is within the
    closed-form band (0.917, 1.0607] of 2^(lambda*s) (times a common factor),
    so the odds ratio w1/w0 is within the squared band of the exact one."""
    lo, hi = 2.0 ** (-1.0 / 8.0), 1.5 / math.sqrt(2.0)
    rng = np.random.default_rng(21)
    vals = np.array(sorted(set(oracle_mod.e4m3_decode(np.arange(0x30, 0x58)).tolist())))
    v = codes_of(np.array([0.0, 1.0], np.float32).reshape(1, 2, 1, 1))
    checked = 0
    for _ in range(300):
        qv = rng.choice(vals) * rng.choice([-1, 1])
        kv = rng.choice(vals, size=2) * rng.choice([-1, 1], size=2)
        q = codes_of(np.array([[qv], [qv]], np.float32).reshape(1, 2, 1, 1))
        k = codes_of(kv.astype(np.float32).reshape(1, 2, 1, 1))
        scale = rng.uniform(0.05, 1.5)
        lp, _ = oracle_mod.emul_leanp(q, k, v, 1.0, 1.0, 1.0, scale=scale)
        ref = oracle_mod.ref_fp64(q, k, v, 1.0, 1.0, 1.0, scale=scale)
        o_lp, o_ref = lp[0, 1, 0, 0], ref[0, 1, 0, 0]
        lam_ds = abs(qv * (kv[1] - kv[0])) * scale / LN2
        if lam_ds > 12.0:  # smaller weight would leave the normal code range
            continue
        checked += 1
        odds = (o_lp / (1 - o_lp)) / (o_ref / (1 - o_ref))
        assert lo / hi * (1 - 1e-12) <= odds <= hi / lo * (1 + 1e-12)
    assert checked > 100


def test_leanp_block_scale_keeps_small_blocks(oracle_mod):
    """[ART-MTP] "Per-block scaling and a rounded row sum": each 64-key block gets
    its own power-of-two scale, so a block 20 binades below the row maximum is
    still represented (one shared scale would round all of it to zero)."""
    S = 128
    q = np.ones((1, S, 1, 1), np.float32)
    k = np.empty((1, S, 1, 1), np.float32)
    rng = np.random.default_rng(3)
    vals = np.array([36.0, 40.0, 44.0, 48.0, 52.0, 56.0, 60.0, 64.0])
    k[0, :64, 0, 0] = 64.0 + rng.choice([0.0, -4.0, -8.0], size=64)
    k[0, 64:, 0, 0] = rng.choice(vals[:3], size=64)
    v = np.zeros((1, S, 1, 1), np.float32)
    v[0, 64:, 0, 0] = 1.0
    qc, kc, vc = codes_of(q), codes_of(k), codes_of(v)
    lo, hi = 2.0 ** (-1.0 / 8.0), 1.5 / math.sqrt(2.0)
    for lam in (1.0, 1.1, 0.93):
        lp, _ = oracle_mod.emul_leanp(qc, kc, vc, 1.0, 1.0, 1.0, scale=lam * LN2)
        ref = oracle_mod.ref_fp64(qc, kc, vc, 1.0, 1.0, 1.0, scale=lam * LN2)
        a, b = lp[0, S - 1, 0, 0], ref[0, S - 1, 0, 0]
        assert 1e-9 < b < 1e-5
        assert lo / hi <= a / b <= hi / lo


def test_ablation_underflow_closed_form(oracle_mod):
    """Exact-softmax FP8 ablation: a probability of 2^-12 rounds to zero in e4m3
    (below half the smallest subnormal 2^-9) but still counts in the unrounded
    row sum, so row 1 gives v1 / (1 + 2^-12)."""
    q = codes_of(np.ones((1, 2, 1, 1), np.float32))
    k = codes_of(np.array([0.0, 12.0], np.float32).reshape(1, 2, 1, 1))
    v = codes_of(np.array([3.0, 5.0], np.float32).reshape(1, 2, 1, 1))
    ab, _ = oracle_mod.emul_exact_fp8(q, k, v, 1.0, 1.0, 1.0, scale=LN2)
    assert ab[0, 0, 0, 0] == 3.0
    assert ab[0, 1, 0, 0] == 5.0 / (1.0 + 2.0 ** -12)
    lp, _ = oracle_mod.emul_leanp(q, k, v, 1.0, 1.0, 1.0, scale=LN2)
    ref = oracle_mod.ref_fp64(q, k, v, 1.0, 1.0, 1.0, scale=LN2)
    want = (3.0 * 2.0 ** -12 + 5.0) / (1.0 + 2.0 ** -12)
    assert abs(ref[0, 1, 0, 0] - want) < 1e-14
    # Lean-P is exact here: both logits sit on integer binades in one block
    assert abs(lp[0, 1, 0, 0] - want) < 1e-14


def test_bf16_emulation_rounds_p(oracle_mod):
    """BF16 path: p = 2^(lambda s - m) rounded to bf16 in P.V, unrounded in the sum."""
    one = np.uint16(0x3F80)
    q = np.full((1, 2, 1, 1), one, np.uint16)
    # k1 = 1/3 in bf16 -> p0 = 2^(-k1 * lambda)
    k = np.array([0x0000, 0x3EAB], np.uint16).reshape(1, 2, 1, 1)
    v = np.array([0x3F80, 0x0000], np.uint16).reshape(1, 2, 1, 1)
    out = oracle_mod.emul_bf16(q, k, v, scale=LN2)
    k1 = oracle_mod.bf16_decode(np.array([0x3EAB]))[0]
    p0 = 2.0 ** (-k1)
    want = oracle_mod.bf16_round([p0])[0] / (p0 + 1.0)
    assert abs(out[0, 1, 0, 0] - want) < 1e-15


def test_errors_vs_fp64_on_gaussian(oracle_mod):
    """All three paths stay within the tolerances of the specification on
    the 2-head, S=256, d128 Gaussian workload (Lean-P and ablation <= 3e-2,
    BF16 <= 5e-3 relative RMS against fp64)."""
    c = wl.make_case("fp8_h2_s256_d128")
    ref, lp, ab = _all_paths(oracle_mod, c.q, c.k, c.v, c.dq, c.dk, c.dv)
    assert rel_rms(lp, ref) < 3e-2
    assert rel_rms(ab, ref) < 3e-2
    b = wl.bf16_gaussian_case(1, 2, 2, 256, 128, 128)
    assert rel_rms(oracle_mod.emul_bf16(b.q, b.k, b.v), oracle_mod.ref_fp64_bf16(b.q, b.k, b.v)) < 5e-3


def test_ambiguity_band(oracle_mod):
    """amb is 0 when no rounding decision is within the band (Q = 0 gives exact
    zero logits), and positive when a code boundary is hit exactly."""
    c = wl.fp8_gaussian_case(1, 1, 1, 70, 8, 8, seeds=(1, 2, 3))
    _, amb = oracle_mod.emul_leanp(np.zeros_like(c.q), c.k, c.v, 1.0, c.dk, c.dv)
    assert np.all(amb == 0.0)
    q = codes_of(np.ones((1, 2, 1, 1), np.float32))
    k = codes_of(np.array([2.0, 1.0], np.float32).reshape(1, 2, 1, 1))
    v = codes_of(np.array([0.0, 1.0], np.float32).reshape(1, 2, 1, 1))
    # lambda = 1: u = (16, 8), e = 2, x = (112, 104): both exactly on integers
    _, amb = oracle_mod.emul_leanp(q, k, v, 1.0, 1.0, 1.0, scale=LN2)
    dec = oracle_mod.e4m3_decode
    w = np.array([dec([112])[0], dec([104])[0]])
    want = ((dec([112])[0] - dec([111])[0]) + (dec([104])[0] - dec([103])[0])
            + 0.0) / w.sum()
    assert amb[0, 1, 0] >= want - 1e-15


def test_sink_input_block_scale_beats_ablation(oracle_mod):
    """With an attention sink (key 0 dominating every row by 15-25 nats) the
    exact-softmax FP8 ablation rounds most other probabilities to zero or to
    subnormals, while the per-block power-of-two scale keeps every 64-key
    block at full e4m3 precision ([ART-MTP] "Per-block scaling and a rounded
    row sum"; "How accurate is ZYFA's FP8 attention?" attributes the ablation's
    larger error to such zeros and subnormals).  Lean-P's error against fp64
    must be well below the ablation's."""
    c = wl.fp8_sink_case(1, 2, 2, 1024, 128, 128)
    rng = np.random.default_rng(4)
    rows = np.stack([np.zeros(96, np.int64), rng.integers(0, 2, 96), rng.integers(64, 1024, 96)], 1)
    ref = oracle_mod.ref_fp64(c.q, c.k, c.v, c.dq, c.dk, c.dv, rows=rows)
    lp, _ = oracle_mod.emul_leanp(c.q, c.k, c.v, c.dq, c.dk, c.dv, rows=rows)
    ab, _ = oracle_mod.emul_exact_fp8(c.q, c.k, c.v, c.dq, c.dk, c.dv, rows=rows)
    e_lp, e_ab = rel_rms(lp, ref), rel_rms(ab, ref)
    assert e_lp < 3e-2
    assert e_lp < 0.3 * e_ab, (e_lp, e_ab)


# --- options for flash_attn_func-style calls: non-causal, per-(batch, kv
# head) descales, log-sum-exp ------------------------------------------------

def _dequant(oracle_mod, c, B, Hkv, dq, dk, dv):
    """Dequantised q, k, v with per-(b, kv head) descales (GQA groups share)."""
    Hq = c.q.shape[2]
    grp = Hq // Hkv
    q = oracle_mod.e4m3_decode(c.q) * np.repeat(np.asarray(dq).reshape(B, 1, Hkv, 1), grp, 2)
    k = oracle_mod.e4m3_decode(c.k) * np.asarray(dk).reshape(B, 1, Hkv, 1)
    v = oracle_mod.e4m3_decode(c.v) * np.asarray(dv).reshape(B, 1, Hkv, 1)
    return q, k, v


def _sdpa(q, k, v, causal, scale):
    Hq, Hkv = q.shape[2], k.shape[2]
    kk = torch.from_numpy(np.repeat(k, Hq // Hkv, axis=2)).permute(0, 2, 1, 3)
    vv = torch.from_numpy(np.repeat(v, Hq // Hkv, axis=2)).permute(0, 2, 1, 3)
    qq = torch.from_numpy(q).permute(0, 2, 1, 3)
    out = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=causal, scale=scale)
    s = torch.einsum("bhid,bhjd->bhij", qq, kk) * scale
    if causal:
        S = s.shape[-1]
        s = s.masked_fill(torch.triu(torch.ones(S, S, dtype=torch.bool), 1), float("-inf"))
    return out.permute(0, 2, 1, 3).numpy(), torch.logsumexp(s, -1).numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_reference_options_match_sdpa_and_logsumexp(oracle_mod, causal):
    """Non-causal rows, per-(batch, kv head) descales and the log-sum-exp of the
    fp64 reference against torch's SDPA and logsumexp in fp64."""
    B, Hq, Hkv, S, D = 2, 4, 2, 70, 32
    c = wl.fp8_gaussian_case(B, Hq, Hkv, S, D, D, seeds=(81, 82, 83))
    rng = np.random.default_rng(84)
    dq, dk, dv = (c.dq * rng.uniform(0.5, 2.0, (B, Hkv)), c.dk * rng.uniform(0.5, 2.0, (B, Hkv)),
                  c.dv * rng.uniform(0.5, 2.0, (B, Hkv)))
    scale = 0.21
    out, _, lse = oracle_mod.attention("ref", c.q, c.k, c.v, dq, dk, dv, scale=scale, causal=causal)
    want, want_lse = _sdpa(*_dequant(oracle_mod, c, B, Hkv, dq, dk, dv), causal, scale)
    assert np.max(np.abs(out - want)) < 1e-12
    assert np.max(np.abs(lse - want_lse)) < 1e-12


@pytest.mark.parametrize("path", ["leanp", "exact_fp8"])
@pytest.mark.parametrize("causal", [True, False])
def test_per_bkv_descales_equal_per_slice_calls(oracle_mod, path, causal):
    """Per-(batch, kv head) descales give, slice by slice, what a call on that
    slice with its scalar descales gives."""
    B, Hq, Hkv, S, D = 2, 4, 2, 150, 64
    c = wl.fp8_gaussian_case(B, Hq, Hkv, S, D, D, seeds=(85, 86, 87))
    rng = np.random.default_rng(88)
    dq, dk, dv = (rng.uniform(0.005, 0.02, (B, Hkv)) for _ in range(3))
    out, amb, lse = oracle_mod.attention(path, c.q, c.k, c.v, dq, dk, dv, causal=causal)
    grp = Hq // Hkv
    for b in range(B):
        for g in range(Hkv):
            sl = lambda a, h0, h1: np.ascontiguousarray(a[b:b + 1, :, h0:h1])
            o2, a2, l2 = oracle_mod.attention(
                path, sl(c.q, g * grp, (g + 1) * grp), sl(c.k, g, g + 1), sl(c.v, g, g + 1),
                dq[b, g], dk[b, g], dv[b, g], causal=causal)
            assert np.array_equal(out[b:b + 1, :, g * grp:(g + 1) * grp], o2)
            assert np.array_equal(lse[b:b + 1, g * grp:(g + 1) * grp], l2)


@pytest.mark.parametrize("causal", [True, False])
def test_lse_of_each_path(oracle_mod, causal):
    """Lean-P's log-sum-exp is the log of the rounded row sum, so it lies in
    the closed-form element band (2^(-1/8), 1.0607] of the fp64 one (plus the
    tiny flushed weights); the exact ablation's (unrounded sum) equals it."""
    c = wl.fp8_gaussian_case(1, 2, 2, 333, 128, 128, seeds=(91, 92, 93))
    _, _, ref = oracle_mod.attention("ref", c.q, c.k, c.v, c.dq, c.dk, c.dv, causal=causal)
    _, _, lp = oracle_mod.attention("leanp", c.q, c.k, c.v, c.dq, c.dk, c.dv, causal=causal)
    _, _, ex = oracle_mod.attention("exact_fp8", c.q, c.k, c.v, c.dq, c.dk, c.dv, causal=causal)
    d = lp - ref
    assert d.min() > math.log(2.0 ** (-1.0 / 8.0)) - 1e-6 and d.max() <= math.log(1.0607) + 1e-9
    assert np.max(np.abs(ex - ref)) < 1e-9


def test_noncausal_q_zero_gives_mean_of_all_keys(oracle_mod):
    S = 200
    c = wl.fp8_gaussian_case(1, 2, 2, S, 128, 128, seeds=(94, 95, 96))
    q0 = np.zeros_like(c.q)
    want = (oracle_mod.e4m3_decode(c.v) * c.dv).mean(axis=1, keepdims=True)
    for path in ("ref", "leanp", "exact_fp8"):
        out, _, _ = oracle_mod.attention(path, q0, c.k, c.v, c.dq, c.dk, c.dv, causal=False)
        assert np.max(np.abs(out - want)) < 1e-12, path


def test_bf16_reference_noncausal_matches_sdpa(oracle_mod):
    b = wl.bf16_gaussian_case(1, 2, 2, 90, 64, 64)
    out, _, lse = oracle_mod.attention("ref_bf16", b.q, b.k, b.v, causal=False)
    q, k, v = (oracle_mod.bf16_decode(a) for a in (b.q, b.k, b.v))
    want, want_lse = _sdpa(q, k, v, False, 1.0 / math.sqrt(64))
    assert np.max(np.abs(out - want)) < 1e-12 and np.max(np.abs(lse - want_lse)) < 1e-12


def test_variant_e_isolates_the_code(oracle_mod):
    """Variant E keeps Lean-P's blocks, exponents and rounded row sum but rounds
    the exact weight to nearest e4m3: with V = 1 it is exactly 1 like Lean-P
    (rounded sum), its weights sit within half an e4m3 ulp of the exact ones,
    and where every logit is an integer number of binades (exact codes) it
    equals Lean-P."""
    c = wl.fp8_gaussian_case(1, 2, 2, 200, 128, 128, seeds=(121, 122, 123))
    ones = np.full_like(c.v, 0x38)
    e1, _, _ = oracle_mod.attention("variant_e", c.q, c.k, ones, c.dq, c.dk, 1.0)
    assert np.max(np.abs(e1 - 1.0)) < 1e-12
    _, _, ref = oracle_mod.attention("ref", c.q, c.k, c.v, c.dq, c.dk, c.dv)
    _, _, le = oracle_mod.attention("variant_e", c.q, c.k, c.v, c.dq, c.dk, c.dv)
    assert np.max(np.abs(le - ref)) < math.log(1.0 + 2.0 ** -4)
    # logits on integer binades: q = 1, k in {0, 1, 2, ...}, scale = ln 2
    S = 64
    q = codes_of(np.ones((1, S, 1, 1), np.float32))
    k = codes_of(np.arange(S, dtype=np.float32).reshape(1, S, 1, 1) % 8)
    v = codes_of(np.linspace(-2, 2, S).astype(np.float32).round(0).reshape(1, S, 1, 1))
    a, _, _ = oracle_mod.attention("variant_e", q, k, v, scale=LN2)
    b, _, _ = oracle_mod.attention("leanp", q, k, v, scale=LN2)
    assert np.array_equal(a, b)
