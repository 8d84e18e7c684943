"""GPU parity of the split schedule (attn_fwd_full with a workspace).

Problems with too few work items to keep every SM busy (few heads, short
sequences) split their longest items along the keys into pieces that run on
different SMs; the piece that finishes last adds the pieces' partial results
(O and the rounded row sum, relative to each piece's power-of-two reference)
and writes the output.  Lean-P's codes and block scales depend on each 64-key
block alone ("Zyphra ZYFA: FP8 FlashAttention for AMD MI355X", "Lean P: one
multiply-add instead of an exponential" and "Per-block scaling and a rounded
row sum"), so a split changes only the order of the fp32 sums.

Checks, on shapes the schedule splits (asserted through workspace_size):
- sampled rows against the oracle's emulation of the same path, with the
  usual per-row gate, and the log-sum-exp;
- the whole output and LSE against the same call without splitting, within
  fp32 reassociation;
- the same bits on every call, with fresh workspaces and with a workspace
  filled with garbage (its counters need no clearing), and for two problems
  that alternate on one workspace;
- bf16 output equal to the fp32 output rounded, and no write outside the
  output;
- a captured call replayed from a CUDA graph, and a stalled call (every
  bounded wait expires) followed by a correct one.
The schedule checks run on Lean-P and on BF16, whose split differs from whole
items by the bf16 rounding of each piece's probabilities (its own test below
bounds that against whole items, fp64 and the emulation).
"""
import numpy as np
import pytest
import torch

import fp8_causal_prefill_flash_gb300 as fa
import oracle
from fp8_causal_prefill_flash_gb300 import workloads as wl

from gpu_helpers import check_rows

pytestmark = pytest.mark.gpu

PATH = {fa.ATTN_VARIANT_LEANP: "leanp", fa.ATTN_VARIANT_BLOCK_EXACT: "variant_e"}

# (B, Hq, Hkv, S, Dqk, causal, per-(batch, kv head) descales)
SHAPES = {
    "h8_s2048": (1, 8, 8, 2048, 128, True, False),
    "gqa_b2_ragged": (2, 4, 2, 2000, 128, True, False),
    "noncausal_h4": (1, 4, 4, 2000, 128, False, False),
    "mla_h4": (1, 4, 4, 2048, 192, True, False),
    "h2_s4096": (1, 2, 2, 4096, 128, True, False),
    "per_bkv_b2": (2, 4, 2, 2048, 128, True, True),
    "h1_s32k": (1, 1, 1, 32768, 128, True, False),  # pieces of about 128 key tiles
    "mla_noncausal_ragged": (1, 2, 2, 3000, 192, False, False),  # every item split, ragged S
}


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


def make(name, seed):
    B, Hq, Hkv, S, Dqk, causal, per_bkv = SHAPES[name]
    case = wl.fp8_gaussian_case(B, Hq, Hkv, S, Dqk, 128, seeds=(seed, seed + 1, seed + 2))
    if per_bkv:
        rng = np.random.default_rng(seed + 3)
        dq, dk, dv = (case.dq * rng.uniform(0.5, 2.0, (B, Hkv)) for _ in range(3))
    else:
        dq, dk, dv = case.dq, case.dk, case.dv
    q, k, v = (torch.from_numpy(a).cuda() for a in (case.q, case.k, case.v))
    d = [torch.from_numpy(np.asarray(x, np.float32).reshape(-1).copy()).cuda() for x in (dq, dk, dv)]
    return case, (q, k, v, *d), (dq, dk, dv), causal


def make_for(variant, name, seed):
    """make() for Lean-P; for BF16 the same shape (head dim 128) with bf16
    Gaussian inputs and no descales."""
    if variant != fa.ATTN_VARIANT_BF16:
        return make(name, seed)
    B, Hq, Hkv, S, Dqk, causal, _ = SHAPES[name]
    assert Dqk == 128
    case = wl.bf16_gaussian_case(B, Hq, Hkv, S, 128, 128, seeds=(seed, seed + 1, seed + 2))
    q, k, v = (torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
               for a in (case.q, case.k, case.v))
    return case, (q, k, v, None, None, None), (None, None, None), causal


# the variants whose split is exercised by the schedule tests below
SCHED_VARIANTS = pytest.mark.parametrize("variant", [fa.ATTN_VARIANT_LEANP, fa.ATTN_VARIANT_BF16],
                                         ids=["leanp", "bf16"])


def call(variant, args, causal, split=True, out_dtype=fa.ATTN_OUT_F32, workspace=None,
         status=None):
    out, lse = fa.attn_fwd_full(variant, *args, out_dtype=out_dtype, causal=causal,
                                return_lse=True, split=split, workspace=workspace,
                                dev_status=status)
    return out, lse


def sample_rows(B, Hq, S, seed, n=700):
    rng = np.random.default_rng(seed)
    edge = [0, 1, 127, 128, 255, 256, S // 2, S - 2, S - 1]
    rows = [(b, h, i) for b in range(B) for h in range(min(Hq, 2)) for i in edge if 0 <= i < S]
    rows += list(zip(rng.integers(0, B, n), rng.integers(0, Hq, n), rng.integers(0, S, n)))
    return np.asarray(rows, dtype=np.int64)


@pytest.mark.parametrize("variant", [fa.ATTN_VARIANT_LEANP, fa.ATTN_VARIANT_BLOCK_EXACT])
@pytest.mark.parametrize("name", list(SHAPES))
def test_split_matches_the_oracle_and_the_whole_items(name, variant):
    case, args, (dq, dk, dv), causal = make(name, 500)
    B, Hq, Hkv, S, Dqk, Dv = case.shape
    need = fa.workspace_size(variant, B, Hq, Hkv, S, Dqk, Dv, causal)
    assert need > 0, "the schedule should split this problem"
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = call(variant, args, causal, status=status)
    plain, plain_lse = call(variant, args, causal, split=False)
    torch.cuda.synchronize()
    assert int(status.item()) == fa.ATTN_OK, fa.status_string(int(status.item()))

    # the whole output: only the order of the fp32 sums differs
    scale = float(plain.abs().max())
    assert float((out - plain).abs().max()) <= 2e-6 * scale + 1e-30
    assert float((lse - plain_lse).abs().max()) <= 2e-6 * (1.0 + float(plain_lse.abs().max()))

    # sampled rows against the emulation of the same path
    rows = sample_rows(B, Hq, S, 501)
    want, amb, want_lse = oracle.attention(PATH[variant], case.q, case.k, case.v, dq, dk, dv,
                                           rows=rows, causal=causal)
    gpu = out.cpu().numpy().astype(np.float64)
    got = np.stack([gpu[b, i, h] for b, h, i in rows])
    vmax = float(np.max(np.abs(oracle.e4m3_decode(case.v)))) * float(np.max(dv))
    check_rows(got, want, amb, vmax)
    glse = lse.cpu().numpy().astype(np.float64)
    got_lse = np.array([glse[b, h, i] for b, h, i in rows])
    a = np.minimum(amb, 0.5)
    assert np.all(np.abs(got_lse - want_lse) <= 2e-5 * (1 + np.abs(want_lse)) + 2.0 * a / (1.0 - a))


@SCHED_VARIANTS
@pytest.mark.parametrize("name", ["h8_s2048", "gqa_b2_ragged", "mla_h4"])
def test_split_is_deterministic_with_any_workspace(name, variant):
    if variant == fa.ATTN_VARIANT_BF16 and SHAPES[name][4] != 128:
        pytest.skip("the BF16 path has head dim 128 only")
    case, args, _, causal = make_for(variant, name, 520)
    B, Hq, Hkv, S, Dqk, Dv = case.shape
    need = fa.workspace_size(variant, B, Hq, Hkv, S, Dqk, Dv, causal)
    assert need > 0
    first = call(variant, args, causal)
    outs = [call(variant, args, causal) for _ in range(3)]  # fresh workspaces
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    outs.append(call(variant, args, causal, workspace=ws))
    ws.random_(0, 256)
    outs.append(call(variant, args, causal, workspace=ws))
    outs.append(call(variant, args, causal, workspace=ws))  # counters left by the call before
    torch.cuda.synchronize()
    for o, l in outs:
        assert torch.equal(o, first[0]) and torch.equal(l, first[1])


@SCHED_VARIANTS
def test_two_problems_alternate_on_one_workspace(variant):
    case_a, args_a, _, causal_a = make_for(variant, "h8_s2048", 540)
    case_b, args_b, _, causal_b = make_for(variant, "h2_s4096", 550)
    need = max(fa.workspace_size(variant, *c.shape, causal) for c, causal in
               ((case_a, causal_a), (case_b, causal_b)))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    want_a = call(variant, args_a, causal_a)
    want_b = call(variant, args_b, causal_b)
    got = []
    for _ in range(3):
        got.append(call(variant, args_a, causal_a, workspace=ws))
        got.append(call(variant, args_b, causal_b, workspace=ws))
    torch.cuda.synchronize()
    for i, (o, l) in enumerate(got):
        want = want_a if i % 2 == 0 else want_b
        assert torch.equal(o, want[0]) and torch.equal(l, want[1]), i


@SCHED_VARIANTS
@pytest.mark.parametrize("name", ["h8_s2048", "gqa_b2_ragged", "noncausal_h4"])
def test_split_bf16_output_is_the_fp32_output_rounded(name, variant):
    """The last piece writes bf16 through the same shared-memory slot and
    TMA stores as a whole item (direct stores for BF16); the values are the
    fp32 output rounded."""
    case, args, _, causal = make_for(variant, name, 560)
    assert fa.workspace_size(variant, *case.shape, causal) > 0
    f32, _ = call(variant, args, causal)
    b16, _ = call(variant, args, causal, out_dtype=fa.ATTN_OUT_BF16)
    torch.cuda.synchronize()
    assert torch.equal(b16, f32.to(torch.bfloat16))


@SCHED_VARIANTS
@pytest.mark.parametrize("out_dtype", [fa.ATTN_OUT_F32, fa.ATTN_OUT_BF16])
def test_split_writes_every_output_element_and_nothing_else(out_dtype, variant):
    case, args, _, causal = make_for(variant, "gqa_b2_ragged", 580)
    B, Hq, Hkv, S, Dqk, Dv = case.shape
    assert fa.workspace_size(variant, *case.shape, causal) > 0
    esz = 4 if out_dtype == fa.ATTN_OUT_F32 else 2
    n_out = B * S * Hq * Dv * esz
    pad = 4096
    raw = torch.full((pad + n_out + pad,), 0xA5, dtype=torch.uint8, device="cuda")
    dt = torch.float32 if out_dtype == fa.ATTN_OUT_F32 else torch.bfloat16
    out = raw[pad:pad + n_out].view(dt).view(B, S, Hq, Dv)
    fa.attn_fwd_full(variant, *args, out=out, out_dtype=out_dtype, causal=causal)
    torch.cuda.synchronize()
    h = raw.cpu().numpy()
    assert np.all(h[:pad] == 0xA5) and np.all(h[-pad:] == 0xA5)
    words = h[pad:pad + n_out].view(np.uint32 if esz == 4 else np.uint16)
    assert not np.any(words == (0xA5A5A5A5 if esz == 4 else 0xA5A5))


@SCHED_VARIANTS
def test_split_call_replays_from_a_cuda_graph(variant):
    """A captured call replays with the same parameters, its per-call tag
    included; the last piece resets the counters, so every replay combines
    its own pieces.  New inputs are copied in between replays."""
    case_a, args_a, _, causal = make_for(variant, "h8_s2048", 590)
    case_b, args_b, _, _ = make_for(variant, "h8_s2048", 595)
    q, k, v, dq, dk, dv = (None if t is None else t.clone() for t in args_a)
    out = torch.empty((1, 2048, 8, 128), dtype=torch.bfloat16, device="cuda")
    need = fa.workspace_size(variant, 1, 8, 8, 2048, 128, 128, causal)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    run = lambda: fa.attn_fwd_full(variant, q, k, v, dq, dk, dv, out=out, causal=causal,
                                   workspace=ws)
    run()  # eager warm-up: library loaded, plan cached
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for src in (args_b, args_a, args_b):
        for dst, x in zip((q, k, v, dq, dk, dv), src):
            if dst is not None:
                dst.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        want = fa.attn_fwd_full(variant, *src, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(out, want)


@SCHED_VARIANTS
def test_split_kernel_reports_a_stall_and_the_next_call_is_correct(variant):
    """Test hook: the load warp issues nothing, every bounded wait of the split
    kernel expires (0.2 s) and the status word reads ATTN_ERR_TIMEOUT; the next
    call on the same workspace is correct (no piece arrived, so no counter
    moved, and the next call's tag differs anyway): the same bits as a call
    on a fresh workspace, and close to whole items."""
    case, args, _, causal = make_for(variant, "h8_s2048", 600)
    need = fa.workspace_size(variant, *case.shape, causal)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fa.attn_fwd_full(variant, *args, causal=causal, flags=fa.ATTN_FLAG_TEST_STALL_LOADS,
                     dev_status=status, workspace=ws)
    torch.cuda.synchronize()
    assert int(status.item()) == fa.ATTN_ERR_TIMEOUT
    status.zero_()
    out, _ = call(variant, args, causal, workspace=ws, status=status)
    fresh, _ = call(variant, args, causal)
    plain, _ = call(variant, args, causal, split=False)
    torch.cuda.synchronize()
    assert int(status.item()) == fa.ATTN_OK
    assert torch.equal(out, fresh)
    # fp32 reassociation for Lean-P; bf16 rounding of the probabilities per
    # piece for BF16 (the bound of the BF16 split test)
    tol = 2e-6 if variant == fa.ATTN_VARIANT_LEANP else 4e-3
    assert float((out - plain).abs().max()) <= tol * float(plain.abs().max())


# BF16 (exact softmax): each piece rounds its probabilities to bf16 relative
# to its own running maximum, and the last piece rescales the pieces by exp2
# of their maxima's differences, so a split result differs from whole items
# by that rounding.  Where every probability is rounded differently on the
# two sides, the difference is two independent round-to-nearest errors of
# relative size up to 2^-9 each, weighted like the output itself: for values
# that average out (the non-causal rows over 2000 keys) its RMS relative to
# the output's RMS is about sqrt(2/3) * 2^-9 = 1.6e-3.  The test allows twice
# one rounding step, 2^-8, and the gate against fp64 (5e-3) still applies.
BF16_SHAPES = {
    "h8_s2048": (1, 8, 8, 2048, True),
    "gqa_b2_ragged": (2, 4, 2, 2000, True),
    "noncausal_h4": (1, 4, 4, 2000, False),
    "h2_s4096": (1, 2, 2, 4096, True),
}


@pytest.mark.parametrize("name", list(BF16_SHAPES))
def test_bf16_split_against_fp64_and_whole_items(name):
    B, Hq, Hkv, S, causal = BF16_SHAPES[name]
    case = wl.bf16_gaussian_case(B, Hq, Hkv, S, 128, 128, seeds=(700, 701, 702))
    q, k, v = (torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
               for a in (case.q, case.k, case.v))
    variant = fa.ATTN_VARIANT_BF16
    assert fa.workspace_size(variant, B, Hq, Hkv, S, 128, 128, causal) > 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = fa.attn_fwd_full(variant, q, k, v, out_dtype=fa.ATTN_OUT_F32, causal=causal,
                                return_lse=True, dev_status=status)
    plain, plain_lse = fa.attn_fwd_full(variant, q, k, v, out_dtype=fa.ATTN_OUT_F32,
                                        causal=causal, return_lse=True, split=False)
    again = fa.attn_fwd_full(variant, q, k, v, out_dtype=fa.ATTN_OUT_F32, causal=causal)
    torch.cuda.synchronize()
    assert int(status.item()) == fa.ATTN_OK
    assert torch.equal(out, again)  # the same bits on every call
    scale = float(plain.abs().max())
    diff = (out - plain).double()
    assert float(diff.abs().max()) <= 4e-3 * scale
    assert float(diff.pow(2).mean().sqrt()) <= 2.0 ** -8 * float(plain.double().pow(2).mean().sqrt())
    assert float((lse - plain_lse).abs().max()) <= 1e-3 * (1.0 + float(plain_lse.abs().max()))
    rows = sample_rows(B, Hq, S, 703, n=500)
    ref, _, ref_lse = oracle.attention("ref_bf16", case.q, case.k, case.v, rows=rows,
                                       causal=causal)
    gpu = out.cpu().numpy().astype(np.float64)
    got = np.stack([gpu[b, i, h] for b, h, i in rows])
    rel = float(np.sqrt(np.mean((got - ref) ** 2)) / np.sqrt(np.mean(ref ** 2)))
    assert rel <= 5e-3, rel
    emul, _, _ = oracle.attention("bf16", case.q, case.k, case.v, rows=rows, causal=causal)
    vmax = float(np.max(np.abs(oracle.bf16_decode(case.v))))
    check_rows(got, emul, np.zeros(len(rows)), vmax)


@pytest.mark.parametrize("variant", [fa.ATTN_VARIANT_LEANP, fa.ATTN_VARIANT_BF16], ids=["leanp", "bf16"])
def test_planner_declines_one_thousand_keys(variant):
    """At 1K keys every forced plan measured slower than whole items on GB300
    (1, 4, 8 and 16 heads, causal and not), so the plan model, with the fitted
    costs of each path, must choose no split there; at 2K keys and few heads
    it must split."""
    for H, causal in ((1, True), (4, True), (16, True), (8, False)):
        assert fa.workspace_size(variant, 1, H, H, 1024, 128, 128, causal) == 0, (H, causal)
    for H in (1, 2, 4):
        assert fa.workspace_size(variant, 1, H, H, 2048, 128, 128, True) > 0, H


@SCHED_VARIANTS
def test_split_calls_on_two_streams_with_their_own_workspaces(variant):
    """Calls on different streams may run at the same time, each with its own
    workspace: every result equals the same call made alone."""
    case_a, args_a, _, causal_a = make_for(variant, "h8_s2048", 610)
    case_b, args_b, _, causal_b = make_for(variant, "h2_s4096", 615)
    want_a = call(variant, args_a, causal_a)
    want_b = call(variant, args_b, causal_b)
    torch.cuda.synchronize()
    ws = [torch.empty(fa.workspace_size(variant, *c.shape, ca), dtype=torch.uint8, device="cuda")
          for c, ca in ((case_a, causal_a), (case_b, causal_b))]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    got = []
    for _ in range(3):
        for s, w, args, ca in zip(streams, ws, (args_a, args_b), (causal_a, causal_b)):
            with torch.cuda.stream(s):
                got.append(call(variant, args, ca, workspace=w))
    torch.cuda.synchronize()
    for i, (o, l) in enumerate(got):
        want = want_a if i % 2 == 0 else want_b
        assert torch.equal(o, want[0]) and torch.equal(l, want[1]), i
