"""The split schedule's choices, through attn_split_plan (host only, no GPU).

attn_fwd_full splits the longest work items along the keys when a problem
has too few items to keep every SM busy.  The plan comes from a model of the
kernel's time (per key tile, per unit, per piece) fitted to GB300 timings,
with a minimum predicted gain per path.  These tests pin:
- the decisions measured on GB300: no split at 1K keys, where every forced
  plan was slower than whole items; the plan of the bench's few-heads leg;
  the per-path thresholds (FP8 needs a larger predicted gain than BF16);
- the schedule's invariants: workspace size, pieces of at least two key
  tiles, the 128 MiB limit, variants that never split;
- the C search against a plain restatement of the model in Python.
"""
import ctypes

import pytest

import fp8_causal_prefill_flash_gb300 as fa

SMS = 152  # GB300
LEANP, BEXACT, BF16 = fa.ATTN_VARIANT_LEANP, fa.ATTN_VARIANT_BLOCK_EXACT, fa.ATTN_VARIANT_BF16
SLOT_FLOATS = 128 * 128 + 2 * 128  # one partial result: O (128 x 128), l and ref per row
LIMIT = 128 << 20


def plan(variant, B, Hq, Hkv, S, causal=True, sms=SMS, Dqk=128, flags=0):
    return fa.split_plan(variant, B, Hq, Hkv, S, Dqk, 128, causal, sms, flags)


# ------------------------------------------------------------------ the model
# (step, unit, piece0, piece_ns in ns; minimum predicted gain in percent)
COSTS = {LEANP: (950, 5000, 3000, 1000, 15), BEXACT: (950, 5000, 3000, 1000, 15),
         BF16: (1580, 6640, 5360, 1300, 8)}


def ws_bytes(n_split, ns):
    return (n_split * 16 + 255) // 256 * 256 + n_split * ns * 2 * SLOT_FLOATS * 4


def makespan(units_bh, nq, nkvt, causal, sq, ns, grid, c):
    """Busiest CTA under the kernel's alternating round-robin order: the
    pieces of the split items first, then the other items, longest first."""
    step, unit, piece0, piece_ns, _ = c
    load = [0] * grid
    pos = 0

    def place(cost):
        nonlocal pos
        rnd, k = divmod(pos, grid)
        load[grid - 1 - k if rnd & 1 else k] += cost + unit
        pos += 1

    def nkv(qb):
        return 2 * qb + 2 if causal and 2 * qb + 2 < nkvt else nkvt

    if ns > 1:
        for qb in range(nq - 1, sq - 1, -1):
            n = nkv(qb)
            for _ in range(units_bh):
                for s in range(ns):
                    place(((s + 1) * n // ns - s * n // ns) * step + piece0 + piece_ns * ns)
    for qb in range((sq if ns > 1 else nq) - 1, -1, -1):
        for _ in range(units_bh):
            place(nkv(qb) * step)
    return max(load)


def model_plan(variant, B, Hq, S, causal, sms=SMS):
    c = COSTS[variant]
    units_bh, nq, nkvt = B * Hq, (S + 255) // 256, (S + 127) // 128
    n_items = units_bh * nq
    if n_items >= 4 * sms:
        return 0, 1, 0
    base = makespan(units_bh, nq, nkvt, causal, 0, 1, min(n_items, sms), c)
    best_t, best = base, (0, 1, 0)
    for ns in (2, 3, 4):
        for sq in range(nq - 1, -1, -1):
            nmin = 2 * sq + 2 if causal and 2 * sq + 2 < nkvt else nkvt
            if nmin < 2 * ns:
                break
            n_split = units_bh * (nq - sq)
            b = ws_bytes(n_split, ns)
            if b > LIMIT:
                break
            t = makespan(units_bh, nq, nkvt, causal, sq, ns,
                         min(n_items + n_split * (ns - 1), sms), c)
            if t < best_t:
                best_t, best = t, (sq, ns, b)
    if best[1] > 1 and best_t * (100 + c[4]) > base * 100:
        return 0, 1, 0
    return best


# ------------------------------------------------------------------ tests
@pytest.mark.parametrize("variant", [LEANP, BEXACT, BF16])
def test_no_split_at_one_thousand_keys(variant):
    for H in (1, 4, 8, 16):
        for causal in (True, False):
            assert plan(variant, 1, H, H, 1024, causal) == (0, 1, 0), (H, causal)


@pytest.mark.parametrize("variant", [LEANP, BF16])
def test_the_few_heads_bench_leg_splits_its_last_query_blocks_in_two(variant):
    # 4 heads at 8K keys: 128 items for 152 SMs; the bench line reports this
    # workspace (13,845,504 bytes) for both paths
    assert plan(variant, 1, 4, 4, 8192) == (19, 2, 13845504)


def test_the_thresholds_differ_by_path():
    # predicted gains 1.15 (FP8) and 1.17 (BF16): below FP8's 15%, above BF16's 8%
    assert plan(LEANP, 1, 8, 8, 2048, causal=False) == (0, 1, 0)
    assert plan(BF16, 1, 8, 8, 2048, causal=False)[1] > 1
    # 2 x 8/2 heads at 1500 keys: 1.11 (FP8), 1.15 (BF16)
    assert plan(LEANP, 2, 8, 2, 1500) == (0, 1, 0)
    assert plan(BF16, 2, 8, 2, 1500)[1] > 1


@pytest.mark.parametrize("variant", [fa.ATTN_VARIANT_EXACT_FP8, fa.ATTN_VARIANT_LEANP_A3])
def test_variants_rounded_against_the_running_maximum_never_split(variant):
    for S in (2048, 4096, 8192):
        assert plan(variant, 1, 2, 2, S) == (0, 1, 0)


def test_enough_items_or_the_chunked_order_run_whole_items():
    assert plan(LEANP, 1, 32, 32, 32768) == (0, 1, 0)   # 4096 items
    assert plan(LEANP, 1, 4, 4, 8192, flags=fa.ATTN_FLAG_TEST_CHUNK_UNITS) == (0, 1, 0)
    # the same problem on 16 SMs has 8 items per SM: nothing to gain
    assert plan(LEANP, 1, 4, 4, 8192, sms=16) == (0, 1, 0)


SHAPES = [(B, H, Hkv, S, causal)
          for B, H, Hkv in ((1, 1, 1), (1, 2, 2), (1, 4, 4), (1, 8, 8), (1, 8, 2), (2, 4, 2),
                            (1, 12, 12), (1, 16, 4))
          for S in (1000, 2048, 3000, 4096, 8192, 16384)
          for causal in (True, False)]


@pytest.mark.parametrize("variant", [LEANP, BF16])
def test_every_plan_keeps_the_schedule_invariants(variant):
    split = 0
    for B, H, Hkv, S, causal in SHAPES:
        sq, ns, nbytes = plan(variant, B, H, Hkv, S, causal)
        if ns == 1:
            assert (sq, nbytes) == (0, 0)
            continue
        split += 1
        nq, nkvt = (S + 255) // 256, (S + 127) // 128
        assert 2 <= ns <= 4 and 0 <= sq < nq
        n_split = B * H * (nq - sq)
        assert nbytes == ws_bytes(n_split, ns) <= LIMIT
        # every piece of every split item gets at least two key tiles
        n_min = min(2 * sq + 2, nkvt) if causal else nkvt
        assert n_min >= 2 * ns, (B, H, S, causal, sq, ns)
        assert B * H * nq < 4 * SMS
    assert split >= 20


@pytest.mark.parametrize("variant", [LEANP, BEXACT, BF16])
def test_the_search_matches_a_restatement_of_the_model(variant):
    for B, H, Hkv, S, causal in SHAPES:
        assert plan(variant, B, H, Hkv, S, causal) == model_plan(variant, B, H, S, causal), \
            (B, H, Hkv, S, causal)
    for sms in (16, 64, 148, 152):
        assert plan(variant, 1, 4, 4, 8192, sms=sms) == model_plan(variant, 1, 4, 8192, True, sms)


def test_invalid_arguments_are_rejected():
    lib = fa.load_library()
    qb, ns, n = ctypes.c_int(7), ctypes.c_int(7), ctypes.c_size_t(7)
    args = (LEANP, 1, 4, 4, 8192, 128, 128, 1, 0)
    assert lib.attn_split_plan(*args, 0, ctypes.byref(qb), ctypes.byref(ns),
                               ctypes.byref(n)) == fa.ATTN_ERR_INVALID_ARG
    assert (qb.value, ns.value, n.value) == (0, 1, 0)
    assert lib.attn_split_plan(*args, SMS, None, ctypes.byref(ns),
                               ctypes.byref(n)) == fa.ATTN_ERR_INVALID_ARG
    bad = (LEANP, 1, 6, 4, 8192, 128, 128, 1, 0)  # Hq not a multiple of Hkv
    assert lib.attn_split_plan(*bad, SMS, ctypes.byref(qb), ctypes.byref(ns),
                               ctypes.byref(n)) == fa.ATTN_ERR_INVALID_ARG
    with pytest.raises(Exception):
        plan(99, 1, 4, 4, 8192)
