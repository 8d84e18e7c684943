"""Race detection for the kernel's synchronisation (CPU): the mbarrier protocol
of attn_fwd.cuh, modelled in ``sync_model`` and explored under random
schedules with random per-role speeds.

- The protocols the kernel ships show no aliased wait, no deadlock and no data
  race: FP8 unordered with 4 and 3 ring stages, and BF16 ordered with 2
  stages and four ``qk_go`` barriers per tile; so do the variants that were
  built, measured and not kept (two Q buffers, P in halves at head dim 128,
  tile 0's epilogue held back until tile 1's last P).
- Mistakes planted in the model are found: two ``qk_go`` barriers per tile
  alias (a first GPU build of that variant ended some launches on the bounded
  wait's timeout), and dropping the S-drain, P.V-done or Q-empty wait is an
  overwrite.
- The failure path: with one bounded wait running out of time at a random
  moment, every role leaves and the CTA exits with no TMA load, MMA or commit
  arrival in flight; without the producer's or an issuing warp's drain it
  does not.
"""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(__file__))
import sync_model as sm  # noqa: E402

SEEDS = range(400)


@pytest.mark.parametrize("proto", [
    sm.Protocol(stages=4, q_bufs=1),                     # FP8, Dqk 128
    sm.Protocol(stages=3, q_bufs=1),                     # FP8, Dqk 192
    sm.Protocol(stages=2, q_bufs=1, order_pv=True, qk_go=4),  # BF16
    sm.Protocol(stages=4, q_bufs=2),                     # FP8 with two Q buffers
    sm.Protocol(stages=4, p_halves=True),                # FP8, P in two halves
    sm.Protocol(stages=3, p_halves=True),                # FP8 Dqk 192, P in two halves
    sm.Protocol(stages=4, order_pv=True, qk_go=4),       # the order with a deeper ring
    sm.Protocol(stages=4, order_pv=True, qk_go=4, split_pv=True),
    sm.Protocol(stages=4, q_bufs=1, epi_after_p1=True),  # tile 0's epilogue after P1 (not kept)
], ids=["fp8", "fp8_mla", "bf16", "fp8_two_q", "fp8_halves", "fp8_mla_halves",
        "ordered_4stages", "ordered_split", "fp8_epi_after_p1"])
def test_kernel_protocols_have_no_race_or_aliasing(proto):
    assert sm.check(proto, SEEDS) is None


@pytest.mark.parametrize("split", [False, True])
def test_two_ordering_barriers_per_tile_alias(split):
    found = sm.check(sm.Protocol(stages=2, order_pv=True, qk_go=2, split_pv=split), SEEDS)
    assert found is not None and "parity wait cannot tell" in found[2], found


def test_three_ordering_barriers_suffice():
    # the bound in the kernel's argument: S_t(n+3) already needs the P.V product
    # that consumes arrival n; the kernel takes four, a power of two
    assert sm.check(sm.Protocol(stages=2, order_pv=True, qk_go=3), SEEDS) is None


def test_epilogue_wait_on_the_p_barrier_aliases():
    # softmax 0 may reach its epilogue while tile 1 has two more P writes to
    # go, so a parity wait on p_full1 for the last one is ambiguous; the
    # variant as built waited on p1_last, one phase per item
    found = sm.check(sm.Protocol(epi_after_p1=True, epi_wait_on_p_full1=True), SEEDS)
    assert found is not None and "parity wait cannot tell" in found[2], found


def test_missing_drain_wait_is_an_overwrite_of_s():
    found = sm.check(sm.Protocol(skip_drain_wait=True), SEEDS)
    assert found is not None and "before it was copied out" in found[2], found


def test_missing_q_empty_wait_is_an_overwrite_of_q():
    # the producer reloading a Q buffer before the S products of its previous
    # item have run
    found = sm.check(sm.Protocol(q_bufs=2, skip_q_empty_wait=True), SEEDS)
    assert found is not None and "Q buffer" in found[2], found


@pytest.mark.parametrize("halves", [False, True])
def test_missing_pv_done_wait_is_an_overwrite_of_p(halves):
    # without halves the overwrite of P shows first; with them the epilogue's
    # wait on o_done can run two phases behind first
    found = sm.check(sm.Protocol(skip_o_done_wait=True, p_halves=halves), SEEDS)
    assert found is not None and ("before its P.V ran" in found[2]
                                  or "phase" in found[2] and "o_done" in found[2]), found


def test_model_reports_a_deadlock():
    # one arrival too few on a barrier every role depends on: the model must
    # stop with a deadlock, not spin
    import random
    items = [(1, 2), (2, 2)]
    m = sm.Model(items, sm.Protocol(), random.Random(0))
    m.bars["q_full0"].count = 2
    m.bars["q_full0"].pending = 2
    with pytest.raises(sm.Violation, match="deadlock"):
        m.run()


@pytest.mark.parametrize("proto", [
    sm.Protocol(stages=4, q_bufs=1, inject_timeout=True),
    sm.Protocol(stages=4, q_bufs=1, epi_after_p1=True, inject_timeout=True),
    sm.Protocol(stages=4, q_bufs=2, inject_timeout=True),
    sm.Protocol(stages=4, p_halves=True, inject_timeout=True),
    sm.Protocol(stages=3, q_bufs=1, inject_timeout=True),
    sm.Protocol(stages=2, q_bufs=1, order_pv=True, inject_timeout=True),
], ids=["fp8", "fp8_epi_after_p1", "fp8_two_q", "fp8_halves", "fp8_mla", "bf16"])
def test_a_timed_out_wait_leaves_nothing_in_flight(proto):
    assert sm.check(proto, range(600)) is None


def test_producer_without_drain_can_exit_with_loads_in_flight():
    found = sm.check(sm.Protocol(inject_timeout=True, skip_producer_drain=True), range(600))
    assert found is not None and "TMA loads in flight" in found[2], found


def test_issuing_warps_without_drain_exit_with_mmas_in_flight():
    found = sm.check(sm.Protocol(inject_timeout=True, skip_mma_drain=True), range(600))
    assert found is not None and ("MMAs in flight" in found[2]
                                  or "commit arrivals pending" in found[2]), found
