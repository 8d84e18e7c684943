"""The split schedule's completion protocol, modelled on the CPU.

Each piece of a split item writes its partial result to the workspace, fences,
and then arrives on a 64-bit counter per (split item, query tile) with one
atomic read-modify-write (a compare-and-swap loop in the kernel,
``split_arrive``).  The counter holds ``(epoch << 3) + arrivals``, where the
epoch is a per-call number.  A word that carries another epoch counts as zero
arrivals: it may be left over from an earlier call (also one that ran out of
time part-way), or it may be garbage in a workspace that was never cleared.
The piece that sees ``ns - 1`` earlier arrivals is the last one. It adds all
the partial results up and sets the counter back to zero. A CUDA graph replays
a launch with its epoch unchanged, so the replay must find the counter at
zero.

These tests explore random arrival orders over sequences of calls on one
workspace. The sequences include calls that stop before every piece has
arrived, workspaces that start as random 64-bit words, and graph replays. In
every call that completes, exactly one piece must find itself last, and only
after all ns pieces of that call have written. The model also plants two
mistakes, and each must fail the same exploration: a counter without the
epoch, and a last piece that does not reset the counter (which fails on
replays).
"""
import random

import pytest

EPOCH_BITS = 61


def arrive(word: int, epoch: int, ns: int):
    """One arrival: the new word and whether this piece is the last (which
    sets the word back to zero)."""
    if word >> 3 == epoch:
        last = (word & 7) == ns - 1
        return (0 if last else word + 1), last
    return (epoch << 3) + 1, ns == 1


def arrive_without_epoch(word: int, epoch: int, ns: int):
    """Planted mistake: a plain counter, reset by the last piece."""
    last = word == ns - 1
    return (0 if last else word + 1), last


def run_calls(seed, arrive_fn, n_calls=40, n_items=6, garbage=True, replays=False):
    """A sequence of calls on one workspace.  With ``replays``, a call that
    follows a completed call may repeat it with the same epoch and pieces, as
    a CUDA graph replays its launch with the same parameters."""
    rng = random.Random(seed)
    counters = [rng.getrandbits(64) if garbage else 0 for _ in range(n_items * 2)]
    epoch = rng.getrandbits(58)
    ns = 2
    aborted = True
    for call in range(n_calls):
        if not (replays and not aborted and rng.random() < 0.5):
            epoch = (epoch + 1) & ((1 << EPOCH_BITS) - 1)
            ns = rng.choice([2, 3, 4])
        aborted = rng.random() < 0.2
        # events: (piece writes, piece arrives) per (item, tile, piece); a
        # piece arrives only after it has written
        pending = [(i, s) for i in range(n_items * 2) for s in range(ns)]
        rng.shuffle(pending)
        if aborted:  # the call runs out of time: some pieces never arrive
            pending = pending[:rng.randrange(len(pending))]
        written = {}
        lasts = {}
        for slot, s in pending:
            written.setdefault(slot, set()).add(s)
            counters[slot], last = arrive_fn(counters[slot], epoch, ns)
            if last:
                if slot in lasts:
                    return f"call {call}: two pieces of slot {slot} found themselves last"
                if written[slot] != set(range(ns)):
                    return f"call {call}: slot {slot} combined before every piece had written"
                lasts[slot] = s
        if not aborted and len(lasts) != n_items * 2:
            return f"call {call}: {n_items * 2 - len(lasts)} slots never combined"
    return None


def arrive_without_reset(word: int, epoch: int, ns: int):
    """Planted mistake: the last piece leaves its count in the word."""
    if word >> 3 == epoch:
        return word + 1, (word & 7) == ns - 1
    return (epoch << 3) + 1, ns == 1


@pytest.mark.parametrize("replays", [False, True])
@pytest.mark.parametrize("garbage", [False, True])
def test_exactly_one_last_piece_per_call(garbage, replays):
    for seed in range(300):
        assert run_calls(seed, arrive, garbage=garbage, replays=replays) is None, seed


def test_graph_replays_need_the_reset():
    """Without the reset, a replay with the same epoch counts the previous
    launch's arrivals and no piece finds itself last."""
    found = [run_calls(seed, arrive_without_reset, replays=True) for seed in range(100)]
    assert any(f is not None and "never combined" in f for f in found)


def test_counter_without_epoch_fails_after_an_aborted_call_or_on_garbage():
    found = [run_calls(seed, arrive_without_epoch, garbage=g) for seed in range(100)
             for g in (False, True)]
    assert any(f is not None for f in found)

