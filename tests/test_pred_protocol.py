"""Model check of the named-barrier protocol of the predicate compaction
(csrc/compact_pred.cu, k_compact_pred): 16 compute warps (one 512-thread
party) and one look-back warp (32 threads) hand each tile over on barrier
kBarAgg + parity and its offsets back on kBarPre + parity, both counting
544 threads.  Hardware barriers have no timeout, so the kernel must never
leave a party waiting; this test replays the kernel's control flow under
every failure it handles (a copy that never arrives at any tile, a look-back
that times out at any tile, both) over random interleavings and checks:

  - no deadlock: some party can always move until both finish;
  - no barrier phase ever receives more than 544 arrivals;
  - no phase is left half complete when both parties have left.

If the kernel's hand-off changes, this model must change with it."""

from __future__ import annotations

import random

import pytest

ALL, CT, LW = 544, 512, 32
AGG, PRE = 2, 4


def compute_warps(count, copy_fails_at, sh):
    """The compute warps' barrier operations: count tile 0 and hand it over;
    then per tile k: count tile k+1 and hand it over, wait for tile k's
    offsets, stop on a failed look-back or on tile k+1's missing copy."""
    def count_tile(k):
        sh["stop"][k & 1] = k == copy_fails_at  # written by the last counting warp
        yield ("arrive", AGG + (k & 1), CT)

    if count > 0:
        yield from count_tile(0)
        if sh["stop"][0]:
            return
    for k in range(count):
        if k + 1 < count:
            yield from count_tile(k + 1)
        yield ("sync", PRE + (k & 1), CT)
        if sh["fail"][k & 1]:
            return
        if k + 1 < count and sh["stop"][(k + 1) & 1]:
            return


def lookback_warp(count, lookback_fails_at, sh):
    """The look-back warp: per tile, wait for the hand-over, leave if the
    compute warps stopped, else publish and hand the offsets back; after a
    failed look-back, take the next tile's hand-over and leave."""
    for k in range(count):
        yield ("sync", AGG + (k & 1), LW)
        if sh["stop"][k & 1]:
            return
        failed = k == lookback_fails_at
        sh["fail"][k & 1] = failed
        yield ("arrive", PRE + (k & 1), LW)
        if failed:
            if k + 1 < count:
                yield ("sync", AGG + ((k + 1) & 1), LW)
            return


def run(count, copy_fails_at, lookback_fails_at, seed):
    rnd = random.Random(seed)
    sh = {"stop": [False, False], "fail": [False, False]}
    parties = {"compute": compute_warps(count, copy_fails_at, sh),
               "lookback": lookback_warp(count, lookback_fails_at, sh)}
    waiting, bars, done = {}, {}, set()

    def step(p):
        try:
            kind, bid, n = next(parties[p])
        except StopIteration:
            done.add(p)
            return
        b = bars.setdefault(bid, [0, 0])  # arrivals in the open phase, phases completed
        b[0] += n
        assert b[0] <= ALL, f"barrier {bid}: more than {ALL} arrivals in one phase"
        if b[0] == ALL:
            b[0] = 0
            b[1] += 1
            for q, (wid, ph) in list(waiting.items()):
                if wid == bid and ph < b[1]:
                    del waiting[q]
        elif kind == "sync":
            waiting[p] = (bid, b[1])

    for _ in range(100_000):
        if len(done) == 2:
            break
        movable = [p for p in parties if p not in done and p not in waiting]
        assert movable, f"deadlock: waiting {waiting}, barriers {bars}"
        step(rnd.choice(movable))
    assert len(done) == 2
    for bid, b in bars.items():
        assert b[0] == 0, f"barrier {bid} left with {b[0]} of {ALL} arrivals"


@pytest.mark.parametrize("count", [1, 2, 3, 4, 6])
def test_protocol_never_hangs(count):
    for copy_fails_at in [None] + list(range(count)):
        for lookback_fails_at in [None] + list(range(count)):
            for seed in range(20):
                run(count, copy_fails_at, lookback_fails_at, seed)


def test_model_catches_a_missing_final_hand_over():
    # the check is not vacuous: drop the look-back warp's last wait after a
    # failure and the compute warps' extra hand-over is left half complete
    def broken_lookback(count, lookback_fails_at, sh):
        for k in range(count):
            yield ("sync", AGG + (k & 1), LW)
            if sh["stop"][k & 1]:
                return
            sh["fail"][k & 1] = k == lookback_fails_at
            yield ("arrive", PRE + (k & 1), LW)
            if sh["fail"][k & 1]:
                return

    global lookback_warp
    saved = lookback_warp
    lookback_warp = broken_lookback
    try:
        with pytest.raises(AssertionError):
            run(3, None, 0, 0)
    finally:
        lookback_warp = saved
