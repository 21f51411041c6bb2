"""Pins for oracle.schedule (circular two-slot prefetch order)."""
import os

import pytest

from oracle import schedule as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "execution_flow_n4.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            a, b = line.split()
            rows.append((int(a), int(b)))
    return rows


def test_execution_flow_table():
    """The page's table: block i prefetches i+1, block n-1 prefetches block 0."""
    ev = S.schedule(4, 0, 1)
    assert ev[0] == ("stage", 0, 0)                 # priming of the first block
    pairs = [(ev[i + 1][1], ev[i][1]) for i in range(1, len(ev), 2)]
    assert pairs == _golden_rows()
    assert [S.next_block(i, 4, 0) for i in range(4)] == [1, 2, 3, 0]


def simulate(events, n, k, steps):
    """Independent check of an event list by simulating the two slots.

    Returns a list of violations (empty when the schedule is valid).
    """
    bad = []
    slot = {0: None, 1: None}          # block currently held by each slot
    pending = {0: False, 1: False}     # staged but not yet executed
    order = []
    n_stage = 0
    for kind, blk, s in events:
        if kind == "stage":
            n_stage += 1
            if not (k <= blk < n):
                bad.append(("staged a non-streamed block", blk))
            if pending[s]:
                bad.append(("clobbered a staged block before use", s, slot[s]))
            slot[s] = blk
            pending[s] = True
        else:
            order.append(blk)
            if blk < k:
                if s is not None:
                    bad.append(("resident block ran from a slot", blk))
                continue
            if slot.get(s) != blk:
                bad.append(("executed from a slot not holding the block", blk, s, slot.get(s)))
            pending[s] = False
    if order != list(range(n)) * steps:
        bad.append(("execution order", order))
    want = 0 if k == n else 1 + steps * (n - k)
    if n_stage != want:
        bad.append(("staging count", n_stage, want))
    if k < n and events[-2][0] == "stage":
        # after the last block of the last step the first streamed block is
        # already staged again, so the next forward starts warm
        if events[-2][1] != k:
            bad.append(("tail prefetch is not the first streamed block", events[-2]))
    return bad


@pytest.mark.parametrize("n", range(1, 7))
def test_brute_force_all_small(n):
    for k in range(0, n + 1):
        for steps in range(1, 4):
            ev = S.schedule(n, k, steps)
            assert simulate(ev, n, k, steps) == [], (n, k, steps)
            # streamed execution j reads slot j % 2
            j = 0
            for kind, blk, s in ev:
                if kind == "exec" and s is not None:
                    assert s == j % 2
                    j += 1


def test_invalid_arguments():
    with pytest.raises(ValueError):
        S.schedule(3, 4, 1)
    with pytest.raises(ValueError):
        S.next_block(0, 4, 1)


def test_simulator_catches_planted_mistakes():
    """The pins above must reject plausible slips in the schedule."""
    n, k, steps = 5, 2, 2

    def wrap_to_zero(i, n, k):          # last block prefetches block 0, not k
        return i + 1 if i < n - 1 else 0

    def same_slot(n, k, steps):          # stages into the slot being read
        ev = [("stage", k, 0)]
        j = 0
        for _ in range(steps):
            for i in range(k):
                ev.append(("exec", i, None))
            for i in range(k, n):
                ev.append(("stage", S.next_block(i, n, k), j % 2))
                ev.append(("exec", i, j % 2))
                j += 1
        return ev

    orig = S.next_block
    try:
        S.next_block = wrap_to_zero
        assert simulate(S.schedule(n, k, steps), n, k, steps) != []
    finally:
        S.next_block = orig
    assert simulate(same_slot(n, k, steps), n, k, steps) != []
    no_prime = S.schedule(n, k, steps)[1:]
    assert simulate(no_prime, n, k, steps) != []
