"""A model of the prefill's K/V ring at D = 128, where slots are released in
pairs, run on the CPU.  Each side takes the index arithmetic the kernel uses.

The ring holds K_0, V_0, K_1, V_1, ... of each item at consecutive positions
(an item of n K/V steps takes positions kb .. kb + 2n - 1, kb even).  With an
even number of stages, positions 2g - 1 (a V) and 2g (the K after it) always
occupy the same two slots, "pair g".  The producer, before loading either
position of pair g, waits on empty[g % NPAIR] with parity
((g / NPAIR) & 1) ^ 1.  The MMA warp releases pair kb / 2 once an item's K_0
is consumed, which also covers the previous item's last V.  Within an item it
releases pair kb / 2 + j + 1 once V_j and K_{j+1} are consumed.

Under random interleavings of the two sides, the model checks three things:
- no slot is overwritten before the tile in it is consumed;
- a parity wait never sees its barrier two phases ahead, which would make it
  wait for the wrong phase;
- both sides finish (no deadlock).
"""
import random

import pytest

NSTAGE = 4
NPAIR = NSTAGE // 2


def barrier_passes(completions, parity):
    # mbarrier parity wait: true once the phase of that parity has completed,
    # i.e. the current (open) phase has the other parity.
    return (completions & 1) != parity


def run(ns, rng):
    # Tiles in item order: (position, kind, item, j).
    loads = []
    kb = 0
    for it, n in enumerate(ns):
        if n == 0:
            continue
        loads.append((kb, "K", it, 0))
        for j in range(n):
            loads.append((kb + 2 * j + 1, "V", it, j))
            if j + 1 < n:
                loads.append((kb + 2 * j + 2, "K", it, j + 1))
        kb += 2 * n
    # MMA events: the positions it consumes, then the pair it releases (or None).
    events = []
    kb = 0
    for it, n in enumerate(ns):
        if n == 0:
            continue
        events.append(([kb], (kb >> 1) % NPAIR))  # S(0) on K_0
        for j in range(n):
            if j + 1 < n:  # PV(j) on V_j, S(j+1) on K_{j+1}, then one commit
                events.append(([kb + 2 * j + 1, kb + 2 * j + 2], ((kb >> 1) + j + 1) % NPAIR))
            else:  # the last PV: V_{n-1} waits for the next item's K_0
                events.append(([kb + 2 * j + 1], None))
        kb += 2 * n

    slot = [None] * NSTAGE          # position held by each slot (None: free)
    consumed = set()
    completions = [0] * NPAIR       # phases completed per pair barrier
    loaded = set()
    pi = mi = 0
    expect_gen = 0                  # pairs must be released in order 0, 1, 2, ...
    steps = 0
    while pi < len(loads) or mi < len(events):
        steps += 1
        assert steps < 100000, "deadlock"
        can_p = False
        if pi < len(loads):
            pos = loads[pi][0]
            g = (pos + 1) >> 1
            b = g % NPAIR
            can_p = barrier_passes(completions[b], ((g // NPAIR) & 1) ^ 1)
        can_m = mi < len(events) and all(p in loaded for p in events[mi][0])
        assert can_p or can_m, "deadlock"
        if can_p and (not can_m or rng.random() < 0.5):
            pos = loads[pi][0]
            g = (pos + 1) >> 1
            b = g % NPAIR
            # The wait passed: the barrier must be exactly at the phase this
            # load needs, never a phase beyond it.
            assert completions[b] == g // NPAIR, (pos, g, completions)
            s = pos % NSTAGE
            assert slot[s] is None or slot[s] in consumed, f"slot {s} overwritten"
            slot[s] = pos
            loaded.add(pos)
            pi += 1
        else:
            used, release = events[mi]
            for p in used:
                consumed.add(p)
            if release is not None:
                # Both positions of the released pair have been consumed.
                gen = expect_gen
                for p in (2 * gen - 1, 2 * gen):
                    if p >= 0:
                        assert p in consumed, (gen, p)
                assert release == gen % NPAIR
                completions[release] += 1
                expect_gen += 1
            mi += 1
    return True


@pytest.mark.parametrize("seed", range(40))
def test_paired_ring_releases_never_overwrite_or_skip_a_phase(seed):
    rng = random.Random(seed)
    ns = [rng.choice([0, 1, 1, 2, 3, 5, 8, 17]) for _ in range(rng.randint(1, 12))]
    assert run(ns, rng)


def test_paired_ring_with_single_step_items_back_to_back():
    # Items of one K/V step each release only the pair of their K_0.
    assert run([1] * 9, random.Random(1))
    assert run([1, 0, 2, 0, 0, 1, 3], random.Random(2))
