"""Pins of the wave buffer's page-cache policy oracle (oracle.wave_buffer).

The pages name LRU replacement and nothing finer, so the pins are a hand-worked
LRU trace, the invariants any cache keeps, and the special cases that reduce to
something known (a cache as large as the working set never evicts; a cache of
no slots never admits).
"""
import random

import pytest

from oracle.wave_buffer import LruPagePolicy, pages_of_rows


def test_hand_worked_lru_trace():
    """Three slots, one page per round, the textbook reference string 1 2 3 1 4 5: page 4 evicts
    2 (the least recently used, since 1 was touched again), page 5 evicts 3."""
    pol = LruPagePolicy(pages=8, slots=3, admit_max=4)
    trace = []
    for t, p in enumerate([1, 2, 3, 1, 4, 5]):
        trace.append(pol.round([p], t))
    assert trace[0] == ([], [(1, 0)])
    assert trace[1] == ([], [(2, 1)])
    assert trace[2] == ([], [(3, 2)])
    assert trace[3] == ([], [])                 # hit
    assert trace[4] == ([(2, 1)], [(4, 1)])     # 2 is least recently used
    assert trace[5] == ([(3, 2)], [(5, 2)])
    assert pol.slot_of == {1: 0, 4: 1, 5: 2}


def test_round_order_and_same_round_protection():
    """Within a round pages go in increasing order; a page touched in this round is never the
    victim, so a round that touches more pages than there are slots stops admitting."""
    pol = LruPagePolicy(pages=16, slots=2, admit_max=8)
    ev, ad = pol.round([9, 3, 5], 0)
    assert ev == [] and ad == [(3, 0), (5, 1)]      # 9 finds no victim: 3 and 5 are this round's
    ev, ad = pol.round([9], 1)
    assert ev == [(3, 0)] and ad == [(9, 0)]        # 3 was made most recent before 5
    ev, ad = pol.round([5, 7], 2)                   # 5 hit (most recent); 7 evicts 9
    assert ev == [(9, 0)] and ad == [(7, 0)]


def test_admission_budget():
    pol = LruPagePolicy(pages=64, slots=32, admit_max=3)
    ev, ad = pol.round(range(10), 0)
    assert ev == [] and ad == [(0, 0), (1, 1), (2, 2)]
    ev, ad = pol.round(range(10), 1)     # 0-2 hit, the next three misses are admitted
    assert ad == [(3, 3), (4, 4), (5, 5)]


def test_free_slot_is_the_lowest():
    pol = LruPagePolicy(pages=8, slots=4, admit_max=4)
    pol.round([0, 1, 2, 3], 0)
    pol.round([4], 1)                    # evicts 0 from slot 0
    assert pol.slot_of[4] == 0


def test_large_cache_never_evicts_and_empty_cache_never_admits():
    rng = random.Random(5)
    big = LruPagePolicy(pages=100, slots=100, admit_max=100)
    none = LruPagePolicy(pages=100, slots=0, admit_max=100)
    for t in range(50):
        touched = rng.sample(range(100), 20)
        ev, ad = big.round(touched, t)
        assert ev == []
        assert none.round(touched, t) == ([], [])
    assert len(big.slot_of) == len({p for p in big.slot_of})


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_brute_force_lru(seed):
    """A second statement of the rounds, by time stamps and argmin instead of a recency list:
    pages in increasing order, a hit re-stamps its page, a miss takes the lowest free slot or
    evicts the cached page of smallest stamp unless that stamp is this round's.  The oracle's
    evictions and admissions equal it over random rounds; slots stay a bijection."""
    rng = random.Random(seed)
    P, S, A = 40, 7, 5
    pol = LruPagePolicy(pages=P, slots=S, admit_max=A)
    slot = {}       # page -> slot
    stamp = {}      # page -> (round, order of touch within the round)
    for t in range(300):
        touched = sorted(set(rng.sample(range(P), rng.randint(1, 9))))
        exp_ev, exp_ad, n = [], [], 0
        for i, p in enumerate(touched):
            if p in slot:
                stamp[p] = (t, i)
                continue
            if n >= A:
                continue
            free = sorted(set(range(S)) - set(slot.values()))
            if free:
                s_ = free[0]
            else:
                if not slot:
                    continue
                victim = min(slot, key=lambda q: stamp[q])
                if stamp[victim][0] == t:
                    continue
                s_ = slot.pop(victim)
                del stamp[victim]
                exp_ev.append((victim, s_))
            slot[p] = s_
            stamp[p] = (t, i)
            exp_ad.append((p, s_))
            n += 1
        ev, ad = pol.round(touched, t)
        assert (ev, ad) == (exp_ev, exp_ad), t
        assert pol.slot_of == slot
        used = list(pol.slot_of.values())
        assert len(used) == len(set(used)) <= S


def test_pages_of_rows():
    assert pages_of_rows(0, 16, 16) == [0]
    assert pages_of_rows(15, 2, 16) == [0, 1]
    assert pages_of_rows(20, 40, 16) == [1, 2, 3]
    assert pages_of_rows(7, 0, 16) == []
