"""The library's page replacement policy (wi_lru_*, run on the host) against the oracle's rounds.

No device is involved: the policy is the host side of the wave buffer, and these calls exercise the
same C++ class the replacement thread runs.
"""
import random

import pytest

import oracle

wi = pytest.importorskip("clustered_sparse_kv_gb300")


@pytest.mark.parametrize("pages,slots,admit,seed", [(40, 7, 5, 0), (64, 64, 64, 1), (200, 16, 3, 2),
                                                     (30, 0, 4, 3), (50, 10, 0, 4), (1, 1, 1, 5)])
def test_policy_matches_oracle(pages, slots, admit, seed):
    rng = random.Random(seed)
    lib_pol = wi.LruPolicy(pages, slots, admit)
    ref = oracle.LruPagePolicy(pages, slots, admit)
    for t in range(400):
        touched = [rng.randrange(pages) for _ in range(rng.randint(0, 12))]  # repeats, any order
        assert lib_pol.round(touched, t) == ref.round(touched, t), t


def test_policy_rounds_with_gaps_in_round_numbers():
    """Round numbers are decode steps: they increase with gaps (rounds run when the thread is free)."""
    rng = random.Random(9)
    lib_pol = wi.LruPolicy(32, 5, 4)
    ref = oracle.LruPagePolicy(32, 5, 4)
    t = 0
    for _ in range(200):
        t += rng.randint(1, 7)
        touched = rng.sample(range(32), rng.randint(1, 8))
        assert lib_pol.round(touched, t) == ref.round(touched, t)


def test_policy_rejects_bad_input():
    with pytest.raises(ValueError):
        wi.LruPolicy(0, 1, 1)
    with pytest.raises(ValueError):
        wi.LruPolicy(4, -1, 1)
    pol = wi.LruPolicy(4, 2, 2)
    with pytest.raises(wi.WiError):
        pol.round([4], 0)
    with pytest.raises(wi.WiError):
        pol.round([-1], 0)
    assert pol.round([], 0) == ([], [])
