"""Round counters ("A drafter inside the artifact", Ignis DFlash2 page,
section "See it, control it", Metrics): the oracle's definition pinned by a
hand-worked case and by the invariants the counts must keep."""
from __future__ import annotations

import numpy as np

import oracle


def test_hand_worked_case():
    # gamma 3, four lanes accepting 0, 3, 1 and 2 drafts, counted by hand:
    # position 0 is accepted by the lanes with a >= 1 (3 of them), position 1
    # by a >= 2 (2), position 2 by a = 3 (1)
    c = oracle.counters(np.array([0, 3, 1, 2]), 3)
    assert c == {"rounds": 4, "drafted_tokens": 12, "accepted_tokens": 6,
                 "position_drafted": [4, 4, 4], "position_accepted": [3, 2, 1]}


def test_golden_verify_lanes():
    # the gamma = 2 lanes of the hand-worked verify examples accept 2, 1, 0, 0
    c = oracle.counters(np.array([2, 1, 0, 0]), 2)
    assert c["position_accepted"] == [2, 1] and c["accepted_tokens"] == 3 and c["drafted_tokens"] == 8


def test_extremes():
    assert oracle.counters(np.zeros(5, dtype=np.int32), 7)["position_accepted"] == [0] * 7
    full = oracle.counters(np.full(5, 7), 7)
    assert full["position_accepted"] == [5] * 7 and full["accepted_tokens"] == full["drafted_tokens"] == 35
    assert oracle.counters(np.zeros(0, dtype=np.int32), 4)["rounds"] == 0


def test_invariants_on_random_lanes():
    rng = np.random.default_rng(5)
    for gamma in (1, 2, 7, 15):
        acc = rng.integers(0, gamma + 1, size=200)
        c = oracle.counters(acc, gamma)
        pa, pd = c["position_accepted"], c["position_drafted"]
        assert sum(pa) == c["accepted_tokens"] == int(acc.sum())
        assert sum(pd) == c["drafted_tokens"] == 200 * gamma
        assert all(pa[i] >= pa[i + 1] for i in range(gamma - 1))       # a lane accepting i+1 accepts i
        assert all(0 <= x <= 200 for x in pa)
        assert [int((acc > i).sum()) for i in range(gamma)] == pa      # closed form per position


def test_rejects_impossible_lengths():
    import pytest
    with pytest.raises(ValueError):
        oracle.counters(np.array([4]), 3)
