"""Pins of the ranking diagnostics (oracle/diagnostics.py) against their
definitions worked out by hand or by brute force: the raw top-B set is the
unique B-subset whose every (-score, slot) key is below every other key;
Jaccard overlaps of small sets; the step counts of a hand example; the
Future Missed Mass of a hand example and of a run that discards nothing; the
Global LIR of a hand-written routing history."""
import itertools

import numpy as np
import pytest

from oracle import diagnostics as D


def test_raw_topb_matches_brute_force_with_ties():
    rng = np.random.default_rng(2)
    for _ in range(200):
        L = int(rng.integers(1, 8))
        raw = rng.choice([0.0, 0.1, 0.1, 0.5, 2.0], size=L)
        B = int(rng.integers(0, L + 2))
        got = D.raw_topb(raw, B)
        n = min(B, L)
        keys = [(-raw[i], i) for i in range(L)]
        valid = [S for S in itertools.combinations(range(L), n)
                 if all(keys[a] < keys[b] for a in S for b in range(L) if b not in S)]
        assert len(valid) == 1 and list(got) == list(valid[0])


def test_jaccard_small_sets():
    assert D.jaccard([1, 2, 3], [2, 3, 4]) == pytest.approx(2 / 4)
    assert D.jaccard([], []) == 1.0
    assert D.jaccard([1], [2]) == 0.0
    assert D.jaccard(range(5), range(5)) == 1.0


def test_step_counts_hand_example():
    # 6 slots after the append (slot 5 is the new token), positions 10..15
    pos = np.array([10, 11, 12, 13, 14, 15])
    c = D.step_counts(raw_set_slots=[0, 2, 5], kept_slots=[0, 1, 2, 5], L=6,
                      prev_raw_pos=[10, 13, 9], prev_raw_size=3, pos=pos)
    assert c == {"n_raw": 3, "n_kept": 4, "raw_and_kept": 3, "raw_and_prev_raw": 1,
                 "n_prev_raw": 3, "kept_and_prev_kept": 3}
    c0 = D.step_counts([1], [1, 2], 3)
    assert c0["raw_and_prev_raw"] == 0 and c0["n_prev_raw"] == 0
    assert c0["kept_and_prev_kept"] == 1       # slot 1 was held before, slot 2 is new


def test_missed_mass_hand_example_and_no_eviction():
    full = [1.0, 2.0, 3.0, 4.0]
    assert D.missed_mass(full, held_pos=[0, 2], new_pos=3) == pytest.approx(0.2)
    assert D.missed_mass(full, held_pos=[0, 1, 2], new_pos=3) == pytest.approx(0.0)
    assert D.missed_mass(full, held_pos=[], new_pos=3) == pytest.approx(0.6)


def test_global_lir_hand_history():
    c = D.LIRCounter(sustain=2)
    history = [{0: "F", 1: "Q", 2: "Q", 3: "U"},
               {0: "Q", 1: "F", 2: "Q", 3: "U"},
               {0: "Q", 1: "F", 2: "E", 3: "Q"},
               {0: "F", 1: "Q", 2: "E", 3: "Q"}]
    for h in history:
        c.route(h)
    # window 0: F, Q, Q, F -> sustained inactive after event 3, revived at 4;
    # window 1: Q, F, F, Q -> never sustained; window 2: Q, Q, E, E -> one
    # span, no revival; window 3: U, U, Q, Q -> one span at event 4
    assert (c.events, c.revivals, c.spans) == (4, 1, 3)
    assert c.lir() == pytest.approx(1 / 3)
    assert D.LIRCounter(3).lir() == 0.0
