"""Ranking diagnostics of an eviction run, restated from their definitions.

TEST INFRASTRUCTURE ONLY (tests, benchmark CPU leg); shares nothing with the
CUDA library.  Every function is the plain definition, in fp64 / exact
integer counts:

  raw top-B      "What Matters for Aggressive Decoding-Time KV Eviction?"
                 (p1) Sec. 5.3 and Appendix I, Table 13: the B tokens the
                 step's raw score ranks highest (the score before any
                 aggregation: here the attention summed over query heads and
                 layers), ties to the lower slot.
  Jaccard, churn p1 Appendix I: raw / EMA Jaccard overlap |R & E| / |R | E|
                 of the raw top-B set R and the retained set E; the churn of a
                 ranking is the Jaccard distance 1 - J between its top-B sets
                 at consecutive scoring steps; "raw-top evicted" is the share
                 of R not retained.
  FMM            QEvict review, Sec. 3 "Diagnosing the problem" (Future Missed
                 Mass): the share of a FullKV run's attention at step t that
                 lands on tokens the compressed policy discarded before step t.
  Global LIR     the same section (Long-term Importance Revival): how often a
                 window inactive (outside the full-precision tier) for a
                 sustained period re-enters it.  Reading: a window is
                 sustained-inactive once it has been outside the Full tier at
                 `sustain` consecutive routing events; a revival is such a
                 window routed to Full; LIR = revivals / sustained-inactive
                 spans.  Windows not yet routable (recent, unrouted) do not
                 count; evicted windows stay inactive.
"""
from __future__ import annotations

import numpy as np


def raw_topb(raw: np.ndarray, budget: int) -> np.ndarray:
    """Ascending slots of the `budget` largest raw scores, ties to the lower
    slot (all slots when there are no more than `budget`)."""
    raw = np.asarray(raw, dtype=np.float64)
    L = raw.shape[0]
    order = sorted(range(L), key=lambda i: (-raw[i], i))
    return np.array(sorted(order[:min(budget, L)]), dtype=np.int64)


def jaccard(a, b) -> float:
    """|A & B| / |A | B| of two sets (1 for two empty sets)."""
    a, b = set(int(x) for x in a), set(int(x) for x in b)
    union = a | b
    return 1.0 if not union else len(a & b) / len(union)


def step_counts(raw_set_slots, kept_slots, L: int, prev_raw_pos=None, prev_raw_size: int = 0,
                pos=None):
    """Exact counts of one scoring step (slots of the cache after the append,
    length L; `pos` maps slots to logical positions, slot order):
    n_raw, n_kept, |R & E|, |R & R_prev| (by position; R_prev the raw set of
    the previous scoring step, tokens since evicted included in its size),
    |R_prev|, |E & E_prev| (E_prev = every cached token but the new one)."""
    pos = np.arange(L) if pos is None else np.asarray(pos)
    R = set(int(x) for x in raw_set_slots)
    E = set(int(x) for x in kept_slots)
    rr = 0
    if prev_raw_pos is not None:
        prev = set(int(p) for p in prev_raw_pos)
        rr = sum(1 for s in R if int(pos[s]) in prev)
    return {"n_raw": len(R), "n_kept": len(E), "raw_and_kept": len(R & E),
            "raw_and_prev_raw": rr, "n_prev_raw": int(prev_raw_size) if prev_raw_pos is not None
            else 0, "kept_and_prev_kept": len(E - {L - 1})}


def missed_mass(full_score, held_pos, new_pos: int) -> float:
    """Future Missed Mass of one step: 1 - (the FullKV run's attention on the
    positions the policy holds, plus the new token's) / (its attention on
    every position so far).  full_score[p] is the FullKV attention on
    position p (any common scale: summed over heads and layers)."""
    full = np.asarray(full_score, dtype=np.float64)
    held = set(int(p) for p in held_pos) | {int(new_pos)}
    tot = float(full.sum())
    return 1.0 - float(sum(full[p] for p in sorted(held))) / tot


class LIRCounter:
    """Global LIR bookkeeping over routing events (see the module header)."""

    def __init__(self, sustain: int):
        self.sustain = int(sustain)
        self.streak = {}
        self.revivals = 0
        self.spans = 0
        self.events = 0

    def route(self, tiers: dict):
        """tiers: window id -> 'F' (full precision), 'Q' (INT2), 'E' (evicted)
        or 'U' (unrouted, skipped), after one routing event."""
        self.events += 1
        for wid, tier in sorted(tiers.items()):
            if tier == "U":
                continue
            s = self.streak.get(wid, 0)
            if tier == "F":
                if s >= self.sustain:
                    self.revivals += 1
                self.streak[wid] = 0
            else:
                self.streak[wid] = s + 1
                if s + 1 == self.sustain:
                    self.spans += 1

    def lir(self) -> float:
        return self.revivals / self.spans if self.spans else 0.0
