"""MemDecay's eviction loop (Algorithm 1: pop the page of least S_p until the
tokens fit the budget) becomes a count on the device.

Every page but the last is full.  Popping j pages removes the j pages of
largest key (key = order bits of -S_p, 0 for a pinned page; equal keys:
the later page first).  The least sufficient j is ceil(excess / P), plus one
when the partial last page is among those j and they still fall short.  The
selection then keeps the other pages.  Restated in numpy, that count gives
the oracle's heap the same evicted set on random page scores.  The cases
include ties, pinned pages, a partial last page and budgets no eviction can
meet."""
import numpy as np
import pytest

from oracle import memdecay as MD


def order_bits(p):
    u = (np.asarray(p, dtype=np.float32) + np.float32(0)).view(np.uint32)
    return np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)


def device_evicted(S, n_tok, pinned, budget, P):
    nb = len(S)
    keys = np.where(pinned, 0, np.maximum(order_bits(-np.asarray(S, np.float32)), 1)).astype(np.uint32)
    excess = int(np.sum(n_tok)) - budget
    if excess <= 0 or nb == 0:
        keep = nb
    else:
        last, kl, rl = nb - 1, keys[-1], int(n_tok[-1])
        n_free = int(np.sum(keys != 0))
        ahead = int(np.sum((np.arange(nb) < last) & (keys <= kl)))
        j0 = min(-(-excess // P), n_free)
        last_goes = kl != 0 and ahead >= nb - j0
        if rl < P and last_goes and P * (j0 - 1) + rl < excess and j0 < n_free:
            j0 += 1
        keep = nb - j0
    order = np.argsort(keys, kind="stable")          # the selection: smallest keys kept
    return set(range(nb)) - set(order[:keep].tolist())


@pytest.mark.parametrize("seed", range(8))
def test_device_count_matches_the_heap(seed):
    rng = np.random.default_rng(seed)
    P = 16
    for trial in range(400):
        nb = int(rng.integers(1, 40))
        n_tok = np.full(nb, P)
        n_tok[-1] = int(rng.integers(1, P + 1))      # the last page may be partial
        if trial % 3 == 0:
            S = rng.choice(np.float32([0.1, 0.2, 0.2, 0.3]), size=nb)   # many ties
        else:
            S = rng.uniform(0, 2, nb).astype(np.float32)
        pinned = rng.random(nb) < (0.15 if trial % 4 else 0.0)
        if trial % 7 == 0:
            pinned[-1] = True                        # a pinned partial page
        total = int(n_tok.sum())
        budget = int(rng.integers(0, total + P))     # 0 .. beyond the cache
        want = set(MD.evict_pages(S.astype(np.float64), n_tok, pinned, budget))
        got = device_evicted(S, n_tok, pinned, budget, P)
        assert got == want, (nb, n_tok[-1], budget, sorted(got), sorted(want))
