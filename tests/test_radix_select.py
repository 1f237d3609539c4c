"""The selection's key mapping and radix select, restated in numpy, equal a
plain sort.

Keys: an fp32 priority p becomes the 32-bit key of bits(p + 0) with the sign
bit set for p >= 0, or all bits inverted for p < 0.  Adding 0 turns -0 into
+0, so the two zeros tie.  Unsigned key order is then the order of p.

Select: four passes over 8-bit digits, most significant first, find the
B-th smallest key T and how many keys equal to T are kept. Each pass takes
the digit whose cumulative count first reaches the wanted rank among the keys
that still match the prefix.  The cluster's CTAs hold contiguous chunks of
the sequence.  Each CTA keeps its keys < T, and the keys == T in slot order
while the count of equal keys in earlier chunks plus its own stays below the
kept number.  It writes them at the offset of the earlier chunks' kept
counts.  The result must be the first B slots of a stable sort by key."""
import numpy as np
import pytest


def order_bits(p):
    u = (np.asarray(p, dtype=np.float32) + np.float32(0)).view(np.uint32)
    return np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)


def radix_select(keys, B, CL=8):
    keys = np.asarray(keys, dtype=np.uint32)
    L = len(keys)
    if B <= 0:
        return np.zeros(0, dtype=np.int64)
    if L <= B:
        return np.arange(L)
    prefix, pmask, want = 0, 0, B
    for shift in (24, 16, 8, 0):
        cand = keys[(keys & np.uint32(pmask)) == np.uint32(prefix)]
        hist = np.bincount((cand >> np.uint32(shift)) & np.uint32(255), minlength=256)
        incl = np.cumsum(hist)
        excl = incl - hist
        d = int(np.nonzero((excl < want) & (want <= incl))[0][0])
        prefix |= d << shift
        pmask |= 255 << shift
        want -= int(excl[d])
    T, keep_eq = np.uint32(prefix), want
    chunk = -(-L // CL)
    out, eq_before = [], 0
    for r in range(CL):                       # CTA r of the cluster, in slot order
        c0, c1 = min(L, r * chunk), min(L, (r + 1) * chunk)
        for i in range(c0, c1):
            if keys[i] < T:
                out.append(i)
            elif keys[i] == T:
                if eq_before < keep_eq:
                    out.append(i)
                eq_before += 1
    return np.array(out, dtype=np.int64)


def sort_select(keys, B):
    order = np.argsort(np.asarray(keys, dtype=np.uint32), kind="stable")
    return np.sort(order[:max(B, 0)])


def test_key_order_is_the_priority_order_and_zeros_tie():
    rng = np.random.default_rng(0)
    p = np.concatenate([rng.standard_normal(5000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, np.inf, -np.inf, 1e-40, -1e-40, 3.4e38, -3.4e38],
                                 dtype=np.float32)])
    k = order_bits(p)
    a, b = np.argsort(p, kind="stable"), np.argsort(k, kind="stable")
    assert np.array_equal(p[a], p[b])
    assert order_bits(np.float32(-0.0)) == order_bits(np.float32(0.0))
    assert order_bits(np.float32(-1e-40)) < order_bits(np.float32(0.0)) < order_bits(np.float32(1e-40))


@pytest.mark.parametrize("CL", [1, 8])
def test_radix_select_equals_a_stable_sort(CL):
    rng = np.random.default_rng(CL)
    for trial in range(300):
        L = int(rng.integers(1, 400))
        B = int(rng.integers(1, L + 3))
        kind = trial % 5
        if kind == 0:       # many exact ties (accessed tokens all have priority 0)
            p = rng.choice(np.float32([0.0, -0.0, 0.25, 0.5]), size=L)
        elif kind == 1:     # keys that differ in the lowest byte only
            k = (np.uint32(0x9A000000) + rng.integers(0, 256, L)).astype(np.uint32)
            assert np.array_equal(radix_select(k, B, CL), sort_select(k, B))
            continue
        elif kind == 2:     # one value everywhere
            p = np.full(L, 0.125, dtype=np.float32)
        else:
            p = (rng.standard_normal(L) * 3).astype(np.float32)
        k = order_bits(p)
        assert np.array_equal(radix_select(k, B, CL), sort_select(k, B)), (L, B, kind)


def test_ties_straddling_cta_chunks_keep_the_lowest_slots():
    L, B = 64, 20
    p = np.full(L, 1.0, dtype=np.float32)
    p[::7] = 0.5                                # 10 clear keeps; the other 10 from the ties
    got = radix_select(order_bits(p), B, CL=8)  # 8 chunks of 8 slots
    assert np.array_equal(got, sort_select(order_bits(p), B))
    clear = set(range(0, L, 7))
    ties = [i for i in range(L) if i not in clear][:B - len(clear)]
    assert list(got) == sorted(clear | set(ties))   # the tied keys kept are the lowest slots
