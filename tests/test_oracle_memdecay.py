"""Pins for the region-aware (MemDecay) page-eviction oracle."""
import itertools
import math

import numpy as np
import pytest

from oracle import memdecay as MD
from workloads import f32_to_bf16_bits, region_spans


def _bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _params(**kw):
    base = dict(n_layers=1, n_q_heads=1, n_kv_heads=1, head_dim=4, budget=1000,
                base=(1.0, 1.0), lam=(math.log(2) / 10.0, math.log(2) / 40.0),
                pinned=(False, False), rho=0.9, attn_weight=0.5, tau_scale=2.0, page=4,
                decode_region=1)
    base.update(kw)
    return MD.MDParams(**base)


def _seq(K, region, page=4, V=None):
    K = _bits(K)
    V = _bits(np.zeros_like(np.asarray(K, dtype=np.float32))) if V is None else _bits(V)
    return MD.MDSequence.from_prefill(K, V, np.asarray(region), page)


def _zeros(P):
    z = np.zeros((P.n_layers, P.n_kv_heads, P.head_dim), np.float32)
    return _bits(z), _bits(z)


def _q(P, x0=0.0):
    q = np.zeros((P.n_layers, P.n_q_heads, P.head_dim), np.float32)
    q[..., 0] = x0
    return _bits(q)


def test_half_life_of_the_structural_prior():
    """Eq. (4) with alpha a = 0 and lambda = ln 2 / t_half (Eq. (7)): a token
    never attended above tau keeps b / 2 after one half-life, b / 4 after two."""
    P = _params(attn_weight=0.0, base=(3.0, 1.0))
    seq = _seq(np.zeros((1, 1, 8, 4)), [0] * 8)
    kn, vn = _zeros(P)
    for t in range(1, 21):
        res = MD.step(P, seq, t, True, _q(P), kn, vn)
        if t == 10:
            assert res["s"][0] == pytest.approx(1.5, rel=1e-12)
    assert res["s"][0] == pytest.approx(0.75, rel=1e-12)   # region 0: half-life 10, t = 20
    # uniform attention 1 / L never reaches tau = 2 / L: the clock never resets
    assert res["t_ref"][0] == 0


def test_attention_above_tau_resets_the_clock():
    """Eq. (3): a token taking almost all attention (A_bar >= 2 / L) gets
    t_ref = t, so its structural term is back to b_r; the others decay."""
    P = _params()
    K = np.zeros((1, 1, 8, 4), np.float32)
    K[0, 0, 3, 0] = 40.0
    seq = _seq(K, [0] * 8)
    kn, vn = _zeros(P)
    res = MD.step(P, seq, 40, True, _q(P, 1.0), kn, vn)
    assert res["accessed"][3] and not res["accessed"][0]
    assert res["t_ref"][3] == 40 and res["t_ref"][0] == 0
    a3 = 0.1 * res["A_bar"][3]                                # (1 - rho) A_bar from a = 0
    assert res["s"][3] == pytest.approx(1.0 + 0.5 * a3, rel=1e-12)
    assert res["s"][0] == pytest.approx(2.0 ** -4 + 0.5 * 0.1 * res["A_bar"][0], rel=1e-12)


def test_importance_ewma_closed_form():
    """Eq. (2) under uniform attention: after n observation steps
    a = sum_k (1 - rho) rho^(n - k) / L_k, L_k the cache size at step k."""
    P = _params(rho=0.8)
    seq = _seq(np.zeros((1, 1, 8, 4)), [1] * 8)
    kn, vn = _zeros(P)
    Ls = []
    for t in range(1, 6):
        res = MD.step(P, seq, t, True, _q(P), kn, vn)
        Ls.append(res["L"])
    want = sum(0.2 * 0.8 ** (5 - k) / Ls[k - 1] for k in range(1, 6))
    assert res["a"][0] == pytest.approx(want, rel=1e-12)


def test_page_score_is_the_mean_of_its_tokens():
    """Eq. (5): a page holding tokens of two regions scores the mean."""
    P = _params(attn_weight=0.0)
    seq = _seq(np.zeros((1, 1, 8, 4)), [0, 0, 1, 1, 1, 1, 1, 1])
    kn, vn = _zeros(P)
    res = MD.step(P, seq, 20, True, _q(P), kn, vn)
    want = (2 * 2.0 ** -2 + 2 * 2.0 ** -0.5) / 4
    assert res["S"][0] == pytest.approx(want, rel=1e-12)
    assert res["S"][1] == pytest.approx(2.0 ** -0.5, rel=1e-12)


def test_greedy_page_eviction_is_optimal_for_equal_pages():
    """Sec. III-D: with equal-size pages, evicting in ascending S_p until the
    budget holds keeps the largest retained score of any admissible set
    (brute force over all subsets of pages)."""
    rng = np.random.default_rng(3)
    for _ in range(30):
        n = 7
        S = rng.random(n)
        pinned = rng.random(n) < 0.2
        n_tok = np.full(n, 4)
        budget = int(rng.integers(4, 24))
        ev = MD.evict_pages(S, n_tok, pinned, budget)
        best, best_set = -1.0, None
        for k in range(n + 1):
            for sub in itertools.combinations([j for j in range(n) if not pinned[j]], k):
                kept = [j for j in range(n) if j not in sub]
                if n_tok[kept].sum() > budget and len(sub) < (~pinned).sum():
                    continue
                val = (S[kept] * n_tok[kept]).sum()
                if val > best + 1e-15:
                    best, best_set = val, set(sub)
        assert set(ev) == best_set


def test_pinned_page_survives_and_protects_its_pagemates():
    """A page with one pinned token is never evicted, whatever its score,
    and keeps its unpinned pagemates (Sec. IV-A)."""
    P = _params(pinned=(True, False), base=(1.0, 1.0), lam=(0.0, 0.0), attn_weight=0.0,
                budget=4)
    region = [1, 1, 1, 1] + [0, 1, 1, 1] + [1] * 8
    seq = _seq(np.zeros((1, 1, 16, 4)), region)
    kn, vn = _zeros(P)
    res = MD.step(P, seq, 1, True, _q(P), kn, vn)
    assert res["pinned"].tolist() == [False, True, False, False, False]
    assert seq.pids() == [1]                                  # only the pinned page is left
    assert seq.n_tokens == 4


def test_equal_scores_evict_the_higher_page_index_first():
    """lambda = 0, alpha = 0: every page scores b, so the lower pages stay."""
    P = _params(lam=(0.0, 0.0), attn_weight=0.0, budget=9)
    seq = _seq(np.zeros((1, 1, 16, 4)), [1] * 16)
    kn, vn = _zeros(P)
    res = MD.step(P, seq, 1, True, _q(P), kn, vn)
    assert res["evicted"] == [4, 3, 2]                       # 17 tokens -> 16 -> 12 -> 8
    assert seq.pids() == [0, 1]


def test_budget_undershoot_is_below_one_page():
    """Whole pages go: after a step B - (page - 1) <= |K| <= B."""
    rng = np.random.default_rng(5)
    P = _params(budget=21, n_q_heads=2, n_kv_heads=1)
    seq = _seq(rng.standard_normal((1, 1, 40, 4)), list(rng.integers(0, 2, 40)))
    for t in range(1, 12):
        q = _bits(rng.standard_normal((1, 2, 4)))
        kn = _bits(rng.standard_normal((1, 1, 4)))
        MD.step(P, seq, t, True, q, kn, kn)
        assert P.budget - (P.page - 1) <= seq.n_tokens <= P.budget


def test_new_tokens_fill_the_partial_page_first():
    P = _params()
    seq = _seq(np.zeros((1, 1, 6, 4)), [0] * 6)              # pages of 4 + 2
    kn, vn = _zeros(P)
    MD.step(P, seq, 1, True, _q(P), kn, vn)
    MD.step(P, seq, 2, True, _q(P), kn, vn)
    assert [p.n for p in seq.pages] == [4, 4]
    MD.step(P, seq, 3, True, _q(P), kn, vn)
    assert [p.n for p in seq.pages] == [4, 4, 1] and seq.pages[-1].region.tolist() == [1]


def test_non_refresh_steps_keep_the_statistics():
    """Off observation steps a and t_ref stay; the prior keeps decaying."""
    P = _params()
    K = np.zeros((1, 1, 8, 4), np.float32)
    K[0, 0, 2, 0] = 40.0
    seq = _seq(K, [0] * 8)
    kn, vn = _zeros(P)
    r1 = MD.step(P, seq, 1, True, _q(P, 1.0), kn, vn)
    r2 = MD.step(P, seq, 2, False, _q(P, 1.0), kn, vn)
    assert np.array_equal(r2["a"][:9], r1["a"][:9]) and r2["a"][9] == 0.0
    assert np.array_equal(r2["t_ref"][:9], r1["t_ref"][:9])
    assert r2["s"][0] == pytest.approx(2.0 ** -0.2 + 0.5 * r1["a"][0], rel=1e-12)


def test_region_spans_of_the_workload():
    assert region_spans(16384) == [819, 819, 1638, 4915, 4915, 3278]
    assert region_spans(1700) == [85, 85, 170, 510, 510, 340]


def test_tau_is_inclusive_and_scaled_to_the_cache():
    """Eq. (3) with tau = tau_scale / |K_t|: under uniform attention A_bar is
    exactly 1 / L, which resets every clock at tau_scale = 1 (>=) and none
    at tau_scale = 2."""
    for scale, want in ((1.0, True), (2.0, False)):
        P = _params(tau_scale=scale, n_layers=2, n_q_heads=2)   # averaged over 2 x 2
        seq = _seq(np.zeros((2, 1, 7, 4)), [0] * 7)
        kn, vn = _zeros(P)
        res = MD.step(P, seq, 5, True, _q(P), kn, vn)
        assert bool(res["accessed"][:7].all()) == want and bool(res["accessed"][:7].any()) == want


def test_budget_met_exactly_stops_the_eviction():
    """17 tokens, budget 12: pages of 1 and 4 tokens go (17 -> 16 -> 12)."""
    P = _params(lam=(0.0, 0.0), attn_weight=0.0, budget=12)
    seq = _seq(np.zeros((1, 1, 16, 4)), [1] * 16)
    kn, vn = _zeros(P)
    res = MD.step(P, seq, 1, True, _q(P), kn, vn)
    assert res["evicted"] == [4, 3] and seq.n_tokens == 12


@pytest.mark.parametrize("L0", [4, 6])
def test_decoded_token_enters_at_full_structural_priority(L0):
    """A new token is inserted at t (t_ref = t_ins = t), so its prior term is
    b of the decode region, plus alpha (1 - rho) A_bar from this step; the
    same whether it opens a page (L0 = 4, pages of 4) or joins the partial
    last page (L0 = 6).  Uniform attention over L0 + 1 tokens."""
    P = _params(base=(1.0, 2.5))
    seq = _seq(np.zeros((1, 1, L0, 4)), [0] * L0)
    kn, vn = _zeros(P)
    res = MD.step(P, seq, 7, True, _q(P), kn, vn)
    assert res["t_ref"][L0] == 7
    assert res["s"][L0] == pytest.approx(2.5 + 0.5 * 0.1 * (1 / (L0 + 1)), rel=1e-12)
