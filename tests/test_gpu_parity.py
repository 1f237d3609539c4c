"""GPU parity of the eviction pass against the fp64 oracle.

Every test runs the CUDA path through the C ABI (Python binding) and the
oracle from the same seeded prefill and inputs, free-running (it never
reads the device's state), and compares every step element by element
(tolerances in tests/parity.py); at a validated near tie the oracle follows
the device's admissible choice.
"""
import math

import numpy as np
import pytest

import oracle as O
from workloads import Geometry, Workload, llama8b_workload, tiny_workload

from parity import (access_alternative, boundary_check, compare_step, follow, load_prefill,
                    oracle_step, to_dev_bf16)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

AGE_NAMES = {O.AGE_SINCE_INSERT: kvev.KVEV_AGE_SINCE_INSERT,
             O.AGE_SINCE_ACCESS: kvev.KVEV_AGE_SINCE_ACCESS}
REFRESH = {"full": (O.REFRESH_FULL, kvev.KVEV_REFRESH_FULL),
           "lazy": (O.REFRESH_LAZY, kvev.KVEV_REFRESH_LAZY),
           "frozen": (O.REFRESH_FROZEN, kvev.KVEV_REFRESH_FROZEN)}


def run_parity(wl: Workload, budget: int, alpha: float, beta: float, steps: int, *,
               age_mode=O.AGE_SINCE_INSERT, refresh="full", period=8, pool_mean=False,
               max_ctx=None, check_every=1, aggregation=O.AGG_EMA, weighting=0,
               m_atol=None, diagnostics=False, fused=False):
    """`diagnostics`: the ranking counters and raw scores are gathered on
    the device every step and checked (check_diagnostics)."""
    g = wl.geom
    max_ctx = max_ctx or max(wl.L0 + steps + 1, budget + 1)
    mode_o, mode_d = REFRESH[refresh]
    ep = kvev.EvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch, max_ctx,
                           budget, alpha, beta, age_mode=AGE_NAMES[age_mode],
                           pool=kvev.KVEV_POOL_MEAN if pool_mean else kvev.KVEV_POOL_SUM,
                           refresh=mode_d, period=period,
                           aggregation={O.AGG_EMA: kvev.KVEV_AGG_EMA,
                                        O.AGG_CUMULATIVE: kvev.KVEV_AGG_CUMULATIVE}[aggregation],
                           weighting=((kvev.KVEV_W_VNORM if weighting & O.W_VNORM else 0) |
                                      (kvev.KVEV_W_ENTROPY if weighting & O.W_ENTROPY else 0)),
                           fused=fused)
    load_prefill(ep, wl)
    ep.begin(wl.L0)
    probs = torch.zeros((g.batch, g.n_layers, g.n_q_heads, max_ctx), dtype=torch.float32,
                        device="cuda")
    prio = torch.zeros((g.batch, max_ctx), dtype=torch.float32, device="cuda")
    kvev.kvev_set_debug(ep.ctx, probs, prio)
    counters = raw_dev = None
    if diagnostics:
        counters = torch.full((g.batch, kvev.KVEV_DIAG_FIELDS), -1, dtype=torch.int32,
                              device="cuda")
        raw_dev = torch.zeros((g.batch, max_ctx), dtype=torch.float32, device="cuda")
        kvev.kvev_set_diagnostics(ep.ctx, counters, raw_dev)
    prev_raw = [None] * g.batch          # positions of the last raw top-B set, its size
    P = O.OracleParams(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, budget, alpha, beta,
                       age_mode, pool_mean, aggregation, weighting)
    K, V = wl.prefill()
    states = [O.SequenceState.from_prefill(K[:, b], V[:, b], wl.L0, max_ctx)
              for b in range(g.batch)]
    del K, V
    totals = {"swaps": 0, "followed": 0, "out_rel": 0.0, "m_abs": 0.0, "p_rel": 0.0,
              "steps": 0}
    for t in range(1, steps + 1):
        L_prev = ep.length()
        check = (t - 1) % check_every == 0 or t == steps
        q, kn, vn = wl.step_inputs(t)
        ep.step(to_dev_bf16(q), to_dev_bf16(kn), to_dev_bf16(vn))
        kvev.kvev_sync(ep.ctx)
        refresh_now = O.is_refresh(mode_o, period, t)
        for b in range(g.batch):
            pre = states[b]
            assert pre.L == L_prev, "oracle and device cache lengths"
            res, new = oracle_step(P, pre, t, refresh_now, q[b], kn[b], vn[b], wl.L0 + t - 1,
                                   want_probs=check)
            if diagnostics:
                totals["diag_swaps"] = totals.get("diag_swaps", 0) + check_diagnostics(
                    res, ep, b, pre, budget, counters, raw_dev, prev_raw, refresh_now, t)
            alt, amb = access_alternative(res, pre, P) if refresh_now else (None, None)
            if check:
                st = compare_step(res, ep, b, pre, budget, probs, prio, refresh_now, alt,
                                  access_amb=amb, **({} if m_atol is None else {"m_atol": m_atol}))
                totals["swaps"] += st["swaps"]
                for k in ("out_rel", "m_abs", "p_rel"):
                    totals[k] = max(totals[k], st.get(k, 0.0))
                totals["steps"] += 1
            # continue the oracle along the device's choice where it was admissible
            n = int(ep.n_retained[b].item())
            kept = ep.retained[b, :n].cpu().numpy().astype(np.int64)
            t_ref_kept = res["t_ref_upd"][kept]
            if amb is not None and amb[kept].any():
                dev = ep.t_ref[b, :n].cpu().numpy().astype(np.int64)
                t_ref_kept = np.where(amb[kept], dev, t_ref_kept)
            if not np.array_equal(kept, res["retained"]) or \
                    not np.array_equal(t_ref_kept, res["t_ref_upd"][kept]):
                if not check:   # the choice is still checked for admissibility
                    compare_step(res, ep, b, pre, budget, None, prio, refresh_now, alt,
                                 access_amb=amb)
                new = follow(res, pre, kept, t_ref_kept)
                totals["followed"] += 1
            states[b] = new
        assert ep.length() == min(L_prev + 1, budget)
    kvev.kvev_check_scratch(ep.ctx)   # no scratch region overran its guard band
    ep.close()
    return totals


def check_diagnostics(res, ep, b, pre, budget, counters, raw_dev, prev_raw, refresh, t):
    """The device's ranking diagnostics of step t, sequence b: its raw
    scores against the oracle's (the head- and layer-summed probabilities,
    the probability tolerance), its raw top-B set (restated on the host from
    its own fp32 scores: the B largest, ties to the lower slot) admissible
    against the oracle's fp64 ranking, and its counters equal to the exact
    counts of its sets (oracle/diagnostics.py).  Returns the near-tie swaps
    of the raw set; updates prev_raw[b]."""
    from oracle import diagnostics as D
    L = res["L"]
    c = counters[b].cpu().numpy()
    n = int(ep.n_retained[b].item())
    kept = ep.retained[b, :n].cpu().numpy().astype(np.int64)
    pos = np.append(pre.pos[:L - 1], res["new_pos"])
    assert c[0] == t and c[1] == int(refresh)
    swaps = 0
    if refresh:
        raw = raw_dev[b, :L].cpu().numpy().astype(np.float64)
        ref = res["score_sum"]
        atol = 1e-9 * ep.layout.n_layers * ep.layout.n_q_heads   # the probabilities' own
        assert (np.abs(raw - ref) <= 2e-3 * ref + atol).all(), "raw scores"
        R = D.raw_topb(raw.astype(np.float32).astype(np.float64), budget)
        swaps = boundary_check(-ref, R, budget, 1e-5)
        prev = prev_raw[b]
        want = D.step_counts(R, kept, L, None if prev is None else prev[0],
                             0 if prev is None else prev[1], pos)
        prev_raw[b] = (pos[R], len(R))
    else:
        want = D.step_counts([], kept, L)
    got = dict(zip(kvev.DIAG_NAMES[2:], (int(x) for x in c[2:])))
    assert got == want, f"step {t}: counters {got} vs {want}"
    return swaps


def test_tiny_token_eviction_64_steps():
    """1 layer, 8 q / 2 KV heads, d 64, 512-token prefill with 8 heavy
    hitters, alpha 0.05, beta 0.001, budget 128, 64 full-refresh steps."""
    tot = run_parity(tiny_workload(0), 128, 0.05, 0.001, 64)
    print("tiny:", tot)
    assert tot["steps"] == 64


@pytest.mark.parametrize("refresh", ["full", "lazy", "frozen"])
@pytest.mark.parametrize("alpha", [0.01, 0.05, 0.15])
def test_llama_geometry_modes(refresh, alpha):
    """Llama-3.1-8B head geometry (32 q / 8 KV, d 128), 3 layers, 1000-token
    prefill (ragged last tile), 10% budget, access-clock ages, 12 steps in
    every refresh mode (lazy period 4 so non-refresh steps occur)."""
    wl = llama8b_workload(0, prefill_len=1000, n_layers=3, needle_period=5)
    tot = run_parity(wl, 100, alpha, 0.001, 12, age_mode=O.AGE_SINCE_ACCESS, refresh=refresh,
                     period=4)
    print(refresh, alpha, tot)


def test_batch_and_ragged_lengths():
    """Four sequences, prefill 47 (not a tile multiple), budget 20."""
    wl = Workload(Geometry(2, 8, 2, 128, 4), 47, seed=3, outliers=4, heavy=3)
    run_parity(wl, 20, 0.05, 0.001, 6)


@pytest.mark.parametrize("L0,budget", [(1, 1), (15, 8), (16, 8), (17, 16), (33, 40)])
def test_edge_lengths(L0, budget):
    """Tiny caches around the 16-token tile: single token, exact tile, one
    past a tile, and a budget larger than the cache (no eviction)."""
    wl = Workload(Geometry(2, 4, 1, 64, 1), L0, seed=L0, heavy=1)
    run_parity(wl, budget, 0.05, 0.001, 4)


@pytest.mark.parametrize("excess", [1, 2, 5, 8, 9, 12])
@pytest.mark.parametrize("beta", [0.0, 0.001])
def test_few_evictions_and_all_ties(excess, beta):
    """Step 1 evicts `excess` tokens (L0 + 1 - B): up to 8 go through the
    selection's block-maxima path, more through the radix select, and every
    later step evicts one.  beta = 0 makes every priority 0, so the tie rule
    alone decides (the lowest B slots are kept) and the device must take the
    oracle's set exactly at every step."""
    L0 = 200
    wl = Workload(Geometry(2, 8, 2, 64, 2), L0, seed=70 + excess, heavy=3)
    totals = run_parity(wl, L0 + 1 - excess, 0.05, beta, 3)
    if beta == 0.0:
        assert totals["followed"] == 0 and totals["swaps"] == 0


@pytest.mark.parametrize("d", [64, 128])
def test_eight_query_heads_per_kv_head(d):
    """Token mode with 8 query heads per KV head (16 q / 2 KV), both head
    sizes, two sequences, ragged prefill 260, access-clock ages."""
    wl = Workload(Geometry(2, 16, 2, d, 2), 260, seed=40 + d, outliers=2, heavy=3)
    run_parity(wl, 64, 0.05, 0.001, 5, age_mode=O.AGE_SINCE_ACCESS)


def test_beta_infinite_and_head_mean():
    """beta = +inf (rank by score, newest token protected) with head-mean
    pooling (Sec. 3.1 Eq. (1))."""
    wl = Workload(Geometry(2, 8, 2, 64, 1), 300, seed=11, heavy=4)
    run_parity(wl, 64, 0.2, math.inf, 5, pool_mean=True)


@pytest.mark.parametrize("aggregation,weighting", [
    (O.AGG_CUMULATIVE, 0), (O.AGG_EMA, O.W_VNORM), (O.AGG_EMA, O.W_ENTROPY),
    (O.AGG_EMA, O.W_VNORM | O.W_ENTROPY), (O.AGG_CUMULATIVE, O.W_VNORM | O.W_ENTROPY)])
def test_scorer_variants(aggregation, weighting):
    """The aggregation and weighting variants of the scorer (Sec. 3.1 Eqs.
    (3)-(4), Appendix E "Per-step scoring"): cumulative sums, VNorm value-norm
    factors, per-layer entropy weights, alone and together, on the
    Llama-3.1-8B head geometry (3 layers, ragged 1000-token prefill; N(0,1)
    value rows, whose norms differ by a few per cent), 10 steps with lazy
    refresh every 3 steps (the statistics are gathered on refresh steps
    only), access-clock ages."""
    wl = llama8b_workload(2, prefill_len=1000, n_layers=3, needle_period=4)
    tot = run_parity(wl, 100, 0.1, 0.001, 10, age_mode=O.AGE_SINCE_ACCESS, refresh="lazy",
                     period=3, aggregation=aggregation, weighting=weighting)
    print(aggregation, weighting, tot)


@pytest.mark.parametrize("weighting", [O.W_VNORM, O.W_ENTROPY])
def test_scorer_weightings_on_small_shapes(weighting):
    """Weightings with head_dim 64, 8 query heads per KV head, a ragged
    prefill, two sequences and head-mean pooling; and a single cached token
    (entropy weight 1)."""
    wl = Workload(Geometry(2, 16, 2, 64, 2), 77, seed=90 + weighting, heavy=2)
    run_parity(wl, 40, 0.2, 0.001, 5, weighting=weighting, pool_mean=True)
    wl1 = Workload(Geometry(1, 4, 1, 128, 1), 0, seed=5)
    run_parity(wl1, 2, 0.3, 0.001, 4, weighting=weighting)


@pytest.mark.parametrize("refresh", ["full", "lazy"])
def test_ranking_diagnostics(refresh):
    """The device's raw top-B / retained-set counters (Sec. 5.3, Appendix I
    Table 13) over 14 steps of the Llama-3.1-8B head geometry (3 layers,
    1000-token prefill, budget 100, a needle re-drawn every 5 steps), full
    refresh or lazy refresh every 3 steps (counts on the scoring steps only,
    the raw-set flags carried through the compactions in between)."""
    wl = llama8b_workload(0, prefill_len=1000, n_layers=3, needle_period=5)
    tot = run_parity(wl, 100, 0.05, 0.001, 14, age_mode=O.AGE_SINCE_ACCESS, refresh=refresh,
                     period=3, diagnostics=True)
    print(refresh, tot)


def test_ranking_diagnostics_tiny_and_below_budget():
    """The tiny workload (heavy hitters, 64 steps) and a cache that stays
    below the budget (the raw set is every token)."""
    run_parity(tiny_workload(0), 128, 0.05, 0.001, 64, diagnostics=True)
    wl = Workload(Geometry(2, 8, 2, 64, 2), 20, seed=9, heavy=2)
    run_parity(wl, 40, 0.05, 0.001, 6, diagnostics=True)


def test_probabilities_sum_to_one():
    """Device probabilities of every (layer, head) sum to 1 (fp32)."""
    wl = Workload(Geometry(2, 8, 2, 128, 1), 777, seed=5, outliers=4)
    g = wl.geom
    ep = kvev.EvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, 1, 800, 100, 0.05,
                           0.001)
    load_prefill(ep, wl)
    ep.begin(wl.L0)
    probs = torch.zeros((1, g.n_layers, g.n_q_heads, 800), device="cuda")
    kvev.kvev_set_debug(ep.ctx, probs, None)
    q, kn, vn = wl.step_inputs(1)
    ep.step(to_dev_bf16(q), to_dev_bf16(kn), to_dev_bf16(vn))
    kvev.kvev_sync(ep.ctx)
    s = probs[0, :, :, :778].sum(-1).cpu().numpy()
    assert np.allclose(s, 1.0, atol=1e-5)
    kvev.kvev_check_scratch(ep.ctx)   # no scratch region overran its guard band
    ep.close()


@pytest.mark.slow
def test_llama8b_32k_step1_full_size():
    """The full Llama-3.1-8B-shaped pass: 32 layers, 32 q / 8 KV heads, d 128,
    32768-token prefill + 1, budget 3277, alpha 0.05, beta 0.001, access
    clock; steps 1 and 2 against the oracle, element by element."""
    wl = llama8b_workload(0, prefill_len=32768)
    tot = run_parity(wl, 3277, 0.05, 0.001, 2, age_mode=O.AGE_SINCE_ACCESS, max_ctx=32768 + 64)
    print("llama8b 32k:", tot)


@pytest.mark.slow
@pytest.mark.parametrize("refresh", ["lazy", "frozen"])
def test_llama8b_32k_lazy_and_frozen_through_step_64(refresh):
    """The full Llama-3.1-8B-shaped pass over the horizon the refresh-mode
    measurements cover: 32768-token prefill, budget 3277, alpha 0.05, beta
    0.001, access clock, 64 steps with lazy refresh every 8 steps (refresh
    at t = 1, 9, ..., 57) or Score-Free (t = 1 only), through the needle
    re-draw at t = 51.  The oracle runs free beside the device on every
    step (and checks every admissible choice it follows); every 4th step
    and the last are compared element by element."""
    wl = llama8b_workload(0, prefill_len=32768)
    tot = run_parity(wl, 3277, 0.05, 0.001, 64, age_mode=O.AGE_SINCE_ACCESS, refresh=refresh,
                     period=8, max_ctx=32768 + 96, check_every=4)
    print(f"llama8b 32k {refresh} x 64:", tot)
    assert tot["steps"] == 17
