"""Pins for the fp64 oracle against what the pages and mathematics fix.

Each test ties one oracle function to something other than itself: values the
"ema-eviction" figure prints, closed forms (logistic function, geometric layer
weights), special cases, and brute force on tiny inputs.  A plausible mistake
in the oracle (a dropped term, a swapped EMA weight, a wrong GQA head index, a
missing 1/sqrt(d), a transposed PV product, an inverted selection order) fails
at least one of them.
"""
import itertools
import math
from decimal import ROUND_HALF_UP, Decimal

import numpy as np
import pytest

import oracle as O
from workloads import f32_to_bf16_bits


def _f(vals):
    return [float(x) for x in vals]


# ----------------------------------------------------------------- EMA rule
def test_ema_worked_row_exact_decimal_values(golden):
    """The EMA row of the figure, state 0, alpha 0.05.  Exact decimal values
    of the recurrence, worked by hand: 0.05*0.45 = 0.0225; 0.006 + 0.95*0.0225
    = 0.027375; 0.015 + 0.02600625; 0.004 + 0.0389559375; 0.0175 +
    0.040808140625."""
    alpha = float(golden["alpha"][0][0])
    xs = _f(golden["ema_inputs"][0])
    exact = [0.0225, 0.027375, 0.04100625, 0.0429559375, 0.058308140625]
    m = 0.0
    for x, e in zip(xs, exact):
        m = O.ema(m, x, alpha)
        assert abs(m - e) < 1e-15
    # the raw average the figure contrasts with
    assert abs(sum(xs) / len(xs) - float(golden["raw_average"][0][0])) < 1e-12


def test_ema_printed_row_is_the_rounded_chain(golden):
    """The printed row equals the chain that rounds the state to 3 decimals
    after every step (the figure's Calculation column multiplies 0.95 by the
    printed state), and the exact chain stays within the accumulated rounding
    bound sum_k 0.5e-3 * 0.95^k of it."""
    alpha = float(golden["alpha"][0][0])
    xs = _f(golden["ema_inputs"][0])
    printed = _f(golden["ema_printed"][0])
    m_r, m_x, bound = 0.0, 0.0, 0.0
    for x, p in zip(xs, printed):
        m_r = float(Decimal(repr(O.ema(m_r, x, alpha))).quantize(Decimal("0.001"), ROUND_HALF_UP))
        m_x = O.ema(m_x, x, alpha)
        bound = 0.5e-3 + (1 - alpha) * bound
        assert m_r == p
        assert abs(m_x - p) <= bound + 1e-12


def test_ema_weight_goes_to_the_new_observation():
    """alpha weights the new score: one step from 0 with input 1 gives alpha,
    not 1-alpha (the opposite convention of p1's Eq. 4 would give 0.95)."""
    assert O.ema(0.0, 1.0, 0.05) == pytest.approx(0.05, abs=1e-15)
    assert O.ema(1.0, 0.0, 0.05) == pytest.approx(0.95, abs=1e-15)


def test_half_life(golden):
    """ln 0.5 / ln 0.95 = 13.51 steps: a unit state with zero inputs is above
    one half after 13 updates and below it after 14."""
    alpha = float(golden["alpha"][0][0])
    hl = float(golden["half_life"][0][0])
    m = 1.0
    trace = []
    for _ in range(14):
        m = O.ema(m, 0.0, alpha)
        trace.append(m)
    assert trace[12] > 0.5 > trace[13]
    assert abs(math.log(0.5) / math.log(1 - alpha) - hl) < 0.05


# ------------------------------------------------------------ LRFU priority
def test_recency_decay_horizon(golden):
    beta = float(golden["beta"][0][0])
    for steps, printed in golden["recency"]:
        got = O.priority(0.0, int(steps), beta)
        assert abs(got - float(printed)) < 0.01
    # 1 - 1/e and 1 - 1/e^2 (closed forms)
    assert abs(O.priority(0.0, 1000, beta) - 0.6321205588285577) < 1e-12
    assert abs(O.priority(0.0, 2000, beta) - 0.8646647167633873) < 1e-12


def test_block_examples(golden):
    """Block A (score 0.059, 50 steps) -> 0.046, kept; block B (score 0.02,
    2000 steps) -> 0.848, evicted.  The page rounds the decay of B to 0.865
    before multiplying, so B is held to 1e-3, A to the 3-decimal rounding."""
    beta = float(golden["beta"][0][0])
    prs = []
    for name, score, steps, printed, fate in golden["block"]:
        pr = O.priority(float(score), int(steps), beta)
        tol = 5e-4 if name == "A" else 1e-3
        assert abs(pr - float(printed)) <= tol
        prs.append((name, pr, fate))
    kept = O.select(np.array([p for _, p, _ in prs]), 1)
    assert [prs[i][0] for i in kept] == [n for n, _, f in prs if f == "kept"]


def test_decision_matrix(golden):
    beta = float(golden["beta"][0][0])
    for score, steps, printed in golden["matrix"]:
        pr = O.priority(float(score), int(steps), beta)
        assert abs(pr - float(printed)) <= 5e-4 + 1e-12


def test_priority_special_cases():
    # steps 0: no decay, whatever beta (also beta = +inf)
    assert O.priority(0.3, 0, 0.001) == 0.0
    assert O.priority(0.3, 0, math.inf) == 0.0
    # beta = +inf, steps >= 1: priority is 1 - score (rank by score alone)
    assert O.priority(0.3, 1, math.inf) == pytest.approx(0.7, abs=1e-15)
    # score above 1 (head-summed probabilities) gives a negative priority
    assert O.priority(1.5, 10, 0.001) < 0.0
    # beta -> 0 removes the recency term: priority -> 0 from above
    assert 0.0 < O.priority(0.2, 5, 1e-9) < 1e-8


# --------------------------------------------------------------- attention
def _bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_attention_two_tokens_is_logistic():
    """Two positions: p_1 = 1 / (1 + exp(l_2 - l_1)).  Integer vectors keep
    every dot product exact; d = 4 so the scale is exactly 1/2."""
    q = _bits([[2, 1, 0, -1]])
    k = _bits([[[1, 0, 0, 0], [0, 3, 1, 0]]])           # dots 2 and 3
    v = _bits([[[1, 0, 0, 0], [0, 1, 0, 0]]])
    p, out = O.attention(q, k, v)
    l1, l2 = 2 / 2.0, 3 / 2.0
    p1 = 1.0 / (1.0 + math.exp(l2 - l1))
    assert p[0, 0] == pytest.approx(p1, abs=1e-15)
    assert p[0, 1] == pytest.approx(1 - p1, abs=1e-15)
    # V rows are unit vectors: the output is the probability vector itself
    assert out[0, :2] == pytest.approx([p1, 1 - p1], abs=1e-15)
    assert out[0, 2:] == pytest.approx([0, 0], abs=1e-15)


def test_attention_scale_is_inverse_sqrt_head_dim():
    for d in (4, 16, 64):
        q = np.zeros((1, d)); q[0, 0] = 4.0
        k = np.zeros((1, 2, d)); k[0, 0, 0] = 1.0     # dots 4 and 0
        v = np.zeros((1, 2, d))
        p, _ = O.attention(_bits(q), _bits(k), _bits(v))
        l1 = 4.0 / math.sqrt(d)
        assert p[0, 0] == pytest.approx(1 / (1 + math.exp(-l1)), abs=1e-14)


def test_attention_uniform_keys_give_uniform_weights_and_mean_value():
    rng = np.random.default_rng(5)
    L, d = 37, 16
    krow = rng.standard_normal(d)
    k = np.repeat(krow[None, None, :], L, axis=1)
    v = rng.standard_normal((1, L, d))
    q = rng.standard_normal((3, d))
    vb = _bits(v)
    p, out = O.attention(_bits(q), _bits(k), vb)
    assert np.allclose(p, 1.0 / L, atol=1e-15)
    vf = (vb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.allclose(out, vf[0].mean(axis=0)[None, :], atol=1e-14)


def test_attention_gqa_groups_are_contiguous():
    """8 query heads over 2 KV heads: heads 0-3 read KV head 0, heads 4-7 read
    KV head 1.  Each KV head's value rows are one constant, so the output of
    head h is that constant whatever the weights."""
    rng = np.random.default_rng(7)
    L, d = 9, 8
    k = rng.standard_normal((2, L, d))
    v = np.empty((2, L, d)); v[0] = 1.5; v[1] = -2.25
    q = rng.standard_normal((8, d))
    _, out = O.attention(_bits(q), _bits(k), _bits(v))
    assert np.allclose(out[:4], 1.5, atol=1e-14)
    assert np.allclose(out[4:], -2.25, atol=1e-14)


def test_attention_probabilities_sum_to_one_and_pick_the_matching_key():
    rng = np.random.default_rng(11)
    L, d = 50, 32
    k = rng.standard_normal((2, L, d))
    q = rng.standard_normal((4, d))
    q[1] = 40.0 * k[0, 17]          # head 1 (KV head 0) locks onto key 17
    q[3] = 40.0 * k[1, 3]           # head 3 (KV head 1) locks onto key 3
    p, _ = O.attention(_bits(q), _bits(k), _bits(rng.standard_normal((2, L, d))))
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-13)
    assert (p >= 0).all()
    assert p[1].argmax() == 17 and p[1, 17] > 0.999
    assert p[3].argmax() == 3 and p[3, 3] > 0.999


# --------------------------------------------------------------- selection
def test_selection_matches_brute_force_on_tiny_inputs():
    """The kept set is the unique B-subset whose every (priority, index) key
    is below every evicted key; enumerated over all subsets."""
    rng = np.random.default_rng(3)
    for trial in range(200):
        L = int(rng.integers(1, 8))
        pr = rng.choice([-0.5, 0.0, 0.1, 0.1, 0.3, 0.7], size=L)
        B = int(rng.integers(0, L + 2))
        kept = O.select(pr, B)
        n = min(B, L)
        keys = [(pr[i], i) for i in range(L)]
        valid = [S for S in itertools.combinations(range(L), n)
                 if all(keys[a] < keys[b] for a in S for b in range(L) if b not in S)]
        assert len(valid) == 1
        assert list(kept) == list(valid[0])     # ascending order too


def test_selection_ties_go_to_the_lower_index():
    kept = O.select(np.zeros(10), 4)
    assert list(kept) == [0, 1, 2, 3]


def test_selection_pinned_units_are_forced_in():
    pr = np.array([0.9, 0.1, 0.8, 0.2, 0.95])
    kept = O.select(pr, 2, pinned=np.array([1, 0, 0, 0, 1]))
    assert list(kept) == [0, 4]
    # forced in even past the budget: three pinned units under B = 2 are all
    # kept, and nothing else
    kept = O.select(pr, 2, pinned=np.array([1, 0, 1, 0, 1]))
    assert list(kept) == [0, 2, 4]


def test_beta_infinite_reduces_to_lowest_score_eviction():
    """beta = +inf: every token older than 0 steps has priority 1 - m, so the
    kept set is the B highest m (ties to the lower index), and a token of age
    0 is always kept (p1 Sec. 3.1 evicts the lowest m)."""
    rng = np.random.default_rng(9)
    m = rng.choice([0.1, 0.2, 0.2, 0.5, 0.9], size=20)
    ages = np.ones(20, dtype=np.int64); ages[-1] = 0
    pr = np.array([O.priority(mi, a, math.inf) for mi, a in zip(m, ages)])
    kept = O.select(pr, 6)
    order = sorted(range(19), key=lambda i: (-m[i], i))
    assert list(kept) == sorted(order[:5] + [19])


# ------------------------------------------------------------------- steps
def _small_params(**kw):
    base = dict(n_layers=1, n_q_heads=1, n_kv_heads=1, head_dim=4, budget=8,
                alpha=0.05, beta=0.001)
    base.update(kw)
    return O.OracleParams(**base)


def _empty_state(Ly, Hkv, cap, d):
    return O.SequenceState.from_prefill(np.zeros((Ly, Hkv, 0, d), np.uint16),
                                        np.zeros((Ly, Hkv, 0, d), np.uint16), 0, cap)


def test_layer_sequential_ema_closed_form_single_token():
    """One cached token attends only to itself: s = 1 in every layer, so the
    state after K layers is 1 - (1 - alpha)^K from m0 = 0 (p1 Appendix E: the
    prior state has weight (1-alpha)^K, layer l has alpha (1-alpha)^(K-l))."""
    for Ly, alpha in ((1, 0.05), (5, 0.05), (32, 0.15)):
        P = _small_params(n_layers=Ly, alpha=alpha)
        st = _empty_state(Ly, 1, 4, 4)
        z = np.zeros((Ly, 1, 4), np.uint16)
        res, _ = O.step(P, st, 1, True, z, z, z, 0)
        assert res["m_upd"][0] == pytest.approx(1 - (1 - alpha) ** Ly, abs=1e-14)


def test_layer_sequential_ema_matches_geometric_layer_weights():
    """Two tokens, per-layer logits set by the query: s_l(i) is a logistic
    value per layer, and the final state is (1-a)^K m0 + sum_l a (1-a)^(K-1-l)
    s_l (layers numbered from 0)."""
    Ly, alpha, d = 6, 0.3, 4
    P = _small_params(n_layers=Ly, alpha=alpha, head_dim=d)
    K = np.zeros((Ly, 1, 1, d), np.float32); K[:, 0, 0, 0] = 1.0   # token 0 key
    st = O.SequenceState.from_prefill(_bits(K), _bits(np.zeros_like(K)), 1, 4)
    st.m[0] = 0.4
    q = np.zeros((Ly, 1, d), np.float32)
    q[:, 0, 0] = [2, -2, 4, 0, 6, -4]             # logit of token 0: q0/2
    kn = np.zeros((Ly, 1, d), np.float32)         # new token: logit 0
    res, _ = O.step(P, st, 1, True, _bits(q), _bits(kn), _bits(kn), 1)
    s0 = [1 / (1 + math.exp(-x / 2.0)) for x in q[:, 0, 0]]
    want0 = (1 - alpha) ** Ly * 0.4 + sum(alpha * (1 - alpha) ** (Ly - 1 - l) * s0[l]
                                          for l in range(Ly))
    want1 = sum(alpha * (1 - alpha) ** (Ly - 1 - l) * (1 - s0[l]) for l in range(Ly))
    assert res["m_upd"][0] == pytest.approx(want0, abs=1e-14)
    assert res["m_upd"][1] == pytest.approx(want1, abs=1e-14)


def test_head_pooling_sum_and_mean():
    """Sum over query heads (the eviction configurations) vs the head mean of
    p1 Eq. (1): with one token every head gives p = 1, so s = Hq or 1."""
    for pool_mean, want in ((False, 4.0), (True, 1.0)):
        P = _small_params(n_q_heads=4, n_kv_heads=2, alpha=1.0, pool_mean=pool_mean)
        st = _empty_state(1, 2, 4, 4)
        res, _ = O.step(P, st, 1, True, np.zeros((1, 4, 4), np.uint16),
                        np.zeros((1, 2, 4), np.uint16), np.zeros((1, 2, 4), np.uint16), 0)
        assert res["m_upd"][0] == pytest.approx(want, abs=1e-15)


def _random_state(rng, Ly, Hkv, L0, cap, d):
    K = _bits(rng.standard_normal((Ly, Hkv, L0, d)))
    V = _bits(rng.standard_normal((Ly, Hkv, L0, d)))
    st = O.SequenceState.from_prefill(K, V, L0, cap)
    st.m[:L0] = rng.uniform(0, 0.5, L0)
    return st


def test_non_refresh_step_freezes_state_and_new_token_takes_the_mean():
    rng = np.random.default_rng(21)
    Ly, Hq, Hkv, d, L0 = 2, 4, 2, 8, 12
    P = _small_params(n_layers=Ly, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, budget=20)
    st = _random_state(rng, Ly, Hkv, L0, 16, d)
    q = _bits(rng.standard_normal((Ly, Hq, d)))
    kn = _bits(rng.standard_normal((Ly, Hkv, d)))
    res, new = O.step(P, st, 5, False, q, kn, kn, L0)
    assert np.array_equal(res["m_upd"][:L0], st.m[:L0])
    assert res["m_upd"][L0] == pytest.approx(np.mean(st.m[:L0]), abs=1e-15)
    assert not res["accessed"].any()
    # the attention output is still produced on non-refresh steps
    assert np.abs(res["out"]).sum() > 0


def test_refresh_schedules():
    assert [t for t in range(1, 30) if O.is_refresh(O.REFRESH_LAZY, 8, t)] == [1, 9, 17, 25]
    assert [t for t in range(1, 6) if O.is_refresh(O.REFRESH_FROZEN, 0, t)] == [1]
    assert all(O.is_refresh(O.REFRESH_FULL, 0, t) for t in range(1, 6))


def test_access_clock_threshold():
    """Uniform attention over L tokens (1/L each) is below the threshold 2/L;
    a token taking almost all the mass is above it and its clock resets."""
    d, L0 = 4, 7
    P = _small_params(n_q_heads=2, n_kv_heads=1, head_dim=d, budget=100,
                      age_mode=O.AGE_SINCE_ACCESS)
    K = np.zeros((1, 1, L0, d), np.float32)
    st = O.SequenceState.from_prefill(_bits(K), _bits(K), L0, 16)
    z = np.zeros((1, 1, d), np.uint16)
    res, _ = O.step(P, st, 3, True, np.zeros((1, 2, d), np.uint16), z, z, L0)
    assert not res["accessed"][:L0].any()           # all 8 tokens get 1/8 < 2/8
    K[0, 0, 2, 0] = 30.0
    st = O.SequenceState.from_prefill(_bits(K), _bits(K), L0, 16)
    q = np.zeros((1, 2, d), np.float32); q[0, :, 0] = 4.0
    res, new = O.step(P, st, 3, True, _bits(q), z, z, L0)
    assert list(np.nonzero(res["accessed"])[0]) == [2]
    assert res["t_ref_upd"][2] == 3 and res["t_ref_upd"][0] == 0
    assert res["priority"][2] == 0.0                # age 0 after the reset


def test_access_threshold_is_inclusive():
    """Attention of exactly 2/L resets the clock (>=): one prefill token and
    the new one (L = 2, threshold 1), logits 100 and 0, so the prefill token
    takes probability exactly 1.0 in fp64 (1 + e^-100 rounds to 1)."""
    d = 16
    P = _small_params(n_q_heads=1, n_kv_heads=1, head_dim=d, budget=100,
                      age_mode=O.AGE_SINCE_ACCESS)
    K = np.zeros((1, 1, 1, d), np.float32)
    K[0, 0, 0, 0] = 40.0
    st = O.SequenceState.from_prefill(_bits(K), _bits(K), 1, 4)
    q = np.zeros((1, 1, d), np.float32); q[0, 0, 0] = 10.0      # logit 10 * 40 / 4
    z = np.zeros((1, 1, d), np.uint16)
    res, _ = O.step(P, st, 5, True, _bits(q), z, z, 1)
    assert res["score_sum"][0] == 1.0
    assert bool(res["accessed"][0]) and res["t_ref_upd"][0] == 5


def test_step_age_since_insertion_and_budget():
    """Step 1 after a prefill inserted at step 0: every prefill token has age
    1, so the priority order is the m order; the new token has age 0 and
    priority 0 and is kept."""
    rng = np.random.default_rng(2)
    Ly, Hq, Hkv, d, L0, B = 1, 2, 1, 8, 30, 10
    P = _small_params(n_layers=Ly, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, budget=B)
    st = _random_state(rng, Ly, Hkv, L0, 40, d)
    q = _bits(rng.standard_normal((Ly, Hq, d)))
    kn = _bits(rng.standard_normal((Ly, Hkv, d)))
    res, new = O.step(P, st, 1, True, q, kn, kn, L0)
    m = res["m_upd"]
    assert res["priority"][L0] == 0.0
    expect = sorted(sorted(range(L0), key=lambda i: (-m[i], i))[:B - 1] + [L0])
    assert list(res["retained"]) == expect
    assert new.L == B


def test_compaction_moves_retained_rows_in_order():
    rng = np.random.default_rng(4)
    Ly, Hq, Hkv, d, L0, B = 2, 4, 2, 8, 25, 7
    P = _small_params(n_layers=Ly, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, budget=B)
    st = _random_state(rng, Ly, Hkv, L0, 32, d)
    q = _bits(rng.standard_normal((Ly, Hq, d)))
    kn = _bits(rng.standard_normal((Ly, Hkv, d)))
    vn = _bits(rng.standard_normal((Ly, Hkv, d)))
    res, new = O.step(P, st, 1, True, q, kn, vn, 99)
    r = res["retained"]
    Kfull = st.K.copy(); Kfull[:, :, L0] = kn
    Vfull = st.V.copy(); Vfull[:, :, L0] = vn
    assert np.array_equal(new.K[:, :, :B], Kfull[:, :, r])
    assert np.array_equal(new.V[:, :, :B], Vfull[:, :, r])
    posfull = np.append(st.pos[:L0], 99)
    assert np.array_equal(new.pos[:B], posfull[r])
    assert np.array_equal(new.m[:B], res["m_upd"][r])


def test_no_eviction_below_budget():
    rng = np.random.default_rng(8)
    P = _small_params(n_q_heads=2, n_kv_heads=1, head_dim=8, budget=50)
    st = _random_state(rng, 1, 1, 10, 16, 8)
    z = _bits(rng.standard_normal((1, 1, 8)))
    res, new = O.step(P, st, 1, True, _bits(rng.standard_normal((1, 2, 8))), z, z, 10)
    assert list(res["retained"]) == list(range(11)) and new.L == 11


def test_threads_leave_every_result_bit_identical():
    """The oracle's attention may run its query heads on several host
    threads; each head's arithmetic is unchanged, so a step's outputs,
    probabilities, scores, priorities and kept set are identical bit for
    bit on one thread and on four."""
    from workloads import Geometry, Workload
    wl = Workload(Geometry(2, 8, 2, 64, 1), 300, seed=77, heavy=3)
    K, V = wl.prefill()
    q, kn, vn = wl.step_inputs(1)
    P = O.OracleParams(2, 8, 2, 64, 50, 0.05, 0.001, O.AGE_SINCE_ACCESS)
    runs = []
    for n in (1, 4):
        O.set_threads(n)
        st = O.SequenceState.from_prefill(K[:, 0], V[:, 0], 300, 310)
        res, _ = O.step(P, st, 1, True, q[0], kn[0], vn[0], 300)
        runs.append(res)
    O.set_threads(0)
    for key in ("out", "probs", "m_upd", "priority", "retained"):
        assert np.array_equal(runs[0][key], runs[1][key]), key
