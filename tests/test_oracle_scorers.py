"""Pins of the oracle's aggregation and weighting variants ("What Matters for
Aggressive Decoding-Time KV Eviction?", Sec. 3.1 Eqs. (2)-(4) and Appendix E
"Per-step scoring"), each against a closed form the pages' definitions fix:

  cumulative   m <- m + s, layer after layer: with two tokens and per-layer
               logits set by the query the state is m0 + the sum over layers
               of the logistic attention values, and a second step adds its
               own sum (nothing is forgotten);
  single-step  Eq. (2) is the EMA with alpha = 1: the state is the last
               layer's score;
  VNorm        each head's attention times ||v_i|| / mean_j ||v_j|| of its KV
               head: value rows of equal norm leave the scores unchanged; two
               tokens with norms a, b weight their attention by 2a/(a+b) and
               2b/(a+b);
  entropy      the layer's pooled score times the heads' mean entropy over
               ln L: a uniform distribution weighs 1 (scores unchanged), two
               tokens weigh the binary entropy of the logistic value over ln 2,
               a single cached token weighs 1.
"""
import math

import numpy as np
import pytest

import oracle as O
from workloads import f32_to_bf16_bits


def _bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _params(**kw):
    base = dict(n_layers=1, n_q_heads=1, n_kv_heads=1, head_dim=4, budget=8, alpha=0.05,
                beta=0.001)
    base.update(kw)
    return O.OracleParams(**base)


def _two_token_case(Ly, qvals, vrows=None, d=4):
    """Token 0 has key e_0; the new token (slot 1) has key 0; the query of
    layer l puts logit qvals[l] / 2 on token 0 (sqrt(d) = 2), so head h's
    attention to token 0 is the logistic of that logit."""
    K = np.zeros((Ly, 1, 1, d), np.float32)
    K[:, 0, 0, 0] = 1.0
    V = np.zeros((Ly, 1, 1, d), np.float32) if vrows is None else vrows[0]
    st = O.SequenceState.from_prefill(_bits(K), _bits(V), 1, 4)
    q = np.zeros((Ly, 1, d), np.float32)
    q[:, 0, 0] = qvals
    kn = np.zeros((Ly, 1, d), np.float32)
    vn = kn if vrows is None else vrows[1]
    return st, _bits(q), _bits(kn), _bits(vn)


def _logistic(x):
    return 1.0 / (1.0 + math.exp(-x))


def test_cumulative_sums_every_layer_and_step():
    Ly = 5
    qv = [2.0, -2.0, 4.0, 0.0, 6.0]
    P = _params(n_layers=Ly, aggregation=O.AGG_CUMULATIVE)
    st, q, kn, vn = _two_token_case(Ly, qv)
    st.m[0] = 0.25
    res, new = O.step(P, st, 1, True, q, kn, vn, 1)
    s0 = [_logistic(x / 2.0) for x in qv]
    assert res["m_upd"][0] == pytest.approx(0.25 + sum(s0), abs=1e-13)
    assert res["m_upd"][1] == pytest.approx(sum(1 - x for x in s0), abs=1e-13)
    # a second step over three tokens adds its own layer sums to the state
    res2, _ = O.step(P, new, 2, True, q, kn, vn, 2, want_probs=True)
    p2 = res2["probs"]                            # [Ly][Hq][3]
    for i in range(2):
        assert res2["m_upd"][i] == pytest.approx(res["m_upd"][i] + p2[:, 0, i].sum(), abs=1e-12)


def test_cumulative_differs_from_the_ema():
    Ly = 3
    st, q, kn, vn = _two_token_case(Ly, [1.0, 2.0, 3.0])
    r_ema, _ = O.step(_params(n_layers=Ly), st, 1, True, q, kn, vn, 1)
    r_cum, _ = O.step(_params(n_layers=Ly, aggregation=O.AGG_CUMULATIVE), st, 1, True, q, kn,
                      vn, 1)
    assert r_cum["m_upd"][0] > 5 * r_ema["m_upd"][0]


def test_single_step_is_the_ema_with_alpha_one():
    Ly = 4
    qv = [3.0, -1.0, 2.0, 5.0]
    st, q, kn, vn = _two_token_case(Ly, qv)
    st.m[0] = 0.9
    res, _ = O.step(_params(n_layers=Ly, alpha=1.0), st, 1, True, q, kn, vn, 1)
    assert res["m_upd"][0] == pytest.approx(_logistic(qv[-1] / 2.0), abs=1e-14)


def test_vnorm_equal_norms_change_nothing():
    """Value rows that are sign flips and permutations of one vector all
    have the same norm: every factor is 1."""
    rng = np.random.default_rng(4)
    Ly, Hq, Hkv, d, L0 = 2, 4, 2, 8, 9
    base = np.array([1.0, -2.0, 0.5, 3.0, 0.0, 1.5, -1.0, 2.0], np.float32)
    V = np.empty((Ly, Hkv, L0, d), np.float32)
    for idx in np.ndindex(Ly, Hkv, L0):
        V[idx] = rng.permutation(base) * rng.choice([-1.0, 1.0], size=d)
    K = rng.standard_normal((Ly, Hkv, L0, d)).astype(np.float32)
    q = _bits(rng.standard_normal((Ly, Hq, d)))
    kn = _bits(rng.standard_normal((Ly, Hkv, d)))
    vn = _bits(rng.permutation(base)[None, None, :].repeat(Ly, 0).repeat(Hkv, 1))
    out = []
    for w in (0, O.W_VNORM):
        P = _params(n_layers=Ly, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, weighting=w)
        st = O.SequenceState.from_prefill(_bits(K), _bits(V), L0, L0 + 2)
        out.append(O.step(P, st, 1, True, q, kn, vn, L0)[0]["m_upd"])
    assert np.allclose(out[0], out[1], atol=1e-15, rtol=1e-13)


def test_vnorm_two_tokens_weighted_by_their_norms():
    Ly, d = 1, 4
    v0 = np.zeros((Ly, 1, 1, d), np.float32)
    v0[..., :] = [3.0, 4.0, 0.0, 0.0]            # norm 5
    vn = np.zeros((Ly, 1, d), np.float32)
    vn[..., 0] = 1.0                              # norm 1
    st, q, kn, vb = _two_token_case(Ly, [2.0], vrows=(v0, vn))
    P = _params(n_layers=Ly, alpha=1.0, weighting=O.W_VNORM)
    res, _ = O.step(P, st, 1, True, q, kn, vb, 1)
    p0 = _logistic(1.0)
    assert res["m_upd"][0] == pytest.approx(p0 * 5 / 3.0, abs=1e-14)       # 2*5/(5+1)
    assert res["m_upd"][1] == pytest.approx((1 - p0) * 1 / 3.0, abs=1e-14)   # 2*1/(5+1)


def test_vnorm_follows_each_heads_kv_head():
    """Two KV heads whose value norms favour opposite tokens: the query
    heads of each group take their own KV head's factors."""
    Ly, Hq, Hkv, d = 1, 2, 2, 4
    K = np.zeros((Ly, Hkv, 1, d), np.float32)
    V = np.zeros((Ly, Hkv, 1, d), np.float32)
    V[0, 0, 0, 0], V[0, 1, 0, 0] = 3.0, 1.0       # token 0: norm 3 (head 0), 1 (head 1)
    vn = np.zeros((Ly, Hkv, d), np.float32)
    vn[0, 0, 0], vn[0, 1, 0] = 1.0, 3.0           # new token: norm 1 (head 0), 3 (head 1)
    st = O.SequenceState.from_prefill(_bits(K), _bits(V), 1, 4)
    z = np.zeros((Ly, Hq, d), np.float32)         # all logits 0: p = 1/2 everywhere
    P = _params(n_q_heads=Hq, n_kv_heads=Hkv, alpha=1.0, weighting=O.W_VNORM)
    res, _ = O.step(P, st, 1, True, _bits(z), _bits(np.zeros((Ly, Hkv, d))), _bits(vn), 1)
    # token 0: 0.5 * 3/2 (head 0) + 0.5 * 1/2 (head 1) = 1; token 1 the same by symmetry
    assert res["m_upd"][0] == pytest.approx(1.0, abs=1e-14)
    assert res["m_upd"][1] == pytest.approx(1.0, abs=1e-14)


def test_entropy_weight_is_one_for_uniform_attention():
    rng = np.random.default_rng(8)
    Ly, Hq, Hkv, d, L0 = 3, 4, 2, 8, 12
    krow = rng.standard_normal(d).astype(np.float32)
    K = np.broadcast_to(krow, (Ly, Hkv, L0, d)).copy()
    V = rng.standard_normal((Ly, Hkv, L0, d)).astype(np.float32)
    q = _bits(rng.standard_normal((Ly, Hq, d)))
    kn = _bits(np.broadcast_to(krow, (Ly, Hkv, d)).copy())
    vn = _bits(rng.standard_normal((Ly, Hkv, d)))
    out = []
    for w in (0, O.W_ENTROPY):
        P = _params(n_layers=Ly, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, weighting=w)
        st = O.SequenceState.from_prefill(_bits(K), _bits(V), L0, L0 + 2)
        out.append(O.step(P, st, 1, True, q, kn, vn, L0)[0]["m_upd"])
    assert np.allclose(out[0], out[1], atol=1e-15, rtol=1e-12)


def test_entropy_weight_of_two_tokens_is_the_binary_entropy():
    Ly = 3
    qv = [2.0, 8.0, -4.0]
    st, q, kn, vn = _two_token_case(Ly, qv)
    P = _params(n_layers=Ly, alpha=1.0, weighting=O.W_ENTROPY)
    res, _ = O.step(P, st, 1, True, q, kn, vn, 1)
    p = _logistic(qv[-1] / 2.0)
    h = -(p * math.log(p) + (1 - p) * math.log(1 - p)) / math.log(2.0)
    assert res["m_upd"][0] == pytest.approx(h * p, abs=1e-14)
    assert res["m_upd"][1] == pytest.approx(h * (1 - p), abs=1e-14)


def test_entropy_weight_of_a_single_token_is_one():
    P = _params(n_layers=2, alpha=1.0, weighting=O.W_ENTROPY | O.W_VNORM)
    st = O.SequenceState.from_prefill(np.zeros((2, 1, 0, 4), np.uint16),
                                      np.zeros((2, 1, 0, 4), np.uint16), 0, 4)
    z = np.zeros((2, 1, 4), np.uint16)
    res, _ = O.step(P, st, 1, True, z, z, z, 0)
    assert res["m_upd"][0] == pytest.approx(1.0, abs=1e-15)   # zero values: VNorm factor 1


def test_access_clock_reads_the_plain_attention():
    """The weightings change the score, not the access test: the clocks of a
    weighted step equal those of the plain one."""
    rng = np.random.default_rng(12)
    Ly, Hq, Hkv, d, L0 = 2, 4, 2, 8, 20
    K = rng.standard_normal((Ly, Hkv, L0, d)).astype(np.float32)
    V = (rng.standard_normal((Ly, Hkv, L0, d)) * rng.uniform(0.1, 3.0, (1, 1, L0, 1))).astype(
        np.float32)
    q = _bits(3 * rng.standard_normal((Ly, Hq, d)))
    kn, vn = _bits(rng.standard_normal((Ly, Hkv, d))), _bits(rng.standard_normal((Ly, Hkv, d)))
    acc = []
    for w in (0, O.W_VNORM | O.W_ENTROPY):
        P = _params(n_layers=Ly, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, weighting=w,
                    age_mode=O.AGE_SINCE_ACCESS)
        st = O.SequenceState.from_prefill(_bits(K), _bits(V), L0, L0 + 2)
        acc.append(O.step(P, st, 3, True, q, kn, vn, L0)[0]["accessed"])
    assert np.array_equal(acc[0], acc[1]) and 0 < acc[0].sum() < L0 + 1
