"""Pins for the block-granular (paged) oracle with score persistence."""
import math

import numpy as np
import pytest

import oracle as O
from oracle import paged as PG
from workloads import f32_to_bf16_bits


def _bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _params(**kw):
    base = dict(n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=8, budget=6, alpha=0.05,
                beta=0.001, age_mode=O.AGE_SINCE_ACCESS)
    base.update(kw)
    return O.OracleParams(**base)


@pytest.mark.parametrize("refresh_pattern", [(True, True, True, True), (True, False, False, True)])
def test_one_token_pages_reduce_to_the_token_oracle(refresh_pattern):
    """With 1-token blocks the max over a block's tokens is the token's own
    score, so every step must equal the (pinned) token-granular oracle:
    same attention, scores, priorities and kept set."""
    rng = np.random.default_rng(1)
    P = _params(budget=7)
    Ly, Hkv, d, L0 = P.n_layers, P.n_kv_heads, P.head_dim, 10
    K = _bits(rng.standard_normal((Ly, Hkv, L0, d)))
    V = _bits(rng.standard_normal((Ly, Hkv, L0, d)))
    seq = PG.PagedSequence.from_prefill(K, V, 1)
    st = O.SequenceState.from_prefill(K, V, L0, 32)
    for t, refresh in enumerate(refresh_pattern, start=1):
        q = _bits(rng.standard_normal((Ly, P.n_q_heads, d)))
        kn = _bits(rng.standard_normal((Ly, Hkv, d)))
        vn = _bits(rng.standard_normal((Ly, Hkv, d)))
        res_t, st = O.step(P, st, t, refresh, q, kn, vn, L0 + t - 1)
        res_p = PG.step(P, seq, t, refresh, q, kn, vn)
        assert np.allclose(res_p["out"], res_t["out"], atol=1e-14)
        assert np.allclose(res_p["m_upd"], res_t["m_upd"], atol=1e-14)
        assert np.allclose(res_p["priority"], res_t["priority"], atol=1e-15)
        assert list(res_p["kept"]) == list(res_t["retained"])
        assert [b.lid for b in seq.blocks] == list(st.pos[:st.L])


def test_block_score_is_the_max_over_its_tokens():
    """Two 2-token blocks, one layer, one head: the new score of a block is
    alpha times the larger of its tokens' probabilities (logistic closed
    forms from integer logits)."""
    P = _params(n_layers=1, n_q_heads=1, n_kv_heads=1, head_dim=4, budget=10, alpha=0.5,
                age_mode=O.AGE_SINCE_INSERT)
    K = np.zeros((1, 1, 4, 4), np.float32)
    K[0, 0, :, 0] = [2, 0, 4, 2]                  # logits q0*k/2 with q0 = 1 -> 1, 0, 2, 1
    seq = PG.PagedSequence.from_prefill(_bits(K), _bits(np.zeros_like(K)), 2)
    q = np.zeros((1, 1, 4), np.float32); q[0, 0, 0] = 1.0
    z = np.zeros((1, 1, 4), np.float32)
    res = PG.step(P, seq, 1, True, _bits(q), _bits(z), _bits(z))
    logits = np.array([1, 0, 2, 1, 0])            # + the new token (logit 0)
    p = np.exp(logits) / np.exp(logits).sum()
    assert res["m_upd"][0] == pytest.approx(0.5 * max(p[0], p[1]), abs=1e-15)
    assert res["m_upd"][1] == pytest.approx(0.5 * max(p[2], p[3]), abs=1e-15)
    assert res["m_upd"][2] == pytest.approx(0.5 * p[4], abs=1e-15)   # the opened block
    assert [b.n for b in seq.blocks] == [2, 2, 1]


def _random_seq(rng, P, L0, page):
    K = _bits(rng.standard_normal((P.n_layers, P.n_kv_heads, L0, P.head_dim)))
    V = _bits(rng.standard_normal((P.n_layers, P.n_kv_heads, L0, P.head_dim)))
    return PG.PagedSequence.from_prefill(K, V, page)


def _inputs(rng, P):
    q = _bits(rng.standard_normal((P.n_layers, P.n_q_heads, P.head_dim)))
    kn = _bits(rng.standard_normal((P.n_layers, P.n_kv_heads, P.head_dim)))
    vn = _bits(rng.standard_normal((P.n_layers, P.n_kv_heads, P.head_dim)))
    return q, kn, vn


def test_persistence_restores_the_evicted_score_exactly():
    """p4: an evicted block's identity key and score persist and come back on
    re-admission (not reset to 0); with persistence off it comes back at 0."""
    rng = np.random.default_rng(4)
    P = _params(budget=3)
    seq = _random_seq(rng, P, 32, 4)              # 8 prefill blocks
    res = PG.step(P, seq, 1, True, *_inputs(rng, P))
    ev = res["evicted_lids"]
    assert len(ev) == 9 - 3
    prefill_ev = [lid for lid in ev if lid < 8]
    lid = prefill_ev[0]
    j = res["lids_before"].index(lid)
    stored = seq.table[lid]
    assert stored == res["m_upd"][j]
    other = seq.copy()
    assert PG.readmit(seq, lid, 2, persist=True)
    blk = [b for b in seq.blocks if b.lid == lid][0]
    assert blk.m == stored and blk.t_ref == 2
    assert PG.readmit(other, lid, 2, persist=False)
    assert [b for b in other.blocks if b.lid == lid][0].m == 0.0
    # the block's contents come back bit for bit from the backing tier
    assert np.array_equal(blk.K, seq.backing_K[lid]) and np.array_equal(blk.V, seq.backing_V[lid])


def test_readmit_keeps_slot_order_and_is_a_noop_when_resident():
    rng = np.random.default_rng(6)
    P = _params(budget=4)
    seq = _random_seq(rng, P, 40, 4)              # 10 prefill blocks
    PG.step(P, seq, 1, True, *_inputs(rng, P))
    resident = seq.lids()
    assert not PG.readmit(seq, resident[0], 2)
    missing = [lid for lid in range(10) if lid not in resident]
    for lid in missing[:3]:
        assert PG.readmit(seq, lid, 2)
    assert seq.lids() == sorted(seq.lids())


def test_budget_counts_blocks_and_open_block_fills_first():
    """Tokens fill the open block before a new one opens; the cache never
    holds more than B blocks after a step."""
    rng = np.random.default_rng(8)
    P = _params(budget=5)
    seq = _random_seq(rng, P, 24, 4)              # 6 prefill blocks
    for t in range(1, 7):
        PG.step(P, seq, t, True, *_inputs(rng, P))
        assert len(seq.blocks) <= 5
    decode = [b for b in seq.blocks if b.lid >= 6]
    assert all(b.n <= 4 for b in decode)
    assert seq.next_lid >= 7


def test_appending_into_the_open_block_is_an_access():
    """Insertion counts as an access: the decode block opened at step 1 takes
    the token of step 2 (a non-refresh step, so no attention decides any
    access) and its clock moves to 2 (age 0, priority 0), while the prefill
    blocks keep the clock of their insertion (step 0)."""
    rng = np.random.default_rng(3)
    P = _params(n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=4, budget=10)
    seq = _random_seq(rng, P, 8, 4)                # 2 prefill blocks
    PG.step(P, seq, 1, True, *_inputs(rng, P))     # opens block 2
    res = PG.step(P, seq, 2, False, *_inputs(rng, P))
    assert [b.n for b in seq.blocks] == [4, 4, 2]
    assert not res["accessed"].any()
    assert [b.t_ref for b in seq.blocks] == [0, 0, 2]
    assert res["priority"][2] == 0.0 and (res["priority"][:2] != 0.0).all()


def test_block_access_when_any_member_token_is_accessed():
    """A block whose one token takes almost all the attention is accessed
    (its clock resets, priority 0); blocks of uniform tokens are not."""
    P = _params(n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=4, budget=10)
    K = np.zeros((1, 1, 8, 4), np.float32)
    K[0, 0, 5, 0] = 30.0
    seq = PG.PagedSequence.from_prefill(_bits(K), _bits(K), 4)
    q = np.zeros((1, 2, 4), np.float32); q[0, :, 0] = 4.0
    z = np.zeros((1, 1, 4), np.float32)
    res = PG.step(P, seq, 3, True, _bits(q), _bits(z), _bits(z))
    assert list(res["accessed"]) == [False, True, False]  # block 1 holds token 5
    assert res["priority"][1] == 0.0 and res["priority"][0] > 0.0
    assert res["priority"][2] == 0.0                       # opened this step: age 0


def _pinned_seq(rng, P, L0, page, region, pinned_regions, decode_region=0, zero_blocks=()):
    K = rng.standard_normal((P.n_layers, P.n_kv_heads, L0, P.head_dim))
    for j in zero_blocks:                          # keys of 0: logits 0, the smallest block max
        K[:, :, j * page:(j + 1) * page] = 0.0
    V = rng.standard_normal((P.n_layers, P.n_kv_heads, L0, P.head_dim))
    return PG.PagedSequence.from_prefill(_bits(K), _bits(V), page, region=region,
                                         pinned_regions=pinned_regions,
                                         decode_region=decode_region)


def test_a_block_with_a_pinned_token_is_never_evicted():
    """MemDecay Sec. III-A / IV-A under LRFU: one token of block 0 is in a
    pinned region, so block 0 survives although its priority is the highest
    (its keys are 0, its block max the smallest); the other slot goes to
    the lowest priority (the new block, age 0; ages since insertion, so every
    prefill block is one step old)."""
    rng = np.random.default_rng(11)
    P = _params(n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=8, budget=2,
                age_mode=O.AGE_SINCE_INSERT)
    region = np.zeros(16, dtype=np.int64)
    region[2] = 1
    seq = _pinned_seq(rng, P, 16, 4, region, (False, True), zero_blocks=(0,))
    res = PG.step(P, seq, 1, True, *_inputs(rng, P))
    assert list(res["pinned"]) == [1, 0, 0, 0, 0]
    assert int(np.argmax(res["priority"])) == 0      # unpinned, block 0 would go first
    assert 0 not in O.select(res["priority"], 2)
    assert seq.lids() == [0, 4]


def test_pinned_blocks_past_the_budget_are_all_kept():
    """Forced in even past the budget: three pinned blocks under B = 2 stay,
    and nothing else does (not even the new block of priority 0)."""
    rng = np.random.default_rng(12)
    P = _params(n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=8, budget=2)
    region = np.repeat([1, 0, 1, 1], 4)
    seq = _pinned_seq(rng, P, 16, 4, region, (False, True))
    res = PG.step(P, seq, 1, True, *_inputs(rng, P))
    assert res["priority"][4] == 0.0
    assert seq.lids() == [0, 2, 3]


def test_decoded_tokens_take_the_decode_region():
    """With a pinned decode region every block opened by decoding is pinned:
    under B = 1 they accumulate while the prefill blocks go."""
    rng = np.random.default_rng(13)
    P = _params(n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=8, budget=1)
    seq = _pinned_seq(rng, P, 8, 2, np.zeros(8, dtype=np.int64), (False, True), decode_region=1)
    for t in range(1, 6):
        PG.step(P, seq, t, True, *_inputs(rng, P))
    assert seq.lids() == [4, 5, 6]                   # tokens 1-2, 3-4 and 5 of decoding
    assert [b.region.tolist() for b in seq.blocks] == [[1, 1], [1, 1], [1]]
    with pytest.raises(ValueError):
        PG.readmit(seq, 0, 6)
