"""GPU parity of block-granular eviction with score persistence.

The CUDA path runs through the C ABI (kvev_paged_begin / kvev_paged_step /
kvev_readmit); the fp64 oracle (oracle/paged.py) runs free from the same
seeded prefill and inputs.  Per step and sequence the two are compared
element by element: attention outputs and probabilities (2e-3 relative),
block priorities and EMA scores (1e-5 absolute), the retained logical ids
(exact away from near ties), per-block clocks and lengths (exact), the K/V
of every live page (bit-exact) and the persisted score table (1e-5).  Where
a decision sits within rounding of a tie (a block's access on the 2/L
threshold, a swap at the budget boundary) the device's choice is checked to
be admissible and the oracle continues along it.
"""
import math

import numpy as np
import pytest

import oracle as O
from oracle import paged as PG
from workloads import Geometry, Workload, needle_blocks, paged_workload

from parity import M_ATOL, OUT_RTOL, P_ATOL, P_RTOL, PR_ATOL, boundary_check, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

PAGE = 16
AMB_REL = 1e-4


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def load_pool(pp, wl, nb0):
    """Prefill block j of sequence b into page b*pps + j and the backing tier."""
    K, V = wl.prefill()                       # [Ly][b][Hkv][L0][d]
    g = wl.geom
    for b in range(g.batch):
        for src, pool, back in ((K, pp.k_pool, pp.backing_k), (V, pp.v_pool, pp.backing_v)):
            x = src[:, b].reshape(g.n_layers, g.n_kv_heads, nb0, PAGE, g.head_dim)
            x = np.ascontiguousarray(x.transpose(2, 0, 1, 3, 4))
            xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
            pool[b * pp.pps:b * pp.pps + nb0].copy_(xt)
            back[b, :nb0].copy_(xt)


def check_pages(pp, b, seq, contents=True):
    """Block table, free stack and (`contents`) page contents of sequence b
    against the oracle's block list."""
    nb = int(pp.n_blocks[b])
    assert nb == len(seq.blocks), "live block count"
    table = pp.block_table[b, :nb].cpu().numpy()
    nf = int(pp.n_free[b])
    free = pp.free_pages[b, :nf].cpu().numpy()
    own = np.arange(b * pp.pps, (b + 1) * pp.pps)
    assert np.array_equal(np.sort(np.concatenate([table, free])), own), \
        "live and free pages must partition the sequence's pages"
    lens = pp.len[b, :nb].cpu().numpy()
    assert list(lens) == [blk.n for blk in seq.blocks], "block lengths"
    assert list(pp.lid[b, :nb].cpu().numpy()) == seq.lids(), "logical ids"
    if not contents:
        return
    for j, blk in enumerate(seq.blocks):
        kd = _bits(pp.k_pool[table[j], :, :, :blk.n])
        vd = _bits(pp.v_pool[table[j], :, :, :blk.n])
        assert np.array_equal(kd, blk.K), f"K of block {blk.lid}"
        assert np.array_equal(vd, blk.V), f"V of block {blk.lid}"


def check_state(pp, b, seq, amb_lids=()):
    nb = len(seq.blocks)
    m = pp.score[b, :nb].cpu().numpy().astype(np.float64)
    ref = np.array([blk.m for blk in seq.blocks])
    m_abs = float(np.abs(m - ref).max(initial=0.0))
    assert m_abs <= M_ATOL, "block EMA scores"
    assert list(pp.t_ins[b, :nb].cpu().numpy()) == [blk.t_ins for blk in seq.blocks], "t_ins"
    tref = pp.t_ref[b, :nb].cpu().numpy()
    for j, blk in enumerate(seq.blocks):
        if tref[j] != blk.t_ref:
            assert blk.lid in amb_lids, f"t_ref of block {blk.lid}: {tref[j]} vs {blk.t_ref}"
            blk.t_ref = int(tref[j])         # the other admissible access decision
    tab = pp.table[b].cpu().numpy().astype(np.float64)
    for lid in range(pp.table_len):
        if lid in seq.table:
            assert abs(tab[lid] - seq.table[lid]) <= M_ATOL, f"persisted score of {lid}"
        else:
            assert math.isnan(tab[lid]), f"table entry {lid} written without an eviction"
    return m_abs


def ambiguous_blocks(res, P):
    """Blocks whose access decision the fp32 device may take either way: a
    token within AMB_REL of the 2/L threshold and no token clearly above."""
    L = res["L"]
    mean = res["token_sum"] / (P.n_layers * P.n_q_heads)
    thr = 2.0 / L
    near = np.abs(mean - thr) <= AMB_REL * thr
    above = mean > thr * (1 + AMB_REL)
    nb = len(res["lids_before"])
    amb = np.zeros(nb, dtype=bool)
    for j in range(nb - 1):                  # the last block took the new token: accessed
        own = res["owner"] == j
        amb[j] = near[own].any() and not above[own].any()
    return amb


def step_and_compare(pp, P, seqs, b, t, ref_now, q, kn, vn, probs, prio, stats, full=True):
    """Run the oracle's step t on sequence b and compare the device's
    (`full`: the probabilities and every live page's K/V too; otherwise
    outputs, priorities, the kept set, block tables and per-block state)."""
    budget, beta, age_mode = P.budget, P.beta, P.age_mode
    pre = seqs[b].copy()
    res = PG.step(P, seqs[b], t, ref_now, q, kn, vn, want_probs=True)
    out = pp.out[b].cpu().numpy().astype(np.float64)
    err = np.abs(out - res["out"]).max(-1) / np.abs(res["out"]).max(-1)
    assert err.max() <= OUT_RTOL, f"step {t} seq {b}: output rel err {err.max():.2e}"
    stats["out_rel"] = max(stats["out_rel"], float(err.max()))
    # slot of every oracle token in the device's block-major layout
    owner = res["owner"]
    first = np.searchsorted(owner, np.arange(len(res["lids_before"])))
    slot = owner * PAGE + (np.arange(res["L"]) - first[owner])
    if ref_now and full:
        p = probs[b].cpu().numpy().astype(np.float64)[:, :, slot]
        bad = np.abs(p - res["probs"]) > P_RTOL * res["probs"] + P_ATOL
        assert not bad.any(), f"step {t} seq {b}: {bad.sum()} probabilities"
    nbb = len(res["lids_before"])
    pr = prio[b, :nbb].cpu().numpy().astype(np.float64)
    amb = ambiguous_blocks(res, P) if ref_now else np.zeros(nbb, dtype=bool)
    alt = res["priority"].copy()
    for j in np.nonzero(amb)[0] if age_mode == O.AGE_SINCE_ACCESS else []:
        blk_tref = pre.blocks[j].t_ref if j < len(pre.blocks) else t
        age = (t - blk_tref) if res["accessed"][j] else 0
        alt[j] = O.priority(res["m_upd"][j], age, beta)
    ok = (np.abs(pr - res["priority"]) <= PR_ATOL) | (amb & (np.abs(pr - alt) <= PR_ATOL))
    assert ok.all(), f"step {t} seq {b}: {(~ok).sum()} block priorities"
    n = int(pp.n_retained[b])
    kept_lids = list(pp.retained_lid[b, :n].cpu().numpy())
    if kept_lids != [res["lids_before"][j] for j in res["kept"]]:
        dev_slots = np.array([res["lids_before"].index(x) for x in kept_lids])
        stats["swaps"] += boundary_check(res["priority"], dev_slots, budget, PR_ATOL,
                                         alt if amb.any() else None)
        seqs[b] = pre.copy()        # continue along the device's admissible choice
        res = PG.step(P, seqs[b], t, ref_now, q, kn, vn, kept=dev_slots)
    stats["amb"] += int(amb.sum())
    amb_lids = {res["lids_before"][j] for j in np.nonzero(amb)[0]}
    check_pages(pp, b, seqs[b], contents=full)
    stats["m_abs"] = max(stats["m_abs"], check_state(pp, b, seqs[b], amb_lids))


def run_paged(wl, budget, alpha, beta, steps, *, pps, age_mode=O.AGE_SINCE_ACCESS,
              refresh=kvev.KVEV_REFRESH_FULL, refresh_o=O.REFRESH_FULL, period=1,
              pool_mean=False, readmit=None, persist=True, pinned_regions=None, labels=None,
              decode_region=0):
    """`pinned_regions` (per label) with `labels` [batch][L0]: LRFU scoring
    with a region table; blocks holding a pinned token are never evicted."""
    g = wl.geom
    nb0 = wl.L0 // PAGE
    regions = None
    if pinned_regions is not None:
        n = len(pinned_regions)
        regions = kvev.region_table([1.0] * n, [0.0] * n, pinned_regions,
                                    score_kind=kvev.KVEV_SCORE_LRFU, decode_region=decode_region)
    pp = kvev.PagedEvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch, pps,
                                PAGE, budget, alpha, beta, n_backing=nb0,
                                table_len=nb0 + steps // PAGE + 4,
                                age_mode=(kvev.KVEV_AGE_SINCE_ACCESS
                                          if age_mode == O.AGE_SINCE_ACCESS
                                          else kvev.KVEV_AGE_SINCE_INSERT),
                                pool=kvev.KVEV_POOL_MEAN if pool_mean else kvev.KVEV_POOL_SUM,
                                refresh=refresh, period=period, regions=regions)
    load_pool(pp, wl, nb0)
    if regions is not None:   # prefill block j of sequence b sits in page b * pps + j
        lab = torch.zeros((g.batch, pps * PAGE), dtype=torch.uint8)
        lab[:, :wl.L0] = torch.from_numpy(np.asarray(labels, dtype=np.uint8))
        pp.region.copy_(lab.reshape(-1))
    pp.begin(wl.L0)
    probs = torch.zeros((g.batch, g.n_layers, g.n_q_heads, pps * PAGE), device="cuda")
    prio = torch.zeros((g.batch, pps), device="cuda")
    kvev.kvev_set_debug(pp.ctx, probs, prio)
    K, V = wl.prefill()
    seqs = [PG.PagedSequence.from_prefill(K[:, b], V[:, b], PAGE,
                                          region=None if labels is None else labels[b],
                                          pinned_regions=pinned_regions,
                                          decode_region=decode_region)
            for b in range(g.batch)]
    P = O.OracleParams(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, budget, alpha, beta,
                       age_mode, pool_mean)
    stats = {"swaps": 0, "amb": 0, "readmitted": 0, "out_rel": 0.0, "m_abs": 0.0}
    for t in range(1, steps + 1):
        for (b, lid) in (readmit(t) if readmit else []):
            pp.readmit(b, lid, persist)
            stats["readmitted"] += int(PG.readmit(seqs[b], lid, t, persist))
        if readmit:
            kvev.kvev_sync(pp.ctx)
            for b in range(g.batch):
                check_pages(pp, b, seqs[b])
                check_state(pp, b, seqs[b])
        q, kn, vn = wl.step_inputs(t)
        pp.step(to_dev_bf16(q), to_dev_bf16(kn), to_dev_bf16(vn))
        kvev.kvev_sync(pp.ctx)
        ref_now = O.is_refresh(refresh_o, period, t)
        for b in range(g.batch):
            step_and_compare(pp, P, seqs, b, t, ref_now, q[b], kn[b], vn[b], probs, prio, stats)
    kvev.kvev_check_scratch(pp.ctx)   # no scratch region overran its guard band
    pp.close()
    return stats


def test_paged_small_full_refresh_with_readmission():
    """3 layers of the Llama-8B geometry, 3 sequences of 640 prefill tokens
    (40 blocks), budget 10 blocks, 40 steps (decode blocks open and fill),
    the needle blocks re-admitted when the needle set is re-drawn."""
    wl = paged_workload(1, prefill_len=640, n_layers=3, batch=3, needle_period=10)
    sched = lambda t: ([(b, int(x)) for b in range(3) for x in needle_blocks(wl, t, PAGE)]
                       if t > 1 and (t - 1) % 10 == 0 else [])
    st = run_paged(wl, 10, 0.05, 0.001, 40, pps=64, readmit=sched)
    print("paged:", st)
    assert st["readmitted"] > 0


def test_paged_persistence_off_and_lazy_refresh():
    """Persistence off (re-admitted blocks restart at score 0), lazy refresh
    every 4 steps, insertion ages, head-mean pooling."""
    wl = paged_workload(2, prefill_len=320, n_layers=2, batch=2, needle_period=6)
    sched = lambda t: ([(b, int(x)) for b in range(2) for x in needle_blocks(wl, t, PAGE)]
                       if t > 1 and (t - 1) % 6 == 0 else [])
    st = run_paged(wl, 6, 0.15, 0.001, 20, pps=40, age_mode=O.AGE_SINCE_INSERT,
                   refresh=kvev.KVEV_REFRESH_LAZY, refresh_o=O.REFRESH_LAZY, period=4,
                   pool_mean=True, readmit=sched, persist=False)
    print("paged lazy:", st)


@pytest.mark.parametrize("L0,budget", [(16, 1), (32, 2), (64, 8)])
def test_paged_edge_sizes(L0, budget):
    """One prefill block with a one-block budget; a budget at least the cache
    (nothing evicted until decoding opens blocks); d 64 geometry."""
    wl = Workload(Geometry(2, 8, 2, 64, 2), L0, seed=L0, heavy=1)
    run_paged(wl, budget, 0.05, 0.001, 20, pps=budget + 8)


def test_paged_many_sequences():
    """24 sequences (the selection then runs one CTA per sequence instead of
    a cluster per sequence), small geometry, 6 steps."""
    wl = Workload(Geometry(2, 8, 2, 64, 24), 96, seed=24, heavy=2)
    run_paged(wl, 3, 0.05, 0.001, 6, pps=12)


def test_paged_beta_infinite():
    wl = paged_workload(3, prefill_len=256, n_layers=2, batch=1, needle_period=50)
    run_paged(wl, 4, 0.2, math.inf, 6, pps=20)


def _labels(batch, L0, pinned_tokens):
    lab = np.zeros((batch, L0), dtype=np.uint8)
    for b, toks in enumerate(pinned_tokens):
        lab[b, list(toks)] = 1
    return lab


def test_paged_lrfu_with_pinned_regions():
    """LRFU block scoring with a region table: blocks holding a token of the
    pinned region 1 stay whatever their priority (one token of block 2 in
    sequence 0; blocks 12, 18 and 19 in sequence 1), the budget's other
    slots go by priority, and decoded tokens (region 0) are not pinned."""
    wl = paged_workload(4, prefill_len=320, n_layers=2, batch=2, needle_period=50)
    lab = _labels(2, 320, [[35], [200, *range(300, 311)]])
    st = run_paged(wl, 6, 0.05, 0.001, 12, pps=40, pinned_regions=(False, True), labels=lab)
    print("paged pinned:", st)


def test_paged_pinned_blocks_past_the_budget_and_a_pinned_decode_region():
    """More pinned blocks than the budget (5 under B = 2 in sequence 0): all
    stay and nothing else; with the decode region pinned too, every block
    opened by decoding stays as well (sequence 1 holds no pinned prefill)."""
    wl = paged_workload(5, prefill_len=160, n_layers=2, batch=2, needle_period=50)
    lab = _labels(2, 160, [[0, 20, 40, 60, 150], []])
    # a pinned decode region makes the host's page bound grow by one block per
    # step, so the pool holds the 10 prefill blocks plus one page per step
    st = run_paged(wl, 2, 0.05, 0.001, 20, pps=32, pinned_regions=(False, True), labels=lab,
                   decode_region=1)
    print("paged pinned past budget:", st)


@pytest.mark.slow
def test_paged_full_size_through_readmission():
    """The full block-granular workload on the device: 32 layers, 64
    sequences of 8192 tokens (512 blocks), budget 128 blocks, through step
    202: at t = 201 the needle is re-drawn and every sequence's new needle
    blocks are re-admitted from the backing tier with their persisted
    scores.  Sequences 0 and 63 run in the oracle beside the device on every
    step; outputs, block priorities, kept sets, block tables, per-block state
    and the persisted score table are compared on every step, the
    probabilities and every live page's K/V on steps 1, 2, every 25th, and
    199 to 202."""
    from workloads.device import PagedDeviceWorkload
    wl = PagedDeviceWorkload(0)
    Ly, b, nb0 = wl.n_layers, wl.batch, wl.n_blocks
    pps, budget, T = nb0 + 8, 128, 202
    pp = kvev.PagedEvictionPass(Ly, 32, 8, 128, b, pps, PAGE, budget, 0.05, 0.001,
                                n_backing=nb0, table_len=nb0,
                                age_mode=kvev.KVEV_AGE_SINCE_ACCESS)
    wl.fill(torch, pp.k_pool, pp.v_pool, pps, pp.backing_k, pp.backing_v)
    pp.begin(wl.prefill)
    probs = torch.zeros((b, Ly, 32, pps * PAGE), device="cuda")
    prio = torch.zeros((b, pps), device="cuda")
    kvev.kvev_set_debug(pp.ctx, probs, prio)
    sample = (0, b - 1)
    seqs = {}
    for s in sample:
        K = _bits(pp.backing_k[s, :nb0]).transpose(1, 2, 0, 3, 4).reshape(Ly, 8, -1, 128)
        V = _bits(pp.backing_v[s, :nb0]).transpose(1, 2, 0, 3, 4).reshape(Ly, 8, -1, 128)
        seqs[s] = PG.PagedSequence.from_prefill(np.ascontiguousarray(K),
                                                np.ascontiguousarray(V), PAGE)
    P = O.OracleParams(Ly, 32, 8, 128, budget, 0.05, 0.001, O.AGE_SINCE_ACCESS, False)
    stats = {"swaps": 0, "amb": 0, "out_rel": 0.0, "m_abs": 0.0, "readmitted": 0}
    for t in range(1, T + 1):
        if t > 1 and (t - 1) % wl.needle_period == 0:
            nd = wl.needle(t)
            for s in range(b):
                for lid in nd[s]:
                    pp.readmit(s, int(lid), True)
                    if s in seqs:
                        stats["readmitted"] += int(PG.readmit(seqs[s], int(lid), t, True))
            kvev.kvev_sync(pp.ctx)
            for s in sample:
                check_pages(pp, s, seqs[s])
                check_state(pp, s, seqs[s])
        q, kn, vn = wl.step_inputs(torch, t, pp.backing_k)
        pp.step(q, kn, vn)
        kvev.kvev_sync(pp.ctx)
        full = t <= 2 or t % 25 == 0 or t >= 199
        for s in sample:
            step_and_compare(pp, P, seqs, s, t, True, _bits(q[s]), _bits(kn[s]), _bits(vn[s]),
                             probs, prio, stats, full=full)
    print("paged full size through re-admission:", stats)
    assert stats["readmitted"] > 0
    kvev.kvev_check_scratch(pp.ctx)   # no scratch region overran its guard band
    pp.close()
