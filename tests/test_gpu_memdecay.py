"""GPU parity of region-aware page eviction (MemDecay) against the oracle.

The CUDA path runs through the C ABI (kvev_create with a region table,
kvev_paged_begin, kvev_paged_step); the fp64 oracle (oracle/memdecay.py)
runs free from the same seeded prefill, labels and inputs.  Per step and
sequence: attention outputs and probabilities (2e-3 relative), page scores
S_p (1e-5 absolute), the kept pages (exact away from near ties), per-token
importance (1e-5) and clocks (exact), labels, page contents (bit-exact) and
the page bookkeeping.  A token whose attention sits within 1e-4 relative of
tau may have its clock reset on either side: the oracle then takes the
device's decision for it; a page-score near tie at the eviction boundary
is checked admissible and followed the same way.
"""
import math

import numpy as np
import pytest

from oracle import memdecay as MD
from workloads import (DECODE_REGION, REGION_HALF_LIVES, REGION_PINNED, memdecay_workload,
                       region_labels)

from parity import OUT_RTOL, P_ATOL, P_RTOL, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

PAGE = 16
S_ATOL = 1e-5
AMB_REL = 1e-4


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def md_params(g, budget, **kw):
    lam = tuple(math.log(2.0) / h for h in REGION_HALF_LIVES)
    return MD.MDParams(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, budget,
                       base=(1.0,) * len(lam), lam=lam, pinned=REGION_PINNED,
                       decode_region=DECODE_REGION, **kw)


def table_of(P):
    return kvev.region_table(P.base, P.lam, P.pinned, score_kind=kvev.KVEV_SCORE_MEMDECAY,
                             rho=P.rho, attn_weight=P.attn_weight, tau_scale=P.tau_scale,
                             decode_region=P.decode_region)


def load(pp, K, V, labels, L0):
    """Prefill of every sequence into pages b*pps + j; labels per token."""
    Ly, batch, Hkv, _, d = K.shape
    nb0 = -(-L0 // PAGE)
    pad = nb0 * PAGE - L0
    lab = np.concatenate([labels, np.zeros(pad, np.uint8)]).reshape(nb0, PAGE)
    for b in range(batch):
        for src, pool in ((K, pp.k_pool), (V, pp.v_pool)):
            x = np.concatenate([src[:, b], np.zeros((Ly, Hkv, pad, d), np.uint16)], axis=2)
            x = np.ascontiguousarray(x.reshape(Ly, Hkv, nb0, PAGE, d).transpose(2, 0, 1, 3, 4))
            pool[b * pp.pps:b * pp.pps + nb0].copy_(
                torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
        r0 = b * pp.pps * PAGE
        pp.region[r0:r0 + nb0 * PAGE].copy_(torch.from_numpy(lab.reshape(-1)))


def admissible_eviction(res, dev_evicted, budget):
    """The device's evicted pages are a greedy prefix under the oracle's page
    scores up to S_ATOL: no pinned page, the budget met, the last page taken
    needed, and no kept page scoring below an evicted one by more than the
    tolerance."""
    S, n_tok, pinned = res["S"], res["n_tok"], res["pinned"]
    ev = set(dev_evicted)
    assert not any(pinned[j] for j in ev), "a pinned page was evicted"
    left = int(n_tok.sum()) - int(sum(n_tok[j] for j in ev))
    free_left = [j for j in range(len(S)) if j not in ev and not pinned[j]]
    assert left <= budget or not free_left, "budget not met"
    if ev:   # the greedy stop: the last page taken (a top score of the set) was needed
        top = max(S[j] for j in ev)
        assert any(left + n_tok[j] > budget for j in ev if S[j] >= top - S_ATOL), \
            "more pages evicted than needed"
    if ev and free_left:
        assert max(S[j] for j in ev) <= min(S[j] for j in free_left) + S_ATOL, \
            "an evicted page outranks a kept one"


def compare(pp, P, seqs, b, t, refresh, q, kn, vn, probs, prio, stats):
    pre = seqs[b].copy()
    res = MD.step(P, seqs[b], t, refresh, q, kn, vn, want_probs=True)
    L = res["L"]
    # positions of the oracle's tokens on the device: block slot j, token k
    owner = res["owner"]
    first = np.searchsorted(owner, np.arange(len(res["pids_before"])))
    within = np.arange(L) - first[owner]
    table = pp.block_table[b].cpu().numpy()          # after compaction: for kept pages
    # clocks: adopt the device's decision where the threshold is within rounding
    if refresh:
        tau = P.tau_scale / L
        amb = np.abs(res["A_bar"] - tau) <= AMB_REL * tau
        amb[L - 1] = False
        if amb.any():
            stats["amb"] += int(amb.sum())
            # device pages of the pre-eviction blocks are not kept for evicted ones:
            # only the tokens of kept pages can be read back
            kept_lids = set(pp.retained_lid[b, :int(pp.n_retained[b])].cpu().numpy().tolist())
            lid_page = {int(pp.lid[b, j]): int(table[j]) for j in range(int(pp.n_blocks[b]))}
            fa = np.full(L, -1)
            for i in np.nonzero(amb)[0]:
                lid = res["pids_before"][owner[i]]
                if lid in kept_lids:
                    tr = int(pp.tok_t_ref[lid_page[lid] * PAGE + within[i]])
                    fa[i] = 1 if tr == t else 0
            if (fa >= 0).any() and (fa != np.where(res["accessed"], 1, 0))[fa >= 0].any():
                seqs[b] = pre.copy()
                res = MD.step(P, seqs[b], t, refresh, q, kn, vn, want_probs=True,
                              forced_access=fa)
    out = pp.out[b].cpu().numpy().astype(np.float64)
    err = np.abs(out - res["out"]).max(-1) / np.abs(res["out"]).max(-1)
    assert err.max() <= OUT_RTOL, f"step {t} seq {b}: output rel err {err.max():.2e}"
    stats["out_rel"] = max(stats["out_rel"], float(err.max()))
    slot = owner * PAGE + within
    if refresh:
        p = probs[b].cpu().numpy().astype(np.float64)[:, :, slot]
        bad = np.abs(p - res["probs"]) > P_RTOL * res["probs"] + P_ATOL
        assert not bad.any(), f"step {t} seq {b}: {bad.sum()} probabilities"
    nbb = len(res["pids_before"])
    S = prio[b, :nbb].cpu().numpy().astype(np.float64)
    serr = np.abs(S - res["S"])
    assert serr.max() <= S_ATOL, f"step {t} seq {b}: page score err {serr.max():.2e}"
    stats["S_abs"] = max(stats["S_abs"], float(serr.max()))
    n = int(pp.n_retained[b])
    kept_lids = list(pp.retained_lid[b, :n].cpu().numpy())
    want = [res["pids_before"][j] for j in res["kept"]]
    if kept_lids != want:
        dev_ev = [j for j, lid in enumerate(res["pids_before"]) if lid not in set(kept_lids)]
        admissible_eviction(res, dev_ev, P.budget)
        stats["swaps"] += 1
        seqs[b] = pre.copy()
        res = MD.step(P, seqs[b], t, refresh, q, kn, vn, forced_access=None, evicted=dev_ev)
    # pages after the step
    seq = seqs[b]
    nb = int(pp.n_blocks[b])
    assert nb == len(seq.pages), "live pages"
    assert list(pp.lid[b, :nb].cpu().numpy()) == seq.pids(), "page ids"
    assert list(pp.len[b, :nb].cpu().numpy()) == [pg.n for pg in seq.pages], "page lengths"
    nf = int(pp.n_free[b])
    own = np.arange(b * pp.pps, (b + 1) * pp.pps)
    live = pp.block_table[b, :nb].cpu().numpy()
    assert np.array_equal(np.sort(np.concatenate([live, pp.free_pages[b, :nf].cpu().numpy()])),
                          own), "live and free pages must partition the sequence's pages"
    tok_a = pp.tok_a.cpu().numpy().astype(np.float64)
    tok_tr = pp.tok_t_ref.cpu().numpy()
    region = pp.region.cpu().numpy()
    for j, pg in enumerate(seq.pages):
        idx = live[j] * PAGE + np.arange(pg.n)
        aerr = np.abs(tok_a[idx] - pg.a).max()
        assert aerr <= S_ATOL, f"importance of page {pg.pid}: {aerr:.2e}"
        stats["a_abs"] = max(stats["a_abs"], float(aerr))
        assert np.array_equal(tok_tr[idx], pg.t_ref), f"clocks of page {pg.pid}"
        assert np.array_equal(region[idx], pg.region), f"labels of page {pg.pid}"
        assert np.array_equal(_bits(pp.k_pool[live[j], :, :, :pg.n]), pg.K), f"K of {pg.pid}"
        assert np.array_equal(_bits(pp.v_pool[live[j], :, :, :pg.n]), pg.V), f"V of {pg.pid}"
    if any(not any(P.pinned[r] for r in pg.region) for pg in seq.pages):
        assert seq.n_tokens <= P.budget, "an unpinned page is left above the budget"


def run_memdecay(wl, budget, steps, *, pps_slack=4, refresh=kvev.KVEV_REFRESH_FULL, period=1,
                 **kw):
    g = wl.geom
    L0 = wl.L0
    P = md_params(g, budget, **kw)
    nb0 = -(-L0 // PAGE)
    pp = kvev.PagedEvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch,
                                nb0 + pps_slack, PAGE, budget, 0.05, 0.001, regions=table_of(P),
                                refresh=refresh, period=period)
    K, V = wl.prefill()
    labels = region_labels(L0)
    load(pp, K, V, labels, L0)
    pp.begin(L0)
    probs = torch.zeros((g.batch, g.n_layers, g.n_q_heads, pp.pps * PAGE), device="cuda")
    prio = torch.zeros((g.batch, pp.pps), device="cuda")
    kvev.kvev_set_debug(pp.ctx, probs, prio)
    seqs = [MD.MDSequence.from_prefill(K[:, b], V[:, b], labels, PAGE) for b in range(g.batch)]
    stats = {"swaps": 0, "amb": 0, "out_rel": 0.0, "S_abs": 0.0, "a_abs": 0.0}
    for t in range(1, steps + 1):
        q, kn, vn = wl.step_inputs(t)
        pp.step(to_dev_bf16(q), to_dev_bf16(kn), to_dev_bf16(vn))
        kvev.kvev_sync(pp.ctx)
        ref_now = refresh == kvev.KVEV_REFRESH_FULL or (t - 1) % period == 0
        for b in range(g.batch):
            compare(pp, P, seqs, b, t, ref_now, q[b], kn[b], vn[b], probs, prio, stats)
    kvev.kvev_check_scratch(pp.ctx)   # no scratch region overran its guard band
    pp.close()
    return stats


def test_memdecay_small_partial_prefill_page():
    """3 layers of the Qwen2.5-3B geometry (16 q / 2 KV heads: 8 per group),
    2 sequences of 200 tokens (last prefill page 8 tokens), 30% budget
    (60 tokens), 40 steps: pages fill, open, get evicted whole."""
    wl = memdecay_workload(0, prefill_len=200, n_layers=3, batch=2)
    st = run_memdecay(wl, 60, 40)
    print("memdecay small:", st)


def test_memdecay_many_sequences():
    """24 sequences (one selection CTA per sequence), 2 layers, 96-token
    prefills, a 28-token budget, 8 steps."""
    wl = memdecay_workload(0, prefill_len=96, n_layers=2, batch=24)
    run_memdecay(wl, 28, 8)


def test_memdecay_1700_full_depth():
    """36 layers, 1700-token contexts (the short tier's length), budget 510,
    6 steps, one sequence."""
    wl = memdecay_workload(1, prefill_len=1700, n_layers=36, batch=1)
    st = run_memdecay(wl, 510, 6)
    print("memdecay 1700:", st)


def test_memdecay_lazy_observation_and_small_budget():
    """Observation every 3 steps (clocks and importance frozen in between,
    the prior keeps decaying), a budget below the pinned span."""
    wl = memdecay_workload(2, prefill_len=96, n_layers=2, batch=2)
    st = run_memdecay(wl, 3, 12, refresh=kvev.KVEV_REFRESH_LAZY, period=3)
    print("memdecay lazy:", st)


@pytest.mark.slow
def test_memdecay_full_size_through_step_16():
    """The full region-aware workload on the device: Qwen2.5-3B geometry (36
    layers, 16 q / 2 KV heads), 32 sequences of 16384 labelled tokens,
    budget 4915 tokens; steps 1 to 16 of sequences 0 and 31 against the
    oracle, element by element (decoded tokens fill the last page, open new
    ones and get evicted with it)."""
    from workloads import Geometry
    from workloads.device import PagedDeviceWorkload
    L0, batch, Ly, budget = 16384, 32, 36, 4915
    wl = PagedDeviceWorkload(0, n_layers=Ly, n_q_heads=16, n_kv_heads=2, batch=batch,
                             prefill=L0, needle_blocks=0)
    g = Geometry(Ly, 16, 2, 128, batch)
    P = md_params(g, budget)
    nb0 = L0 // PAGE
    pp = kvev.PagedEvictionPass(Ly, 16, 2, 128, batch, nb0 + 8, PAGE, budget, 0.05, 0.001,
                                regions=table_of(P))
    wl.fill(torch, pp.k_pool, pp.v_pool, pp.pps)
    labels = region_labels(L0)
    lab_t = torch.from_numpy(labels).cuda()
    for b in range(batch):
        pp.region[b * pp.pps * PAGE:b * pp.pps * PAGE + L0].copy_(lab_t)
    pp.begin(L0)
    probs = torch.zeros((batch, Ly, 16, pp.pps * PAGE), device="cuda")
    prio = torch.zeros((batch, pp.pps), device="cuda")
    kvev.kvev_set_debug(pp.ctx, probs, prio)
    sample = (0, batch - 1)
    seqs = {}
    for s in sample:
        pages = slice(s * pp.pps, s * pp.pps + nb0)
        K = _bits(pp.k_pool[pages]).transpose(1, 2, 0, 3, 4).reshape(Ly, 2, -1, 128)
        V = _bits(pp.v_pool[pages]).transpose(1, 2, 0, 3, 4).reshape(Ly, 2, -1, 128)
        seqs[s] = MD.MDSequence.from_prefill(np.ascontiguousarray(K), np.ascontiguousarray(V),
                                             labels, PAGE)
    stats = {"swaps": 0, "amb": 0, "out_rel": 0.0, "S_abs": 0.0, "a_abs": 0.0}
    for t in range(1, 17):
        q, kn, vn = wl.step_inputs(torch, t, None)
        pp.step(q, kn, vn)
        kvev.kvev_sync(pp.ctx)
        for s in sample:
            compare(pp, P, seqs, s, t, True, _bits(q[s]), _bits(kn[s]), _bits(vn[s]), probs,
                    prio, stats)
    print("memdecay full size:", stats)
    kvev.kvev_check_scratch(pp.ctx)   # no scratch region overran its guard band
    pp.close()
