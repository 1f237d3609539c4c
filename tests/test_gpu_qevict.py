"""GPU parity of two-tier window routing with an INT2 tier (QEvict).

The CUDA path runs through the C ABI (kvev_set_tiers, kvev_tier_begin,
kvev_tier_step); the fp64 oracle (oracle/qevict.py) runs free from the same
seeded prefill and inputs.  Per step and sequence: attention outputs
(2e-3 relative per vector), window scores (1e-5 absolute), tiers (exact
away from near ties), the INT2 ledger of every quantized window (codes and
fp16 scale/zero bit-exact) and the bf16 pages of every full-precision window
(bit-exact, promoted copies included).  Where two windows' scores sit within
the tolerance across a tier boundary the device's ranking is checked
admissible and the oracle continues along it.
"""
import copy

import numpy as np
import pytest

from oracle import qevict as QE
from workloads import Geometry, Workload

from ledger_codec import decode_ledger
from parity import OUT_RTOL, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

M_ATOL = 1e-5
TIER_NAME = {kvev.KVEV_TIER_UNROUTED: "U", kvev.KVEV_TIER_FULL: "F", kvev.KVEV_TIER_QUANT: "Q",
             kvev.KVEV_TIER_EVICTED: "E"}


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def load(tp, K, V, L0):
    """Prefill into the windowed page layout: sinks in page b*pps, token
    5 + 16 i + r in row r of page b*pps + 1 + i."""
    Ly, batch, Hkv, _, d = K.shape
    hist = L0 - 5
    n_pages = -(-hist // 16)
    for b in range(batch):
        for src, pool in ((K, tp.k_pool), (V, tp.v_pool)):
            sink = np.zeros((Ly, Hkv, 16, d), np.uint16)
            sink[:, :, :5] = src[:, b, :, :5]
            rest = np.zeros((Ly, Hkv, n_pages * 16, d), np.uint16)
            rest[:, :, :hist] = src[:, b, :, 5:]
            pages = rest.reshape(Ly, Hkv, n_pages, 16, d).transpose(2, 0, 1, 3, 4)
            allp = np.concatenate([sink[None], pages], axis=0)
            pool[b * tp.pps:b * tp.pps + 1 + n_pages].copy_(
                torch.from_numpy(np.ascontiguousarray(allp).view(np.int16)).view(torch.bfloat16))


def admissible(m: dict, dev_tiers: dict, tol: float):
    """Every window the device placed higher scores at least as much as
    every window it placed lower, up to tol."""
    rank = {"F": 0, "Q": 1, "E": 2}
    for a, ta in dev_tiers.items():
        for b, tb in dev_tiers.items():
            if rank[ta] < rank[tb]:
                assert m[a] >= m[b] - tol, f"window {a} ({ta}) below {b} ({tb})"


def score_tol(P, m):
    """Window-score tolerance: 1e-5 absolute for the EMA; the cumulative
    score grows with every step and layer, where fp32 keeps 1e-5 relative."""
    return M_ATOL * max(1.0, abs(m)) if P.cumulative else M_ATOL


def compare(tp, P, seqs, b, t, q, kn, vn, stats, check_windows=None, lir=None):
    """check_windows: ids whose pages / ledger entries are compared (all when
    None); lir: (oracle LIRCounter per sequence, device counters) to check
    after routing events."""
    pre = copy.deepcopy(seqs[b])
    res = QE.step(P, seqs[b], t, q, kn, vn)
    seq = seqs[b]
    dev_tier = [TIER_NAME.get(int(x), "-") for x in tp.tier[b, :len(seq.windows)].cpu().numpy()]
    if res["routed"] and dev_tier != seq.tiers():
        # a near tie at a tier boundary: check the device's choice, then follow it
        cand = {w.wid: res["m"][w.wid] for w in pre.windows if w.wid in res["m"]}
        new_t = {wid: dev_tier[wid] for wid in cand if dev_tier[wid] in ("F", "Q", "E")}
        admissible(cand, new_t, max(score_tol(P, m) for m in cand.values()))
        order = sorted(new_t, key=lambda wid: ({"F": 0, "Q": 1, "E": 2}[new_t[wid]], -cand[wid], wid))
        seqs[b] = pre
        res = QE.step(P, seqs[b], t, q, kn, vn, ranking=order)
        seq = seqs[b]
        stats["swaps"] += 1
    assert dev_tier == seq.tiers(), f"step {t} seq {b}: tiers {dev_tier} vs {seq.tiers()}"
    for w0, w in zip(pre.windows, seq.windows):
        stats["promoted"] += w0.tier == "Q" and w.tier == "F"
        stats["redemoted"] += w0.tier == "F" and w.tier == "Q" and w0.ledger is not None
    out = tp.out[b].cpu().numpy().astype(np.float64)
    err = np.abs(out - res["out"]).max(-1) / np.abs(res["out"]).max(-1)
    assert err.max() <= OUT_RTOL, f"step {t} seq {b}: output rel err {err.max():.2e}"
    if float(err.max()) > stats["out_rel"]:   # where the largest error sits
        layer, head = np.unravel_index(int(np.argmax(err)), err.shape)
        stats["out_rel_at"] = (t, int(layer), int(head),
                               float(np.abs(res["out"][layer, head]).max()))
    stats["out_rel"] = max(stats["out_rel"], float(err.max()))
    sc = tp.score[b].cpu().numpy().astype(np.float64)
    for wid, m in res["m"].items():
        assert abs(sc[wid] - m) <= score_tol(P, m), f"step {t} seq {b}: score of window {wid}"
        stats["m_abs"] = max(stats["m_abs"], abs(sc[wid] - m))
    if lir is not None and res["routed"]:
        counter, dev = lir
        counter[b].route({w.wid: w.tier for w in seq.windows})
        got = dev[b].cpu().numpy().tolist()
        assert got == [counter[b].events, counter[b].revivals, counter[b].spans], \
            f"step {t} seq {b}: LIR counts {got}"
        stats["revivals"] = stats.get("revivals", 0) + 0   # reported at the end
    assert int(tp.n_windows[b]) == len(seq.windows)
    assert int(tp.tail_len[b]) == seq.K_tail.shape[2]
    wp = tp.win_pages[b].cpu().numpy()
    for w in seq.windows:
        if check_windows is not None and w.wid not in check_windows:
            continue
        if w.tier in ("U", "F"):
            for i in range(8):
                page = wp[w.wid, i]
                assert np.array_equal(_bits(tp.k_pool[page]), w.K[:, :, 16 * i:16 * i + 16]), \
                    f"K pages of window {w.wid} ({w.tier})"
                assert np.array_equal(_bits(tp.v_pool[page]), w.V[:, :, 16 * i:16 * i + 16])
        if w.tier == "Q":
            for l in range(P.n_layers):
                for g in range(P.n_kv_heads):
                    kq, ks, kz, vq, vs, vz = decode_ledger(tp.ledger[b, w.wid, l, g].cpu().numpy())
                    L = w.ledger
                    assert np.array_equal(kq, L["kq"][l, g]), f"key codes of window {w.wid}"
                    assert np.array_equal(ks.view(np.uint16), L["ks"][l, g].view(np.uint16))
                    assert np.array_equal(kz.view(np.uint16), L["kz"][l, g].view(np.uint16))
                    assert np.array_equal(vq, L["vq"][l, g]), f"value codes of window {w.wid}"
                    assert np.array_equal(vs.view(np.uint16), L["vs"][l, g].view(np.uint16))
                    assert np.array_equal(vz.view(np.uint16), L["vz"][l, g].view(np.uint16))
            stats["ledgers"] += 1


def check_reconstructions(tp, P, seq, b):
    """Rotary mode: each INT2 window of sequence b has a reconstruction slot
    of its own among the last 8 K_q pages of the sequence's range, holding
    the window dequantized with keys rotated forward, keys and values rounded
    to bf16, bit for bit (the oracle's dequantize_window with the window's
    (cos, sin) rows).  Slots are the device's to assign: each window's is
    found by its content."""
    n_slots = P.k_quant
    base = b * tp.pps + tp.pps - 8 * n_slots
    kp = _bits(tp.k_pool[base:base + 8 * n_slots])    # [slot * 8 + i][Ly][Hkv][16][d]
    vp = _bits(tp.v_pool[base:base + 8 * n_slots])
    used = set()
    for w in [w for w in seq.windows if w.tier == "Q"]:
        k, v = QE.dequantize_window(w.ledger, cs=QE.window_cs(P, w.wid))
        kb, vb = QE._f32_to_bf16_bits(k), QE._f32_to_bf16_bits(v)
        want_k = kb.reshape(P.n_layers, P.n_kv_heads, 8, 16, -1).transpose(2, 0, 1, 3, 4)
        want_v = vb.reshape(P.n_layers, P.n_kv_heads, 8, 16, -1).transpose(2, 0, 1, 3, 4)
        slots = [s_ for s_ in range(n_slots)
                 if np.array_equal(kp[8 * s_:8 * s_ + 8], want_k)]
        assert slots, f"no slot holds the reconstructed keys of window {w.wid}"
        s_ = slots[0]
        assert s_ not in used, f"window {w.wid} shares slot {s_}"
        used.add(s_)
        assert np.array_equal(vp[8 * s_:8 * s_ + 8], want_v), \
            f"reconstructed values of window {w.wid}"
    return len(used)


def run_tiers(wl, k_full, k_quant, omega, steps, alpha=0.05, pps_slack=24, cumulative=False,
              sustain=None):
    """sustain: check the Global LIR counts with that span length.  With
    wl.rope_base set the run is in rotary mode (the workload's table), and
    after every step the reconstruction pages are checked."""
    g = wl.geom
    L0 = wl.L0
    max_ctx = L0 + steps + 8
    rope = None if wl.rope_base is None else wl.rope_table(max_ctx)
    pps = 1 + -(-(L0 - 5) // 16) + pps_slack + (0 if rope is None else 8 * k_quant)
    tp = kvev.TierEvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch,
                               max_ctx, pps, k_full, k_quant, omega, alpha,
                               aggregation=kvev.KVEV_AGG_CUMULATIVE if cumulative
                               else kvev.KVEV_AGG_EMA, rope=rope)
    lir = None
    if sustain is not None:
        from oracle import diagnostics as D
        dev = torch.full((g.batch, 3), -1, dtype=torch.int32, device="cuda")
        kvev.kvev_tier_diagnostics(tp.ctx, sustain, dev)
        lir = ([D.LIRCounter(sustain) for _ in range(g.batch)], dev)
    K, V = wl.prefill()
    load(tp, K, V, L0)
    tp.begin(L0)
    P = QE.QParams(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, k_full, k_quant,
                   alpha=alpha, omega=omega, cumulative=cumulative, rope=rope)
    seqs = [QE.QSequence.from_prefill(P, K[:, b], V[:, b]) for b in range(g.batch)]
    stats = {"swaps": 0, "out_rel": 0.0, "m_abs": 0.0, "ledgers": 0, "promoted": 0,
             "redemoted": 0, "recon": 0}
    for t in range(1, steps + 1):
        q, kn, vn = wl.step_inputs(t)
        tp.step(to_dev_bf16(q), to_dev_bf16(kn), to_dev_bf16(vn))
        kvev.kvev_sync(tp.ctx)
        for b in range(g.batch):
            compare(tp, P, seqs, b, t, q[b], kn[b], vn[b], stats, lir=lir)
            if rope is not None:
                stats["recon"] += check_reconstructions(tp, P, seqs[b], b)
    if lir is not None:
        stats["lir"] = [(c.events, c.revivals, c.spans) for c in lir[0]]
    kvev.kvev_check_scratch(tp.ctx)   # no scratch region overran its guard band
    tp.close()
    return stats


def test_tiers_small_routing_promotion_and_new_window():
    """2 layers of the Llama-8B geometry, 2 sequences of 1325 tokens (10
    windows + a 40-token tail), K_f 2, K_q 3, routing every 4 steps, 100
    steps: windows get quantized, promoted back, re-demoted (ledger reuse),
    evicted, and one new window forms from decoded tokens."""
    wl = Workload(Geometry(2, 32, 8, 128, 2), 5 + 128 * 10 + 40, seed=7, outliers=4, needle=16,
                  needle_period=16)
    st = run_tiers(wl, 2, 3, 4, 100)
    print("tiers:", st)
    assert st["ledgers"] > 0 and st["promoted"] > 0 and st["redemoted"] > 0


def test_tiers_cumulative_window_score_and_global_lir():
    """The review's Sec. 4.2 Eq. (1) cumulative window score (sums over steps
    and layers, never decays) driving the routing, with the Global LIR counts
    (Sec. 3) checked after every routing event against the oracle's
    restatement; then the EMA score with LIR counts over a drifting needle,
    where windows leave the Full tier and come back."""
    wl = Workload(Geometry(2, 32, 8, 128, 2), 5 + 128 * 10 + 40, seed=7, outliers=4, needle=16,
                  needle_period=16)
    st = run_tiers(wl, 2, 3, 4, 60, cumulative=True, sustain=2)
    print("tiers cumulative:", st)
    st = run_tiers(wl, 2, 3, 4, 100, sustain=2)
    print("tiers EMA + LIR:", st)
    assert any(r > 0 for _, r, _ in st["lir"]), "no revival in 100 steps of needle drift"


def test_tiers_rotary_positions():
    """Rotary mode (the review's Sec. 4.4): the cache holds rotated keys
    (rope base 10000); windows are quantized rotated back by position (the
    ledger bit-exact against the oracle), promoted windows come back rotated
    forward (bf16 pages bit-exact), the INT2 windows are attended through
    bf16 reconstructions, made as windows enter the INT2 tier (checked bit
    for bit after every step), and the outputs stay within the attention
    tolerance."""
    wl = Workload(Geometry(2, 32, 8, 128, 2), 5 + 128 * 10 + 40, seed=7, outliers=4, needle=16,
                  needle_period=16, rope_base=10000.0)
    st = run_tiers(wl, 2, 3, 4, 60)
    print("tiers rotary:", st)
    assert st["ledgers"] > 0 and st["promoted"] > 0 and st["recon"] > 0


def test_tiers_no_quantized_tier_and_large_capacity():
    """K_q = 0 (two tiers: Full or evicted) and K_f covering every window."""
    wl = Workload(Geometry(2, 32, 8, 128, 1), 5 + 128 * 6 + 3, seed=8, needle=16, needle_period=8)
    run_tiers(wl, 2, 0, 2, 20)
    run_tiers(wl, 6, 0, 3, 12)


def test_tiers_route_every_step():
    """Omega 1: routing, first demotions, promotions and evictions at the end
    of every step, with a needle that moves every 3 steps."""
    wl = Workload(Geometry(2, 32, 8, 128, 2), 5 + 128 * 8 + 7, seed=21, needle=16,
                  needle_period=3)
    st = run_tiers(wl, 2, 3, 1, 16)
    assert st["ledgers"] > 0 and st["promoted"] > 0


def test_tiers_quantizer_exact_ties():
    """Groups whose quotients (x - zero) / scale land exactly on 0.5, 1.5 and
    2.5 (scale 1 and 2: min 0, max 3 or 6) in the keys of channels 0-15 and
    the values of channel group 0, in every window: rint's ties to even
    decide codes 0, 2, 2 on both sides (the quantizer's exact-division path)."""
    wl = Workload(Geometry(2, 32, 8, 128, 1), 5 + 128 * 4 + 20, seed=12, needle=16,
                  needle_period=8)
    K, V = wl.prefill()      # cached arrays: edited in place for both sides
    bf = {0: 0x0000, 0.5: 0x3F00, 1: 0x3F80, 1.5: 0x3FC0, 2: 0x4000, 2.5: 0x4020,
          3: 0x4040, 5: 0x40A0, 6: 0x40C0}
    pat1 = [0, 3, 0.5, 1.5, 2.5, 1, 2, 0.5] * 4             # scale 1
    pat2 = [0, 6, 1, 3, 5, 2, 0, 6] * 4                     # scale 2: ties at 1, 3, 5
    for w in range(4):
        t0 = 5 + 128 * w
        for i in range(32):
            K[:, :, :, t0 + i, 0:8] = bf[pat1[i]]
            K[:, :, :, t0 + i, 8:16] = bf[pat2[i]]
        for i in range(16):
            V[:, :, :, t0 + i, 0:32] = np.array([bf[x] for x in (pat1 if i % 2 else pat2)],
                                                np.uint16)
    st = run_tiers(wl, 1, 3, 4, 12)
    assert st["ledgers"] > 0


@pytest.mark.slow
def test_tiers_full_size_three_routing_events():
    """The full two-tier workload on the device: 32 layers, 4 sequences of
    131072 tokens (1023 windows), K_f 51, K_q 204, routing every 8 steps;
    steps 1-24 of sequence 0 against the oracle: the first routing event
    (t = 8) quantizes 204 windows, the next ones (t = 16, 24) move windows
    between the tiers (promotions from the ledger included), and the steps
    in between attend the mixed bf16 / INT2 cache."""
    from workloads.device import TierDeviceWorkload
    L0, batch, Ly = 131072, 4, 32
    wl = TierDeviceWorkload(0, n_layers=Ly, batch=batch, prefill=L0)
    pps = wl.n_pages + 16 + 8 * 51
    tp = kvev.TierEvictionPass(Ly, 32, 8, 128, batch, L0 + 32, pps, 51, 204, 8, 0.05)
    wl.fill(torch, tp.k_pool, tp.v_pool, pps)
    T = 24
    inputs = [wl.step_inputs(torch, t, tp.k_pool, pps) for t in range(1, T + 1)]
    # sequence 0's prefill in token order, from the windowed pages
    hist = L0 - 5
    pages = slice(0, wl.n_pages)
    kp, vp = _bits(tp.k_pool[pages]), _bits(tp.v_pool[pages])
    def tokens(p):
        rest = p[1:].transpose(1, 2, 0, 3, 4).reshape(Ly, 8, -1, 128)[:, :, :hist]
        return np.concatenate([p[0, :, :, :5], rest], axis=2)
    P = QE.QParams(Ly, 32, 8, 128, 51, 204, alpha=0.05, omega=8)
    seqs = [QE.QSequence.from_prefill(P, tokens(kp), tokens(vp))]
    del kp, vp
    tp.begin(L0)
    stats = {"swaps": 0, "out_rel": 0.0, "m_abs": 0.0, "ledgers": 0, "promoted": 0,
             "redemoted": 0}
    for t in range(1, T + 1):
        q, kn, vn = inputs[t - 1]
        tp.step(q, kn, vn)
        kvev.kvev_sync(tp.ctx)
        compare(tp, P, seqs, 0, t, _bits(q[0]), _bits(kn[0]), _bits(vn[0]), stats,
                check_windows=set(range(0, 1023, 61)))
    print("tiers full size:", stats)
    assert stats["ledgers"] > 0
    kvev.kvev_check_scratch(tp.ctx)   # no scratch region overran its guard band
    tp.close()


@pytest.mark.slow
def test_tiers_full_size_rotary_two_routing_events():
    """Rotary mode on the full two-tier workload: 32 layers, 4 sequences of
    131072 tokens (positions up to 131087 in the table), K_f 51, K_q 204,
    routing every 8 steps; steps 1-16 of sequence 0 against the oracle with
    the same table: the first routing event quantizes 204 windows rotated
    back and reconstructs them rotated forward, the second moves windows
    between the tiers (promotions rotated forward, reconstructions of the
    windows entering INT2).  Ledger entries, bf16 pages and reconstructions
    are compared bit for bit on sampled windows, outputs within 2e-3.  The
    device draws of the keys carry no rotation: the rotation's arithmetic
    is the same for any key values."""
    from workloads import rope_table
    from workloads.device import TierDeviceWorkload
    L0, batch, Ly = 131072, 4, 32
    max_ctx = L0 + 32
    rope = rope_table(max_ctx, 128, 10000.0)
    wl = TierDeviceWorkload(0, n_layers=Ly, batch=batch, prefill=L0)
    pps = wl.n_pages + 16 + 8 * 51 + 8 * 204
    tp = kvev.TierEvictionPass(Ly, 32, 8, 128, batch, max_ctx, pps, 51, 204, 8, 0.05, rope=rope)
    wl.fill(torch, tp.k_pool, tp.v_pool, pps)
    T = 16
    inputs = [wl.step_inputs(torch, t, tp.k_pool, pps) for t in range(1, T + 1)]
    hist = L0 - 5
    pages = slice(0, wl.n_pages)
    kp, vp = _bits(tp.k_pool[pages]), _bits(tp.v_pool[pages])
    def tokens(p):
        rest = p[1:].transpose(1, 2, 0, 3, 4).reshape(Ly, 8, -1, 128)[:, :, :hist]
        return np.concatenate([p[0, :, :, :5], rest], axis=2)
    P = QE.QParams(Ly, 32, 8, 128, 51, 204, alpha=0.05, omega=8, rope=rope)
    seqs = [QE.QSequence.from_prefill(P, tokens(kp), tokens(vp))]
    del kp, vp
    tp.begin(L0)
    sample = set(range(0, 1023, 61))
    stats = {"swaps": 0, "out_rel": 0.0, "m_abs": 0.0, "ledgers": 0, "promoted": 0,
             "redemoted": 0, "recon": 0}
    base = tp.pps - 8 * 204                      # sequence 0's reconstruction slots
    for t in range(1, T + 1):
        q, kn, vn = inputs[t - 1]
        tp.step(q, kn, vn)
        kvev.kvev_sync(tp.ctx)
        compare(tp, P, seqs, 0, t, _bits(q[0]), _bits(kn[0]), _bits(vn[0]), stats,
                check_windows=sample)
        if t % 8 == 0:   # sampled INT2 windows: a slot holds the reconstruction
            probe = _bits(tp.k_pool[base:base + 8 * 204:8, 0, 0])   # first page, layer 0, head 0
            for w in seqs[0].windows:
                if w.tier != "Q" or w.wid not in sample:
                    continue
                k, v = QE.dequantize_window(w.ledger, cs=QE.window_cs(P, w.wid))
                kb, vb = QE._f32_to_bf16_bits(k), QE._f32_to_bf16_bits(v)
                hits = [s_ for s_ in range(204) if np.array_equal(probe[s_], kb[0, 0, :16])]
                assert hits, f"step {t}: no slot holds window {w.wid}"
                s_ = hits[0]
                for i in range(8):
                    page = base + 8 * s_ + i
                    assert np.array_equal(_bits(tp.k_pool[page]), kb[:, :, 16 * i:16 * i + 16])
                    assert np.array_equal(_bits(tp.v_pool[page]), vb[:, :, 16 * i:16 * i + 16])
                stats["recon"] += 1
    print("tiers full size rotary:", stats)
    assert stats["ledgers"] > 0 and stats["recon"] > 0
    kvev.kvev_check_scratch(tp.ctx)   # no scratch region overran its guard band
    tp.close()
