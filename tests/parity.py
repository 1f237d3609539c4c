"""Shared helpers of the GPU parity tests: load a seeded workload into the
CUDA path, run the oracle beside it from the same seeded inputs, and compare
one step element by element under the stated tolerances.  The oracle never
reads the device's state: where the device took one of several admissible
outcomes (a near tie at the budget boundary, an access decision on the
threshold) the test checks it is admissible and continues the oracle from
its own pre-selection values along that choice (`follow`).

Tolerances (bf16 inputs, fp32 device arithmetic, fp64 oracle):
  attention output   per (layer, head) vector: max|d| / max|ref| <= 2e-3
  probabilities      |d p| <= 2e-3 * p_ref + 1e-9
  EMA score          |d m| <= 1e-5
  priority           |d pr| <= 1e-5
  retained set       identical wherever the priority gap at the budget
                     boundary exceeds the priority tolerance; otherwise the
                     swaps among units within the tolerance of the boundary
                     are counted and the rest must match
  compacted K/V      bit-exact given the device's retained indices
"""
from __future__ import annotations

import numpy as np

import oracle as O

OUT_RTOL = 2e-3
P_RTOL, P_ATOL = 2e-3, 1e-9
M_ATOL = 1e-5
PR_ATOL = 1e-5


def load_prefill(ep, wl):
    """Copy the workload's prefill into buffer 0 of an EvictionPass."""
    import torch
    K, V = wl.prefill()
    L0 = wl.L0
    kt = torch.from_numpy(K.view(np.int16)).view(torch.bfloat16)
    vt = torch.from_numpy(V.view(np.int16)).view(torch.bfloat16)
    for layer in range(K.shape[0]):
        ep.k[0][layer, :, :, :L0].copy_(kt[layer], non_blocking=False)
        ep.v[0][layer, :, :, :L0].copy_(vt[layer], non_blocking=False)


def to_dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def boundary_check(pr_ref: np.ndarray, kept_dev: np.ndarray, budget: int, tol: float,
                   pr_alt: np.ndarray | None = None):
    """Check a device retained set against oracle priorities.

    pr_ref: oracle priority per slot; pr_alt: admissible alternative priority
    (slots whose access decision sits on the threshold), else None.
    Returns the number of near-tie swaps; raises AssertionError otherwise."""
    L = pr_ref.shape[0]
    n = min(budget, L)
    kept = np.zeros(L, dtype=bool)
    kept[kept_dev] = True
    assert kept.sum() == n == len(kept_dev), "retained count"
    assert np.all(np.diff(kept_dev) > 0), "retained list must be ascending"
    if n == L:
        return 0
    lo = pr_ref if pr_alt is None else np.minimum(pr_ref, pr_alt)
    hi = pr_ref if pr_alt is None else np.maximum(pr_ref, pr_alt)
    order = np.lexsort((np.arange(L), pr_ref))
    want = np.zeros(L, dtype=bool)
    want[order[:n]] = True
    if pr_alt is None:
        s = pr_ref[order]
        gap = s[n] - s[n - 1]
        if gap > tol:
            assert np.array_equal(kept, want), "retained set differs away from near-ties"
            return 0
    # consistency: every kept unit could rank no worse than every evicted one
    theta_kept = lo[kept].max()
    theta_evict = hi[~kept].min()
    assert theta_kept <= theta_evict + tol, (
        f"kept unit with priority {theta_kept} above evicted {theta_evict}")
    return int((kept & ~want).sum())


def compare_step(res, ep, b: int, pre: O.SequenceState, budget: int, dbg_probs=None,
                 dbg_prio=None, refresh: bool = True, pr_alt=None, m_atol: float = M_ATOL,
                 access_amb=None):
    """Compare one device step of sequence b with the oracle result `res`
    computed from the same pre-step state.  Returns a dict of counters."""
    import torch
    L = res["L"]
    stats = {}
    out = ep.out[b].float().cpu().numpy().astype(np.float64)   # fp32 or bf16 output
    ref = res["out"]
    err = np.abs(out - ref).max(axis=-1) / np.abs(ref).max(axis=-1)
    stats["out_rel"] = float(err.max())
    assert err.max() <= OUT_RTOL, f"attention output rel err {err.max():.3e}"
    if refresh and dbg_probs is not None:
        p = dbg_probs[b, :, :, :L].cpu().numpy().astype(np.float64)
        pref = res["probs"]
        bad = np.abs(p - pref) > P_RTOL * pref + P_ATOL
        stats["p_rel"] = float((np.abs(p - pref) / np.maximum(pref, 1e-30)).max())
        assert not bad.any(), f"{bad.sum()} probabilities out of tolerance"
    if dbg_prio is not None:
        pr = dbg_prio[b, :L].cpu().numpy().astype(np.float64)
        ok = np.abs(pr - res["priority"]) <= PR_ATOL
        if pr_alt is not None:
            ok |= np.abs(pr - pr_alt) <= PR_ATOL
        stats["pr_abs"] = float(np.abs(pr - res["priority"]).max())
        assert ok.all(), f"{(~ok).sum()} priorities out of tolerance"
    n = int(ep.n_retained[b].item())
    kept = ep.retained[b, :n].cpu().numpy().astype(np.int64)
    stats["swaps"] = boundary_check(res["priority"], kept, budget, PR_ATOL, pr_alt)
    # state after compaction, gathered with the device's own indices
    m_dev = ep.score[b, :n].cpu().numpy().astype(np.float64)
    merr = np.abs(m_dev - res["m_upd"][kept])
    stats["m_abs"] = float(merr.max()) if n else 0.0
    assert stats["m_abs"] <= m_atol, f"EMA score abs err {stats['m_abs']:.3e}"
    pos_full = np.append(pre.pos[:L - 1], res["new_pos"])
    assert np.array_equal(ep.pos[b, :n].cpu().numpy(), pos_full[kept]), "compacted pos"
    tins_full = np.append(pre.t_ins[:L - 1], res["t"])
    assert np.array_equal(ep.t_ins[b, :n].cpu().numpy(), tins_full[kept]), "compacted t_ins"
    tref_dev = ep.t_ref[b, :n].cpu().numpy()
    tref_ok = tref_dev == res["t_ref_upd"][kept]
    if access_amb is not None:
        tref_ok |= access_amb[kept]
    assert tref_ok.all(), f"compacted t_ref: {(~tref_ok).sum()} differ"
    # K/V after compaction: the device's pre-step rows (plus the appended row)
    # at the device's retained indices, bit for bit
    Kd = ep.live_k()[:, b, :, :n].view(torch.int16).cpu().numpy().view(np.uint16)
    Vd = ep.live_v()[:, b, :, :n].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(Kd, res["K_full"][:, :, kept]), "compacted K differs"
    assert np.array_equal(Vd, res["V_full"][:, :, kept]), "compacted V differs"
    return stats


def oracle_step(P, pre: O.SequenceState, t: int, refresh: bool, q, kn, vn, new_pos: int,
                forced_access=None, want_probs=True):
    res, new = O.step(P, pre, t, refresh, q, kn, vn, new_pos, forced_access, want_probs)
    L = res["L"]
    Kf = pre.K[:, :, :L].copy()
    Vf = pre.V[:, :, :L].copy()
    Kf[:, :, L - 1] = kn
    Vf[:, :, L - 1] = vn
    res["K_full"], res["V_full"], res["new_pos"], res["t"] = Kf, Vf, new_pos, t
    return res, new


def follow(res, pre: O.SequenceState, kept, t_ref_kept=None) -> O.SequenceState:
    """The oracle's post-step state built from its own pre-selection values
    (cache with the new token, updated scores and clocks) at the slots
    `kept` (ascending), optionally with the clocks of those slots replaced
    by `t_ref_kept` (an admissible access decision taken the other way)."""
    L = res["L"]
    kept = np.asarray(kept, dtype=np.int64)
    n = len(kept)
    cap = pre.K.shape[2]
    new = O.SequenceState(np.zeros_like(pre.K), np.zeros_like(pre.V), np.zeros(cap),
                          np.zeros(cap, np.int64), np.zeros(cap, np.int64),
                          np.zeros(cap, np.int64), n)
    new.K[:, :, :n] = res["K_full"][:, :, kept]
    new.V[:, :, :n] = res["V_full"][:, :, kept]
    new.m[:n] = res["m_upd"][kept]
    new.t_ins[:n] = np.append(pre.t_ins[:L - 1], res["t"])[kept]
    new.t_ref[:n] = res["t_ref_upd"][kept] if t_ref_kept is None else t_ref_kept
    new.pos[:n] = np.append(pre.pos[:L - 1], res["new_pos"])[kept]
    return new


def access_alternative(res, pre: O.SequenceState, P, rel: float = 1e-4):
    """Slots whose head- and layer-averaged attention is within `rel` of the
    2/L threshold, where fp32 on the device and fp64 here may decide the
    access either way.  Returns (priorities under the other decision, or None
    when the age does not depend on it or no slot is ambiguous; the mask)."""
    L = res["L"]
    mean_attn = res["score_sum"] / (P.n_layers * P.n_q_heads)
    thr = 2.0 / L
    amb = np.abs(mean_attn - thr) <= rel * thr
    amb[L - 1] = False                       # the new token is accessed by insertion
    if not amb.any() or P.age_mode != O.AGE_SINCE_ACCESS:
        return None, amb
    alt = res["priority"].copy()
    t = res["t"]
    for i in np.nonzero(amb)[0]:
        if res["accessed"][i]:
            age = t - int(pre.t_ref[i])      # clock not reset
        else:
            age = 0                          # clock reset this step
        alt[i] = O.priority(res["m_upd"][i], age, P.beta)
    return alt, amb
