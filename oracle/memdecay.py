"""fp64 oracle of region-aware page eviction (MemDecay).

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU leg).  The
attention is the C oracle's (kvev_oracle.c); this module keeps one
sequence's pages and applies, in the order of "MemDecay: Region-Aware KV
Cache Eviction for Efficient LLM Agent Inference":

  * Sec. III-C Eq. (2): at an observation step every cached token's
    importance a <- rho * a + (1 - rho) * A_bar, with A_bar the attention
    mass the token receives averaged over heads and layers (window of one
    step: every refresh step is an observation step);
  * Eq. (3): the decay clock t_ref becomes the observation step when
    A_bar >= tau, tau = tau_scale / |K_t| (the scaled form, Sec. IV-A);
    otherwise it stays at its last value (the insertion step at first);
  * Eq. (4): retention score s = b_r * exp(-lambda_r * (t - t_ref)) +
    alpha * a, b_r and lambda_r of the token's region;
  * Eq. (5): page score S_p = mean of s over the page's tokens;
  * Sec. III-D and Algorithm 1: when the cache holds more than B tokens,
    the non-pinned pages are evicted in ascending S_p until |K| <= B
    (a min-heap); a page holding any pinned token is pinned (Sec. IV-A:
    pinning protects whole pages).

Parity unpinned: the per-region base priorities b_r.  The page prints the
caption of its Table I without the values; this oracle reads b_r = 1 for every
region (any b_r enters the same Eq. (4), whose structure the pins check), so
no test can tie the values themselves to the page.

Readings where the paper is silent: decoded tokens take the label
``decode_region`` (scratchpad); a new token joins the last page while it has
room, else opens a page; among equal page scores the higher page index is
evicted first (the lower kept); the scores and eviction are applied every
step, the attention statistics (a, t_ref) only on refresh steps.
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass

import numpy as np

from . import oracle as O


@dataclass
class MDParams:
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    budget: int                  # tokens
    base: tuple                  # b_r per region
    lam: tuple                   # lambda_r per region (per decode step)
    pinned: tuple                # bool per region
    rho: float = 0.9
    attn_weight: float = 0.5     # alpha of Eq. (4)
    tau_scale: float = 2.0       # tau = tau_scale / |K_t|
    page: int = 16
    decode_region: int = 0


@dataclass
class MDPage:
    pid: int                     # logical page id (ascending = slot order)
    K: np.ndarray                # [Ly][Hkv][n][d] bf16 bits
    V: np.ndarray
    region: np.ndarray           # [n] int
    a: np.ndarray                # [n] float64 importance
    t_ref: np.ndarray            # [n] int

    @property
    def n(self) -> int:
        return self.K.shape[2]


@dataclass
class MDSequence:
    pages: list
    page: int
    next_pid: int

    @staticmethod
    def from_prefill(K, V, region, page: int) -> "MDSequence":
        """K, V: [Ly][Hkv][L0][d] bits; region: [L0] labels.  Prefill tokens
        have insertion step 0 and importance 0; the last page may be partial."""
        L0 = K.shape[2]
        pages = []
        for pid, s in enumerate(range(0, L0, page)):
            e = min(L0, s + page)
            pages.append(MDPage(pid, K[:, :, s:e].copy(), V[:, :, s:e].copy(),
                                np.asarray(region[s:e], dtype=np.int64).copy(),
                                np.zeros(e - s), np.zeros(e - s, dtype=np.int64)))
        return MDSequence(pages, page, len(pages))

    def copy(self) -> "MDSequence":
        return MDSequence([MDPage(p.pid, p.K.copy(), p.V.copy(), p.region.copy(), p.a.copy(),
                                  p.t_ref.copy()) for p in self.pages], self.page, self.next_pid)

    @property
    def n_tokens(self) -> int:
        return sum(p.n for p in self.pages)

    def pids(self):
        return [p.pid for p in self.pages]


def retention(P: MDParams, region, a, t_ref, t: int) -> np.ndarray:
    """Eq. (4) for arrays of tokens."""
    b = np.array([P.base[r] for r in region], dtype=np.float64)
    lam = np.array([P.lam[r] for r in region], dtype=np.float64)
    return b * np.exp(-lam * (t - np.asarray(t_ref, dtype=np.float64))) + P.attn_weight * a


def evict_pages(S, n_tok, pinned, budget: int):
    """Algorithm 1's eviction loop: pop non-pinned pages of minimum score
    (ties: higher index first) until the token count is within the budget.
    Returns the evicted page indexes in eviction order."""
    total = int(sum(n_tok))
    heap = [(float(S[j]), -j) for j in range(len(S)) if not pinned[j]]
    heapq.heapify(heap)
    evicted = []
    while total > budget and heap:
        _, mj = heapq.heappop(heap)
        evicted.append(-mj)
        total -= int(n_tok[-mj])
    return evicted


def step(P: MDParams, seq: MDSequence, t: int, refresh: bool, q_bits, knew_bits, vnew_bits,
         want_probs: bool = False, forced_access=None, evicted=None):
    """One decode step of one sequence; `seq` is updated in place.

    forced_access: per token, -1 = the threshold decides, 0/1 = the clock
    decision taken instead; evicted: the page indexes to evict instead of
    this function's own choice (a caller continuing along another
    admissible outcome at a near tie)."""
    Ly, Hq, Hkv, d = P.n_layers, P.n_q_heads, P.n_kv_heads, P.head_dim
    kn = np.ascontiguousarray(knew_bits, dtype=np.uint16).reshape(Ly, Hkv, 1, d)
    vn = np.ascontiguousarray(vnew_bits, dtype=np.uint16).reshape(Ly, Hkv, 1, d)
    # append
    if not seq.pages or seq.pages[-1].n == seq.page:
        seq.pages.append(MDPage(seq.next_pid, kn.copy(), vn.copy(),
                                np.array([P.decode_region]), np.zeros(1),
                                np.array([t], dtype=np.int64)))
        seq.next_pid += 1
    else:
        pg = seq.pages[-1]
        pg.K = np.concatenate([pg.K, kn], axis=2)
        pg.V = np.concatenate([pg.V, vn], axis=2)
        pg.region = np.append(pg.region, P.decode_region)
        pg.a = np.append(pg.a, 0.0)
        pg.t_ref = np.append(pg.t_ref, t)
    Kall = np.concatenate([p.K for p in seq.pages], axis=2)
    Vall = np.concatenate([p.V for p in seq.pages], axis=2)
    L = Kall.shape[2]
    owner = np.concatenate([np.full(p.n, j) for j, p in enumerate(seq.pages)])
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    out = np.zeros((Ly, Hq, d))
    probs = np.zeros((Ly, Hq, L)) if want_probs else None
    mass = np.zeros(L)
    for layer in range(Ly):
        p, o = O.attention(q[layer], Kall[layer], Vall[layer])
        out[layer] = o
        if want_probs:
            probs[layer] = p
        mass += p.sum(axis=0)
    a = np.concatenate([p.a for p in seq.pages])
    t_ref = np.concatenate([p.t_ref for p in seq.pages])
    region = np.concatenate([p.region for p in seq.pages])
    A_bar = mass / (Ly * Hq)
    accessed = np.zeros(L, dtype=bool)
    if refresh:
        a = P.rho * a + (1.0 - P.rho) * A_bar
        accessed = A_bar >= P.tau_scale / L
        if forced_access is not None:
            fa = np.asarray(forced_access)
            accessed = np.where(fa >= 0, fa.astype(bool), accessed)
        t_ref = np.where(accessed, t, t_ref)
    s = retention(P, region, a, t_ref, t)
    nb = len(seq.pages)
    S = np.array([s[owner == j].mean() for j in range(nb)])
    n_tok = np.array([p.n for p in seq.pages])
    pinned = np.array([any(P.pinned[r] for r in p.region) for p in seq.pages])
    for j, pg in enumerate(seq.pages):
        pg.a = a[owner == j].copy()
        pg.t_ref = t_ref[owner == j].copy()
    ev = evict_pages(S, n_tok, pinned, P.budget) if evicted is None else list(evicted)
    pids_before = seq.pids()
    evs = set(ev)
    kept = [j for j in range(nb) if j not in evs]
    seq.pages = [seq.pages[j] for j in kept]
    return dict(out=out, probs=probs, L=L, owner=owner, A_bar=A_bar, a=a, t_ref=t_ref, s=s,
                S=S, pinned=pinned, n_tok=n_tok, accessed=accessed, evicted=ev,
                kept=np.array(kept, dtype=np.int64), pids_before=pids_before)
