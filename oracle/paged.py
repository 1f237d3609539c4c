"""fp64 oracle of block-granular (paged) eviction with score persistence.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU leg).  The
attention and the selection are the C oracle's (kvev_oracle.c); this module
keeps one sequence's block list and applies, in the pages' order:

  * the kv-cache-docs figure "ema-eviction" (LRFU per (sequence, token
    block)): score = alpha * new + (1 - alpha) * score; priority = (1 -
    score) * (1 - exp(-beta * steps since access)); a higher priority is
    evicted; when a block is evicted its identity key and score persist and
    are restored on re-admission rather than reset;
  * the block's new score is the max over its tokens of the head-summed
    attention probability, folded layer by layer in ascending order ("What
    Matters for Aggressive Decoding-Time KV Eviction?" Appendix E "Layer
    scoring");
  * a block is accessed at a refresh step when any of its tokens' attention,
    averaged over heads and layers, reaches 2/L (MemDecay Sec. III-C Eq. (3)
    with the scaled threshold); a re-admitted or newly opened block counts as
    accessed when it enters;
  * whenever the cache holds more than B blocks, the B of lowest priority are
    kept, ties to the lower slot (Sec. 3.1 of the first paper);
  * with pinned regions (optional): every token carries a region label and
    a block holding a token of a pinned region is never evicted (MemDecay
    Sec. III-A and IV-A: pinning protects whole pages); pinned blocks are
    forced into the kept set, past the budget when they outnumber it.
    Decoded tokens take ``decode_region``.  Re-admission is not combined with
    regions (the backing tier keeps no labels).

Block order is slot order: ascending logical id (prefill blocks first, then
blocks opened by decoding); a re-admitted block returns to its sorted place.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import oracle as O


@dataclass
class Block:
    lid: int                 # logical block id
    K: np.ndarray            # [Ly][Hkv][n][d] bf16 bits, n <= page tokens
    V: np.ndarray
    m: float = 0.0
    t_ins: int = 0
    t_ref: int = 0
    region: np.ndarray = None   # [n] labels, with pinned regions only

    @property
    def n(self) -> int:
        return self.K.shape[2]


@dataclass
class PagedSequence:
    """One sequence: live blocks in slot order, the persistent score table,
    and the backing tier (full copies of the prefill blocks)."""
    blocks: list
    page: int
    next_lid: int
    backing_K: np.ndarray            # [n_prefill_blocks][Ly][Hkv][page][d]
    backing_V: np.ndarray
    table: dict = field(default_factory=dict)   # lid -> persisted score
    pinned_regions: tuple = None     # per region label: pinned or not
    decode_region: int = 0

    @staticmethod
    def from_prefill(K, V, page: int, region=None, pinned_regions=None,
                     decode_region: int = 0) -> "PagedSequence":
        """K, V: [Ly][Hkv][L0][d] bits, L0 a multiple of `page`; `region`:
        [L0] labels, given together with `pinned_regions`."""
        Ly, Hkv, L0, d = K.shape
        nb = L0 // page
        bk = K.reshape(Ly, Hkv, nb, page, d).transpose(2, 0, 1, 3, 4).copy()
        bv = V.reshape(Ly, Hkv, nb, page, d).transpose(2, 0, 1, 3, 4).copy()
        lab = (None if pinned_regions is None
               else np.asarray(region, dtype=np.int64).reshape(nb, page))
        blocks = [Block(j, bk[j].copy(), bv[j].copy(),
                        region=None if lab is None else lab[j].copy()) for j in range(nb)]
        return PagedSequence(blocks, page, nb, bk, bv, {},
                             None if pinned_regions is None else tuple(pinned_regions),
                             int(decode_region))

    def copy(self) -> "PagedSequence":
        return PagedSequence([Block(b.lid, b.K.copy(), b.V.copy(), b.m, b.t_ins, b.t_ref,
                                    None if b.region is None else b.region.copy())
                              for b in self.blocks], self.page, self.next_lid, self.backing_K,
                             self.backing_V, dict(self.table), self.pinned_regions,
                             self.decode_region)

    def pinned_blocks(self) -> np.ndarray:
        """Per live block: whether it holds a token of a pinned region."""
        return np.array([any(self.pinned_regions[r] for r in b.region) for b in self.blocks],
                        dtype=np.uint8)

    @property
    def n_tokens(self) -> int:
        return sum(b.n for b in self.blocks)

    def lids(self):
        return [b.lid for b in self.blocks]


def readmit(seq: PagedSequence, lid: int, t: int, persist: bool = True) -> bool:
    """Bring prefill block `lid` back from the backing tier (no-op when it is
    resident).  Its score is the persisted one (0 when persistence is off or
    it was never evicted); its access time is t."""
    if seq.pinned_regions is not None:
        raise ValueError("re-admission is not combined with pinned regions")
    if lid in seq.lids():
        return False
    m = seq.table.get(lid, 0.0) if persist else 0.0
    blk = Block(lid, seq.backing_K[lid].copy(), seq.backing_V[lid].copy(), m, 0, t)
    pos = 0
    while pos < len(seq.blocks) and seq.blocks[pos].lid < lid:
        pos += 1
    seq.blocks.insert(pos, blk)
    return True


def step(P: O.OracleParams, seq: PagedSequence, t: int, refresh: bool, q_bits, knew_bits,
         vnew_bits, want_probs: bool = False, forced_access=None, kept=None):
    """One decode step of one sequence.  P.budget counts blocks.  Returns the
    result dict; `seq` is updated in place (append, scores, eviction).

    forced_access: per token, -1 = the threshold decides, 0/1 = the decision
    taken instead; kept: the block slots to keep instead of this function's
    own selection.  Both let a caller continue along another admissible
    outcome where the decision sits within rounding of a tie."""
    Ly, Hq, Hkv, d = P.n_layers, P.n_q_heads, P.n_kv_heads, P.head_dim
    page = seq.page
    kn = np.ascontiguousarray(knew_bits, dtype=np.uint16).reshape(Ly, Hkv, 1, d)
    vn = np.ascontiguousarray(vnew_bits, dtype=np.uint16).reshape(Ly, Hkv, 1, d)
    # 1. append: into the open block, else open a new one
    if not seq.blocks or seq.blocks[-1].n == page or seq.blocks[-1].lid < len(seq.backing_K):
        if refresh or not seq.blocks:
            m0 = 0.0
        else:
            m0 = float(np.mean([b.m for b in seq.blocks]))
        lab = None if seq.pinned_regions is None else np.array([seq.decode_region])
        seq.blocks.append(Block(seq.next_lid, kn.copy(), vn.copy(), m0, t, t, lab))
        seq.next_lid += 1
    else:
        ob = seq.blocks[-1]
        ob.K = np.concatenate([ob.K, kn], axis=2)
        ob.V = np.concatenate([ob.V, vn], axis=2)
        ob.t_ref = t
        if seq.pinned_regions is not None:
            ob.region = np.append(ob.region, seq.decode_region)
    # 2. attention over every live token, slot order
    Kall = np.concatenate([b.K for b in seq.blocks], axis=2)   # [Ly][Hkv][L][d]
    Vall = np.concatenate([b.V for b in seq.blocks], axis=2)
    L = Kall.shape[2]
    owner = np.concatenate([np.full(b.n, j) for j, b in enumerate(seq.blocks)])
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    out = np.zeros((Ly, Hq, d))
    probs = np.zeros((Ly, Hq, L)) if want_probs else None
    nb = len(seq.blocks)
    m = np.array([b.m for b in seq.blocks])
    tok_sum = np.zeros(L)
    for layer in range(Ly):
        p, o = O.attention(q[layer], Kall[layer], Vall[layer])
        out[layer] = o
        if want_probs:
            probs[layer] = p
        if not refresh:
            continue
        s_tok = p.sum(axis=0)
        tok_sum += s_tok
        s_blk = np.array([s_tok[owner == j].max() for j in range(nb)])
        if P.pool_mean:
            s_blk = s_blk / Hq
        m = np.array([O.ema(m[j], s_blk[j], P.alpha) for j in range(nb)])
    accessed = np.zeros(nb, dtype=bool)
    if refresh:
        tok_acc = tok_sum / (Ly * Hq) >= 2.0 / L
        if forced_access is not None:
            fa = np.asarray(forced_access)
            tok_acc = np.where(fa >= 0, fa.astype(bool), tok_acc)
        accessed = np.array([tok_acc[owner == j].any() for j in range(nb)])
    for j, b in enumerate(seq.blocks):
        b.m = float(m[j])
        if accessed[j]:
            b.t_ref = t
    pr = np.array([O.priority(b.m, t - (b.t_ref if P.age_mode == O.AGE_SINCE_ACCESS else b.t_ins),
                              P.beta) for b in seq.blocks])
    pinned = None if seq.pinned_regions is None else seq.pinned_blocks()
    if kept is None:
        kept = O.select(pr, P.budget, pinned=pinned)
    kept = np.asarray(kept, dtype=np.int64)
    evicted = [j for j in range(nb) if j not in set(kept.tolist())]
    for j in evicted:
        seq.table[seq.blocks[j].lid] = seq.blocks[j].m
    lids_before = [b.lid for b in seq.blocks]
    seq.blocks = [seq.blocks[j] for j in kept]
    return dict(out=out, probs=probs, priority=pr, m_upd=m, accessed=accessed, kept=kept,
                pinned=pinned,
                lids_before=lids_before, evicted_lids=[lids_before[j] for j in evicted],
                L=L, owner=owner, token_sum=tok_sum)
