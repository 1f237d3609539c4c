"""fp64 oracle of two-tier window routing with an INT2 tier (QEvict).

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU leg).  One
sequence, following "QEvict: Recoverable Quantized KV Eviction for
Attention-Drift-Robust Long-Context Decoding" (the review page), Sec. 4:

  * Sec. 4.1: a protected sink prefix and a protected recent region stay in
    full precision; the rest of the cache is cut into contiguous windows,
    each in state Full, Quantized or Evicted; attention (eq. "Attention")
    runs over the accessible keys and values: the full-precision tokens plus
    the dequantized INT2 windows;
  * window score: the head-averaged attention a window's tokens receive
    (the inner sums of Eq. (1)), folded per step into an EMA with weight
    alpha on the new value, layer after layer in ascending order, kept
    across steps (the LRFU EMA of the kv-cache-docs figure "ema-eviction",
    the reading taken here of "EMA accumulated-attention score"); or,
    with `cumulative`, Sec. 4.2 Eq. (1) itself: the head-averaged window
    attention added up over steps and, since one routing decision covers
    every layer, over layers too (a sum that never forgets);
  * Eq. (3): tier capacities K_f = floor((1-q) B_hist / M_f) and
    K_q = floor(q B_hist / M_q);
  * Eqs. (4)-(5) and the routing algorithm: every Omega steps the candidates
    (Full and Quantized windows plus windows that have aged out of the recent
    region) are ranked by score; the top K_f are Full, the next K_q
    Quantized, the rest evicted for good;
  * migration-stable quantization: a window is quantized on its first
    demotion only; its codes and scale/zero stay in a ledger and are reused on
    every later demotion; a promoted window is dequantized from the ledger.

Parity unpinned: the window geometry and routing interval (sinks 5, recent
32, windows of 128 tokens on the grid after the sinks, routing every Omega = 8
steps at the end of the step).  The page gives the sink and recent counts and
Omega but not where windows start or when in a step routing happens; these
are the readings taken here, and no pin ties them to the page beyond the
capacity example of Eq. (3).

INT2 codec (asymmetric, as the page's KIVI-style scheme: per-channel keys,
per-token values, groups of 32): for each group zero = fp16(min), scale =
fp16((max - min) / 3) with the difference and division in fp32, code =
clamp(rint((x - zero) / scale), 0, 3) with the subtraction and division in
fp32 (round half to even), code 0 when scale is 0; dequantized value =
code * scale + zero in fp32.  A promoted window's full-precision copy is
that value rounded to bf16.

Rotary positions (Sec. 4.4, "Positional handling for promoted keys" and the
routing algorithm's promotion step), with `rope` set: the cached keys are the
model's rotated keys; a window is quantized in the pre-rotation domain, each
key rotated back by its position p before the codec, and every use of an
INT2 window rotates the dequantized key forward again: a promoted window's
bf16 key is the rotated value rounded to bf16, and attention runs over the
INT2 windows reconstructed the same way (keys rotated, keys and values
rounded to bf16), the review's "reconstruct (dequantize, re-apply RoPE) the
active low-bit windows" before attention.  Rotation of channel pair
(j, j + d/2) by the table's (cos, sin) at position p, every product and sum
rounded to fp32 in this order:
    forward  y_j = x_j cos - x_{j+d/2} sin,  y_{j+d/2} = x_{j+d/2} cos + x_j sin
    back     x_j = y_j cos + y_{j+d/2} sin,  x_{j+d/2} = y_{j+d/2} cos - y_j sin.
The table is the model's own (cos, sin) cache, an input: [positions][d/2][2]
fp32.

Readings where the page is silent: sinks are tokens [0, n_sink); windows
are [n_sink + W j, n_sink + W (j + 1)); a window exists (score 0, Full
precision, not yet routed) from the step its last token is appended and is
scored from that step on; it becomes a routing candidate once its last
position is below L - n_recent; a routing event happens at the end of every
step t with t mod Omega = 0 and takes effect from the next step; ties in
the ranking go to the lower window index.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

UNROUTED, FULL, QUANT, EVICTED = "U", "F", "Q", "E"


@dataclass
class QParams:
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    k_full: int
    k_quant: int
    alpha: float = 0.05
    window: int = 128
    n_sink: int = 5
    n_recent: int = 32
    omega: int = 8
    group: int = 32
    cumulative: bool = False      # Eq. (1): the window score sums, never decays
    rope: np.ndarray = None       # [positions][d/2][2] fp32 (cos, sin), or None


def capacities(b_hist: float, q: float, m_full: float, m_quant: float):
    """Eq. (3): (K_f, K_q)."""
    return int(np.floor((1.0 - q) * b_hist / m_full)), int(np.floor(q * b_hist / m_quant))


def int2_bytes_per_token_layer(n_kv_heads: int, head_dim: int, group: int = 32) -> int:
    """Bytes one token of one layer costs in the INT2 tier: 2-bit key and
    value codes plus fp16 scale and zero (keys per channel per `group`
    tokens, values per token per `group` channels)."""
    codes = 2 * n_kv_heads * head_dim * 2 // 8
    k_meta = n_kv_heads * head_dim * 2 * 2 // group
    v_meta = n_kv_heads * (head_dim // group) * 2 * 2
    return codes + k_meta + v_meta


# ------------------------------------------------------------------ codec
def _bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _f32_to_bf16_bits(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def quantize_groups(x, axis: int):
    """Asymmetric 2-bit quantization of fp32 `x` in groups along `axis`
    (the group's elements are that axis).  Returns (codes uint8, scale
    float16, zero float16) with scale/zero reduced over `axis`."""
    x = np.asarray(x, dtype=np.float32)
    mn = x.min(axis=axis, keepdims=True)
    mx = x.max(axis=axis, keepdims=True)
    zero = mn.astype(np.float16)
    scale = ((mx - mn) / np.float32(3.0)).astype(np.float16)
    z32 = zero.astype(np.float32)
    s32 = scale.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint((x - z32) / s32)
    r = np.where(s32 == 0, 0.0, r)
    codes = np.clip(r, 0, 3).astype(np.uint8)
    return codes, np.squeeze(scale, axis=axis), np.squeeze(zero, axis=axis)


def dequantize(codes, scale, zero, axis: int):
    """fp32 code * scale + zero, scale/zero broadcast along `axis`."""
    s = np.expand_dims(np.asarray(scale, dtype=np.float16).astype(np.float32), axis)
    z = np.expand_dims(np.asarray(zero, dtype=np.float16).astype(np.float32), axis)
    return (codes.astype(np.float32) * s + z).astype(np.float32)


def rotate(x, cs, back: bool = False):
    """Rotate fp32 keys x [..., W, d] by the (cos, sin) rows cs [W][d/2][2]
    of their positions, pairs (j, j + d/2), each product and sum rounded to
    fp32 (forward, or back with the sine negated)."""
    x = np.asarray(x, dtype=np.float32)
    h = x.shape[-1] // 2
    c = np.asarray(cs[..., 0], dtype=np.float32)
    s = np.asarray(cs[..., 1], dtype=np.float32)
    a, b = x[..., :h], x[..., h:]
    if back:
        ya = (a * c).astype(np.float32) + (b * s).astype(np.float32)
        yb = (b * c).astype(np.float32) - (a * s).astype(np.float32)
    else:
        ya = (a * c).astype(np.float32) - (b * s).astype(np.float32)
        yb = (b * c).astype(np.float32) + (a * s).astype(np.float32)
    return np.concatenate([ya.astype(np.float32), yb.astype(np.float32)], axis=-1)


def quantize_window(K_bits, V_bits, group: int = 32, cs=None):
    """Ledger entry of one window.  K, V: [Ly][Hkv][W][d] bf16 bits.
    Keys per channel over groups of `group` tokens; values per token over
    groups of `group` channels.  cs: the (cos, sin) rows of the window's
    positions [W][d/2][2]: the keys are rotated back first."""
    Ly, Hkv, W, d = K_bits.shape
    kf = _bits_to_f32(K_bits)
    if cs is not None:
        kf = rotate(kf, cs, back=True)
    k = kf.reshape(Ly, Hkv, W // group, group, d)
    v = _bits_to_f32(V_bits).reshape(Ly, Hkv, W, d // group, group)
    kq, ks, kz = quantize_groups(k, axis=3)             # scale/zero [Ly][Hkv][W/g][d]
    vq, vs, vz = quantize_groups(v, axis=4)             # scale/zero [Ly][Hkv][W][d/g]
    return dict(kq=kq.reshape(Ly, Hkv, W, d), ks=ks, kz=kz,
                vq=vq.reshape(Ly, Hkv, W, d), vs=vs, vz=vz, group=group)


def dequantize_window(led, layer=None, cs=None):
    """fp32 (K, V) [Ly][Hkv][W][d] of a ledger entry ([Hkv][W][d] of one
    layer when `layer` is given); cs: the window's (cos, sin) rows, the keys
    rotated forward."""
    g = led["group"]
    sel = slice(None) if layer is None else slice(layer, layer + 1)
    kq, vq = led["kq"][sel], led["vq"][sel]
    Ly, Hkv, W, d = kq.shape
    k = dequantize(kq.reshape(Ly, Hkv, W // g, g, d), led["ks"][sel], led["kz"][sel], axis=3)
    v = dequantize(vq.reshape(Ly, Hkv, W, d // g, g), led["vs"][sel], led["vz"][sel], axis=4)
    k, v = k.reshape(Ly, Hkv, W, d), v.reshape(Ly, Hkv, W, d)
    if cs is not None:
        k = rotate(k, cs)
    return (k, v) if layer is None else (k[0], v[0])


def window_cs(P: QParams, wid: int):
    """The (cos, sin) rows of window wid's positions, or None without rope."""
    if P.rope is None:
        return None
    p0 = P.n_sink + P.window * wid
    return P.rope[p0:p0 + P.window]


# ------------------------------------------------------------------ state
@dataclass
class QWindow:
    wid: int
    tier: str
    m: float = 0.0
    K: np.ndarray = None        # full-precision copy, bf16 bits [Ly][Hkv][W][d] (U and F)
    V: np.ndarray = None
    ledger: dict = None         # codes, once quantized


@dataclass
class QSequence:
    K_sink: np.ndarray          # [Ly][Hkv][n_sink][d] bits
    V_sink: np.ndarray
    windows: list
    K_tail: np.ndarray          # tokens after the last formed window
    V_tail: np.ndarray
    L: int                      # positions so far (evicted tokens included)

    @staticmethod
    def from_prefill(P: QParams, K, V) -> "QSequence":
        """K, V: [Ly][Hkv][L0][d] bits, L0 >= n_sink."""
        L0 = K.shape[2]
        ns, W = P.n_sink, P.window
        nw = (L0 - ns) // W
        wins = [QWindow(j, UNROUTED, 0.0, K[:, :, ns + W * j:ns + W * (j + 1)].copy(),
                        V[:, :, ns + W * j:ns + W * (j + 1)].copy()) for j in range(nw)]
        t0 = ns + W * nw
        return QSequence(K[:, :, :ns].copy(), V[:, :, :ns].copy(), wins,
                         K[:, :, t0:].copy(), V[:, :, t0:].copy(), L0)

    def window_end(self, P: QParams, w: QWindow) -> int:
        return P.n_sink + P.window * (w.wid + 1)

    def tiers(self):
        return [w.tier for w in self.windows]


def accessible(P: QParams, seq: QSequence, layer: int):
    """fp32 (K, V) [Hkv][n][d] of every accessible token of one layer in
    position order, and the window index of each (-1: sink or tail)."""
    ks, vs, owner = [_bits_to_f32(seq.K_sink[layer])], [_bits_to_f32(seq.V_sink[layer])], [
        np.full(P.n_sink, -1)]
    for j, w in enumerate(seq.windows):
        if w.tier in (UNROUTED, FULL):
            ks.append(_bits_to_f32(w.K[layer]))
            vs.append(_bits_to_f32(w.V[layer]))
        elif w.tier == QUANT:
            k, v = dequantize_window(w.ledger, layer, window_cs(P, w.wid))
            if P.rope is not None:   # reconstructed as bf16 before attention
                k = _bits_to_f32(_f32_to_bf16_bits(k))
                v = _bits_to_f32(_f32_to_bf16_bits(v))
            ks.append(k)
            vs.append(v)
        else:
            continue
        owner.append(np.full(P.window, j))
    ks.append(_bits_to_f32(seq.K_tail[layer]))
    vs.append(_bits_to_f32(seq.V_tail[layer]))
    owner.append(np.full(seq.K_tail.shape[2], -1))
    return np.concatenate(ks, axis=1), np.concatenate(vs, axis=1), np.concatenate(owner)


def attention_f64(q, K, V):
    """Single-query GQA attention in fp64 over fp32 keys/values.
    q [Hq][d] fp32, K/V [Hkv][n][d] -> (p [Hq][n], out [Hq][d])."""
    Hq, d = q.shape
    Hkv = K.shape[0]
    G = Hq // Hkv                                # query heads h of KV head h // G
    p = np.zeros((Hq, K.shape[1]))
    out = np.zeros((Hq, d))
    for g in range(Hkv):
        k64, v64 = K[g].astype(np.float64), V[g].astype(np.float64)
        heads = slice(g * G, (g + 1) * G)
        lg = (k64 @ q[heads].astype(np.float64).T).T / np.sqrt(d)     # [G][n]
        e = np.exp(lg - lg.max(axis=1, keepdims=True))
        p[heads] = e / e.sum(axis=1, keepdims=True)
        out[heads] = p[heads] @ v64
    return p, out


def route(P: QParams, seq: QSequence):
    """One routing event (Eqs. (4)-(5) and the routing algorithm)."""
    horizon = seq.L - P.n_recent
    cand = [w for w in seq.windows
            if w.tier in (FULL, QUANT) or (w.tier == UNROUTED and seq.window_end(P, w) <= horizon)]
    cand.sort(key=lambda w: (-w.m, w.wid))
    new_f, new_q = cand[:P.k_full], cand[P.k_full:P.k_full + P.k_quant]
    for w in new_q:
        if w.tier != QUANT:
            if w.ledger is None:                 # first demotion: quantize once
                w.ledger = quantize_window(w.K, w.V, P.group, window_cs(P, w.wid))
            w.K = w.V = None
            w.tier = QUANT
    for w in new_f:
        if w.tier == QUANT:                      # promotion: from the ledger
            k, v = dequantize_window(w.ledger, cs=window_cs(P, w.wid))
            w.K, w.V = _f32_to_bf16_bits(k), _f32_to_bf16_bits(v)
        w.tier = FULL
    for w in cand[P.k_full + P.k_quant:]:
        w.tier = EVICTED
        w.K = w.V = w.ledger = None


def step(P: QParams, seq: QSequence, t: int, q_bits, knew_bits, vnew_bits,
         want_probs: bool = False, ranking=None):
    """One decode step; `seq` is updated in place.  `ranking`: candidate
    window ids in rank order to route by instead of the scores (a caller
    following another admissible order at a near tie)."""
    Ly, Hq, Hkv, d = P.n_layers, P.n_q_heads, P.n_kv_heads, P.head_dim
    kn = np.asarray(knew_bits, dtype=np.uint16).reshape(Ly, Hkv, 1, d)
    vn = np.asarray(vnew_bits, dtype=np.uint16).reshape(Ly, Hkv, 1, d)
    seq.K_tail = np.concatenate([seq.K_tail, kn], axis=2)
    seq.V_tail = np.concatenate([seq.V_tail, vn], axis=2)
    seq.L += 1
    if seq.K_tail.shape[2] == P.window:          # the tail completes a window
        seq.windows.append(QWindow(len(seq.windows), UNROUTED, 0.0, seq.K_tail, seq.V_tail))
        seq.K_tail = seq.K_tail[:, :, :0].copy()
        seq.V_tail = seq.V_tail[:, :, :0].copy()
    q = _bits_to_f32(q_bits)
    out = np.zeros((Ly, Hq, d))
    probs = None
    live = [j for j, w in enumerate(seq.windows) if w.tier != EVICTED]
    m = np.array([seq.windows[j].m for j in live])
    s_layers = np.zeros((Ly, len(live)))
    for layer in range(Ly):
        K, V, owner = accessible(P, seq, layer)
        p, o = attention_f64(q[layer], K, V)
        out[layer] = o
        if want_probs:
            probs = np.zeros((Ly, Hq, K.shape[1])) if probs is None else probs
            probs[layer] = p
        tok = p.sum(axis=0) / Hq                 # head-averaged attention per token
        inw = owner >= 0                         # window sums: a library bin-count
        per_window = np.bincount(owner[inw], weights=tok[inw], minlength=len(seq.windows))
        s = per_window[live]
        s_layers[layer] = s
        if P.cumulative:                         # Eq. (1): add the layer's mass
            m = m + s
        else:
            m = P.alpha * s + (1.0 - P.alpha) * m
    for k, j in enumerate(live):
        seq.windows[j].m = float(m[k])
    routed = t % P.omega == 0
    scores_before = {seq.windows[j].wid: float(m[k]) for k, j in enumerate(live)}
    if routed:
        if ranking is None:
            route(P, seq)
        else:
            _route_in_order(P, seq, ranking)
    return dict(out=out, probs=probs, owner=owner, m=scores_before, routed=routed,
                tiers=seq.tiers(), s_layers=s_layers, live=live)


def _route_in_order(P: QParams, seq: QSequence, ranking):
    byid = {w.wid: w for w in seq.windows}
    saved = {w.wid: w.m for w in seq.windows}
    n = len(ranking)
    for r, wid in enumerate(ranking):            # scores that reproduce the given order
        byid[wid].m = float(n - r)
    route(P, seq)
    for w in seq.windows:
        w.m = saved[w.wid]
