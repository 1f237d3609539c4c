"""Seeded generators for the synthetic decode workloads.

Every tensor family has its own independent PCG64 stream, keyed by
``SeedSequence(entropy=seed, spawn_key=(family, index))`` so any single step's
inputs can be drawn without replaying earlier steps.  Values are drawn in fp32
and rounded to bf16 with round-to-nearest-even; arrays hold the raw bf16 bit
patterns as ``uint16``.

Layouts (row-major, last index fastest):
  prefill K/V  : [n_layers][batch][n_kv_heads][L0][head_dim]
  q            : [batch][n_layers][n_q_heads][head_dim]
  k_new, v_new : [batch][n_layers][n_kv_heads][head_dim]

Workload shapes follow the pages' evaluation setups (Llama-3.1-8B GQA geometry,
a needle that the query is drawn toward, heavy-hitter keys); no benchmark item
is reproduced, every value is random.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# stream families (the integer is part of the seed key; never reorder)
_F_K, _F_V, _F_OUTLIER, _F_HEAVY, _F_NEEDLE, _F_Q, _F_KNEW, _F_VNEW = range(8)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def rope_table(n_pos: int, head_dim: int, base: float) -> np.ndarray:
    """[n_pos][head_dim/2][2] fp32 (cos, sin) of p * base^(-2 j / head_dim),
    formed in fp64 and rounded once (a model's rotary cache)."""
    inv = float(base) ** (-2.0 * np.arange(head_dim // 2, dtype=np.float64) / head_dim)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)


def _rng(seed: int, family: int, index: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence(entropy=seed, spawn_key=(family, index))
    return np.random.Generator(np.random.PCG64(ss))


@dataclass(frozen=True)
class Geometry:
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    batch: int = 1

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


class Workload:
    """A seeded decode workload: a prefilled cache plus per-step q/k/v.

    Options:
      outliers      number of key channels drawn with std ``outlier_sigma``
                    (the same channels in every layer and head)
      heavy         number of prefill positions whose key rows are scaled by
                    ``heavy_scale`` (all channels, all KV heads, all layers)
      needle        number of prefill positions whose mean key, times
                    ``needle_weight``, is added to every query; the set is
                    re-drawn at steps 1, 1+P, 1+2P, ... (P = ``needle_period``)
      rope_base     rotary positions: every key (prefill and new) is the drawn
                    key rotated by its position with the table of
                    ``rope_table`` (pairs (j, j + d/2), the rotation in fp64,
                    then rounded to bf16), as a model's cache holds them
    """

    def __init__(self, geom: Geometry, prefill_len: int, seed: int = 0, *,
                 outliers: int = 0, outlier_sigma: float = 8.0,
                 heavy: int = 0, heavy_scale: float = 4.0,
                 needle: int = 0, needle_period: int = 50,
                 needle_weight: float = 0.5, rope_base: float = None):
        self.geom = geom
        self.L0 = int(prefill_len)
        self.seed = int(seed)
        self.needle = int(needle)
        self.needle_period = int(needle_period)
        self.needle_weight = float(needle_weight)
        self.outlier_sigma = float(outlier_sigma)
        self.heavy_scale = float(heavy_scale)
        self.rope_base = None if rope_base is None else float(rope_base)
        d = geom.head_dim
        if outliers:
            ch = _rng(seed, _F_OUTLIER).choice(d, size=outliers, replace=False)
            self.outlier_channels = np.sort(ch)
        else:
            self.outlier_channels = np.zeros(0, dtype=np.int64)
        if heavy:
            pos = _rng(seed, _F_HEAVY).choice(self.L0, size=heavy, replace=False)
            self.heavy_positions = np.sort(pos)
        else:
            self.heavy_positions = np.zeros(0, dtype=np.int64)
        self._k = None
        self._v = None
        self._needle_cache = {}

    # ---------------------------------------------------------------- prefill
    def _key_block(self, rng: np.random.Generator, shape) -> np.ndarray:
        x = rng.standard_normal(shape, dtype=np.float32)
        if self.outlier_channels.size:
            x[..., self.outlier_channels] *= np.float32(self.outlier_sigma)
        return x

    def rope_table(self, n_pos: int) -> np.ndarray:
        """The rotary table of this workload's keys (see ``rope_table``)."""
        return rope_table(n_pos, self.geom.head_dim, self.rope_base)

    def _rotate(self, x: np.ndarray, pos: np.ndarray) -> np.ndarray:
        """Keys x [..., n, d] rotated by the table rows of positions pos [n]."""
        cs = self.rope_table(int(pos.max()) + 1)[pos].astype(np.float64)
        h = x.shape[-1] // 2
        a, b = x[..., :h].astype(np.float64), x[..., h:].astype(np.float64)
        c, s_ = cs[..., 0], cs[..., 1]
        return np.concatenate([a * c - b * s_, b * c + a * s_], axis=-1).astype(np.float32)

    def prefill_layer(self, layer: int):
        """bf16 bits of (K, V) for one layer: each [batch][n_kv][L0][d]."""
        g = self.geom
        shape = (g.batch, g.n_kv_heads, self.L0, g.head_dim)
        k = self._key_block(_rng(self.seed, _F_K, layer), shape)
        if self.heavy_positions.size:
            k[:, :, self.heavy_positions, :] *= np.float32(self.heavy_scale)
        if self.rope_base is not None:
            k = self._rotate(k, np.arange(self.L0))
        v = _rng(self.seed, _F_V, layer).standard_normal(shape, dtype=np.float32)
        return f32_to_bf16_bits(k), f32_to_bf16_bits(v)

    def prefill(self):
        """Full prefill (K, V) bits, [n_layers][batch][n_kv][L0][d]; cached."""
        if self._k is None:
            g = self.geom
            shape = (g.n_layers, g.batch, g.n_kv_heads, self.L0, g.head_dim)
            self._k = np.empty(shape, dtype=np.uint16)
            self._v = np.empty(shape, dtype=np.uint16)
            for layer in range(g.n_layers):
                self._k[layer], self._v[layer] = self.prefill_layer(layer)
        return self._k, self._v

    # ---------------------------------------------------------------- decode
    def needle_positions(self, step: int) -> np.ndarray:
        epoch = (step - 1) // self.needle_period
        pos = _rng(self.seed, _F_NEEDLE, epoch).choice(
            self.L0, size=self.needle, replace=False)
        return np.sort(pos)

    def _needle_mean(self, step: int) -> np.ndarray:
        """[batch][n_layers][n_kv][d] fp32 mean of the prefill keys at the
        needle positions (the original prefill keys, evicted or not)."""
        epoch = (step - 1) // self.needle_period
        if epoch not in self._needle_cache:
            k, _ = self.prefill()
            pos = self.needle_positions(step)
            kf = bf16_bits_to_f32(k[:, :, :, pos, :])   # [Ly][b][g][n][d]
            mean = kf.astype(np.float64).mean(axis=3).astype(np.float32)
            self._needle_cache = {epoch: np.ascontiguousarray(
                mean.transpose(1, 0, 2, 3))}
        return self._needle_cache[epoch]

    def step_inputs(self, step: int):
        """(q, k_new, v_new) bf16 bits for decode step ``step`` (1-based)."""
        if step < 1:
            raise ValueError("decode steps are numbered from 1")
        g = self.geom
        q = _rng(self.seed, _F_Q, step).standard_normal(
            (g.batch, g.n_layers, g.n_q_heads, g.head_dim), dtype=np.float32)
        if self.needle:
            nm = self._needle_mean(step)                     # [b][Ly][g][d]
            nm = np.repeat(nm, g.group, axis=2)              # [b][Ly][Hq][d]
            q = q + np.float32(self.needle_weight) * nm
        kv_shape = (g.batch, g.n_layers, g.n_kv_heads, g.head_dim)
        kn = self._key_block(_rng(self.seed, _F_KNEW, step), kv_shape)
        if self.rope_base is not None:   # the new token sits at position L0 + step - 1
            kn = self._rotate(kn[..., None, :], np.array([self.L0 + step - 1]))[..., 0, :]
        vn = _rng(self.seed, _F_VNEW, step).standard_normal(kv_shape, dtype=np.float32)
        return f32_to_bf16_bits(q), f32_to_bf16_bits(kn), f32_to_bf16_bits(vn)


def tiny_workload(seed: int = 0) -> Workload:
    """Token-granular tiny case: 1 layer, 8 q / 2 KV heads, head_dim 64,
    batch 1, a 512-token prefill of N(0,1) keys and values with 8 heavy-hitter
    key rows scaled by 4; per-step q, k, v ~ N(0,1)."""
    return Workload(Geometry(1, 8, 2, 64, 1), 512, seed, heavy=8, heavy_scale=4.0)


def llama8b_workload(seed: int = 0, prefill_len: int = 32768, *, n_layers: int = 32,
                     batch: int = 1, needle_period: int = 50) -> Workload:
    """Llama-3.1-8B attention geometry (32 q / 8 KV heads, head_dim 128): keys
    N(0,1) with 4 outlier channels of std 8, values N(0,1); each query is
    N(0,1) plus half the mean key of a 16-position needle re-drawn every
    ``needle_period`` steps."""
    return Workload(Geometry(n_layers, 32, 8, 128, batch), prefill_len, seed,
                    outliers=4, outlier_sigma=8.0, needle=16,
                    needle_period=needle_period, needle_weight=0.5)


def paged_workload(seed: int = 0, prefill_len: int = 8192, *, n_layers: int = 32,
                   batch: int = 64, needle_period: int = 200) -> Workload:
    """Block-granular workload: Llama-3.1-8B attention geometry, keys with 4
    outlier channels, queries drawn toward a 16-position needle set that is
    re-drawn every ``needle_period`` steps (the blocks holding the new set
    are the ones a caller re-admits when they were evicted)."""
    return Workload(Geometry(n_layers, 32, 8, 128, batch), prefill_len, seed,
                    outliers=4, outlier_sigma=8.0, needle=16,
                    needle_period=needle_period, needle_weight=0.5)


def needle_blocks(wl: Workload, step: int, page: int) -> np.ndarray:
    """Logical ids of the prefill blocks holding step ``step``'s needle set."""
    return np.unique(wl.needle_positions(step) // page)


# Region-aware workload: labelled contiguous spans of an agent context, in
# this order, each floor(fraction * n) tokens, the remainder scratchpad;
# half-lives in decode steps; the system span is pinned and decoded tokens
# are scratchpad.
REGION_NAMES = ("system", "plan", "user", "tool", "retrieved", "scratchpad")
REGION_FRACTIONS = (0.05, 0.05, 0.10, 0.30, 0.30)
REGION_HALF_LIVES = (160.0, 80.0, 60.0, 30.0, 40.0, 15.0)
REGION_PINNED = (True, False, False, False, False, False)
DECODE_REGION = 5


def region_spans(n: int):
    """Token counts of the six spans of an n-token context."""
    counts = [int(np.floor(f * n)) for f in REGION_FRACTIONS]
    return counts + [n - sum(counts)]


def region_labels(n: int) -> np.ndarray:
    """[n] uint8 region label of every prefill position."""
    return np.repeat(np.arange(len(REGION_NAMES), dtype=np.uint8), region_spans(n))


def memdecay_workload(seed: int = 0, prefill_len: int = 1700, *, n_layers: int = 36,
                      batch: int = 32) -> Workload:
    """Qwen2.5-3B attention geometry (16 q / 2 KV heads, head_dim 128); q, K,
    V ~ N(0,1); labels from ``region_labels``."""
    return Workload(Geometry(n_layers, 16, 2, 128, batch), prefill_len, seed)
