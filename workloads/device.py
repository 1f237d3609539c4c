"""Seeded synthetic inputs drawn on the GPU, for workloads too large to draw
on the host (the 64-sequence, 8192-token block-granular workload holds
68.7 GB of K/V).

Values come from torch's CUDA generator (Philox), one generator per tensor
family and index, seeded from ``SeedSequence(entropy=seed, spawn_key=(family,
index))`` so any sequence's prefill or any step's inputs can be drawn alone.
Draws are fp32 N(0,1) rounded to bf16 by torch's round-to-nearest-even.  The
tensors land directly in the layouts the block-granular entry points take;
tests copy them to the host for the oracle.  Like ``gen``, this module holds
none of the eviction method's arithmetic.

Layouts:
  page pools    [batch * pps][n_layers][n_kv_heads][page][head_dim] bf16;
                prefill block j of sequence b at page b * pps + j
  backing tier  [batch][n_blocks][n_layers][n_kv_heads][page][head_dim] bf16
  q             [batch][n_layers][n_q_heads][head_dim] bf16
  k_new, v_new  [batch][n_layers][n_kv_heads][head_dim] bf16
"""
from __future__ import annotations

import numpy as np

# stream families of this module (part of the seed key; never reorder)
_D_K, _D_V, _D_NEEDLE, _D_Q, _D_KNEW, _D_VNEW = range(100, 106)


def _seed(seed: int, family: int, index: int) -> int:
    ss = np.random.SeedSequence(entropy=seed, spawn_key=(family, index))
    return int(ss.generate_state(1, np.uint64)[0] & np.uint64((1 << 63) - 1))


class PagedDeviceWorkload:
    """Block-granular workload: every sequence has ``prefill`` tokens of
    N(0,1) keys and values in ``page``-token blocks (rows past the prefill in
    a partial last block are drawn too and never read); each step's query is
    N(0,1) plus ``needle_weight`` times the mean prefill key of the sequence's
    needle blocks (``needle_blocks`` distinct prefill blocks, re-drawn at
    steps 1, 1 + P, 1 + 2P, ... with P = ``needle_period``; none when 0); new
    keys and values are N(0,1)."""

    def __init__(self, seed: int = 0, *, n_layers: int = 32, n_q_heads: int = 32,
                 n_kv_heads: int = 8, head_dim: int = 128, batch: int = 64,
                 prefill: int = 8192, page: int = 16, needle_blocks: int = 4,
                 needle_period: int = 200, needle_weight: float = 0.5):
        self.seed = int(seed)
        self.n_layers, self.n_q_heads, self.n_kv_heads = n_layers, n_q_heads, n_kv_heads
        self.head_dim, self.batch, self.prefill, self.page = head_dim, batch, prefill, page
        self.n_blocks = -(-prefill // page)   # the last block may be partial
        self.needle_blocks_n = int(needle_blocks)
        self.needle_period = int(needle_period)
        self.needle_weight = float(needle_weight)

    # ------------------------------------------------------------- prefill
    def _normal(self, torch, shape, family, index, device):
        g = torch.Generator(device=device)
        g.manual_seed(_seed(self.seed, family, index))
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(
            torch.bfloat16)

    def prefill_sequence(self, torch, b: int, device="cuda"):
        """(K, V) of sequence b: [n_blocks][n_layers][n_kv_heads][page][head_dim] bf16."""
        shape = (self.n_blocks, self.n_layers, self.n_kv_heads, self.page, self.head_dim)
        return (self._normal(torch, shape, _D_K, b, device),
                self._normal(torch, shape, _D_V, b, device))

    def fill(self, torch, k_pool, v_pool, pps: int, backing_k=None, backing_v=None):
        """Write every sequence's prefill into its pages (and the backing tier)."""
        for b in range(self.batch):
            k, v = self.prefill_sequence(torch, b, k_pool.device)
            k_pool[b * pps:b * pps + self.n_blocks].copy_(k)
            v_pool[b * pps:b * pps + self.n_blocks].copy_(v)
            if backing_k is not None:
                backing_k[b, :self.n_blocks].copy_(k)
                backing_v[b, :self.n_blocks].copy_(v)
            del k, v

    # -------------------------------------------------------------- decode
    def needle(self, step: int) -> np.ndarray:
        """[batch][needle_blocks] sorted logical ids of step ``step``'s needle."""
        epoch = (step - 1) // self.needle_period
        out = np.empty((self.batch, self.needle_blocks_n), dtype=np.int64)
        for b in range(self.batch):
            rng = np.random.Generator(np.random.PCG64(
                np.random.SeedSequence(entropy=self.seed, spawn_key=(_D_NEEDLE, epoch, b))))
            out[b] = np.sort(rng.choice(self.n_blocks, size=self.needle_blocks_n,
                                        replace=False))
        return out

    def step_inputs(self, torch, step: int, backing_k, device="cuda"):
        """(q, k_new, v_new) bf16 device tensors of decode step ``step``; the
        needle's mean key is taken from the backing tier (the original
        prefill keys, evicted or not)."""
        g = self.n_q_heads // self.n_kv_heads
        q = self._normal(torch, (self.batch, self.n_layers, self.n_q_heads, self.head_dim),
                         _D_Q, step, device).float()
        if self.needle_blocks_n:
            idx = torch.from_numpy(self.needle(step)).to(device)
            sel = backing_k[torch.arange(self.batch, device=device)[:, None], idx]
            mean = sel.float().mean(dim=(1, 4))                # [b][Ly][Hkv][d]
            q = q + self.needle_weight * mean.repeat_interleave(g, dim=2)
        kv = (self.batch, self.n_layers, self.n_kv_heads, self.head_dim)
        return (q.to(torch.bfloat16), self._normal(torch, kv, _D_KNEW, step, device),
                self._normal(torch, kv, _D_VNEW, step, device))


class TierDeviceWorkload:
    """Two-tier workload on the device: Llama-3.1-8B attention geometry,
    ``batch`` sequences of ``prefill`` tokens written in the windowed page
    layout (page 0 of a sequence holds the 5 sinks in rows 0-4, page 1 + i
    holds tokens 5 + 16 i .. 5 + 16 i + 15); keys N(0,1) with ``outliers``
    channels of std ``outlier_sigma``, values N(0,1); each step's query is
    N(0,1) plus ``needle_weight`` times the mean prefill key of 16 positions
    re-drawn every ``needle_period`` steps; new keys and values drawn like
    the prefill."""

    def __init__(self, seed: int = 0, *, n_layers: int = 32, n_q_heads: int = 32,
                 n_kv_heads: int = 8, head_dim: int = 128, batch: int = 4,
                 prefill: int = 131072, outliers: int = 4, outlier_sigma: float = 8.0,
                 needle: int = 16, needle_period: int = 64, needle_weight: float = 0.5):
        self.seed = int(seed)
        self.n_layers, self.n_q_heads, self.n_kv_heads = n_layers, n_q_heads, n_kv_heads
        self.head_dim, self.batch, self.prefill = head_dim, batch, prefill
        self.n_pages = 1 + -(-(prefill - 5) // 16)
        rng = np.random.Generator(np.random.PCG64(
            np.random.SeedSequence(entropy=self.seed, spawn_key=(_D_NEEDLE, 1 << 20))))
        self.outlier_channels = np.sort(rng.choice(head_dim, size=outliers, replace=False))
        self.outlier_sigma = float(outlier_sigma)
        self.needle_n, self.needle_period = int(needle), int(needle_period)
        self.needle_weight = float(needle_weight)

    def _normal(self, torch, shape, family, index, device):
        g = torch.Generator(device=device)
        g.manual_seed(_seed(self.seed, family, index))
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32)

    def _keys(self, torch, shape, family, index, device):
        k = self._normal(torch, shape, family, index, device)
        if len(self.outlier_channels):
            ch = torch.from_numpy(self.outlier_channels).to(device)
            k[..., ch] *= self.outlier_sigma
        return k.to(torch.bfloat16)

    def fill(self, torch, k_pool, v_pool, pps: int, chunk: int = 1024):
        """Draw the prefill pages in chunks of `chunk` pages (one generator
        per sequence and chunk)."""
        for b in range(self.batch):
            for c0 in range(0, self.n_pages, chunk):
                n = min(chunk, self.n_pages - c0)
                shape = (n, self.n_layers, self.n_kv_heads, 16, self.head_dim)
                idx = b * (1 << 16) + c0 // chunk
                dst = slice(b * pps + c0, b * pps + c0 + n)
                k_pool[dst].copy_(self._keys(torch, shape, _D_K, idx, k_pool.device))
                v_pool[dst].copy_(
                    self._normal(torch, shape, _D_V, idx, v_pool.device).to(torch.bfloat16))

    def needle(self, step: int) -> np.ndarray:
        """[batch][needle] sorted prefill positions of step ``step``'s needle."""
        epoch = (step - 1) // self.needle_period
        out = np.empty((self.batch, self.needle_n), dtype=np.int64)
        for b in range(self.batch):
            rng = np.random.Generator(np.random.PCG64(
                np.random.SeedSequence(entropy=self.seed, spawn_key=(_D_NEEDLE, epoch, b))))
            out[b] = np.sort(rng.choice(self.prefill, size=self.needle_n, replace=False))
        return out

    def step_inputs(self, torch, step: int, k_pool, pps: int, device="cuda"):
        """(q, k_new, v_new) of decode step ``step``; the needle's keys are read
        from the untouched prefill pages (call before any page is reused)."""
        g = self.n_q_heads // self.n_kv_heads
        q = self._normal(torch, (self.batch, self.n_layers, self.n_q_heads, self.head_dim),
                         _D_Q, step, device)
        if self.needle_n:
            pos = self.needle(step)
            page = np.where(pos < 5, 0, 1 + (pos - 5) // 16)
            row = np.where(pos < 5, pos, (pos - 5) % 16)
            pages = torch.from_numpy(page + np.arange(self.batch)[:, None] * pps).to(device)
            rows = torch.from_numpy(row).to(device)
            sel = k_pool[pages, :, :, rows].float()          # [b][needle][Ly][Hkv][d]
            q = q + self.needle_weight * sel.mean(dim=1).repeat_interleave(g, dim=2)
        kv = (self.batch, self.n_layers, self.n_kv_heads, self.head_dim)
        return (q.to(torch.bfloat16), self._keys(torch, kv, _D_KNEW, step, device),
                self._normal(torch, kv, _D_VNEW, step, device).to(torch.bfloat16))
