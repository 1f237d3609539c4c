"""Python binding of the kvev C ABI (include/kvev.h).

Argument marshalling only: every function has the C entry point's name,
takes torch tensors (or raw integer pointers) and raises KvevError on a
non-OK status.  Nothing here computes any part of the eviction pass; the
library must be built (``python -m decoding_kv_cache_split_gb300.build``)
and the binding refuses to run without it.

``EvictionPass`` is a convenience owner of the device buffers (ping-pong
cache, per-token state, outputs) for one context; it, too, only allocates
torch tensors and forwards to the C calls.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvev.so")

KVEV_OK, KVEV_EINVAL, KVEV_ENOMEM, KVEV_ECUDA, KVEV_ESTATE, KVEV_ETIMEOUT, KVEV_EUNSUPPORTED = range(7)
STATUS_NAMES = ["OK", "EINVAL", "ENOMEM", "ECUDA", "ESTATE", "ETIMEOUT", "EUNSUPPORTED"]
KVEV_REFRESH_FULL, KVEV_REFRESH_LAZY, KVEV_REFRESH_FROZEN = 0, 1, 2
KVEV_AGE_SINCE_INSERT, KVEV_AGE_SINCE_ACCESS = 0, 1
KVEV_POOL_SUM, KVEV_POOL_MEAN = 0, 1
KVEV_OUT_F32, KVEV_OUT_BF16 = 0, 1
KVEV_AGG_EMA, KVEV_AGG_CUMULATIVE = 0, 1
KVEV_W_VNORM, KVEV_W_ENTROPY = 1, 2
KVEV_DIAG_FIELDS = 8
KVEV_FUSED_OFF, KVEV_FUSED_ALL, KVEV_FUSED_ATTN_COMBINE = 0, 1, 2
DIAG_NAMES = ["step", "refreshed", "n_raw", "n_kept", "raw_and_kept", "raw_and_prev_raw",
              "n_prev_raw", "kept_and_prev_kept"]
KVEV_BF16 = 0
KVEV_MAX_REGIONS = 16
KVEV_SCORE_LRFU, KVEV_SCORE_MEMDECAY = 0, 1
KVEV_TIER_NONE, KVEV_TIER_UNROUTED, KVEV_TIER_FULL, KVEV_TIER_QUANT, KVEV_TIER_EVICTED = range(5)
KVEV_TIER_SINKS, KVEV_TIER_RECENT, KVEV_TIER_WINDOW = 5, 32, 128
TIER_LEDGER_BYTES = 12288   # one (window, layer, KV head) entry at head_dim 128
KVEV_PROFILE_SLOTS = 8
PROFILE_NAMES = ["append", "attention", "combine", "score", "select", "compact", "init_state",
                 "readmit"]

# every entry point declared in include/kvev.h
EXPORTS = ["kvev_create", "kvev_destroy", "kvev_last_error", "kvev_workspace_size",
           "kvev_refresh_mode", "kvev_configure", "kvev_set_output", "kvev_set_scorer",
           "kvev_set_fused_step", "kvev_test_barrier_timeout",
           "kvev_begin",
           "kvev_length",
           "kvev_init_state", "kvev_step", "kvev_step_host", "kvev_set_debug",
           "kvev_set_diagnostics", "kvev_missed_mass",
           "kvev_profile", "kvev_profile_read", "kvev_launch_count", "kvev_test_wait_timeout",
           "kvev_check_scratch", "kvev_sync",
           "kvev_paged_begin", "kvev_paged_step", "kvev_readmit", "kvev_set_tiers",
           "kvev_tier_diagnostics", "kvev_set_rope",
           "kvev_tier_begin", "kvev_tier_step", "kvev_export_state", "kvev_import_state",
           "kvev_attend_noalloc"]


class KvevError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"KVEV_{name}: {message}")


class kvev_layout(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("max_ctx", ctypes.c_int32),
                ("page_tokens", ctypes.c_int32), ("kv_dtype", ctypes.c_int32)]


class kvev_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p * 2), ("v", ctypes.c_void_p * 2), ("cur", ctypes.c_int32)]


class kvev_state(ctypes.Structure):
    _fields_ = [("score", ctypes.c_void_p), ("t_ins", ctypes.c_void_p),
                ("t_ref", ctypes.c_void_p), ("pos", ctypes.c_void_p)]


class kvev_paged_cache(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("pages_per_seq", ctypes.c_int32), ("block_table", ctypes.c_void_p),
                ("n_blocks", ctypes.c_void_p), ("free_pages", ctypes.c_void_p),
                ("n_free", ctypes.c_void_p), ("next_lid", ctypes.c_void_p),
                ("backing_k", ctypes.c_void_p), ("backing_v", ctypes.c_void_p),
                ("n_backing", ctypes.c_int32)]


class kvev_block_state(ctypes.Structure):
    _fields_ = [("score", ctypes.c_void_p), ("t_ins", ctypes.c_void_p),
                ("t_ref", ctypes.c_void_p), ("lid", ctypes.c_void_p), ("len", ctypes.c_void_p),
                ("table", ctypes.c_void_p), ("table_len", ctypes.c_int32),
                ("region", ctypes.c_void_p), ("tok_a", ctypes.c_void_p),
                ("tok_t_ref", ctypes.c_void_p)]


class kvev_region_table(ctypes.Structure):
    _fields_ = [("n_regions", ctypes.c_int32),
                ("base_priority", ctypes.c_float * KVEV_MAX_REGIONS),
                ("decay_lambda", ctypes.c_float * KVEV_MAX_REGIONS),
                ("pinned", ctypes.c_uint8 * KVEV_MAX_REGIONS),
                ("score_kind", ctypes.c_int32), ("rho", ctypes.c_float),
                ("attn_weight", ctypes.c_float), ("tau_scale", ctypes.c_float),
                ("decode_region", ctypes.c_int32)]


def region_table(base, lam, pinned, *, score_kind=KVEV_SCORE_MEMDECAY, rho=0.9,
                 attn_weight=0.5, tau_scale=2.0, decode_region=0) -> kvev_region_table:
    """A kvev_region_table from per-region lists."""
    n = len(base)
    t = kvev_region_table()
    t.n_regions = n
    for r in range(n):
        t.base_priority[r] = float(base[r])
        t.decay_lambda[r] = float(lam[r])
        t.pinned[r] = 1 if pinned[r] else 0
    t.score_kind, t.rho, t.attn_weight = int(score_kind), float(rho), float(attn_weight)
    t.tau_scale, t.decode_region = float(tau_scale), int(decode_region)
    return t


class kvev_tier_cache(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("pages_per_seq", ctypes.c_int32), ("free_pages", ctypes.c_void_p),
                ("n_free", ctypes.c_void_p), ("ledger", ctypes.c_void_p),
                ("max_windows", ctypes.c_int32)]


class kvev_tier_state(ctypes.Structure):
    _fields_ = [("score", ctypes.c_void_p), ("tier", ctypes.c_void_p),
                ("has_codes", ctypes.c_void_p), ("win_pages", ctypes.c_void_p),
                ("n_windows", ctypes.c_void_p), ("tail_pages", ctypes.c_void_p),
                ("tail_len", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                               "(python -m decoding_kv_cache_split_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        sig = {
            "kvev_create": ([P, I64, I32, F, F, P, P], I32),
            "kvev_destroy": ([P], None),
            "kvev_last_error": ([P], ctypes.c_char_p),
            "kvev_workspace_size": ([P, I64, P], I32),
            "kvev_refresh_mode": ([P, I32, I32], I32),
            "kvev_configure": ([P, I32, I32], I32),
            "kvev_set_output": ([P, I32], I32),
            "kvev_set_scorer": ([P, I32, I32], I32),
            "kvev_set_fused_step": ([P, I32], I32),
            "kvev_test_barrier_timeout": ([P, I32, ctypes.c_uint32], I32),
            "kvev_begin": ([P, I32], I32),
            "kvev_length": ([P, P], I32),
            "kvev_init_state": ([P, P, P], I32),
            "kvev_step": ([P, P, P, P, P, P, I64, P, P, P, P], I32),
            "kvev_step_host": ([P, P, P, P, P, P, I64, P, P, P, P], I32),
            "kvev_set_debug": ([P, P, P], I32),
            "kvev_set_diagnostics": ([P, P, P], I32),
            "kvev_missed_mass": ([P, I32, I32, P, I32, I32, I32, P, P], I32),
            "kvev_profile": ([P, I32], I32),
            "kvev_profile_read": ([P, P, P], I32),
            "kvev_launch_count": ([P, P], I32),
            "kvev_test_wait_timeout": ([P, I64, ctypes.c_uint32], I32),
            "kvev_check_scratch": ([P, P], I32),
            "kvev_sync": ([P, P], I32),
            "kvev_paged_begin": ([P, P, P, I32, P], I32),
            "kvev_paged_step": ([P, P, P, P, P, P, I64, P, P, P, P], I32),
            "kvev_readmit": ([P, P, P, I32, I32, I32, P], I32),
            "kvev_set_tiers": ([P, I64, I64, I32], I32),
            "kvev_tier_diagnostics": ([P, I32, P, P], I32),
            "kvev_set_rope": ([P, P, I32], I32),
            "kvev_tier_begin": ([P, P, P, I32, P], I32),
            "kvev_tier_step": ([P, P, P, P, P, P, I64, P, P], I32),
            "kvev_export_state": ([P, P, P], I32),
            "kvev_import_state": ([P, P, ctypes.c_size_t, P], I32),
            "kvev_attend_noalloc": ([P, P, P, P, I32, P, P, P], I32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, ctx=None):
    if status != KVEV_OK:
        raise KvevError(status, lib().kvev_last_error(ctx).decode())


# ------------------------------------------------------------------ C calls
def kvev_create(layout: kvev_layout, budget: int, granularity: int, alpha: float, beta: float,
                regions=None):
    out = ctypes.c_void_p()
    reg = ctypes.byref(regions) if isinstance(regions, kvev_region_table) else _ptr(regions)
    _check(lib().kvev_create(ctypes.byref(layout), int(budget), int(granularity), float(alpha),
                             float(beta), reg, ctypes.byref(out)))
    return out


def kvev_destroy(ctx) -> None:
    lib().kvev_destroy(ctx)


def kvev_last_error(ctx=None) -> str:
    return lib().kvev_last_error(ctx).decode()


def kvev_workspace_size(layout: kvev_layout, budget: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().kvev_workspace_size(ctypes.byref(layout), int(budget), ctypes.byref(n)))
    return n.value


def kvev_refresh_mode(ctx, mode: int, period: int = 1) -> None:
    _check(lib().kvev_refresh_mode(ctx, int(mode), int(period)), ctx)


def kvev_configure(ctx, age_mode: int, pool: int) -> None:
    _check(lib().kvev_configure(ctx, int(age_mode), int(pool)), ctx)


def kvev_set_output(ctx, out_type: int) -> None:
    _check(lib().kvev_set_output(ctx, int(out_type)), ctx)


def kvev_set_scorer(ctx, aggregation: int, weighting: int = 0) -> None:
    _check(lib().kvev_set_scorer(ctx, int(aggregation), int(weighting)), ctx)


def kvev_set_fused_step(ctx, mode: int) -> None:
    """KVEV_FUSED_OFF, KVEV_FUSED_ALL or KVEV_FUSED_ATTN_COMBINE (True: ALL)."""
    _check(lib().kvev_set_fused_step(ctx, int(mode)), ctx)


def kvev_test_barrier_timeout(ctx, cta: int, wait_limit: int) -> None:
    """Test-only barrier timeout injection for the next fused step."""
    _check(lib().kvev_test_barrier_timeout(ctx, int(cta), int(wait_limit)), ctx)


def kvev_begin(ctx, prefill_len: int) -> None:
    _check(lib().kvev_begin(ctx, int(prefill_len)), ctx)


def kvev_length(ctx) -> int:
    n = ctypes.c_int32()
    _check(lib().kvev_length(ctx, ctypes.byref(n)), ctx)
    return n.value


def kvev_init_state(ctx, state: kvev_state, stream=None) -> None:
    _check(lib().kvev_init_state(ctx, ctypes.byref(state), _stream(stream)), ctx)


def kvev_step(ctx, q, k_new, v_new, cache: kvev_cache, state: kvev_state, step: int, out,
              retained_idx, n_retained, stream=None) -> None:
    _check(lib().kvev_step(ctx, _ptr(q), _ptr(k_new), _ptr(v_new), ctypes.byref(cache),
                           ctypes.byref(state), int(step), _ptr(out), _ptr(retained_idx),
                           _ptr(n_retained), _stream(stream)), ctx)


def kvev_step_host(ctx, q, k_new, v_new, cache: kvev_cache, state: kvev_state, step: int, out,
                   retained_idx, n_retained, stream=None) -> None:
    _check(lib().kvev_step_host(ctx, _ptr(q), _ptr(k_new), _ptr(v_new), ctypes.byref(cache),
                                ctypes.byref(state), int(step), _ptr(out), _ptr(retained_idx),
                                _ptr(n_retained), _stream(stream)), ctx)


def kvev_set_debug(ctx, probs=None, priority=None) -> None:
    _check(lib().kvev_set_debug(ctx, _ptr(probs), _ptr(priority)), ctx)


def kvev_set_diagnostics(ctx, counters=None, raw_score=None) -> None:
    _check(lib().kvev_set_diagnostics(ctx, _ptr(counters), _ptr(raw_score)), ctx)


def kvev_missed_mass(full_score, score_ld: int, n_pos: int, pos, pos_ld: int, n_cached: int,
                     batch: int, out, stream=None) -> None:
    """Future Missed Mass of one step (see include/kvev.h)."""
    _check(lib().kvev_missed_mass(_ptr(full_score), int(score_ld), int(n_pos), _ptr(pos),
                                  int(pos_ld), int(n_cached), int(batch), _ptr(out),
                                  _stream(stream)))


def kvev_profile(ctx, enable: bool) -> None:
    _check(lib().kvev_profile(ctx, int(bool(enable))), ctx)


def kvev_profile_read(ctx):
    ms = (ctypes.c_float * KVEV_PROFILE_SLOTS)()
    n = (ctypes.c_int64 * KVEV_PROFILE_SLOTS)()
    _check(lib().kvev_profile_read(ctx, ms, n), ctx)
    return {PROFILE_NAMES[i]: (ms[i], n[i]) for i in range(KVEV_PROFILE_SLOTS) if n[i]}


def kvev_launch_count(ctx) -> int:
    n = ctypes.c_int64()
    _check(lib().kvev_launch_count(ctx, ctypes.byref(n)), ctx)
    return n.value


def kvev_test_wait_timeout(ctx, tile: int, wait_limit: int) -> None:
    """Test-only timeout injection for the next step (see include/kvev.h)."""
    _check(lib().kvev_test_wait_timeout(ctx, int(tile), int(wait_limit)), ctx)


def kvev_check_scratch(ctx, stream=None) -> None:
    """Raise KvevError if a guard band of the context's scratch was overwritten."""
    _check(lib().kvev_check_scratch(ctx, _stream(stream)), ctx)


def kvev_sync(ctx, stream=None) -> None:
    _check(lib().kvev_sync(ctx, _stream(stream)), ctx)


def kvev_paged_begin(ctx, cache: kvev_paged_cache, state: kvev_block_state, prefill_tokens: int,
                     stream=None) -> None:
    _check(lib().kvev_paged_begin(ctx, ctypes.byref(cache), ctypes.byref(state),
                                  int(prefill_tokens), _stream(stream)), ctx)


def kvev_paged_step(ctx, q, k_new, v_new, cache: kvev_paged_cache, state: kvev_block_state,
                    step: int, out, retained_lid, n_retained, stream=None) -> None:
    _check(lib().kvev_paged_step(ctx, _ptr(q), _ptr(k_new), _ptr(v_new), ctypes.byref(cache),
                                 ctypes.byref(state), int(step), _ptr(out), _ptr(retained_lid),
                                 _ptr(n_retained), _stream(stream)), ctx)


def kvev_readmit(ctx, cache: kvev_paged_cache, state: kvev_block_state, seq: int, lid: int,
                 persist: bool = True, stream=None) -> None:
    _check(lib().kvev_readmit(ctx, ctypes.byref(cache), ctypes.byref(state), int(seq), int(lid),
                              int(bool(persist)), _stream(stream)), ctx)


def kvev_set_tiers(ctx, k_full: int, k_quant: int, omega: int) -> None:
    _check(lib().kvev_set_tiers(ctx, int(k_full), int(k_quant), int(omega)), ctx)


def kvev_tier_diagnostics(ctx, sustain: int, counters=None, stream=None) -> None:
    _check(lib().kvev_tier_diagnostics(ctx, int(sustain), _ptr(counters), _stream(stream)), ctx)


def kvev_set_rope(ctx, table, n_pos: int) -> None:
    """table: the model's (cos, sin) cache [n_pos][d/2][2] fp32 on the device
    (kept alive by the caller), or None to turn rotary mode off."""
    _check(lib().kvev_set_rope(ctx, _ptr(table), int(n_pos)), ctx)


def kvev_tier_begin(ctx, cache: kvev_tier_cache, state: kvev_tier_state, prefill_tokens: int,
                    stream=None) -> None:
    _check(lib().kvev_tier_begin(ctx, ctypes.byref(cache), ctypes.byref(state),
                                 int(prefill_tokens), _stream(stream)), ctx)


def kvev_tier_step(ctx, q, k_new, v_new, cache: kvev_tier_cache, state: kvev_tier_state,
                   step: int, out, stream=None) -> None:
    _check(lib().kvev_tier_step(ctx, _ptr(q), _ptr(k_new), _ptr(v_new), ctypes.byref(cache),
                                ctypes.byref(state), int(step), _ptr(out), _stream(stream)), ctx)


def kvev_export_state(ctx) -> bytes:
    """The context's own state as a byte string (see include/kvev.h)."""
    n = ctypes.c_size_t()
    _check(lib().kvev_export_state(ctx, None, ctypes.byref(n)), ctx)
    buf = ctypes.create_string_buffer(n.value)
    _check(lib().kvev_export_state(ctx, buf, ctypes.byref(n)), ctx)
    return buf.raw[:n.value]


def kvev_import_state(ctx, blob: bytes, stream=None) -> None:
    buf = ctypes.create_string_buffer(blob, len(blob))
    _check(lib().kvev_import_state(ctx, buf, len(blob), _stream(stream)), ctx)


def kvev_attend_noalloc(layout: kvev_layout, q, k, v, length: int, out, lse2, stream=None) -> None:
    """Attention of the pass with no allocation (see include/kvev.h)."""
    _check(lib().kvev_attend_noalloc(ctypes.byref(layout), _ptr(q), _ptr(k), _ptr(v), int(length),
                                     _ptr(out), _ptr(lse2), _stream(stream)))


# ------------------------------------------------------------- buffer owner
class EvictionPass:
    """Device buffers plus a context for one decode run (token granularity).

    Cache buffers: k[2], v[2] each [Ly][b][Hkv][max_ctx][d] bf16; state arrays
    [b][max_ctx]; outputs out [b][Ly][Hq][d] fp32 (bf16 with out_type
    KVEV_OUT_BF16), retained [b][budget] int32, n_retained [b] int32.  All
    torch tensors on the current CUDA device."""

    def __init__(self, n_layers, n_q_heads, n_kv_heads, head_dim, batch, max_ctx, budget,
                 alpha, beta, *, age_mode=KVEV_AGE_SINCE_INSERT, pool=KVEV_POOL_SUM,
                 refresh=KVEV_REFRESH_FULL, period=1, out_type=KVEV_OUT_F32,
                 aggregation=KVEV_AGG_EMA, weighting=0, fused=False, device="cuda"):
        import torch
        self.torch = torch
        self.layout = kvev_layout(n_layers, n_q_heads, n_kv_heads, head_dim, batch, max_ctx, 1,
                                  KVEV_BF16)
        self.budget = int(budget)
        self.ctx = kvev_create(self.layout, budget, 1, alpha, beta)
        kvev_configure(self.ctx, age_mode, pool)
        kvev_refresh_mode(self.ctx, refresh, period)
        kvev_set_output(self.ctx, out_type)
        kvev_set_scorer(self.ctx, aggregation, weighting)
        if fused:
            kvev_set_fused_step(self.ctx, KVEV_FUSED_ALL if fused is True else int(fused))
        shape = (n_layers, batch, n_kv_heads, max_ctx, head_dim)
        self.k = [torch.zeros(shape, dtype=torch.bfloat16, device=device) for _ in range(2)]
        self.v = [torch.zeros(shape, dtype=torch.bfloat16, device=device) for _ in range(2)]
        self.score = torch.zeros((batch, max_ctx), dtype=torch.float32, device=device)
        self.t_ins = torch.zeros((batch, max_ctx), dtype=torch.int32, device=device)
        self.t_ref = torch.zeros((batch, max_ctx), dtype=torch.int32, device=device)
        self.pos = torch.zeros((batch, max_ctx), dtype=torch.int32, device=device)
        self.out = torch.zeros((batch, n_layers, n_q_heads, head_dim),
                               dtype=torch.bfloat16 if out_type == KVEV_OUT_BF16 else torch.float32,
                               device=device)
        self.retained = torch.zeros((batch, self.budget), dtype=torch.int32, device=device)
        self.n_retained = torch.zeros((batch,), dtype=torch.int32, device=device)
        self.cache = kvev_cache((ctypes.c_void_p * 2)(self.k[0].data_ptr(), self.k[1].data_ptr()),
                                (ctypes.c_void_p * 2)(self.v[0].data_ptr(), self.v[1].data_ptr()),
                                0)
        self.state = kvev_state(self.score.data_ptr(), self.t_ins.data_ptr(),
                                self.t_ref.data_ptr(), self.pos.data_ptr())
        self.step_no = 0

    @property
    def cur(self) -> int:
        return self.cache.cur

    def live_k(self):
        return self.k[self.cache.cur]

    def live_v(self):
        return self.v[self.cache.cur]

    def begin(self, prefill_len: int, stream=None, cur: int = 0):
        """Start a run over the prefill already written into buffer ``cur``."""
        self.cache.cur = cur
        kvev_begin(self.ctx, prefill_len)
        kvev_init_state(self.ctx, self.state, stream)
        self.step_no = 0

    def length(self) -> int:
        return kvev_length(self.ctx)

    def step(self, q, k_new, v_new, stream=None):
        self.step_no += 1
        kvev_step(self.ctx, q, k_new, v_new, self.cache, self.state, self.step_no, self.out,
                  self.retained, self.n_retained, stream)
        return self.out, self.retained, self.n_retained

    def close(self):
        if self.ctx is not None:
            kvev_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class PagedEvictionPass:
    """Device buffers plus a context for one block-granular run.

    Page pools k_pool, v_pool [batch * pps][Ly][Hkv][P][d] bf16; block table,
    free stack and per-block state [batch][pps]; persisted scores
    [batch][table_len]; the backing tier (prefill blocks, for re-admission)
    [batch][n_backing][Ly][Hkv][P][d] bf16.  All torch tensors on the
    current CUDA device."""

    def __init__(self, n_layers, n_q_heads, n_kv_heads, head_dim, batch, pages_per_seq, page,
                 budget, alpha, beta, *, n_backing=0, table_len=None,
                 age_mode=KVEV_AGE_SINCE_ACCESS, pool=KVEV_POOL_SUM, refresh=KVEV_REFRESH_FULL,
                 period=1, regions=None, device="cuda"):
        import torch
        self.torch = torch
        self.page, self.pps, self.budget = int(page), int(pages_per_seq), int(budget)
        self.layout = kvev_layout(n_layers, n_q_heads, n_kv_heads, head_dim, batch,
                                  self.pps * self.page, self.page, KVEV_BF16)
        self.regions = regions
        self.ctx = kvev_create(self.layout, budget, self.page, alpha, beta, regions)
        kvev_configure(self.ctx, age_mode, pool)
        kvev_refresh_mode(self.ctx, refresh, period)
        pshape = (batch * self.pps, n_layers, n_kv_heads, self.page, head_dim)
        self.k_pool = torch.zeros(pshape, dtype=torch.bfloat16, device=device)
        self.v_pool = torch.zeros(pshape, dtype=torch.bfloat16, device=device)
        i32 = dict(dtype=torch.int32, device=device)
        self.block_table = torch.zeros((batch, self.pps), **i32)
        self.n_blocks = torch.zeros((batch,), **i32)
        self.free_pages = torch.zeros((batch, self.pps), **i32)
        self.n_free = torch.zeros((batch,), **i32)
        self.next_lid = torch.zeros((batch,), **i32)
        bshape = (batch, max(int(n_backing), 1), n_layers, n_kv_heads, self.page, head_dim)
        self.backing_k = torch.zeros(bshape, dtype=torch.bfloat16, device=device)
        self.backing_v = torch.zeros(bshape, dtype=torch.bfloat16, device=device)
        self.score = torch.zeros((batch, self.pps), dtype=torch.float32, device=device)
        self.t_ins = torch.zeros((batch, self.pps), **i32)
        self.t_ref = torch.zeros((batch, self.pps), **i32)
        self.lid = torch.zeros((batch, self.pps), **i32)
        self.len = torch.zeros((batch, self.pps), **i32)
        self.table_len = int(table_len if table_len is not None else max(int(n_backing), 1))
        self.table = torch.zeros((batch, self.table_len), dtype=torch.float32, device=device)
        self.out = torch.zeros((batch, n_layers, n_q_heads, head_dim), dtype=torch.float32,
                               device=device)
        ntok = batch * self.pps * self.page
        self.region = torch.zeros((ntok,), dtype=torch.uint8, device=device)
        self.tok_a = torch.zeros((ntok,), dtype=torch.float32, device=device)
        self.tok_t_ref = torch.zeros((ntok,), **i32)
        self.retained_lid = torch.zeros((batch, self.pps if regions is not None else self.budget),
                                        **i32)
        self.n_retained = torch.zeros((batch,), **i32)
        self.cache = kvev_paged_cache(
            self.k_pool.data_ptr(), self.v_pool.data_ptr(), self.pps, self.block_table.data_ptr(),
            self.n_blocks.data_ptr(), self.free_pages.data_ptr(), self.n_free.data_ptr(),
            self.next_lid.data_ptr(), self.backing_k.data_ptr(), self.backing_v.data_ptr(),
            int(n_backing))
        self.state = kvev_block_state(self.score.data_ptr(), self.t_ins.data_ptr(),
                                      self.t_ref.data_ptr(), self.lid.data_ptr(),
                                      self.len.data_ptr(), self.table.data_ptr(), self.table_len,
                                      self.region.data_ptr(), self.tok_a.data_ptr(),
                                      self.tok_t_ref.data_ptr())
        self.step_no = 0

    def begin(self, prefill_tokens: int, stream=None):
        """Start a run over the prefill already written into pages b*pps + j."""
        kvev_paged_begin(self.ctx, self.cache, self.state, prefill_tokens, stream)
        self.step_no = 0

    def step(self, q, k_new, v_new, stream=None):
        self.step_no += 1
        kvev_paged_step(self.ctx, q, k_new, v_new, self.cache, self.state, self.step_no, self.out,
                        self.retained_lid, self.n_retained, stream)
        return self.out, self.retained_lid, self.n_retained

    def readmit(self, seq: int, lid: int, persist: bool = True, stream=None):
        kvev_readmit(self.ctx, self.cache, self.state, seq, lid, persist, stream)

    def close(self):
        if self.ctx is not None:
            kvev_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class TierEvictionPass:
    """Device buffers plus a context for one two-tier (bf16 + INT2) run.

    bf16 page pools [batch * pps][Ly][Hkv][16][d] (page b*pps holds the 5
    sinks, page b*pps + 1 + i tokens 5 + 16 i ..); the INT2 ledger
    [batch][max_windows][Ly][Hkv][12288] bytes; per-window score, tier,
    ledger flag and pages; outputs out [b][Ly][Hq][d] fp32.  All torch
    tensors on the current CUDA device.  rope: the model's rotary table
    [positions >= max_ctx][d/2][2] (cos, sin) for rotary mode (the pools
    then hold rotated keys, and pages_per_seq must also hold the 8 k_quant
    reconstruction pages at the end of each sequence's range)."""

    def __init__(self, n_layers, n_q_heads, n_kv_heads, head_dim, batch, max_ctx, pages_per_seq,
                 k_full, k_quant, omega, alpha, aggregation=KVEV_AGG_EMA, rope=None,
                 device="cuda"):
        import torch
        self.torch = torch
        self.pps, self.max_ctx = int(pages_per_seq), int(max_ctx)
        self.max_windows = (self.max_ctx - KVEV_TIER_SINKS) // KVEV_TIER_WINDOW
        self.layout = kvev_layout(n_layers, n_q_heads, n_kv_heads, head_dim, batch, self.max_ctx,
                                  KVEV_TIER_WINDOW, KVEV_BF16)
        self.ctx = kvev_create(self.layout, k_full, KVEV_TIER_WINDOW, alpha, 0.0)
        kvev_set_tiers(self.ctx, k_full, k_quant, omega)
        kvev_set_scorer(self.ctx, aggregation, 0)
        self.rope = None
        if rope is not None:   # [positions][d/2][2] (cos, sin): rotated keys in the pools
            self.rope = torch.as_tensor(rope, dtype=torch.float32).to(device).contiguous()
            kvev_set_rope(self.ctx, self.rope, self.rope.shape[0])
        i32 = dict(dtype=torch.int32, device=device)
        pshape = (batch * self.pps, n_layers, n_kv_heads, 16, head_dim)
        self.k_pool = torch.zeros(pshape, dtype=torch.bfloat16, device=device)
        self.v_pool = torch.zeros(pshape, dtype=torch.bfloat16, device=device)
        self.free_pages = torch.zeros((batch, self.pps), **i32)
        self.n_free = torch.zeros((batch,), **i32)
        MW = self.max_windows
        self.ledger = torch.zeros((batch, MW, n_layers, n_kv_heads, TIER_LEDGER_BYTES),
                                  dtype=torch.uint8, device=device)
        self.score = torch.zeros((batch, MW), dtype=torch.float32, device=device)
        self.tier = torch.zeros((batch, MW), dtype=torch.uint8, device=device)
        self.has_codes = torch.zeros((batch, MW), dtype=torch.uint8, device=device)
        self.win_pages = torch.zeros((batch, MW, 8), **i32)
        self.n_windows = torch.zeros((batch,), **i32)
        self.tail_pages = torch.zeros((batch, 8), **i32)
        self.tail_len = torch.zeros((batch,), **i32)
        self.out = torch.zeros((batch, n_layers, n_q_heads, head_dim), dtype=torch.float32,
                               device=device)
        self.cache = kvev_tier_cache(self.k_pool.data_ptr(), self.v_pool.data_ptr(), self.pps,
                                     self.free_pages.data_ptr(), self.n_free.data_ptr(),
                                     self.ledger.data_ptr(), MW)
        self.state = kvev_tier_state(self.score.data_ptr(), self.tier.data_ptr(),
                                     self.has_codes.data_ptr(), self.win_pages.data_ptr(),
                                     self.n_windows.data_ptr(), self.tail_pages.data_ptr(),
                                     self.tail_len.data_ptr())
        self.step_no = 0

    def begin(self, prefill_tokens: int, stream=None):
        kvev_tier_begin(self.ctx, self.cache, self.state, prefill_tokens, stream)
        self.step_no = 0

    def step(self, q, k_new, v_new, stream=None):
        self.step_no += 1
        kvev_tier_step(self.ctx, q, k_new, v_new, self.cache, self.state, self.step_no, self.out,
                       stream)
        return self.out

    def close(self):
        if self.ctx is not None:
            kvev_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
