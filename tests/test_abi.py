"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point that include/kvev.h declares, and rejects
bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from decoding_kv_cache_split_gb300 import build as kbuild
from decoding_kv_cache_split_gb300 import kvev

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kvev.lib()


def declared_entry_points():
    text = open(os.path.join(ROOT, "include", "kvev.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvev_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_what_the_binding_wraps():
    assert declared_entry_points() == sorted(kvev.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), name


def layout(**kw):
    base = dict(n_layers=2, n_q_heads=8, n_kv_heads=2, head_dim=128, batch=1, max_ctx=64,
                page_tokens=1, kv_dtype=0)
    base.update(kw)
    return kvev.kvev_layout(*[base[f] for f, _ in kvev.kvev_layout._fields_])


@pytest.mark.parametrize("kw,budget,status", [
    (dict(head_dim=96), 8, kvev.KVEV_EUNSUPPORTED),
    (dict(n_q_heads=7), 8, kvev.KVEV_EINVAL),
    (dict(n_q_heads=32), 8, kvev.KVEV_EUNSUPPORTED),             # 16 query heads per KV head
    (dict(batch=0), 8, kvev.KVEV_EINVAL),
    (dict(page_tokens=8), 4, kvev.KVEV_EUNSUPPORTED),
    (dict(page_tokens=16), 4, kvev.KVEV_EINVAL),                # budget counts pages: 4 of 4
    (dict(page_tokens=16, max_ctx=72), 2, kvev.KVEV_EINVAL),    # not whole pages
    ({}, 0, kvev.KVEV_EINVAL),
    ({}, 64, kvev.KVEV_EINVAL),
])
def test_create_rejects_bad_layouts(lib, kw, budget, status):
    out = ctypes.c_void_p()
    lay = layout(**kw)
    rc = lib.kvev_create(ctypes.byref(lay), budget, lay.page_tokens, 0.05, 0.001, None,
                         ctypes.byref(out))
    assert rc == status
    assert out.value is None
    assert kvev.kvev_last_error()


def test_create_rejects_bad_scalars(lib):
    out = ctypes.c_void_p()
    lay = layout()
    assert lib.kvev_create(ctypes.byref(lay), 8, 1, 0.0, 0.001, None, ctypes.byref(out)) == kvev.KVEV_EINVAL
    assert lib.kvev_create(ctypes.byref(lay), 8, 1, 1.5, 0.001, None, ctypes.byref(out)) == kvev.KVEV_EINVAL
    assert lib.kvev_create(ctypes.byref(lay), 8, 1, 0.05, -1.0, None, ctypes.byref(out)) == kvev.KVEV_EINVAL
    assert lib.kvev_create(ctypes.byref(lay), 8, 2, 0.05, 0.001, None, ctypes.byref(out)) == kvev.KVEV_EINVAL
    assert lib.kvev_create(None, 8, 1, 0.05, 0.001, None, ctypes.byref(out)) == kvev.KVEV_EINVAL
    assert lib.kvev_create(ctypes.byref(lay), 8, 1, 0.05, 0.001, None, None) == kvev.KVEV_EINVAL


def test_null_context_is_rejected(lib):
    assert lib.kvev_refresh_mode(None, 0, 1) == kvev.KVEV_EINVAL
    assert lib.kvev_configure(None, 0, 0) == kvev.KVEV_EINVAL
    assert lib.kvev_begin(None, 0) == kvev.KVEV_EINVAL
    assert lib.kvev_step(None, None, None, None, None, None, 1, None, None, None, None) == kvev.KVEV_EINVAL
    assert lib.kvev_sync(None, None) == kvev.KVEV_EINVAL
    lib.kvev_destroy(None)   # no-op


def _out():
    return ctypes.byref(ctypes.c_int64())


# every entry point that takes a context, called with a NULL one (and NULL
# for its other pointers): KVEV_EINVAL with a message, before any CUDA call
NULL_CTX_CALLS = {
    "kvev_length": lambda L: L.kvev_length(None, _out()),
    "kvev_init_state": lambda L: L.kvev_init_state(None, None, None),
    "kvev_step_host": lambda L: L.kvev_step_host(None, None, None, None, None, None, 1, None,
                                                 None, None, None),
    "kvev_set_debug": lambda L: L.kvev_set_debug(None, None, None),
    "kvev_set_output": lambda L: L.kvev_set_output(None, 1),
    "kvev_set_scorer": lambda L: L.kvev_set_scorer(None, 1, 0),
    "kvev_set_diagnostics": lambda L: L.kvev_set_diagnostics(None, None, None),
    "kvev_set_fused_step": lambda L: L.kvev_set_fused_step(None, 1),
    "kvev_test_barrier_timeout": lambda L: L.kvev_test_barrier_timeout(None, 0, 10),
    "kvev_profile": lambda L: L.kvev_profile(None, 1),
    "kvev_profile_read": lambda L: L.kvev_profile_read(None, None, None),
    "kvev_launch_count": lambda L: L.kvev_launch_count(None, _out()),
    "kvev_test_wait_timeout": lambda L: L.kvev_test_wait_timeout(None, 0, 1),
    "kvev_check_scratch": lambda L: L.kvev_check_scratch(None, None),
    "kvev_paged_begin": lambda L: L.kvev_paged_begin(None, None, None, 0, None),
    "kvev_paged_step": lambda L: L.kvev_paged_step(None, None, None, None, None, None, 1, None,
                                                   None, None, None),
    "kvev_readmit": lambda L: L.kvev_readmit(None, None, None, 0, 0, 1, None),
    "kvev_set_tiers": lambda L: L.kvev_set_tiers(None, 1, 1, 8),
    "kvev_tier_diagnostics": lambda L: L.kvev_tier_diagnostics(None, 4, None, None),
    "kvev_set_rope": lambda L: L.kvev_set_rope(None, None, 0),
    "kvev_tier_begin": lambda L: L.kvev_tier_begin(None, None, None, 0, None),
    "kvev_tier_step": lambda L: L.kvev_tier_step(None, None, None, None, None, None, 1, None, None),
    "kvev_export_state": lambda L: L.kvev_export_state(None, None, _out()),
    "kvev_import_state": lambda L: L.kvev_import_state(None, None, 0, None),
}


def test_every_context_call_is_covered():
    with_ctx = {"kvev_refresh_mode", "kvev_configure", "kvev_begin", "kvev_step", "kvev_sync"}
    no_ctx = {"kvev_create", "kvev_destroy", "kvev_last_error", "kvev_workspace_size",
              "kvev_attend_noalloc", "kvev_missed_mass"}
    assert set(NULL_CTX_CALLS) | with_ctx | no_ctx == set(kvev.EXPORTS)


@pytest.mark.parametrize("name", sorted(NULL_CTX_CALLS))
def test_every_entry_point_rejects_a_null_context(lib, name):
    assert NULL_CTX_CALLS[name](lib) == kvev.KVEV_EINVAL
    assert kvev.kvev_last_error()


def test_noalloc_rejects_null_buffers_and_bad_layouts(lib):
    lay = layout(max_ctx=64)
    one = ctypes.c_void_p(16)          # never dereferenced: refused before any access
    assert lib.kvev_attend_noalloc(None, one, one, one, 8, one, one, None) == kvev.KVEV_EINVAL
    assert lib.kvev_attend_noalloc(ctypes.byref(lay), None, one, one, 8, one, one, None) == kvev.KVEV_EINVAL
    assert lib.kvev_attend_noalloc(ctypes.byref(lay), one, one, one, 0, one, one, None) == kvev.KVEV_EINVAL
    assert lib.kvev_attend_noalloc(ctypes.byref(lay), one, one, one, 65, one, one, None) == kvev.KVEV_EINVAL
    bad = layout(head_dim=96)
    assert lib.kvev_attend_noalloc(ctypes.byref(bad), one, one, one, 8, one, one, None) == \
        kvev.KVEV_EUNSUPPORTED


def test_binding_raises_with_message(lib):
    with pytest.raises(kvev.KvevError) as ei:
        kvev.kvev_create(layout(head_dim=80), 8, 1, 0.05, 0.001)
    assert ei.value.status == kvev.KVEV_EUNSUPPORTED
    assert "head_dim" in str(ei.value)


def _table(**kw):
    t = kvev.region_table([1.0, 1.0], [0.1, 0.2], [True, False], decode_region=1)
    for k, v in kw.items():
        setattr(t, k, v)
    return t


@pytest.mark.parametrize("lay_kw,table_kw,status", [
    ({}, {}, kvev.KVEV_EUNSUPPORTED),                                  # token granularity
    (dict(page_tokens=16), dict(n_regions=0), kvev.KVEV_EINVAL),
    (dict(page_tokens=16), dict(n_regions=17), kvev.KVEV_EINVAL),
    (dict(page_tokens=16), dict(decode_region=2), kvev.KVEV_EINVAL),
    (dict(page_tokens=16), dict(rho=1.0), kvev.KVEV_EINVAL),
    (dict(page_tokens=16), dict(score_kind=7), kvev.KVEV_EINVAL),
])
def test_create_rejects_bad_region_tables(lib, lay_kw, table_kw, status):
    out = ctypes.c_void_p()
    lay = layout(max_ctx=256, **lay_kw)
    t = _table(**table_kw)
    rc = lib.kvev_create(ctypes.byref(lay), 8, lay.page_tokens, 0.05, 0.001, ctypes.byref(t),
                         ctypes.byref(out))
    assert rc == status
    assert out.value is None


def test_region_table_layout_matches_the_header():
    """Field offsets of the ctypes mirror (the C struct has no padding
    before score_kind: 4 + 64 + 64 + 16 bytes)."""
    T = kvev.kvev_region_table
    assert T.base_priority.offset == 4 and T.decay_lambda.offset == 68
    assert T.pinned.offset == 132 and T.score_kind.offset == 148
    assert ctypes.sizeof(T) == 168


def test_missed_mass_rejects_bad_arguments(lib):
    one = ctypes.c_void_p(16)          # never dereferenced: refused before any launch
    assert lib.kvev_missed_mass(None, 8, 4, one, 4, 2, 1, one, None) == kvev.KVEV_EINVAL
    assert lib.kvev_missed_mass(one, 8, 4, one, 4, 2, 1, None, None) == kvev.KVEV_EINVAL
    assert lib.kvev_missed_mass(one, 8, 0, one, 4, 2, 1, one, None) == kvev.KVEV_EINVAL
    assert lib.kvev_missed_mass(one, 3, 4, one, 4, 2, 1, one, None) == kvev.KVEV_EINVAL
    assert lib.kvev_missed_mass(one, 8, 4, one, 1, 2, 1, one, None) == kvev.KVEV_EINVAL
    assert lib.kvev_missed_mass(one, 8, 4, one, 4, 2, 0, one, None) == kvev.KVEV_EINVAL
    assert lib.kvev_missed_mass(one, 8, 4, None, 4, 2, 1, one, None) == kvev.KVEV_EINVAL
