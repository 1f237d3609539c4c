"""Checkpoint / resume: a run stopped after step n, its device buffers copied
and its context state exported, continues in a fresh context (state
imported) exactly as the uninterrupted run does: outputs, kept sets and
state bit for bit, in the token, block and two-tier modes."""
import numpy as np
import pytest

from workloads import Geometry, Workload, paged_workload

from parity import load_prefill, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

OUTPUTS = ("out", "retained", "n_retained", "retained_lid")


def _tensors(obj):
    """Every device tensor the pass object owns (lists of tensors flattened)."""
    out = {}
    for k, v in vars(obj).items():
        if isinstance(v, torch.Tensor):
            out[k] = v
        elif isinstance(v, (list, tuple)) and v and all(isinstance(x, torch.Tensor) for x in v):
            out.update({f"{k}{i}": x for i, x in enumerate(v)})
    return out


def _same(x, y) -> bool:
    """Bit-for-bit equality (NaN entries of the score table included)."""
    if x.is_floating_point():
        iv = {2: torch.int16, 4: torch.int32, 8: torch.int64}[x.element_size()]
        return torch.equal(x.view(iv), y.view(iv))
    return torch.equal(x, y)


def _snapshot(obj):
    return {k: v.clone() for k, v in _tensors(obj).items() if k not in OUTPUTS}


def _restore(obj, snap):
    dst = _tensors(obj)
    for k, v in snap.items():
        dst[k].copy_(v)


def _run(obj, wl, steps, collect):
    for t in steps:
        q, kn, vn = (to_dev_bf16(x) for x in wl.step_inputs(t))
        obj.step_no = t - 1
        obj.step(q, kn, vn)
        kvev.kvev_sync(obj.ctx)
        collect.append({k: v.clone() for k, v in _tensors(obj).items() if k in OUTPUTS})


def _check_resume(make, load, wl, n_first=5, n_more=7, ignore=()):
    """ignore: buffers left out of the final state comparison."""
    a = make()
    load(a)
    _run(a, wl, range(1, n_first + 1), [])
    snap = _snapshot(a)
    cur = getattr(getattr(a, "cache", None), "cur", None)
    blob = kvev.kvev_export_state(a.ctx)
    want = []
    _run(a, wl, range(n_first + 1, n_first + n_more + 1), want)
    final_a = _snapshot(a)
    b = make()
    _restore(b, snap)
    if cur is not None and hasattr(b.cache, "cur"):
        b.cache.cur = cur
    kvev.kvev_import_state(b.ctx, blob)
    got = []
    _run(b, wl, range(n_first + 1, n_first + n_more + 1), got)
    for w, g in zip(want, got):
        for k in w:
            assert _same(w[k], g[k]), f"resumed run differs in {k}"
    final_b = _snapshot(b)
    for k in final_a:
        if k not in ignore:
            assert _same(final_a[k], final_b[k]), f"resumed state differs in {k}"
    a.close()
    b.close()


def test_resume_token_mode():
    wl = Workload(Geometry(2, 8, 2, 128, 2), 200, seed=21, heavy=3)
    make = lambda: kvev.EvictionPass(2, 8, 2, 128, 2, 240, 64, 0.05, 0.001,
                                     age_mode=kvev.KVEV_AGE_SINCE_ACCESS,
                                     refresh=kvev.KVEV_REFRESH_LAZY, period=3)
    def load(ep):
        load_prefill(ep, wl)
        ep.begin(wl.L0)
    _check_resume(make, load, wl)


def test_resume_block_mode_with_readmission_state():
    wl = paged_workload(5, prefill_len=320, n_layers=2, batch=2, needle_period=4)
    K, V = wl.prefill()
    def make():
        return kvev.PagedEvictionPass(2, 32, 8, 128, 2, 40, 16, 6, 0.05, 0.001, n_backing=20,
                                      table_len=30)
    def load(pp):
        for b in range(2):
            for src, pool, back in ((K, pp.k_pool, pp.backing_k), (V, pp.v_pool, pp.backing_v)):
                x = np.ascontiguousarray(src[:, b].reshape(2, 8, 20, 16, 128).transpose(2, 0, 1, 3, 4))
                xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
                pool[b * pp.pps:b * pp.pps + 20].copy_(xt)
                back[b, :20].copy_(xt)
        pp.begin(320)
    _check_resume(make, load, wl)


def test_resume_two_tier_mode_across_routing_events():
    wl = Workload(Geometry(2, 32, 8, 128, 1), 5 + 128 * 6 + 20, seed=9, needle=16,
                  needle_period=6)
    L0 = wl.L0
    def make():
        return kvev.TierEvictionPass(2, 32, 8, 128, 1, L0 + 40, 1 + 49 + 24, 2, 2, 3, 0.05)
    def load(tp):
        from test_gpu_qevict import load as tload
        K, V = wl.prefill()
        tload(tp, K, V, L0)
        tp.begin(L0)
    _check_resume(make, load, wl, n_first=7, n_more=9)


def test_resume_two_tier_rotary_mode():
    """Rotary mode: the reconstruction slots are not part of a checkpoint;
    the resumed run gives every INT2 window a slot anew and rebuilds the
    reconstructions, and the attention reads them in the same order, so
    outputs and tier state match bit for bit (the pools are left out: the
    slots may differ)."""
    wl = Workload(Geometry(2, 32, 8, 128, 1), 5 + 128 * 6 + 20, seed=9, needle=16,
                  needle_period=6, rope_base=10000.0)
    L0 = wl.L0
    rope = wl.rope_table(L0 + 40)
    def make():
        return kvev.TierEvictionPass(2, 32, 8, 128, 1, L0 + 40, 1 + 49 + 24 + 16, 2, 2, 3, 0.05,
                                     rope=rope)
    def load(tp):
        from test_gpu_qevict import load as tload
        K, V = wl.prefill()
        tload(tp, K, V, L0)
        tp.begin(L0)
    _check_resume(make, load, wl, n_first=7, n_more=9, ignore=("k_pool", "v_pool"))
