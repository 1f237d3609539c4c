"""Host-side error detection on a live context: calls out of order, calls of
the wrong mode, misaligned or missing buffers and a scratch allocation that
cannot succeed are refused with their status and a message before anything
is launched, and the context then continues as if the refused call had not
been made (bit for bit against an untouched context)."""
import pytest

from workloads import Geometry, Workload

from parity import load_prefill, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

STATE = ("out", "retained", "n_retained", "score", "t_ins", "t_ref", "pos")


def _status(fn, *args):
    with pytest.raises(kvev.KvevError) as err:
        fn(*args)
    assert kvev.kvev_last_error(None)   # a message accompanies the status
    return err.value.status


def _token_pass(wl):
    g = wl.geom
    ep = kvev.EvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch,
                           wl.L0 + 8, 64, 0.05, 0.001)
    load_prefill(ep, wl)
    return ep


def _step(ep, q, kn, vn, step):
    kvev.kvev_step(ep.ctx, q, kn, vn, ep.cache, ep.state, step, ep.out, ep.retained,
                   ep.n_retained)


def test_token_mode_refusals_leave_the_run_intact():
    wl = Workload(Geometry(2, 8, 2, 128, 1), 150, seed=4)
    ins = [tuple(to_dev_bf16(x) for x in wl.step_inputs(t)) for t in (1, 2, 3)]
    a = _token_pass(wl)
    q, kn, vn = ins[0]
    assert _status(_step, a, q, kn, vn, 1) == kvev.KVEV_ESTATE          # before kvev_begin
    a.begin(wl.L0)
    assert _status(_step, a, q, kn, vn, 2) == kvev.KVEV_ESTATE          # skips step 1
    assert _status(_step, a, q, kn, vn, 0) == kvev.KVEV_ESTATE
    raw = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    q_odd = raw[1:1 + q.numel()].view_as(q)                               # 2-byte offset
    q_odd.copy_(q)
    assert _status(_step, a, q_odd, kn, vn, 1) == kvev.KVEV_EINVAL      # misaligned q
    with pytest.raises(kvev.KvevError) as err:
        kvev.kvev_step(a.ctx, q, None, vn, a.cache, a.state, 1, a.out, a.retained, a.n_retained)
    assert err.value.status == kvev.KVEV_EINVAL                          # missing k_new
    for t in (1, 2, 3):
        _step(a, *ins[t - 1], t)
        if t == 2:   # a repeated step number is refused mid-run too
            assert _status(_step, a, *ins[1], 2) == kvev.KVEV_ESTATE
    kvev.kvev_sync(a.ctx)
    b = _token_pass(wl)
    b.begin(wl.L0)
    for t in (1, 2, 3):
        _step(b, *ins[t - 1], t)
    kvev.kvev_sync(b.ctx)
    for k in STATE:
        assert torch.equal(getattr(a, k), getattr(b, k)), f"refused calls changed {k}"
    kvev.kvev_check_scratch(a.ctx)
    a.close()
    b.close()


def test_block_and_tier_contexts_refuse_the_other_modes():
    wl = Workload(Geometry(2, 32, 8, 128, 1), 64, seed=6)
    q, kn, vn = (to_dev_bf16(x) for x in wl.step_inputs(1))
    pp = kvev.PagedEvictionPass(2, 32, 8, 128, 1, 8, 16, 2, 0.05, 0.001, n_backing=4)
    assert _status(pp.step, q, kn, vn) == kvev.KVEV_ESTATE               # before paged_begin
    assert _status(pp.readmit, 0, 1) == kvev.KVEV_ESTATE
    assert _status(kvev.kvev_begin, pp.ctx, 16) == kvev.KVEV_ESTATE      # token-mode call
    pp.close()
    tp = kvev.TierEvictionPass(2, 32, 8, 128, 1, 5 + 128 * 2 + 40, 1 + 16 + 8, 1, 1, 4, 0.05)
    assert _status(tp.step, q, kn, vn) == kvev.KVEV_ESTATE               # before tier_begin
    assert _status(kvev.kvev_begin, tp.ctx, 16) == kvev.KVEV_ESTATE
    tp.close()


def test_readmission_is_refused_with_a_region_table():
    """The backing tier keeps no region labels, so a context with a region
    table refuses kvev_readmit (before launching anything)."""
    table = kvev.region_table([1.0, 1.0], [0.0, 0.0], [False, True],
                              score_kind=kvev.KVEV_SCORE_LRFU)
    pp = kvev.PagedEvictionPass(2, 8, 2, 64, 1, 8, 16, 2, 0.05, 0.001, n_backing=4,
                                regions=table)
    pp.begin(64)
    assert _status(pp.readmit, 0, 1) == kvev.KVEV_EUNSUPPORTED
    kvev.kvev_sync(pp.ctx)
    pp.close()


def test_scratch_that_cannot_be_allocated_is_reported():
    """A layout whose scratch exceeds the device (hundreds of TB): the
    allocation fails, KVEV_ENOMEM comes back, and the device stays usable."""
    lay = kvev.kvev_layout(32, 32, 8, 128, 64, 1 << 30, 1, kvev.KVEV_BF16)
    with pytest.raises(kvev.KvevError) as err:
        kvev.kvev_create(lay, 1024, 1, 0.05, 0.001)
    assert err.value.status in (kvev.KVEV_ENOMEM, kvev.KVEV_EINVAL)
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0


def test_rotary_table_refusals():
    """kvev_set_rope refuses a token-granular context (KVEV_ESTATE), a table
    shorter than max_ctx or not 16-byte aligned (KVEV_EINVAL); in rotary mode
    kvev_tier_begin refuses a page range without room for the 8 K_q
    reconstruction pages, and after it K_q cannot grow past them (KVEV_ESTATE)
    while it may shrink."""
    L0 = 5 + 128 * 3 + 20
    max_ctx = L0 + 16
    table = torch.zeros((max_ctx, 64, 2), dtype=torch.float32, device="cuda")
    ep = kvev.EvictionPass(2, 8, 2, 128, 1, 64, 32, 0.05, 0.001)
    assert _status(kvev.kvev_set_rope, ep.ctx, table, max_ctx) == kvev.KVEV_ESTATE
    ep.close()
    used = 1 + -(-(L0 - 5) // 16)
    tight = kvev.TierEvictionPass(2, 32, 8, 128, 1, max_ctx, used + 4, 1, 2, 4, 0.05)
    assert _status(kvev.kvev_set_rope, tight.ctx, table, max_ctx - 1) == kvev.KVEV_EINVAL
    assert _status(kvev.kvev_set_rope, tight.ctx, table.data_ptr() + 4, max_ctx) == kvev.KVEV_EINVAL
    kvev.kvev_set_rope(tight.ctx, table, max_ctx)
    assert _status(tight.begin, L0) == kvev.KVEV_EINVAL          # no room for 16 scratch pages
    tight.close()
    tp = kvev.TierEvictionPass(2, 32, 8, 128, 1, max_ctx, used + 4 + 16, 1, 2, 4, 0.05,
                               rope=table)
    tp.begin(L0)
    assert _status(kvev.kvev_set_tiers, tp.ctx, 1, 3, 4) == kvev.KVEV_ESTATE
    kvev.kvev_set_tiers(tp.ctx, 1, 1, 4)                         # shrinking is allowed
    kvev.kvev_sync(tp.ctx)
    tp.close()
