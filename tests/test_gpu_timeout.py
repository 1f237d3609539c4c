"""Failure detection without a fault: one tile of the attention launch has its
copies withheld (test-only injection through the C ABI), the warp waiting on
it gives up after its bounded wait, the step reports KVEV_ETIMEOUT, and the
same context then runs a fresh decode that matches a second, untouched
context bit for bit."""
import pytest

from workloads import Geometry, Workload

from parity import load_prefill, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

OUTPUTS = ("out", "retained", "n_retained", "score", "t_ins", "t_ref", "pos")


def _make(wl):
    g = wl.geom
    return kvev.EvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch,
                             wl.L0 + 16, 96, 0.05, 0.001)


def _restart(ep, wl):
    for buf in ep.k + ep.v:
        buf.zero_()
    load_prefill(ep, wl)
    ep.begin(wl.L0)


def _run(ep, wl, steps):
    got = []
    for t in range(1, steps + 1):
        q, kn, vn = (to_dev_bf16(x) for x in wl.step_inputs(t))
        ep.step(q, kn, vn)
        kvev.kvev_sync(ep.ctx)
        got.append({k: getattr(ep, k).clone() for k in OUTPUTS})
        got[-1]["k"] = ep.live_k().clone()
    return got


@pytest.mark.parametrize("tile", [0, 5, 37])
def test_injected_wait_timeout_is_reported_and_context_recovers(tile):
    wl = Workload(Geometry(2, 8, 2, 128, 2), 300, seed=31, heavy=2)
    a = _make(wl)
    _restart(a, wl)
    q, kn, vn = (to_dev_bf16(x) for x in wl.step_inputs(1))
    kvev.kvev_test_wait_timeout(a.ctx, tile, 2000)
    a.step(q, kn, vn)
    with pytest.raises(kvev.KvevError) as err:
        kvev.kvev_sync(a.ctx)
    assert err.value.status == kvev.KVEV_ETIMEOUT
    # the warp that gave up poisoned its split slots: the row of the withheld
    # tile (layer, sequence, KV head) comes out NaN instead of a partial merge
    g = wl.geom
    tiles_per_row = -(-(wl.L0 + 1) // 16)
    row = tile // tiles_per_row
    kvh, lb = row % g.n_kv_heads, row // g.n_kv_heads
    b, layer = lb % g.batch, lb // g.batch
    G = g.n_q_heads // g.n_kv_heads
    assert torch.isnan(a.out[b, layer, kvh * G:(kvh + 1) * G]).all()
    # the injection covers one step only, and the status word was cleared
    _restart(a, wl)
    got = _run(a, wl, 6)
    b = _make(wl)
    _restart(b, wl)
    want = _run(b, wl, 6)
    for w, g in zip(want, got):
        for k in w:
            assert torch.equal(w[k], g[k]), f"after the timeout the run differs in {k}"
    kvev.kvev_check_scratch(a.ctx)
    a.close()
    b.close()


def test_injection_arguments_are_validated():
    wl = Workload(Geometry(1, 8, 2, 128, 1), 200, seed=3)
    a = _make(wl)
    with pytest.raises(kvev.KvevError):
        kvev.kvev_test_wait_timeout(a.ctx, -1, 100)
    with pytest.raises(kvev.KvevError):
        kvev.kvev_test_wait_timeout(a.ctx, 0, 0)
    a.close()
