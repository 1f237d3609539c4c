"""A decode step can be captured in a CUDA graph: the context's launches on
the capturing stream (state reset and step, with their programmatic
dependencies) replay to the same outputs and state, bit for bit, as the
eager step."""
import pytest

from workloads import Geometry, Workload

from parity import load_prefill, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

STATE = ("out", "retained", "n_retained", "score", "t_ins", "t_ref", "pos")


def test_step_replays_from_a_cuda_graph():
    wl = Workload(Geometry(2, 8, 2, 128, 2), 700, seed=17, heavy=4)
    g_ = wl.geom
    ep = kvev.EvictionPass(g_.n_layers, g_.n_q_heads, g_.n_kv_heads, g_.head_dim, g_.batch,
                           wl.L0 + 8, 200, 0.05, 0.001, age_mode=kvev.KVEV_AGE_SINCE_ACCESS)
    load_prefill(ep, wl)
    q, kn, vn = (to_dev_bf16(x) for x in wl.step_inputs(1))
    ep.begin(wl.L0)
    ep.step(q, kn, vn)
    kvev.kvev_sync(ep.ctx)
    want = {k: getattr(ep, k).clone() for k in STATE}
    want["k"] = ep.live_k().clone()
    for k in STATE:
        getattr(ep, k).zero_()
    ep.k[1].zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        ep.begin(wl.L0, side)
        ep.step(q, kn, vn, side)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    kvev.kvev_sync(ep.ctx)
    for k in STATE:
        assert torch.equal(getattr(ep, k), want[k]), f"graph replay differs in {k}"
    assert torch.equal(ep.k[1], want["k"]), "graph replay differs in the compacted keys"
    kvev.kvev_check_scratch(ep.ctx)   # no scratch region overran its guard band
    ep.close()
