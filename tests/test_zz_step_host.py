"""kvev_step_host, the host-buffer entry point that the benchmark's end-to-end
figure goes through, matches kvev_step on the same inputs bit for bit: the
attention output, the retained lists, the per-token state and the live K/V.
Each call copies the step's inputs in from pinned host memory and the
results back to it."""
import numpy as np
import pytest

from workloads import Geometry, Workload

from parity import load_prefill, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

STATE = ("score", "t_ins", "t_ref", "pos")


def _host_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).pin_memory()


def test_host_buffer_step_matches_the_device_step():
    wl = Workload(Geometry(2, 8, 2, 128, 2), 300, seed=19, heavy=3)
    g = wl.geom
    budget = 64

    def make():
        ep = kvev.EvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch,
                               wl.L0 + 8, budget, 0.05, 0.001,
                               age_mode=kvev.KVEV_AGE_SINCE_ACCESS)
        load_prefill(ep, wl)
        ep.begin(wl.L0)
        return ep

    dev, host = make(), make()
    out_h = torch.empty((g.batch, g.n_layers, g.n_q_heads, g.head_dim),
                        dtype=torch.float32).pin_memory()
    ret_h = torch.empty((g.batch, budget), dtype=torch.int32).pin_memory()
    nret_h = torch.empty((g.batch,), dtype=torch.int32).pin_memory()
    for t in (1, 2, 3):
        q, kn, vn = wl.step_inputs(t)
        dev.step(to_dev_bf16(q), to_dev_bf16(kn), to_dev_bf16(vn))
        kvev.kvev_step_host(host.ctx, _host_bf16(q), _host_bf16(kn), _host_bf16(vn), host.cache,
                            host.state, t, out_h, ret_h, nret_h)   # synchronises its stream
        kvev.kvev_sync(dev.ctx)
        assert torch.equal(out_h, dev.out.cpu()), f"step {t}: output"
        n = dev.n_retained.cpu()
        assert torch.equal(nret_h, n), f"step {t}: retained counts"
        for b in range(g.batch):
            k = int(n[b])
            assert torch.equal(ret_h[b, :k], dev.retained[b, :k].cpu()), f"step {t}: retained"
        for name in STATE:
            assert torch.equal(getattr(host, name), getattr(dev, name)), f"step {t}: {name}"
        assert host.cache.cur == dev.cache.cur
        assert torch.equal(host.live_k(), dev.live_k()) and torch.equal(host.live_v(),
                                                                        dev.live_v())
    kvev.kvev_check_scratch(host.ctx)   # no scratch region overran its guard band
    dev.close()
    host.close()
