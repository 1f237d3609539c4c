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


def test_bf16_output_is_the_rounded_fp32_output():
    """With KVEV_OUT_BF16 the step writes its fp32 result rounded to bf16
    (nearest even), bit for bit, through kvev_step and kvev_step_host alike
    (the host copy then moves half the bytes); everything else is unchanged.
    Against the oracle the rounded output is within the attention tolerance
    plus bf16's unit roundoff 2^-8 (rounding to 8 significant bits)."""
    import oracle as O
    from parity import compare_step, oracle_step
    wl = Workload(Geometry(2, 8, 2, 128, 2), 300, seed=23, heavy=3)
    g = wl.geom
    budget = 64

    def make(out_type):
        ep = kvev.EvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch,
                               wl.L0 + 8, budget, 0.05, 0.001, out_type=out_type)
        load_prefill(ep, wl)
        ep.begin(wl.L0)
        return ep

    f32, b16, host = make(kvev.KVEV_OUT_F32), make(kvev.KVEV_OUT_BF16), make(kvev.KVEV_OUT_BF16)
    assert b16.out.dtype == torch.bfloat16
    out_h = torch.empty((g.batch, g.n_layers, g.n_q_heads, g.head_dim),
                        dtype=torch.bfloat16).pin_memory()
    ret_h = torch.empty((g.batch, budget), dtype=torch.int32).pin_memory()
    nret_h = torch.empty((g.batch,), dtype=torch.int32).pin_memory()
    K, V = wl.prefill()
    P = O.OracleParams(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, budget, 0.05, 0.001)
    pre = [O.SequenceState.from_prefill(K[:, b], V[:, b], wl.L0, wl.L0 + 8)
           for b in range(g.batch)]
    q, kn, vn = wl.step_inputs(1)
    f32.step(to_dev_bf16(q), to_dev_bf16(kn), to_dev_bf16(vn))
    b16.step(to_dev_bf16(q), to_dev_bf16(kn), to_dev_bf16(vn))
    kvev.kvev_step_host(host.ctx, _host_bf16(q), _host_bf16(kn), _host_bf16(vn), host.cache,
                        host.state, 1, out_h, ret_h, nret_h)
    kvev.kvev_sync(f32.ctx)
    want = f32.out.to(torch.bfloat16)                    # round to nearest even
    assert torch.equal(b16.out.view(torch.int16), want.view(torch.int16))
    assert torch.equal(out_h.view(torch.int16), want.cpu().view(torch.int16))
    assert torch.equal(b16.retained, f32.retained) and torch.equal(b16.score, f32.score)
    for b in range(g.batch):
        res, _ = oracle_step(P, pre[b], 1, True, q[b], kn[b], vn[b], wl.L0)
        compare_step(res, f32, b, pre[b], budget)          # the fp32 output, as every test
        out = b16.out[b].float().cpu().numpy().astype(np.float64)
        err = np.abs(out - res["out"]).max(-1) / np.abs(res["out"]).max(-1)
        assert err.max() <= 2e-3 + 2.0 ** -8, f"bf16 output rel err {err.max():.3e}"
    for ep in (f32, b16, host):
        ep.close()
