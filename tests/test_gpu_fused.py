"""The fused refresh step (attention, split combine and scoring in one
cooperative launch with grid barriers): parity with the oracle in every
refresh mode and shape it is built for, equality with the three-launch path
bit for bit where the attention splits its tiles the same way, graph replay,
and the bounded barrier wait (a CTA withheld from a barrier: the step reports
KVEV_ETIMEOUT and the context recovers), all through the C ABI."""
import math

import pytest

import oracle as O
from workloads import Geometry, Workload, llama8b_workload, tiny_workload

from parity import load_prefill, to_dev_bf16
from test_gpu_parity import run_parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

OUTPUTS = ("out", "retained", "n_retained", "score", "t_ins", "t_ref", "pos")


@pytest.mark.parametrize("mode", ["all", "attn_combine"])
def test_fused_tiny_64_steps(mode):
    m = kvev.KVEV_FUSED_ALL if mode == "all" else kvev.KVEV_FUSED_ATTN_COMBINE
    tot = run_parity(tiny_workload(0), 128, 0.05, 0.001, 64, fused=m)
    assert tot["steps"] == 64


@pytest.mark.parametrize("refresh", ["full", "lazy"])
def test_fused_llama_geometry(refresh):
    """3 layers of the Llama-3.1-8B geometry, ragged 1000-token prefill,
    access clock, ranking diagnostics on (their raw keys come from the fused
    scorer)."""
    wl = llama8b_workload(0, prefill_len=1000, n_layers=3, needle_period=5)
    run_parity(wl, 100, 0.05, 0.001, 12, age_mode=O.AGE_SINCE_ACCESS, refresh=refresh,
               period=4, diagnostics=True, fused=True)


@pytest.mark.slow
def test_fused_llama8b_32k_steps_1_to_4():
    """The full 32-layer, 32768-token pass with the fused step (many tiles
    per warp at step 1), steps 1-4 against the oracle."""
    wl = llama8b_workload(0, prefill_len=32768)
    run_parity(wl, 3277, 0.05, 0.001, 4, age_mode=O.AGE_SINCE_ACCESS, max_ctx=32768 + 64,
               fused=True)


@pytest.mark.parametrize("d", [64, 128])
def test_fused_eight_query_heads_and_batches(d):
    wl = Workload(Geometry(2, 16, 2, d, 2), 260, seed=40 + d, outliers=2, heavy=3)
    run_parity(wl, 64, 0.05, 0.001, 5, age_mode=O.AGE_SINCE_ACCESS, fused=True)
    wl4 = Workload(Geometry(2, 8, 2, d, 4), 47, seed=3, outliers=4, heavy=3)
    run_parity(wl4, 20, 0.05, 0.001, 6, fused=True, pool_mean=True)


@pytest.mark.parametrize("L0,budget", [(1, 1), (17, 16), (33, 40)])
def test_fused_edge_lengths(L0, budget):
    wl = Workload(Geometry(2, 8, 2, 64, 1), L0, seed=L0, heavy=1)
    run_parity(wl, budget, 0.05, math.inf, 4, fused=True)


def _make(wl, budget, fused):
    g = wl.geom
    ep = kvev.EvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch,
                           wl.L0 + 16, budget, 0.05, 0.001, age_mode=kvev.KVEV_AGE_SINCE_ACCESS,
                           fused=fused)
    load_prefill(ep, wl)
    ep.begin(wl.L0)
    return ep


def _run(ep, wl, steps):
    got = []
    for t in range(1, steps + 1):
        q, kn, vn = (to_dev_bf16(x) for x in wl.step_inputs(t))
        ep.step(q, kn, vn)
        kvev.kvev_sync(ep.ctx)
        got.append({k: getattr(ep, k).clone() for k in OUTPUTS})
        got[-1]["k"] = ep.live_k().clone()
    return got


@pytest.mark.parametrize("mode", [1, 2])
def test_fused_equals_the_three_launches_bit_for_bit(mode):
    """Llama-3.1-8B head geometry (32 q / 8 KV, d 128), several tiles per
    warp: the fused step runs on the attention kernel's grid, so both split
    the tiles alike and every output, kept list, state array and compacted
    K/V row agrees; no scratch region overran its guard band."""
    wl = llama8b_workload(1, prefill_len=2000, n_layers=4, needle_period=3)
    a, b = _make(wl, 200, False), _make(wl, 200, mode)
    want, got = _run(a, wl, 6), _run(b, wl, 6)
    for t, (w, g) in enumerate(zip(want, got), start=1):
        for k in w:
            assert torch.equal(w[k], g[k]), f"step {t}: {k} differs"
    kvev.kvev_check_scratch(b.ctx)
    a.close()
    b.close()


def test_fused_step_replays_from_a_cuda_graph():
    """A fused step captured in a CUDA graph replays bit for bit (the grid
    barrier leaves its counters at zero after every use)."""
    wl = llama8b_workload(2, prefill_len=700, n_layers=2)
    ep = _make(wl, 80, True)
    q, kn, vn = (to_dev_bf16(x) for x in wl.step_inputs(1))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        ep.begin(wl.L0, stream)
        ep.step(q, kn, vn, stream)
    stream.synchronize()
    ref = ep.out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        ep.begin(wl.L0, cs)
        ep.step(q, kn, vn, cs)
    for _ in range(3):
        ep.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(ep.out, ref)
    kvev.kvev_sync(ep.ctx)
    ep.close()


@pytest.mark.parametrize("cta", [0, 7])
def test_fused_barrier_timeout_is_reported_and_context_recovers(cta):
    wl = Workload(Geometry(2, 8, 2, 128, 2), 300, seed=31, heavy=2)
    a = _make(wl, 96, True)
    q, kn, vn = (to_dev_bf16(x) for x in wl.step_inputs(1))
    kvev.kvev_test_barrier_timeout(a.ctx, cta, 2000)
    a.step(q, kn, vn)
    with pytest.raises(kvev.KvevError) as err:
        kvev.kvev_sync(a.ctx)
    assert err.value.status == kvev.KVEV_ETIMEOUT
    # the barrier state was reset with the status: a fresh run matches an
    # untouched context bit for bit
    for buf in a.k + a.v:
        buf.zero_()
    load_prefill(a, wl)
    a.begin(wl.L0)
    got = _run(a, wl, 5)
    b = _make(wl, 96, True)
    want = _run(b, wl, 5)
    for w, g in zip(want, got):
        for k in w:
            assert torch.equal(w[k], g[k]), f"after the timeout the run differs in {k}"
    a.close()
    b.close()


def test_fused_step_refuses_shapes_it_is_not_built_for():
    lay = kvev.kvev_layout(2, 16, 4, 128, 1, 64, 1, kvev.KVEV_BF16)   # 4 KV heads
    ctx = kvev.kvev_create(lay, 8, 1, 0.05, 0.001)
    with pytest.raises(kvev.KvevError) as ei:
        kvev.kvev_set_fused_step(ctx, True)
    assert ei.value.status == kvev.KVEV_EUNSUPPORTED
    kvev.kvev_destroy(ctx)
