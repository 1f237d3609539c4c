"""Future Missed Mass on the device (QEvict review, Sec. 3): a FullKV run
(a context whose budget is never reached, so slot = position) and a policy
run decode the same seeded inputs; before each policy step the device
computes the share of the FullKV step's attention on positions the policy
already discarded, which must match the oracle's FullKV attention summed
over heads and layers (oracle/diagnostics.py missed_mass, fp64) within 1e-5,
and the same formula on the device's own raw scores within fp32 rounding."""
import numpy as np
import pytest

import oracle as O
from oracle import diagnostics as D
from workloads import Geometry, Workload, tiny_workload

from parity import load_prefill, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402


@pytest.mark.parametrize("case", ["tiny", "two_sequences"])
def test_missed_mass_against_a_fullkv_run(case):
    if case == "tiny":
        wl, budget, steps = tiny_workload(0), 128, 24
    else:
        wl, budget, steps = Workload(Geometry(2, 8, 2, 128, 2), 300, seed=14, heavy=4), 64, 10
    g = wl.geom
    max_ctx = wl.L0 + steps + 8
    full = kvev.EvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch, max_ctx,
                             max_ctx - 1, 0.05, 0.001)
    pol = kvev.EvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch, max_ctx,
                            budget, 0.05, 0.001)
    for ep in (full, pol):
        load_prefill(ep, wl)
        ep.begin(wl.L0)
    counters = torch.zeros((g.batch, kvev.KVEV_DIAG_FIELDS), dtype=torch.int32, device="cuda")
    raw = torch.zeros((g.batch, max_ctx), dtype=torch.float32, device="cuda")
    kvev.kvev_set_diagnostics(full.ctx, counters, raw)
    fmm = torch.zeros((g.batch,), dtype=torch.float32, device="cuda")
    K, V = wl.prefill()
    P = O.OracleParams(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, max_ctx - 1, 0.05,
                       0.001)
    shadow = [O.SequenceState.from_prefill(K[:, b], V[:, b], wl.L0, max_ctx)
              for b in range(g.batch)]
    worst = 0.0
    for t in range(1, steps + 1):
        q, kn, vn = (to_dev_bf16(x) for x in wl.step_inputs(t))
        full.step(q, kn, vn)
        n_pos = full.length()
        held = pol.pos.clone()                  # before the policy's own step
        n_cached = pol.length()
        kvev.kvev_missed_mass(raw, max_ctx, n_pos, pol.pos, max_ctx, n_cached, g.batch, fmm)
        pol.step(q, kn, vn)
        kvev.kvev_sync(pol.ctx)
        qh, knh, vnh = wl.step_inputs(t)
        for b in range(g.batch):
            res, shadow[b] = O.step(P, shadow[b], t, True, qh[b], knh[b], vnh[b],
                                    wl.L0 + t - 1, want_probs=False)
            hp = held[b, :n_cached].cpu().numpy()
            want = D.missed_mass(res["score_sum"], hp, n_pos - 1)
            own = D.missed_mass(raw[b, :n_pos].double().cpu().numpy(), hp, n_pos - 1)
            got = float(fmm[b])
            assert abs(got - want) <= 1e-5, f"step {t} seq {b}: FMM {got} vs {want}"
            assert abs(got - own) <= 1e-6
            worst = max(worst, abs(got - want))
            if t == 1:
                assert abs(got) <= 1e-6        # nothing discarded before the first step
    print(case, "FMM max |err|", worst, "last", fmm.cpu().numpy())
    full.close()
    pol.close()
