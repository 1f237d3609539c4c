"""kvev_attend_noalloc: the pass's attention for callers that cannot
allocate device memory (engines whose allocator owns all of the GPU's memory,
latency-critical paths that cannot take cudaMalloc's implicit
synchronisation).  It keeps its split partials in a fixed array inside the
library and must give the same attention output as kvev_step.

This file is collected last on purpose: the entry point's scratch array is
shared by every call in the process, and a run that stops at the first
failure has then already run every other test.
"""
import ctypes

import numpy as np
import pytest

from workloads import llama8b_workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

OUT_RTOL = 2e-3     # the attention-output tolerance of every parity test


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _rel_err(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float((np.abs(a - b).max(axis=-1) / np.abs(b).max(axis=-1)).max())


def test_noalloc_attention_matches_kvev_step_on_two_calls():
    """Two decode steps through kvev_step; for each, the allocation-free
    call attends over the same appended cache (a copy of the buffer the step
    read, with the step's new K/V written at its slot: the step's compaction
    may rewrite that buffer in place) and must give the step's output."""
    wl = llama8b_workload(0, prefill_len=3000, n_layers=4)
    g = wl.geom
    max_ctx, budget = 3100, 300
    ep = kvev.EvictionPass(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.batch, max_ctx,
                           budget, 0.05, 0.001, age_mode=kvev.KVEV_AGE_SINCE_ACCESS)
    K, V = wl.prefill()
    ep.k[0][:, :, :, :wl.L0].copy_(torch.from_numpy(K.view(np.int16)).view(torch.bfloat16))
    ep.v[0][:, :, :, :wl.L0].copy_(torch.from_numpy(V.view(np.int16)).view(torch.bfloat16))
    ep.begin(wl.L0)
    out = torch.empty_like(ep.out)
    lse2 = torch.empty((g.n_layers, g.batch, g.n_q_heads), dtype=torch.float32, device="cuda")
    for t in (1, 2):
        L = ep.length() + 1
        q, kn, vn = wl.step_inputs(t)
        qd, knd, vnd = _dev(q), _dev(kn), _dev(vn)
        kc, vc = ep.live_k().clone(), ep.live_v().clone()   # [Ly][b][Hkv][slot][d]
        kc[:, :, :, L - 1] = knd.transpose(0, 1)             # new rows are [b][Ly][Hkv][d]
        vc[:, :, :, L - 1] = vnd.transpose(0, 1)
        ep.step(qd, knd, vnd)
        out.fill_(float("nan"))
        kvev.kvev_attend_noalloc(ep.layout, qd, kc, vc, L, out, lse2)
        torch.cuda.synchronize()
        err = _rel_err(out, ep.out)
        assert err <= OUT_RTOL, f"call {t}: rel err {err:.3e}"
        assert torch.isfinite(lse2).all()
    ep.close()


def test_noalloc_rejects_layouts_beyond_its_scratch():
    """A layout whose split partials would not fit the 16 MiB array is
    refused with KVEV_EINVAL and a message, before anything is launched."""
    lay = kvev.kvev_layout(64, 32, 8, 128, 16, 1024, 1, kvev.KVEV_BF16)   # 8192 rows
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(kvev.KvevError) as ei:
        kvev.kvev_attend_noalloc(lay, x, x, x, 10, o, o)
    assert ei.value.status == kvev.KVEV_EINVAL
    assert "16 MiB" in str(ei.value)
