"""kvev_attend_noalloc: the pass's attention for callers that cannot
allocate device memory (engines whose allocator owns all of the GPU's memory,
latency-critical paths that cannot take cudaMalloc's implicit
synchronisation).  It keeps its split partials in a fixed array inside the
library and must give the same attention output as kvev_step.

This file is collected last on purpose: the entry point's scratch array is
shared by every call in the process, and a run that stops at the first
failure has then already run every other test.
"""
import numpy as np
import pytest

import oracle as O
from workloads import Geometry, Workload, llama8b_workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from decoding_kv_cache_split_gb300 import kvev  # noqa: E402

OUT_RTOL = 2e-3     # the attention-output tolerance of every parity test
LSE_RTOL = 2e-3


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _rel_err(a, b):
    a = a.double().cpu().numpy()
    b = np.asarray(b, dtype=np.float64)
    return float((np.abs(a - b).max(axis=-1) / np.abs(b).max(axis=-1)).max())


def _bf16(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _oracle_lse2(q, K, V, L):
    """log2 of each head's softmax normaliser and the attention outputs,
    from the oracle's probabilities: p_i = exp(l_i - lse) for every token,
    so lse = l_i - ln p_i, taken at the most probable token (l_i its plain
    fp64 logit q.k_i / sqrt(d))."""
    Ly, Hq, d = q.shape
    Hkv = K.shape[1]
    lse2 = np.zeros((Ly, Hq))
    out = np.zeros((Ly, Hq, d))
    for layer in range(Ly):
        p, o = O.attention(q[layer], K[layer, :, :L], V[layer, :, :L])
        out[layer] = o
        for h in range(Hq):
            g = h * Hkv // Hq
            i = int(np.argmax(p[h]))
            li = float(np.dot(_bf16(q[layer, h]), _bf16(K[layer, g, i]))) / np.sqrt(d)
            lse2[layer, h] = (li - np.log(p[h, i])) / np.log(2.0)
    return lse2, out


def test_noalloc_attention_matches_kvev_step_on_two_calls():
    """Two decode steps through kvev_step; for each, the allocation-free
    call attends over the same appended cache (a copy of the buffer the step
    read, with the step's new K/V written at its slot: the step's compaction
    may rewrite that buffer in place) and must give the step's output bit
    for bit (the same kernels split the same way), and its log2-sum-exp must
    match the oracle's normaliser."""
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
        lse2.fill_(float("nan"))
        kvev.kvev_attend_noalloc(ep.layout, qd, kc, vc, L, out, lse2)
        torch.cuda.synchronize()
        assert torch.equal(out, ep.out), f"call {t}: output differs from kvev_step's"
        if t == 1:   # the oracle's normaliser over the same appended cache
            kh = kc[:, 0, :, :L].view(torch.int16).cpu().numpy().view(np.uint16)
            vh = vc[:, 0, :, :L].view(torch.int16).cpu().numpy().view(np.uint16)
            ref_lse2, ref_out = _oracle_lse2(q[0], kh, vh, L)
            got = lse2[:, 0].double().cpu().numpy()
            assert np.abs(got - ref_lse2).max() <= LSE_RTOL * np.abs(ref_lse2).max()
            assert _rel_err(out[0], ref_out) <= OUT_RTOL
    ep.close()


@pytest.mark.parametrize("d,G,L,max_ctx", [(64, 4, 1, 16), (64, 4, 37, 40), (128, 8, 203, 256),
                                           (64, 8, 17, 17)])
def test_noalloc_small_shapes_against_the_oracle(d, G, L, max_ctx):
    """head_dim 64 and 128, 4 and 8 query heads per KV head, one token, a
    ragged last tile and a cache filled to max_ctx: outputs and log2-sum-exp
    against the oracle, two calls in a row on the shared array."""
    wl = Workload(Geometry(2, 2 * G, 2, d, 2), L, seed=60 + d + G + L, heavy=1)
    g = wl.geom
    lay = kvev.kvev_layout(g.n_layers, g.n_q_heads, g.n_kv_heads, d, g.batch, max_ctx, 1,
                           kvev.KVEV_BF16)
    K, V = wl.prefill()                                     # [Ly][b][Hkv][L][d]
    kc = np.zeros((g.n_layers, g.batch, g.n_kv_heads, max_ctx, d), np.uint16)
    vc = np.zeros_like(kc)
    kc[:, :, :, :L] = K
    vc[:, :, :, :L] = V
    kd, vd = _dev(kc), _dev(vc)
    out = torch.empty((g.batch, g.n_layers, g.n_q_heads, d), dtype=torch.float32, device="cuda")
    lse2 = torch.empty((g.n_layers, g.batch, g.n_q_heads), dtype=torch.float32, device="cuda")
    for t in (1, 2):
        q, _, _ = wl.step_inputs(t)
        out.fill_(float("nan"))
        kvev.kvev_attend_noalloc(lay, _dev(q), kd, vd, L, out, lse2)
        torch.cuda.synchronize()
        for b in range(g.batch):
            ref_lse2, ref_out = _oracle_lse2(q[b], kc[:, b, :, :L], vc[:, b, :, :L], L)
            assert _rel_err(out[b], ref_out) <= OUT_RTOL
            got = lse2[:, b].double().cpu().numpy()
            assert np.abs(got - ref_lse2).max() <= LSE_RTOL * max(1.0, np.abs(ref_lse2).max())


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
