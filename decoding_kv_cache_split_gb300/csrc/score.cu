// Per-token scoring: probabilities, head pooling, layer-sequential EMA,
// access clock, eviction priority and its sortable key.
//
//  p_h(i)   = exp2(logit2_h(i) - lse2_h)      (the softmax of the attention
//             kernel, from the logits it kept and the log2-sum-exp of the
//             split combine; "What Matters for Aggressive Decoding-Time KV
//             Eviction?" Sec. 3.1 Eq. (1))
//  s_l(i)   = sum_h p_h(i)   (or the head mean, Eq. (1)); optionally each
//             head's p_h(i) times ||v_i|| / mean_j ||v_j|| of its KV head
//             (VNorm), and the layer's s_l times the mean over heads of the
//             normalized entropy of p_h (Appendix E "Per-step scoring")
//  m(i)    <- alpha * s_l(i) + (1 - alpha) * m(i) for l = 0 .. Ly-1 in order
//             (kv-cache-docs "ema-eviction" EMA table; Appendix E "Layer
//             scoring" of the same paper: every layer updates the shared
//             state immediately); cumulative aggregation (Sec. 3.1 Eq. (3))
//             takes m(i) <- s_l(i) + m(i): both weights 1
//  access   sum_l s_l(i) >= 2 Hq Ly / L  (attention averaged over heads and
//             layers at least twice uniform: MemDecay Sec. III-C Eq. (3))
//  pr(i)    = (1 - m(i)) * (1 - exp(-beta * age))  ("ema-eviction" priority)
//  key(i)   = order-preserving bits of pr(i); ties are broken by slot index
//             in the selection kernel.
// On non-refresh steps (lazy refresh, Score-Free: Sec. 3.2 Eq. (6)) the
// probabilities are not formed and m is unchanged; the kernel only forms
// the priorities and the block sums of the old tokens' m, from which the
// selection kernel sets the new token's score to their mean (Appendix E
// "New token insertion during non-refresh steps").
#include <math.h>

#include "kvev_internal.h"
#include "score_refresh.cuh"

namespace kvev {
namespace {

template <int G, int NKV, bool VN>
__global__ void __launch_bounds__(kScoreSegs * 32) score_refresh_kernel(const ScoreArgs a) {
    extern __shared__ float s_tab[];
    __shared__ float s_c[kScoreSegs][32], s_tot[kScoreSegs][32];
    griddep_wait();
    griddep_release();
    score_tables<G, NKV, VN>(a, blockIdx.y, s_tab);
    score_block<G, NKV, VN, kScoreSegs, kScoreSegs>(a, blockIdx.y, blockIdx.x, s_tab, s_c,
                                                    s_tot);
}

template <int G, bool VN>
void* refresh_kernel_for(int nkv) {
    switch (nkv) {
        case 1: return (void*)score_refresh_kernel<G, 1, VN>;
        case 2: return (void*)score_refresh_kernel<G, 2, VN>;
        case 4: return (void*)score_refresh_kernel<G, 4, VN>;
        case 8: return (void*)score_refresh_kernel<G, 8, VN>;
        default: return nullptr;
    }
}

// Non-refresh steps: no probabilities, the state is frozen; one thread per
// token forms the priority from the stale score, and each block adds up its
// old tokens' scores (for the new token's mean, taken by the selection).
__global__ void __launch_bounds__(kScoreThreads) score_stale_kernel(const ScoreArgs a) {
    griddep_wait();
    griddep_release();
    const int b = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = i < a.L;
    const bool is_new = i == a.L - 1;
    const size_t si = (size_t)b * a.max_ctx + i;
    float old_m = 0.f;
    if (live) {
        const float m = a.st.score[si];
        const int t_ref = a.st.t_ref[si];
        const int t_ins = a.st.t_ins[si];
        if (!is_new) old_m = m;
        const int age = a.t - (a.age_mode == KVEV_AGE_SINCE_ACCESS ? t_ref : t_ins);
        const float pr = age == 0 ? 0.0f : (1.0f - m) * -expm1f(-a.beta * (float)age);
        a.keys[si] = order_bits(pr);
        a.m_s[si] = m;
        a.tref_s[si] = t_ref;
        a.tins_s[si] = t_ins;
        a.pos_s[si] = a.st.pos[si];
        if (a.dbg_prio) a.dbg_prio[si] = pr + 0.0f;
    }
    __shared__ float red[kScoreThreads / 32];   // deterministic block sum
    float v = old_m;
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int k = 0; k < kScoreThreads / 32; ++k) s += red[k];
        a.msum_part[(size_t)b * gridDim.x + blockIdx.x] = s;
    }
}

}  // namespace

cudaError_t launch_score(const ScoreArgs& a, int group, int* n_blocks, cudaStream_t s) {
    if (a.refresh) {
        const int nb = (a.L + 31) / 32;   // 32 tokens per CTA
        *n_blocks = nb;
        const dim3 grid(nb, a.batch);
        const size_t smem = sizeof(float) * (size_t)a.n_layers * (a.n_q + 1 + a.n_kv);
        const bool vn = a.vnorm != nullptr;
        void* kern = group == 4 ? (vn ? refresh_kernel_for<4, true>(a.n_kv)
                                      : refresh_kernel_for<4, false>(a.n_kv))
                   : group == 8 ? (vn ? refresh_kernel_for<8, true>(a.n_kv)
                                      : refresh_kernel_for<8, false>(a.n_kv))
                   : nullptr;
        if (!kern) return cudaErrorInvalidValue;
        return launch_pdl(reinterpret_cast<void (*)(ScoreArgs)>(kern), grid,
                          dim3(kScoreSegs * 32), smem, s, a);
    }
    const int nb = (a.L + kScoreThreads - 1) / kScoreThreads;
    *n_blocks = nb;
    (void)group;
    return launch_pdl(score_stale_kernel, dim3(nb, a.batch), dim3(kScoreThreads), 0, s, a);
}

}  // namespace kvev
