// Per-token scoring: probabilities, head pooling, layer-sequential EMA,
// access clock, eviction priority and its sortable key.
//
//  p_h(i)   = exp2(logit2_h(i) - lse2_h)      (the softmax of the attention
//             kernel, from the logits it kept; "What Matters for Aggressive
//             Decoding-Time KV Eviction?" Sec. 3.1 Eq. (1))
//  s_l(i)   = sum_h p_h(i)   (or the head mean, Eq. (1))
//  m(i)    <- alpha * s_l(i) + (1 - alpha) * m(i) for l = 0 .. Ly-1 in order
//             (kv-cache-docs "ema-eviction" EMA table; Appendix E "Layer
//             scoring" of the same paper: every layer updates the shared
//             state immediately)
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

namespace kvev {
namespace {

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t order_bits(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Refresh steps: two threads per token (adjacent lanes), each summing the
// heads of half of the KV heads; lanes cover consecutive tokens so every load
// instruction reads two 256-byte runs.  The (layer, KV head) logit rows are
// visited in layer order in batches whose loads are all issued before any is
// used (kBatch 16-byte loads in flight per thread); each completed layer is
// combined across the pair with one shuffle and folded into the EMA.
constexpr int kRefreshThreads = 128;

template <int G, int kSplit>   // kSplit threads per token (1 or 2)
__global__ void __launch_bounds__(kRefreshThreads, 4) score_refresh_kernel(const ScoreArgs a) {
    constexpr int V4 = G / 4;                          // float4 per (layer, KV head)
    constexpr int kBatch = 16 / V4;                    // (layer, KV head) pairs in flight
    extern __shared__ float s_lse[];                   // [Ly][Hq] of this sequence
    griddep_wait();
    griddep_release();
    const int b = blockIdx.y;
    const int nlse = a.n_layers * a.n_q;
    for (int k = threadIdx.x; k < nlse; k += blockDim.x) {
        const int l = k / a.n_q, h = k % a.n_q;
        s_lse[k] = a.lse2[((size_t)l * a.batch + b) * a.n_q + h];
    }
    __syncthreads();
    const int half = kSplit == 2 ? (threadIdx.x & 1) : 0;
    const int i = (blockIdx.x * kRefreshThreads + threadIdx.x) / kSplit;
    const bool live = i < a.L;                         // both lanes of a pair agree
    const int kv_half = a.n_kv / kSplit;               // KV heads per thread
    const int n_pairs = a.n_layers * kv_half;

    const size_t si = (size_t)b * a.max_ctx + (live ? i : 0);
    float m = live ? a.st.score[si] : 0.f;
    const float oma = 1.0f - a.alpha;
    const float inv_hq = 1.0f / (float)a.n_q;
    float tot = 0.f, s = 0.f;
    for (int k0 = 0; k0 < n_pairs; k0 += kBatch) {
        float4 xb[kBatch][V4];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {           // all loads of the batch first ...
            const int k = k0 + u;
            const int l = k / kv_half, g = half * kv_half + (k - l * kv_half);
            const size_t row = ((size_t)l * a.batch + b) * a.n_kv + g;
            const float4* x = reinterpret_cast<const float4*>(a.logits + (row * a.max_ctx + i) * G);
#pragma unroll
            for (int c = 0; c < V4; ++c)
                xb[u][c] = (live && k < n_pairs) ? __ldcs(x + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {           // ... then the arithmetic, in layer order
            const int k = k0 + u;
            if (k >= n_pairs) break;
            const int l = k / kv_half, gl = k - l * kv_half, g = half * kv_half + gl;
            const float* lg = s_lse + l * a.n_q + g * G;
            const float* xv = reinterpret_cast<const float*>(&xb[u][0]);
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float p = fast_exp2(xv[hh] - lg[hh]);
                if (a.dbg_probs && live)
                    a.dbg_probs[(((size_t)b * a.n_layers + l) * a.n_q + g * G + hh) * a.max_ctx + i] = p;
                s += p;
            }
            if (gl == kv_half - 1) {                 // layer l complete: fold it
                if (kSplit == 2) s += __shfl_xor_sync(0xffffffffu, s, 1);
                tot += s;
                m = fmaf(a.alpha, a.pool_mean ? s * inv_hq : s, oma * m);
                s = 0.f;
            }
        }
    }
    if (!live || half) return;
    int t_ref = a.st.t_ref[si];
    const int t_ins = a.st.t_ins[si];
    if (tot >= a.access_thr) t_ref = a.t;   // the clock runs in every age mode
    const int age = a.t - (a.age_mode == KVEV_AGE_SINCE_ACCESS ? t_ref : t_ins);
    const float pr = age == 0 ? 0.0f : (1.0f - m) * -expm1f(-a.beta * (float)age);
    a.keys[si] = order_bits(pr);
    a.m_s[si] = m;
    a.tref_s[si] = t_ref;
    a.tins_s[si] = t_ins;
    a.pos_s[si] = a.st.pos[si];
    if (a.dbg_prio) a.dbg_prio[si] = pr + 0.0f;
}

// Non-refresh steps (and the general one-thread-per-token form).
template <int G>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(const ScoreArgs a) {
    extern __shared__ float s_lse[];  // [Ly][Hq] of this sequence
    griddep_wait();
    griddep_release();
    const int b = blockIdx.y;
    const int nlse = a.n_layers * a.n_q;
    for (int k = threadIdx.x; k < nlse; k += blockDim.x) {
        const int l = k / a.n_q, h = k % a.n_q;
        s_lse[k] = a.lse2[((size_t)l * a.batch + b) * a.n_q + h];
    }
    __syncthreads();

    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = i < a.L;
    const bool is_new = i == a.L - 1;
    const size_t si = (size_t)b * a.max_ctx + i;
    float old_m = 0.f;
    if (live) {
        float m = a.st.score[si];
        int t_ref = a.st.t_ref[si];
        const int t_ins = a.st.t_ins[si];
        const int pos = a.st.pos[si];
        if (a.refresh) {
            const float oma = 1.0f - a.alpha;
            const float inv_hq = 1.0f / (float)a.n_q;
            float tot = 0.f;
            for (int l = 0; l < a.n_layers; ++l) {
                float s = 0.f;
                const float* lrow = s_lse + l * a.n_q;
                for (int g = 0; g < a.n_kv; ++g) {
                    const size_t row = ((size_t)l * a.batch + b) * a.n_kv + g;
                    const float* x = a.logits + (row * a.max_ctx + i) * G;
                    float xv[G];
                    if constexpr (G == 4) {
                        const float4 x4 = *reinterpret_cast<const float4*>(x);
                        xv[0] = x4.x; xv[1] = x4.y; xv[2] = x4.z; xv[3] = x4.w;
                    } else {
#pragma unroll
                        for (int hh = 0; hh < G; ++hh) xv[hh] = x[hh];
                    }
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        const float p = fast_exp2(xv[hh] - lrow[g * G + hh]);
                        if (a.dbg_probs)
                            a.dbg_probs[(((size_t)b * a.n_layers + l) * a.n_q + g * G + hh) *
                                            a.max_ctx + i] = p;
                        s += p;
                    }
                }
                tot += s;
                const float sp = a.pool_mean ? s * inv_hq : s;
                m = fmaf(a.alpha, sp, oma * m);
            }
            if (tot >= a.access_thr) t_ref = a.t;   // the clock runs in every age mode
        } else if (!is_new) {
            old_m = m;
        }
        const int age = a.t - (a.age_mode == KVEV_AGE_SINCE_ACCESS ? t_ref : t_ins);
        const float pr = age == 0 ? 0.0f : (1.0f - m) * -expm1f(-a.beta * (float)age);
        a.keys[si] = order_bits(pr);
        a.m_s[si] = m;
        a.tref_s[si] = t_ref;
        a.tins_s[si] = t_ins;
        a.pos_s[si] = pos;
        if (a.dbg_prio) a.dbg_prio[si] = pr + 0.0f;
    }
    if (!a.refresh) {  // deterministic block sum of the old tokens' scores
        __shared__ float red[kScoreThreads / 32];
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
}

}  // namespace

cudaError_t launch_score(const ScoreArgs& a, int group, int* n_blocks, cudaStream_t s) {
    if (a.refresh) {
        const int split = a.n_kv % 2 == 0 ? 2 : 1;
        const int nb = (a.L * split + kRefreshThreads - 1) / kRefreshThreads;
        *n_blocks = nb;
        const dim3 grid(nb, a.batch);
        const size_t smem = sizeof(float) * (size_t)a.n_layers * a.n_q;
        void (*kern)(ScoreArgs) = nullptr;
        if (group == 4) kern = split == 2 ? score_refresh_kernel<4, 2> : score_refresh_kernel<4, 1>;
        if (group == 8) kern = split == 2 ? score_refresh_kernel<8, 2> : score_refresh_kernel<8, 1>;
        if (!kern) return cudaErrorInvalidValue;
        return launch_pdl(kern, grid, dim3(kRefreshThreads), smem, s, a);
    }
    const int nb = (a.L + kScoreThreads - 1) / kScoreThreads;
    *n_blocks = nb;
    const dim3 grid(nb, a.batch);
    const size_t smem = sizeof(float) * (size_t)a.n_layers * a.n_q;
    if (group == 4) return launch_pdl(score_kernel<4>, grid, dim3(kScoreThreads), smem, s, a);
    if (group == 8) return launch_pdl(score_kernel<8>, grid, dim3(kScoreThreads), smem, s, a);
    return cudaErrorInvalidValue;
}

}  // namespace kvev
