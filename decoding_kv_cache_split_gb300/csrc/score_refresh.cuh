// The refresh-step scorer's per-token work, shared by the scoring kernel
// (score.cu) and the fused attention step (attn.cu).  See score.cu for the
// method and its sources.
#pragma once

#include "kvev_internal.h"
#include "mma_ops.h"

namespace kvev {
namespace {

__device__ __forceinline__ uint32_t order_bits(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Refresh steps: a CTA takes 32 consecutive tokens (a warp's lanes, so
// every load instruction of a warp reads 512 contiguous bytes) and splits
// the layers into 4 consecutive segments, one per warp (the fused step's
// CTAs have the same 4 warps).  The EMA over a segment is affine in the
// score it starts from, m_out = (1 - alpha)^n m_in + c, so each segment is
// folded in order starting from 0 (the first from the token's score itself)
// and the first warp chains the segments with (1 - alpha)^n from the host:
// the layer order of the recurrence is kept and 4x more threads share the
// loads.  The number of KV heads is a template parameter so a
// layer's heads are an unrolled loop with no index arithmetic; the loads of
// kLB layers are all issued before any is used.

// Shared-memory tables of sequence b (every thread of the CTA takes part;
// ends with a barrier): [n_layers][NKV * G] log2-sum-exp, then [n_layers]
// layer weights, then [n_layers][NKV] inverse mean value norms (VN).
template <int G, int NKV, bool VN>
__device__ __forceinline__ void score_tables(const ScoreArgs& a, int b, float* s_lse) {
    float* s_lw = s_lse + a.n_layers * NKV * G;
    float* s_ivm = s_lw + a.n_layers;
    const int n_lay = a.n_layers;
    const int nlse = n_lay * NKV * G;
    for (int k = threadIdx.x; k < nlse; k += blockDim.x) {
        const int l = k / (NKV * G), h = k % (NKV * G);
        s_lse[k] = a.lse2[((size_t)l * a.batch + b) * a.n_q + h];
    }
    for (int l = threadIdx.x; l < n_lay; l += blockDim.x) {   // entropy weight: head mean
        float w = 1.f;
        if (a.ent) {
            w = 0.f;
            for (int h = 0; h < NKV * G; ++h) w += a.ent[((size_t)l * a.batch + b) * a.n_q + h];
            w /= (float)(NKV * G);
        }
        s_lw[l] = w;
    }
    if constexpr (VN) {
        for (int k = threadIdx.x; k < n_lay * NKV; k += blockDim.x) {
            const float vm = a.vmean[((size_t)(k / NKV) * a.batch + b) * NKV + k % NKV];
            s_ivm[k] = vm > 0.f ? 1.0f / vm : -1.0f;   // -1: every norm 0, factor 1
        }
    }
    __syncthreads();
}

// The 32 tokens of block `blk` of sequence b, folded in SEGS layer segments
// by the CTA's WARPS warps (warp w takes segments w, w + WARPS, ...; the
// arithmetic of a segment does not depend on which warp runs it), with the
// tables of score_tables in s_lse.
template <int G, int NKV, bool VN, int SEGS, int WARPS>
__device__ __forceinline__ void score_block(const ScoreArgs& a, int b, int blk,
                                            const float* s_lse, float (*s_c)[32],
                                            float (*s_tot)[32]) {
    static_assert(SEGS % WARPS == 0, "every warp takes the same number of segments");
    constexpr int V4 = G / 4;                               // float4 per (layer, KV head)
    constexpr int kLB = NKV * V4 >= 16 ? 1 : (16 / (NKV * V4) > 4 ? 4 : 16 / (NKV * V4));  // layers in flight
    constexpr int kPerLine = 128 / (G * 4);                 // tokens per 128-byte line
    const float* s_lw = s_lse + a.n_layers * NKV * G;
    const float* s_ivm = s_lw + a.n_layers;
    const int n_lay = a.n_layers;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blk * 32 + lane;
    const bool live = i < a.L;
    const size_t si = (size_t)b * a.max_ctx + i;
    const float oma = a.oma;
    const float inv_hq = 1.0f / (float)a.n_q;
    const size_t head_stride = (size_t)a.logit_ld * G;                  // one (layer, KV head) row
    const size_t layer_stride = (size_t)a.batch * NKV * head_stride;
    const float* base = a.logits + (size_t)b * NKV * head_stride + (size_t)i * G;
    const bool drop = i % kPerLine == 0 && i + kPerLine <= a.L;         // this thread drops lines

    float c = 0.f, tot = 0.f;
#pragma unroll
    for (int k = 0; k < SEGS / WARPS; ++k) {
        const int seg = warp + k * WARPS;
        const int la = seg * n_lay / SEGS, lb = (seg + 1) * n_lay / SEGS;
        c = live && seg == 0 ? a.st.score[si] : 0.f;   // the first segment starts from
        tot = 0.f;                                      // the score itself, the others at 0
        if (live) {
            for (int l0 = la; l0 < lb; l0 += kLB) {
                float4 xb[kLB][NKV][V4];
                float vb[kLB][NKV];
#pragma unroll
                for (int u = 0; u < kLB; ++u)                 // all loads of the batch first ...
#pragma unroll
                    for (int g = 0; g < NKV; ++g) {
#pragma unroll
                        for (int cc = 0; cc < V4; ++cc)
                            xb[u][g][cc] = l0 + u < lb
                                ? __ldcs(reinterpret_cast<const float4*>(
                                      base + (size_t)(l0 + u) * layer_stride + g * head_stride) + cc)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
                        if constexpr (VN)
                            vb[u][g] = l0 + u < lb
                                ? __ldcs(a.vnorm + (((size_t)(l0 + u) * a.batch + b) * NKV + g) *
                                                       a.logit_ld + i)
                                : 0.f;
                    }
#pragma unroll
                for (int u = 0; u < kLB; ++u) {               // ... then the layers in order
                    const int lr = l0 + u;
                    if (lr >= lb) break;
                    const float4* lg = reinterpret_cast<const float4*>(s_lse + lr * NKV * G);
                    float s = 0.f, sw = 0.f;   // head sum; with VNorm, weighted by the value norms
#pragma unroll
                    for (int g = 0; g < NKV; ++g) {
                        float sg = 0.f;
#pragma unroll
                        for (int cc = 0; cc < V4; ++cc) {
                            const float4 x = xb[u][g][cc], e = lg[g * V4 + cc];
                            const float p0 = fast_exp2(x.x - e.x), p1 = fast_exp2(x.y - e.y);
                            const float p2 = fast_exp2(x.z - e.z), p3 = fast_exp2(x.w - e.w);
                            if (a.dbg_probs) {
                                float* dp = a.dbg_probs +
                                            (((size_t)b * a.n_layers + lr) * a.n_q + g * G + 4 * cc) *
                                                a.max_ctx + i;
                                dp[0] = p0;
                                dp[(size_t)a.max_ctx] = p1;
                                dp[2 * (size_t)a.max_ctx] = p2;
                                dp[3 * (size_t)a.max_ctx] = p3;
                            }
                            sg += (p0 + p1) + (p2 + p3);
                        }
                        s += sg;
                        if constexpr (VN) {
                            const float iv = s_ivm[lr * NKV + g];
                            sw = fmaf(iv >= 0.f ? vb[u][g] * iv : 1.0f, sg, sw);
                        }
                    }
                    // The logits are dead once read: drop their L2 lines without
                    // writing them back.  A 128-byte line holds kPerLine tokens of
                    // one (layer, KV head) row (rows start on a line), all loaded by
                    // this warp's load, which has completed since its values were
                    // just used (the discard takes `s` as an operand, so it cannot
                    // move above that use).  The line's first token's thread drops it.
                    if (drop) {
#pragma unroll
                        for (int g = 0; g < NKV; ++g)
                            asm volatile("discard.global.L2 [%0], 128;" ::"l"(
                                             base + (size_t)lr * layer_stride + g * head_stride),
                                         "f"(s)
                                         : "memory");
                    }
                    tot += s;                  // the access test reads the plain attention
                    float sl = VN ? sw : s;
                    if (a.pool_mean) sl *= inv_hq;
                    c = fmaf(a.alpha, sl * s_lw[lr], oma * c);
                }
            }
        }
        s_c[seg][lane] = c;
        s_tot[seg][lane] = tot;
    }
    __syncthreads();
    if (warp != 0 || !live) return;
    c = s_c[0][lane];
    // chain the segments in layer order: m <- (1 - alpha)^(layers of k) m + c_k
    float m = c;
    tot = s_tot[0][lane];
#pragma unroll
    for (int k = 1; k < SEGS; ++k) {
        m = fmaf(a.seg_decay[k], m, s_c[k][lane]);
        tot += s_tot[k][lane];
    }
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
    if (a.raw_keys) a.raw_keys[si] = order_bits(-tot);   // the largest raw score first
    if (a.dbg_raw) a.dbg_raw[si] = tot;
}

}  // namespace
}  // namespace kvev
