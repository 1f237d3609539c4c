// Attention over the INT2 windows of the two-tier cache ("QEvict: ...",
// Sec. 4.1: the accessible keys and values include the dequantized INT2
// windows), with the dequantization folded into the tensor-core products.
//
// A key is k_c = code_c * s_c + z_c = s_c (code_c - 1.5) + (z_c + 1.5 s_c)
// with (s, z) per channel over a 32-token group, so within a group
//     q . k = sum_c (q_c s_c)(code_c - 1.5) + sum_c q_c (z_c + 1.5 s_c) :
// the A operand is q * s (bf16 hi + lo, the product is exact in fp32), the
// B operand the centred codes (exact in bf16), plus a per-head bias.  A
// value is v_c = s_g (code_c - 1.5) + (z_g + 1.5 s_g) with (s, z) per token
// over a 32-channel group g, so
//     sum_i p_i v_ic = sum_i (p_i s_ig)(code_ic - 1.5) + sum_i p_i (z_ig + 1.5 s_ig) :
// per channel group the A operand is p * s (hi + lo), B the centred codes,
// plus a per-head, per-group bias carried through the online softmax like
// the output.  Centring keeps both sums near the size of the result, so the
// hi + lo rounding of the products is not magnified by cancellation between
// a large code sum and a large zero-point sum.
//
// Work: every (layer, sequence, KV head) row has `slots` units, one INT2
// window each (past the sequence's INT2 list a unit is empty); warps take
// equal contiguous ranges of units (split-K over windows), double-buffer a
// unit's 12 KiB ledger entry in shared memory with cp.async, and leave a
// softmax partial per (warp, row) piece for the split combine, plus the
// per-16-token-tile statistics the window scores are formed from.
#include <cuda_fp16.h>

#include "kvev_internal.h"
#include "mma_ops.h"

namespace kvev {
namespace {

constexpr int kI2Warps = 4;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_prior() {   // all but the newest group
    asm volatile("cp.async.wait_group 1;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}
// Two 2-bit codes at bits 1-2 and 17-18 of x (other bits clear) -> bf16x2 of
// the centred codes c - 1.5 (exact): ORed into the mantissa of 64 (unit 0.5)
// the field 2c reads 64 + c, and 64 + c - 65.5 = c - 1.5.
__device__ __forceinline__ uint32_t centred_bf16x2(uint32_t x) {
    uint32_t r;
    const uint32_t biased = x | 0x42804280u;   // 64 + c
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(biased), "r"(0x42834283u));   // - 65.5
    return r;
}
// The lane's code word: rotated so that its two code pairs sit at bits 1-2 / 17-18
// (b0) and 9-10 / 25-26 (b1) for a lane with column pair t.
__device__ __forceinline__ uint32_t lane_codes(uint32_t u, int t) {
    return __funnelshift_r(u, u, (2 * t + 31) & 31);
}

// The 16 x 8 x 16 tensor-core tile has 8 A rows and a group has 4 query
// heads, so rows 0-3 carry the bf16 "hi" part of each head's operand and
// rows 4-7 the "lo" part (operand - hi): one MMA per operand pair instead of
// two, the halves summed with one shuffle (lane g and lane g + 4, i.e. xor
// 16) where the full value is needed.  Lanes g and g + 4 therefore hold the
// same head (g & 3) and run identical softmax bookkeeping.
template <int D, int G>
__global__ void __launch_bounds__(kI2Warps * 32) attn_int2_kernel(const Int2Args a) {
    static_assert(G == 4, "hi / lo rows need 4 query heads per KV head");
    using Lay = LedgerLayout<D>;
    constexpr int KS = D / 16, NB = D / 8, NG = D / kQGroup;
    extern __shared__ __align__(128) unsigned char smem[];
    griddep_wait();
    griddep_release();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* wbuf = smem + (size_t)warp * 2 * Lay::BYTES;
    const int w = blockIdx.x * kI2Warps + warp;
    const int64_t N = a.n_units;
    const int64_t x0 = (int64_t)w * N / a.total_warps, x1 = (int64_t)(w + 1) * N / a.total_warps;
    if (x0 >= x1) return;

    const int g = lane >> 2, t = lane & 3;   // fragment row, column pair
    const int head = g & 3;                  // query head of the group
    const bool lo_row = g >= 4;              // this row carries the "lo" parts
    // window id of unit x (-1: empty), and its ledger entry
    auto unit_window = [&](int64_t x, const unsigned char** src) -> int {
        const int64_t row = x / a.slots;
        const int j = (int)(x - row * a.slots);
        const int gk = (int)(row % a.n_kv);
        const int64_t lb = row / a.n_kv;
        const int b = (int)(lb % a.batch), l = (int)(lb / a.batch);
        if (j >= a.n_qwin[b]) return -1;
        const int wi = a.q_list[(size_t)b * a.q_ld + j];
        *src = a.ledger +
               ((((size_t)b * a.max_windows + wi) * a.n_layers + l) * a.n_kv + gk) * Lay::BYTES;
        return wi;
    };
    auto issue = [&](int64_t x, int bi) {
        const unsigned char* src = nullptr;
        if (unit_window(x, &src) >= 0) {
            const uint32_t dst = smem_addr(wbuf + (size_t)bi * Lay::BYTES);
            for (int i = lane; i < Lay::BYTES / 16; i += 32) cp_async16(dst + 16 * i, src + 16 * i);
        }
        cp_async_commit();
    };
    // the lane's half (hi or lo) of a product pair
    auto half_pair = [&](float x0v, float x1v) -> uint32_t {
        const uint32_t hi = pack_bf16x2(x0v, x1v);
        return lo_row ? pack_bf16x2(x0v - bf16_lo(hi), x1v - bf16_hi(hi)) : hi;
    };

    uint32_t qa0[KS], qa2[KS];               // Q (bf16x2) of the lane's head
    float o[NB][2];                          // hi or lo part of O[head][8j + 2t, +1]
    float vbias[NG];                         // sum_i p_i z_ig of the head, per channel group
    float m_run = -INFINITY, l_run = 0.f;
    int64_t cur_row = -1;

    auto flush = [&](int64_t row) {
        float l = l_run;
        l += __shfl_xor_sync(kFull, l, 1);
        l += __shfl_xor_sync(kFull, l, 2);
        const int64_t slot = (int64_t)w + row;
        float* po = a.part_o + ((size_t)slot * G + head) * D;
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const float v0 = o[j][0] + __shfl_xor_sync(kFull, o[j][0], 16);
            const float v1 = o[j][1] + __shfl_xor_sync(kFull, o[j][1], 16);
            if (!lo_row)
                *reinterpret_cast<float2*>(po + 8 * j + 2 * t) =
                    make_float2(v0 + vbias[j / 4], v1 + vbias[j / 4]);
        }
        if (!lo_row && t == 0) {
            float* pml = a.part_ml + ((size_t)slot * G + head) * 2;
            pml[0] = m_run;
            pml[1] = l;
        }
    };

    issue(x0, 0);
    int bi = 0;
    for (int64_t x = x0; x < x1; ++x, bi ^= 1) {
        if (x + 1 < x1) issue(x + 1, bi ^ 1);
        else cp_async_commit();              // keep one group per iteration
        cp_async_wait_prior();
        __syncwarp();
        const int64_t row = x / a.slots;
        if (row != cur_row) {
            if (cur_row >= 0) flush(cur_row);
            cur_row = row;
            const int gk = (int)(row % a.n_kv);
            const int64_t lb = row / a.n_kv;
            const int b = (int)(lb % a.batch), l = (int)(lb / a.batch);
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                a.q + (((size_t)b * a.n_layers + l) * a.n_q + (size_t)gk * G + head) * D);
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                qa0[s] = qrow[8 * s + t];       // dims 16s + 2t, +1
                qa2[s] = qrow[8 * s + 4 + t];   // dims 16s + 8 + 2t, +1
            }
#pragma unroll
            for (int j = 0; j < NB; ++j) o[j][0] = o[j][1] = 0.f;
#pragma unroll
            for (int c = 0; c < NG; ++c) vbias[c] = 0.f;
            m_run = -INFINITY;
            l_run = 0.f;
        }
        const unsigned char* src = nullptr;
        const int wid = unit_window(x, &src);
        if (wid >= 0) {
            const unsigned char* buf = wbuf + (size_t)bi * Lay::BYTES;
            const uint32_t* kc = reinterpret_cast<const uint32_t*>(buf + Lay::KC);
            const uint32_t* vc = reinterpret_cast<const uint32_t*>(buf + Lay::VC);
            const __half2* ks2 = reinterpret_cast<const __half2*>(buf + Lay::KS);
            const __half2* kz2 = reinterpret_cast<const __half2*>(buf + Lay::KZ);
            const uint2* vs4 = reinterpret_cast<const uint2*>(buf + Lay::VS);   // 4 fp16 per token
            const uint2* vz4 = reinterpret_cast<const uint2*>(buf + Lay::VZ);
            for (int grp = 0; grp < kTierW / kQGroup; ++grp) {
                // A' = q * s of this group's key scales (the lane's hi or lo part),
                // and the key bias sum_c q_c z_c
                uint32_t af[KS][2];
                float kb = 0.f;
#pragma unroll
                for (int s = 0; s < KS; ++s) {
                    const int c0 = 16 * s + 2 * t, c2 = c0 + 8;
                    const float2 s01 = __half22float2(ks2[(grp * D + c0) / 2]);
                    const float2 s23 = __half22float2(ks2[(grp * D + c2) / 2]);
                    const float2 z01 = __half22float2(kz2[(grp * D + c0) / 2]);
                    const float2 z23 = __half22float2(kz2[(grp * D + c2) / 2]);
                    const float q0 = bf16_lo(qa0[s]), q1 = bf16_hi(qa0[s]);
                    const float q2 = bf16_lo(qa2[s]), q3 = bf16_hi(qa2[s]);
                    af[s][0] = half_pair(q0 * s01.x, q1 * s01.y);
                    af[s][1] = half_pair(q2 * s23.x, q3 * s23.y);
                    kb = fmaf(q0, fmaf(1.5f, s01.x, z01.x), kb);
                    kb = fmaf(q1, fmaf(1.5f, s01.y, z01.y), kb);
                    kb = fmaf(q2, fmaf(1.5f, s23.x, z23.x), kb);
                    kb = fmaf(q3, fmaf(1.5f, s23.y, z23.y), kb);
                }
                kb += __shfl_xor_sync(kFull, kb, 1);
                kb += __shfl_xor_sync(kFull, kb, 2);
#pragma unroll 1
                for (int tt = 0; tt < kQGroup / kTile; ++tt) {
                    const int ti = grp * (kQGroup / kTile) + tt;   // 16-token tile of the window
                    const int tok0 = ti * kTile;
                    // ---- S = A' codes (two 8-token blocks; even and odd k-steps in
                    //      separate accumulators) + bias
                    float acc[2][2][2] = {};
#pragma unroll
                    for (int s = 0; s < KS; ++s)
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const uint32_t y = lane_codes(kc[(tok0 + 8 * i + g) * KS + s], t);
                            const uint32_t b0 = centred_bf16x2(y & 0x00060006u);
                            const uint32_t b1 = centred_bf16x2((y >> 8) & 0x00060006u);
                            mma_rows8(acc[s & 1][i][0], acc[s & 1][i][1], af[s][0], af[s][1], b0, b1);
                        }
                    float sc[2][2];
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float part = acc[0][i][e] + acc[1][i][e];
                            sc[i][e] = (part + __shfl_xor_sync(kFull, part, 16) + kb) * a.q_scale;
                        }
                    // ---- online softmax of the head
                    float mt = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
                    mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
                    mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
                    if (mt > m_run) {
                        const float f = fast_exp2(m_run - mt);
                        m_run = mt;
                        l_run *= f;
#pragma unroll
                        for (int j = 0; j < NB; ++j) {
                            o[j][0] *= f;
                            o[j][1] *= f;
                        }
#pragma unroll
                        for (int c = 0; c < NG; ++c) vbias[c] *= f;
                    }
                    float pv[4];
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            pv[2 * i + e] = fast_exp2(sc[i][e] - m_run);
                            l_run += pv[2 * i + e];
                        }
                    if (a.tile_stats) {   // (running max, tile sum) of the head for the window score
                        float ts = (pv[0] + pv[1]) + (pv[2] + pv[3]);
                        ts += __shfl_xor_sync(kFull, ts, 1);
                        ts += __shfl_xor_sync(kFull, ts, 2);
                        if (!lo_row && t == 0)
                            a.tile_stats[((size_t)row * a.stats_tiles + (size_t)wid * (kTierW / kTile) +
                                          ti) * G + head] = make_float2(m_run, ts);
                    }
                    // ---- O += (p * s_v) codes + p * z_v, per 32-channel group
                    uint2 vsr[4], vzr[4];   // the 4 fp16 scales / zeros of the lane's tokens
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int tk = tok0 + (k >> 1) * 8 + 2 * t + (k & 1);
                        vsr[k] = vs4[tk];
                        vzr[k] = vz4[tk];
                    }
#pragma unroll
                    for (int cg = 0; cg < NG; ++cg) {
                        float sv[4], vb = 0.f;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t ws = (cg < 2 ? vsr[k].x : vsr[k].y) >> (16 * (cg & 1));
                            const uint32_t wz = (cg < 2 ? vzr[k].x : vzr[k].y) >> (16 * (cg & 1));
                            sv[k] = __half2float(__ushort_as_half((unsigned short)(ws & 0xffffu)));
                            const float zc = __half2float(__ushort_as_half((unsigned short)(wz & 0xffffu)));
                            vb = fmaf(pv[k], fmaf(1.5f, sv[k], zc), vb);
                        }
                        vb += __shfl_xor_sync(kFull, vb, 1);
                        vb += __shfl_xor_sync(kFull, vb, 2);
                        vbias[cg] += vb;
                        const uint32_t pa0 = half_pair(pv[0] * sv[0], pv[1] * sv[1]);
                        const uint32_t pa2 = half_pair(pv[2] * sv[2], pv[3] * sv[3]);
#pragma unroll
                        for (int jj = 0; jj < kQGroup / 8; ++jj) {
                            const int j = cg * (kQGroup / 8) + jj;      // 8-channel block
                            const uint32_t y = lane_codes(vc[ti * D + 8 * j + g], t);
                            const uint32_t b0 = centred_bf16x2(y & 0x00060006u);
                            const uint32_t b1 = centred_bf16x2((y >> 8) & 0x00060006u);
                            mma_rows8(o[j][0], o[j][1], pa0, pa2, b0, b1);
                        }
                    }
                }
            }
        }
        __syncwarp();   // every lane is done with this buffer before it is refilled
    }
    cp_async_wait_all();
    flush(cur_row);
}

template <int D, int G>
int ctas_per_sm_int2() {
    auto kern = attn_int2_kernel<D, G>;
    const int smem = kI2Warps * 2 * LedgerLayout<D>::BYTES;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kI2Warps * 32, smem) !=
        cudaSuccess)
        return 0;
    return n;
}

}  // namespace

int int2_warps_per_cta() { return kI2Warps; }

int int2_ctas_per_sm(int head_dim, int group) {
    if (head_dim == 128 && group == 4) return ctas_per_sm_int2<128, 4>();
    return 0;
}

cudaError_t launch_attn_int2(const Int2Args& a, int head_dim, int group, int grid,
                             cudaStream_t s) {
    if (head_dim != 128 || group != 4) return cudaErrorInvalidValue;
    auto kern = attn_int2_kernel<128, 4>;
    const int smem = kI2Warps * 2 * LedgerLayout<128>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kI2Warps * 32), (size_t)smem, s, a);
}

}  // namespace kvev
