// Attention over the INT2 windows of the two-tier cache ("QEvict: ...",
// Sec. 4.1: the accessible keys and values include the dequantized INT2
// windows), with the dequantization folded into the tensor-core products.
//
// A key is k_c = code_c * s_c + z_c with (s, z) per channel over a 32-token
// group, so within a group
//     q . k = sum_c (q_c s_c) code_c + sum_c q_c z_c :
// the A operand is q * s (bf16 hi + lo), the B operand the codes, plus a
// per-head bias (q has both signs and a logit sums 128 channels afresh, so
// the codes need no centring here).  A value is v_c = s_g (code_c - 1.5) + (z_g + 1.5 s_g)
// with (s, z) per token over a 32-channel group g, so
//     sum_i p_i v_ic = sum_i (p_i s_ig)(code_ic - 1.5) + sum_i p_i (z_ig + 1.5 s_ig) :
// per channel group the A operand is p * s (hi + lo), B the centred codes,
// plus a per-head, per-group bias carried through the online softmax like
// the output.  Centring keeps the value sums, which run over whole rows,
// near the size of the result.
//
// The ledger stores each key code as a plain 2-bit number at the bit
// positions of its tensor-core register (see LedgerLayout): a word shifted by
// 0, 6 or 12 and masked gives a bf16 pair of exact subnormals c 2^(2 k)
// 2^-133, k the register's scale class, two shifts and eight masks per word;
// the A operand of k-step s carries 2^(96 - 2 k(s)), so every key product is
// code * q s * 2^-37.  Each value code is a sign and a magnitude bit at the
// positions of its register: one rotate and one mask-and-OR turn a word into
// a bf16 pair of exact subnormals (2 c - 3) * 2^-128; the value A operands
// carry 2^96, so the output products are the centred terms times 2^-31,
// rescaled once per row.
//
// Work: every (layer, sequence, KV head) row has `slots` units, one INT2
// window each (past the sequence's INT2 list a unit is empty); warps take
// equal contiguous ranges of units (split-K over windows), double-buffer a
// unit's 12 KiB ledger entry in shared memory with cp.async, and leave a
// softmax partial per (warp, row) piece for the split combine, plus the
// per-16-token-tile statistics the window scores are formed from.
//
// The bias terms run on the tensor cores too, as fp16 products (fp16 scale and
// zero times q or p split into fp16 hi + lo rows: exact products, fp32 sums):
// per unit one 8-k-step MMA of q against a B operand whose columns are the
// four key groups' zeros (and scales, unused) gives every group's
// sum_c q_c z_c; per tile one MMA of p 2^10 (the scaling keeps its fp16 lo
// part out of the subnormal range) against the tokens' group centres
// z + 1.5 s as fp16 hi and lo columns adds sum_i p_i (z_ig + 1.5 s_ig) to an
// accumulator that the online softmax rescales like the output.  The centres
// take both signs, so the tensor cores' accumulation, which drops low bits as
// it adds, does not build up a one-signed error the way separate sums of p z
// and p s do over a long row.
#include <cuda_fp16.h>

#include "kvev_internal.h"
#include "mma_ops.h"

namespace kvev {
namespace {

constexpr int kI2Warps = 4;
constexpr int kQhBytes = 32 * 16 * 4;   // per warp: q as fp16 hi / lo operand pairs
constexpr unsigned kFull = 0xffffffffu;
constexpr float kAScale = 0x1p96f;    // A operands carry 2^96 (keys: divided by the class scale)
constexpr float kProdScale = 0x1p31f; // undoes 2^96 * 2^-127 (code - 1.5 in a value B operand)
constexpr float kKeyScale = 0x1p37f;  // undoes 2^96 * 2^-133 (a code in a key B operand)
constexpr float kPScale = 0x1p10f;    // p in the value-bias MMA: its fp16 lo part stays normal

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
// Register of field f of a key code word: the bf16 pair c 2^(2 (f % 3)) 2^-133.
// f is a compile-time constant in every use; the shifts of a word are shared.
__device__ __forceinline__ uint32_t field_reg(uint32_t w, int f) {
    return (w >> (6 * (f / 3))) & (0x00030003u << (2 * (f % 3)));
}
// Register `slot` of a value code word: the bf16 pair (2 c - 3) * 2^-128.
__device__ __forceinline__ uint32_t code_reg(uint32_t w, int slot) {
    const uint32_t x = slot == 0 ? w : __funnelshift_r(w, w, 2 * slot);
    return (x & 0x80408040u) | 0x00200020u;
}
__device__ __forceinline__ float2 h2f(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
// Two independent fp32 operations in one instruction (each correctly
// rounded, as the scalar ones).
__device__ __forceinline__ uint64_t pk2(float2 a) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
    return r;
}
__device__ __forceinline__ float2 up2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)), "l"(pk2(c)));
    return up2(r);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)));
    return up2(r);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)));
    return up2(r);
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
    static_assert(D == 128, "ledger registers are laid out for head_dim 128");
    using Lay = LedgerLayout<D>;
    constexpr int KS = D / 16, NB = D / 8, NG = Lay::NG;
    extern __shared__ __align__(128) unsigned char smem[];
    griddep_wait();
    griddep_release();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* wbuf = smem + (size_t)warp * (2 * Lay::BYTES + kQhBytes);
    // q of the current row as fp16 operand pairs, k-step major: uint4 k of lane l
    // at qh4[32 k + l] holds (s, h) = (2k, 0), (2k, 1), (2k + 1, 0), (2k + 1, 1)
    uint4* qh4 = reinterpret_cast<uint4*>(wbuf + 2 * Lay::BYTES);
    const int w = blockIdx.x * kI2Warps + warp;
    const int64_t N = a.n_units;
    const int64_t x0 = (int64_t)w * N / a.total_warps, x1 = (int64_t)(w + 1) * N / a.total_warps;
    if (x0 >= x1) return;

    const int g = lane >> 2, t = lane & 3;   // fragment row, column pair
    const int head = g & 3;                  // query head of the group
    const bool lo_row = g >= 4;              // this row carries the "lo" parts
    const float lom = lo_row ? 1.f : 0.f;
    // Unit x is INT2 slot j of row (layer l, sequence b, KV head gk), rows
    // ordered ((l batch) + b) n_kv + gk; a warp's units are consecutive, so
    // the position is divided out once and then stepped.
    struct UnitPos {
        int64_t row;
        int j, b, l, gk;
    };
    auto locate = [&](int64_t x) {
        UnitPos u;
        u.row = x / a.slots;
        u.j = (int)(x - u.row * a.slots);
        u.gk = (int)(u.row % a.n_kv);
        const int64_t lb = u.row / a.n_kv;
        u.b = (int)(lb % a.batch);
        u.l = (int)(lb / a.batch);
        return u;
    };
    auto advance = [&](UnitPos& u) {
        if (++u.j < a.slots) return;
        u.j = 0;
        ++u.row;
        if (++u.gk < a.n_kv) return;
        u.gk = 0;
        if (++u.b < a.batch) return;
        u.b = 0;
        ++u.l;
    };
    // window id of a unit (-1: past the sequence's INT2 list), and its ledger entry
    auto unit_window = [&](const UnitPos& u, const unsigned char** src) -> int {
        if (u.j >= a.n_qwin[u.b]) return -1;
        const int wi = a.q_list[(size_t)u.b * a.q_ld + u.j];
        *src = a.ledger +
               ((((size_t)u.b * a.max_windows + wi) * a.n_layers + u.l) * a.n_kv + u.gk) *
                   Lay::BYTES;
        return wi;
    };
    auto issue = [&](const unsigned char* src, int wid, int bi) {
        if (wid >= 0) {
            const uint32_t dst = smem_addr(wbuf + (size_t)bi * Lay::BYTES);
            for (int i = lane; i < Lay::BYTES / 16; i += 32) cp_async16(dst + 16 * i, src + 16 * i);
        }
        cp_async_commit();
    };
    // the lane's half (hi or lo) of a product pair: the hi part is the pair
    // truncated to bf16 (exact), the lo part what it leaves (exact in fp32)
    // rounded to bf16; hi rows form 0 * x + hi, lo rows 1 * x + (-hi)
    const uint32_t hi_sign = lo_row ? 0x80000000u : 0u;
    const float2 lo_sel = make_float2(lom, lom);
    auto half_pair = [&](float2 xv) -> uint32_t {
        const float2 hb = make_float2(__uint_as_float((__float_as_uint(xv.x) & 0xffff0000u) ^ hi_sign),
                                      __uint_as_float((__float_as_uint(xv.y) & 0xffff0000u) ^ hi_sign));
        const float2 r = fma2(lo_sel, xv, hb);
        return pack_bf16x2(r.x, r.y);
    };

    uint32_t qa[KS][2];                      // Q * 2^(96 - 2 class(s)) (bf16x2) of the lane's head
    float2 o[NB];                            // hi or lo part of O[head][8j + 2t, +1] * 2^-31
    // value-bias accumulator (fp16 MMA): row g, columns 2t, 2t+1; column c < 4
    // sum_i p_i mid_ic, c >= 4 the same sum over what the fp16 mid_i(c-4)
    // leaves, mid = z + 1.5 s the group's centre (centred terms: a tensor-core
    // sum of one-signed terms, sum p z or sum p s, loses low bits every add)
    float2 vbc = make_float2(0.f, 0.f);
    float m_run = -INFINITY, l_run = 0.f;
    int64_t cur_row = -1;

    auto flush = [&](int64_t row) {
        float l = l_run;
        l += __shfl_xor_sync(kFull, l, 1);
        l += __shfl_xor_sync(kFull, l, 2);
        // the head's value bias of group c: the centre sum's hi + lo columns (and rows)
        float2 vt = add2(vbc, make_float2(__shfl_xor_sync(kFull, vbc.x, 16),
                                          __shfl_xor_sync(kFull, vbc.y, 16)));
        vt = mul2(vt, make_float2(1.0f / kPScale, 1.0f / kPScale));   // exact
        float vb[NG];
#pragma unroll
        for (int c = 0; c < NG; ++c) {
            const float mh = __shfl_sync(kFull, (c & 1) ? vt.y : vt.x, (lane & ~3) + (c >> 1));
            const float ml = __shfl_sync(kFull, (c & 1) ? vt.y : vt.x, (lane & ~3) + 2 + (c >> 1));
            vb[c] = mh + ml;
        }
        const int64_t slot = (int64_t)w + row;
        float* po = a.part_o + ((size_t)slot * G + head) * D;
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const float2 v = make_float2(o[j].x + __shfl_xor_sync(kFull, o[j].x, 16),
                                         o[j].y + __shfl_xor_sync(kFull, o[j].y, 16));
            if (!lo_row)
                *reinterpret_cast<float2*>(po + 8 * j + 2 * t) =
                    fma2(v, make_float2(kProdScale, kProdScale), make_float2(vb[j / 4], vb[j / 4]));
        }
        if (!lo_row && t == 0) {
            float* pml = a.part_ml + ((size_t)slot * G + head) * 2;
            pml[0] = m_run;
            pml[1] = l;
        }
    };
    const float acc_scale = a.q_scale * kKeyScale;    // logits from the code products

    UnitPos cur = locate(x0), nxt = cur;
    const unsigned char* src = nullptr;
    int wid = unit_window(cur, &src);
    issue(src, wid, 0);
    int bi = 0;
    for (int64_t x = x0; x < x1; ++x, bi ^= 1) {
        advance(nxt);                        // unit x + 1
        const unsigned char* src_next = nullptr;
        int wid_next = -1;
        if (x + 1 < x1) {
            wid_next = unit_window(nxt, &src_next);
            issue(src_next, wid_next, bi ^ 1);
        } else {
            cp_async_commit();               // keep one group per iteration
        }
        cp_async_wait_prior();
        __syncwarp();
        const int64_t row = cur.row;
        if (row != cur_row) {
            if (cur_row >= 0) flush(cur_row);
            cur_row = row;
            const int gk = cur.gk, b = cur.b, l = cur.l;
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                a.q + (((size_t)b * a.n_layers + l) * a.n_q + (size_t)gk * G + head) * D);
            uint32_t qhw[KS][2];
#pragma unroll
            for (int s = 0; s < KS; ++s)
#pragma unroll
                for (int h = 0; h < 2; ++h) {   // dims 16s + 8h + 2t, +1 (exact scaling)
                    const uint32_t qw = qrow[8 * s + 4 * h + t];
                    // fp16 hi (rows 0-3) or what it leaves (rows 4-7) of the same q
                    const float q0 = bf16_lo(qw), q1 = bf16_hi(qw);
                    // the key-side A operand of k-step s carries 2^(96 - 2 class(s))
                    const float ka = s < 3 ? kAScale : s < 6 ? 0x1p94f : 0x1p92f;
                    qa[s][h] = pack_bf16x2(q0 * ka, q1 * ka);
                    const uint32_t hw = pack_f16x2(q0, q1);
                    const float2 hf = unpack_f16x2(hw);
                    qhw[s][h] = lo_row ? pack_f16x2(q0 - hf.x, q1 - hf.y) : hw;
                }
            __syncwarp();   // the previous row's q pairs are no longer read
#pragma unroll
            for (int k = 0; k < KS / 2; ++k)
                qh4[32 * k + lane] = make_uint4(qhw[2 * k][0], qhw[2 * k][1], qhw[2 * k + 1][0],
                                                qhw[2 * k + 1][1]);
            __syncwarp();
#pragma unroll
            for (int j = 0; j < NB; ++j) o[j] = make_float2(0.f, 0.f);
            vbc = make_float2(0.f, 0.f);
            m_run = -INFINITY;
            l_run = 0.f;
        }
        if (wid >= 0) {
            const unsigned char* buf = wbuf + (size_t)bi * Lay::BYTES;
            const uint4* kc4 = reinterpret_cast<const uint4*>(buf + Lay::KC) + lane;
            const uint4* vc4 = reinterpret_cast<const uint4*>(buf + Lay::VC) + lane;
            const uint4* ks4 = reinterpret_cast<const uint4*>(buf + Lay::KS) + 4 * t;
            const uint4* vs4 = reinterpret_cast<const uint4*>(buf + Lay::VS) + 2 * t;
            // the value bias's B operand for tokens (2t, 2t+1) + 8 h of a tile:
            // the fp16 hi (columns 0-3) or lo (columns 4-7) part of the centre
            // z + 1.5 s (fp32) of channel group g & 3
            const uint32_t* vz32 = reinterpret_cast<const uint32_t*>(buf + Lay::VZ) +
                                   t * (4 * NG / 2) + (g & 3);
            const uint32_t* vs32 = reinterpret_cast<const uint32_t*>(buf + Lay::VS) +
                                   t * (4 * NG / 2) + (g & 3);
            auto centre_reg = [&](int idx) -> uint32_t {
                const float2 m = fma2(make_float2(1.5f, 1.5f), h2f(vs32[idx]), h2f(vz32[idx]));
                const uint32_t hi = pack_f16x2(m.x, m.y);
                const float2 hf = unpack_f16x2(hi);
                return lo_row ? pack_f16x2(m.x - hf.x, m.y - hf.y) : hi;
            };
            // key biases of the four groups: sum_c q_c z_c (columns 0-3; columns
            // 4-7 take the scales and are not read), one fp16 MMA chain
            float2 kbc = make_float2(0.f, 0.f);
            {
                const uint4* zs4 = reinterpret_cast<const uint4*>(buf + (lo_row ? Lay::KS : Lay::KZ)) +
                                   (g & 3) * (D / 8) + t * (D / 32);
#pragma unroll
                for (int k = 0; k < KS / 2; ++k) {
                    const uint4 qw = qh4[32 * k + lane], zw = zs4[k];
                    mma_rows8_f16(kbc.x, kbc.y, qw.x, qw.y, zw.x, zw.y);
                    mma_rows8_f16(kbc.x, kbc.y, qw.z, qw.w, zw.z, zw.w);
                }
                kbc = add2(kbc, make_float2(__shfl_xor_sync(kFull, kbc.x, 16),
                                            __shfl_xor_sync(kFull, kbc.y, 16)));
            }
            for (int grp = 0; grp < kTierW / kQGroup; ++grp) {
                // A' = q * s * 2^(96 - 2 class(s)) of this group's key scales (the
                // lane's hi or lo part); the key bias sum_c q_c z_c of the head
                uint32_t af[KS][2];
#pragma unroll
                for (int s2 = 0; s2 < KS / 2; ++s2) {
                    const uint4 sw = ks4[grp * (D / 8) + s2];
                    const uint32_t sws[4] = {sw.x, sw.y, sw.z, sw.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {   // (s, h) = (2 s2 + k / 2, k % 2)
                        const int s = 2 * s2 + k / 2, h = k % 2;
                        const float2 sc = h2f(sws[k]);
                        const float2 q01 = make_float2(bf16_lo(qa[s][h]), bf16_hi(qa[s][h]));
                        af[s][h] = half_pair(mul2(q01, sc));
                    }
                }
                const float kz = __shfl_sync(kFull, (grp & 1) ? kbc.y : kbc.x, (lane & ~3) + (grp >> 1));
                const float kb = kz * a.q_scale;   // the head's key bias sum_c q_c z_c
                // ---- S = A' codes + bias for both tiles of the group (two 8-token
                //      blocks each; even and odd k-steps in separate accumulators):
                //      their 32 MMAs are independent of the softmax below
                constexpr int TT = kQGroup / kTile;            // tiles per key group
                float sc[TT][2][2];
#pragma unroll
                for (int tt = 0; tt < TT; ++tt) {
                    const int ti = grp * TT + tt;               // 16-token tile of the window
                    const uint4 kq = kc4[ti * 32];
                    const uint32_t kw[4] = {kq.x, kq.y, kq.z, kq.w};
                    float acc[2][2][2] = {};
#pragma unroll
                    for (int s = 0; s < KS; ++s)
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const uint32_t b0 = field_reg(kw[2 * i], Lay::key_field(s));
                            const uint32_t b1 = field_reg(kw[2 * i + 1], Lay::key_field(s));
                            mma_rows8(acc[s & 1][i][0], acc[s & 1][i][1], af[s][0], af[s][1], b0, b1);
                        }
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        float2 part = add2(make_float2(acc[0][i][0], acc[0][i][1]),
                                           make_float2(acc[1][i][0], acc[1][i][1]));
                        part = add2(part, make_float2(__shfl_xor_sync(kFull, part.x, 16),
                                                      __shfl_xor_sync(kFull, part.y, 16)));
                        const float2 v = fma2(part, make_float2(acc_scale, acc_scale),
                                              make_float2(kb, kb));
                        sc[tt][i][0] = v.x;
                        sc[tt][i][1] = v.y;
                    }
                }
                // ---- online softmax of the head, one update for the group's 32 tokens
                float mt = -INFINITY;
#pragma unroll
                for (int tt = 0; tt < TT; ++tt)
                    mt = fmaxf(mt, fmaxf(fmaxf(sc[tt][0][0], sc[tt][0][1]),
                                         fmaxf(sc[tt][1][0], sc[tt][1][1])));
                mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
                mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
                if (mt > m_run) {
                    const float f = fast_exp2(m_run - mt);
                    m_run = mt;
                    l_run *= f;
#pragma unroll
                    for (int j = 0; j < NB; ++j) o[j] = mul2(o[j], make_float2(f, f));
                    vbc = mul2(vbc, make_float2(f, f));
                }
                float pv[TT][4];
#pragma unroll
                for (int tt = 0; tt < TT; ++tt)
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            pv[tt][2 * i + e] = fast_exp2(sc[tt][i][e] - m_run);
                            l_run += pv[tt][2 * i + e];
                        }
                if (a.tile_stats) {   // (running max, tile sum) per head and tile, for the window score
#pragma unroll
                    for (int tt = 0; tt < TT; ++tt) {
                        float ts = (pv[tt][0] + pv[tt][1]) + (pv[tt][2] + pv[tt][3]);
                        ts += __shfl_xor_sync(kFull, ts, 1);
                        ts += __shfl_xor_sync(kFull, ts, 2);
                        if (!lo_row && t == 0)
                            a.tile_stats[((size_t)row * a.stats_tiles + (size_t)wid * (kTierW / kTile) +
                                          grp * TT + tt) * G + head] = make_float2(m_run, ts);
                    }
                }
#pragma unroll
                for (int tt = 0; tt < TT; ++tt) {
                    const int ti = grp * TT + tt;
                    // ---- O += (p * s_v) codes, per 32-channel group; the value bias
                    //      sum_i p_i (z_ig, s_ig) by one fp16 MMA (p as hi / lo rows)
                    const uint4 vq = vc4[ti * 32];
                    const uint32_t vw[4] = {vq.x, vq.y, vq.z, vq.w};
                    const uint4 s0 = vs4[ti * 8], s1 = vs4[ti * 8 + 1];   // tokens 2t(+1), 2t+8(+1)
                    const uint32_t s0w[4] = {s0.x, s0.y, s0.z, s0.w}, s1w[4] = {s1.x, s1.y, s1.z, s1.w};
                    const float2 p01 = make_float2(pv[tt][0], pv[tt][1]);
                    const float2 p23 = make_float2(pv[tt][2], pv[tt][3]);
                    {   // p 2^10 (exact) as fp16 hi or lo
                        const float2 q01 = mul2(p01, make_float2(kPScale, kPScale));
                        const float2 q23 = mul2(p23, make_float2(kPScale, kPScale));
                        const uint32_t h01 = pack_f16x2(q01.x, q01.y), h23 = pack_f16x2(q23.x, q23.y);
                        uint32_t a0 = h01, a2 = h23;
                        if (lo_row) {
                            const float2 f01 = unpack_f16x2(h01), f23 = unpack_f16x2(h23);
                            a0 = pack_f16x2(q01.x - f01.x, q01.y - f01.y);
                            a2 = pack_f16x2(q23.x - f23.x, q23.y - f23.y);
                        }
                        mma_rows8_f16(vbc.x, vbc.y, a0, a2, centre_reg(ti * 32),
                                      centre_reg(ti * 32 + 4));
                    }
                    const float2 ps01 = mul2(p01, make_float2(kAScale, kAScale));
                    const float2 ps23 = mul2(p23, make_float2(kAScale, kAScale));
#pragma unroll
                    for (int cg = 0; cg < NG; ++cg) {
                        const float2 sa = h2f(s0w[cg]), sb = h2f(s1w[cg]);
                        const uint32_t pa0 = half_pair(mul2(ps01, sa));
                        const uint32_t pa2 = half_pair(mul2(ps23, sb));
#pragma unroll
                        for (int jj = 0; jj < kQGroup / 8; ++jj) {
                            const int j = cg * (kQGroup / 8) + jj;      // 8-channel block
                            const uint32_t b0 = code_reg(vw[cg], 2 * jj);
                            const uint32_t b1 = code_reg(vw[cg], 2 * jj + 1);
                            mma_rows8(o[j].x, o[j].y, pa0, pa2, b0, b1);
                        }
                    }
                }
            }
        }
        __syncwarp();   // every lane is done with this buffer before it is refilled
        cur = nxt;
        wid = wid_next;
    }
    cp_async_wait_all();
    flush(cur_row);
}

template <int D, int G>
int ctas_per_sm_int2() {
    auto kern = attn_int2_kernel<D, G>;
    const int smem = kI2Warps * (2 * LedgerLayout<D>::BYTES + kQhBytes);
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
    const int smem = kI2Warps * (2 * LedgerLayout<128>::BYTES + kQhBytes);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kI2Warps * 32), (size_t)smem, s, a);
}

}  // namespace kvev
