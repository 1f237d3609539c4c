// Split-K single-query GQA attention that keeps its logits.
//
// Computes, for every (layer, sequence, KV head) row of the cache and every
// query head h of that KV head's group, the last-query attention of
// "What Matters for Aggressive Decoding-Time KV Eviction?" Sec. 3.1 Eq. (1):
// logits q_h.k_i/sqrt(d), softmax over the live slots, output sum_i p_i v_i.
// Instead of discarding the logits as a fused decode kernel would, the
// kernel writes them (fp32, pre-scaled into the log2 domain) on refresh
// steps, so the scoring kernel turns them into probabilities with the
// combined normaliser without recomputing q.k (the pages name the
// recomputation, "attention fallback", as the largest per-step cost:
// Appendix J "Hook-level profiling").
//
// Design (GB300, sm_103a):
//  * The op is a GEMV over bf16 K/V: 4 flop per byte at GQA group 4, far
//    below the tensor-core ridge, so it runs on the FP32 pipes with packed
//    fma.rn.f32x2, and the goal is HBM bandwidth.
//  * Every warp owns an equal contiguous range of 16-token tiles of the
//    concatenated rows (no tail imbalance at any length) and streams them
//    through its own double buffer in shared memory with cp.async.bulk
//    (TMA bulk copies, completion on an mbarrier, L2 evict-first).  No
//    block-level barrier exists in the main loop.
//  * A row is read by D/8 lanes, 16 bytes each (LDS.128, conflict-free).
//    Partial dot products are combined by a shuffle reduce-scatter; the
//    lane-dependent index permutation that makes it select-free is folded
//    into the order in which each lane visits its rows and into the slot
//    order of its query registers.
//  * Softmax partials (running max, sum, output) of each warp's piece of a
//    row go to a slot; the last warp to finish a row (an atomic counter per
//    row) merges the row's partials and writes the output and the per-head
//    log2-sum-exp.  A standalone combine kernel does the same for callers
//    without counters.
#include <math.h>

#include "kvev_internal.h"

namespace kvev {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Bounded wait on a phase of an mbarrier; false if the phase never completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_test(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rc, rd;\n"
        " mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
        " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// 8 bf16 (one 16-byte word) -> 4 float pairs, exactly.
__device__ __forceinline__ void unpack8(uint4 w, float2 (&f)[4]) {
    f[0] = make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
    f[1] = make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    f[2] = make_float2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u));
    f[3] = make_float2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
}

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

template <int D, int G, int STAGES, int WARPS>
struct AttnCfg {
    static constexpr int T = kTile;
    static constexpr int LPR = D / 8;        // lanes per cache row (16 B each)
    static constexpr int RPW = 32 / LPR;     // rows covered by one warp-wide load
    static constexpr int RPL = T / RPW;      // rows a lane visits per tile
    static constexpr int NV = RPL * G;       // partial dot products per lane per tile
    static constexpr int NVF = NV / LPR;     // complete dot products per lane per tile
    static constexpr int LOG_NVF = ilog2(NVF);
    static constexpr int NSTEP = ilog2(LPR);
    static constexpr int TILE_BYTES = T * D * 2;
    static constexpr size_t SMEM = (size_t)WARPS * STAGES * 2 * TILE_BYTES +
                                   (size_t)WARPS * STAGES * sizeof(uint64_t);
    static_assert(NVF * 2 == G, "the lane layout splits each tile's heads into two groups");
    static_assert(RPL * RPW == T && NV % LPR == 0, "tile shape");
};

// Warps of the split whose tile range is empty write no partial.
__device__ __forceinline__ bool warp_has_tiles(int64_t w, int64_t N, int64_t W) {
    return w * N / W != (w + 1) * N / W;
}

// Called by every warp after it wrote its partial of `row`: the last of the
// row's warps to arrive merges all of the row's partials into the output and
// the log2-sum-exp, then resets the row's counter for the next launch.
struct CombineView {   // what the fused combine needs, passed by value
    const float* part_o;
    const float* part_ml;
    int32_t* row_done;
    float* out;
    float* lse2;
    int64_t N, W;
    int32_t tiles_per_row, n_kv, batch, n_layers, n_q;
};

template <int D, int G>
__device__ __noinline__ void fused_combine(const CombineView a, int64_t row, int lane) {
    constexpr int VPL = D / 32;   // output dims per lane
    const int64_t N = a.N, W = a.W;
    const int64_t first = row * a.tiles_per_row, last = first + a.tiles_per_row - 1;
    const int64_t w_lo = ((first + 1) * W - 1) / N, w_hi = ((last + 1) * W - 1) / N;
    __threadfence();   // this warp's partial is visible before it is counted
    __syncwarp();
    int is_last = 0;
    if (lane == 0) {
        int need = 0;
        for (int64_t w = w_lo; w <= w_hi; ++w) need += warp_has_tiles(w, N, W);
        is_last = atomicAdd(&a.row_done[row], 1) == need - 1;
    }
    if (!__shfl_sync(kFull, is_last, 0)) return;
    __threadfence();

    float M[G], lsum[G], acc[G][VPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        M[h] = -INFINITY;
        lsum[h] = 0.f;
#pragma unroll
        for (int v = 0; v < VPL; ++v) acc[h][v] = 0.f;
    }
    for (int64_t base = w_lo; base <= w_hi; base += 32) {   // segments, 32 at a time
        const int64_t w = base + lane;
        const bool valid = w <= w_hi && warp_has_tiles(w, N, W);
        float mj[G], lj[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mj[h] = valid ? __ldcg(a.part_ml + ((w + row) * G + h) * 2) : -INFINITY;
            lj[h] = valid ? __ldcg(a.part_ml + ((w + row) * G + h) * 2 + 1) : 0.f;
        }
        float Mn[G], fj[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float mm = mj[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(kFull, mm, o));
            Mn[h] = fmaxf(M[h], mm);
            const float fo = M[h] == -INFINITY ? 0.f : fast_exp2(M[h] - Mn[h]);
            lsum[h] *= fo;
#pragma unroll
            for (int v = 0; v < VPL; ++v) acc[h][v] *= fo;
            M[h] = Mn[h];
            fj[h] = valid ? fast_exp2(mj[h] - Mn[h]) : 0.f;
            float ls = lj[h] * fj[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(kFull, ls, o);
            lsum[h] += ls;
        }
        unsigned vm = __ballot_sync(kFull, valid);
        while (vm) {
            const int j = __ffs(vm) - 1;
            vm &= vm - 1;
            const int64_t slot = base + j + row;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float f = __shfl_sync(kFull, fj[h], j);
                const float* src = a.part_o + (slot * G + h) * D + lane * VPL;
#pragma unroll
                for (int v = 0; v < VPL; ++v) acc[h][v] += __ldcg(src + v) * f;
            }
        }
    }
    const int g = (int)(row % a.n_kv);
    const int64_t lb = row / a.n_kv;
    const int b = (int)(lb % a.batch), l = (int)(lb / a.batch);
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float* dst = a.out + (((size_t)b * a.n_layers + l) * a.n_q + (size_t)g * G + h) * D +
                     lane * VPL;
#pragma unroll
        for (int v = 0; v < VPL; ++v) dst[v] = acc[h][v] / lsum[h];
        if (lane == 0) a.lse2[row * G + h] = M[h] + log2f(lsum[h]);
    }
    if (lane == 0) a.row_done[row] = 0;
}

template <int D, int G, int STAGES, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
    attn_splitk_kernel(const AttnArgs a) {
    using C = AttnCfg<D, G, STAGES, WARPS>;
    constexpr int T = C::T, LPR = C::LPR, RPW = C::RPW, RPL = C::RPL, NV = C::NV,
                  NVF = C::NVF, TB = C::TILE_BYTES;

    extern __shared__ __align__(128) unsigned char smem[];
    griddep_wait();      // the append of this step is complete and visible
    griddep_release();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* wbuf = smem + (size_t)warp * STAGES * 2 * TB;
    uint64_t* bars =
        reinterpret_cast<uint64_t*>(smem + (size_t)WARPS * STAGES * 2 * TB) + warp * STAGES;

    const int w = blockIdx.x * WARPS + warp;
    const int64_t N = a.n_tiles_total;
    const int64_t x0 = (int64_t)w * N / a.total_warps;
    const int64_t x1 = (int64_t)(w + 1) * N / a.total_warps;
    if (x0 >= x1) return;  // this warp has no tiles (tiny problems)

    if (lane == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t pol = evict_first_policy();

    auto issue = [&](int64_t x, int stage) {  // lane 0 only
        const int64_t row = x / a.tiles_per_row;
        const int tok0 = (int)(x - row * a.tiles_per_row) * T;
        const int nv = min(T, a.L - tok0);
        const uint32_t bytes = (uint32_t)nv * D * 2;
        const size_t off = ((size_t)row * a.max_ctx + tok0) * D;
        unsigned char* dst = wbuf + (size_t)stage * 2 * TB;
        mbar_expect_tx(&bars[stage], 2 * bytes);
        bulk_load(dst, a.k + off, bytes, &bars[stage], pol);
        bulk_load(dst + TB, a.v + off, bytes, &bars[stage], pol);
    };
    if (lane == 0)
        for (int s = 0; s < STAGES && x0 + s < x1; ++s) issue(x0 + s, s);

    const int hl = lane % LPR, hr = lane / LPR;
    // Reduce-scatter bookkeeping: the lane stores the partial for (local row
    // j, head h) at index (j*G + h) ^ pmask, so each halving step keeps the
    // lower half; afterwards it owns rows j_own = hl>>1, heads h0..h0+NVF-1.
    const int pmask = hl << C::LOG_NVF;
    const int pmask_r = pmask / G, h0 = pmask % G;
    const bool odd = (hl & 1) != 0;

    float2 q2[G][4];   // slot h' holds head h' ^ h0, dims hl*8 .. hl*8+7, scaled
    float2 o2[G][4];   // running output, head h (natural order)
    float m_run[G];    // running max per head (log2 domain), same in every lane
    float l_part[NVF]; // this lane's share of the running sum, heads h0+e
    int64_t cur_row = -1;

    auto flush = [&](int64_t row) {
        // sum the output over lanes that read different rows of the same dims
#pragma unroll
        for (int m = LPR; m < 32; m <<= 1)
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    o2[h][c].x += __shfl_xor_sync(kFull, o2[h][c].x, m);
                    o2[h][c].y += __shfl_xor_sync(kFull, o2[h][c].y, m);
                }
#pragma unroll
        for (int e = 0; e < NVF; ++e)
#pragma unroll
            for (int m = 2; m < 32; m <<= 1) l_part[e] += __shfl_xor_sync(kFull, l_part[e], m);
        const int64_t slot = (int64_t)w + row;
        float* po = a.part_o + (size_t)slot * G * D;
        if (hr == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float4* dst = reinterpret_cast<float4*>(po + h * D + hl * 8);
                dst[0] = make_float4(o2[h][0].x, o2[h][0].y, o2[h][1].x, o2[h][1].y);
                dst[1] = make_float4(o2[h][2].x, o2[h][2].y, o2[h][3].x, o2[h][3].y);
            }
        }
        float* pml = a.part_ml + (size_t)slot * G * 2;
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) pml[h * 2] = m_run[h];
        }
        if (lane < 2) {  // lane 0 owns heads 0..NVF-1, lane 1 heads NVF..G-1
#pragma unroll
            for (int e = 0; e < NVF; ++e) pml[(h0 + e) * 2 + 1] = l_part[e];
        }
        if (a.row_done) {
            const CombineView cv{a.part_o, a.part_ml, a.row_done, a.out, a.lse2,
                                 a.n_tiles_total, a.total_warps, a.tiles_per_row,
                                 a.n_kv, a.batch, a.n_layers, a.n_q};
            fused_combine<D, G>(cv, row, lane);
        }
    };

    bool ok = true;
    int64_t it = 0;
    for (int64_t x = x0; x < x1; ++x, ++it) {
        const int stage = (int)(it % STAGES);
        const uint32_t parity = (uint32_t)((it / STAGES) & 1);
        const int64_t row = x / a.tiles_per_row;
        const int tok0 = (int)(x - row * a.tiles_per_row) * T;

        if (row != cur_row) {
            if (cur_row >= 0) flush(cur_row);
            cur_row = row;
            const int g = (int)(row % a.n_kv);
            const int64_t lb = row / a.n_kv;
            const int b = (int)(lb % a.batch), l = (int)(lb / a.batch);
            const uint16_t* qrow =
                a.q + (((size_t)b * a.n_layers + l) * a.n_q + (size_t)g * G) * D + hl * 8;
#pragma unroll
            for (int hs = 0; hs < G; ++hs) {
                const uint4 qw = *reinterpret_cast<const uint4*>(qrow + (size_t)(hs ^ h0) * D);
                float2 qf[4];
                unpack8(qw, qf);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    q2[hs][c] = make_float2(qf[c].x * a.q_scale, qf[c].y * a.q_scale);
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                m_run[h] = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c) o2[h][c] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int e = 0; e < NVF; ++e) l_part[e] = 0.f;
        }

        if (!mbar_wait(&bars[stage], parity)) {
            ok = false;
            break;
        }
        const unsigned char* Ks = wbuf + (size_t)stage * 2 * TB;
        const unsigned char* Vs = Ks + TB;
        const int nvalid = min(T, a.L - tok0);

        // ---- q.k for this lane's rows and slice of dims
        float acc[NV];
#pragma unroll
        for (int rp = 0; rp < RPL; ++rp) {
            const int j = rp ^ pmask_r;
            const uint4 kw =
                *reinterpret_cast<const uint4*>(Ks + ((j * RPW + hr) * D + hl * 8) * 2);
            float2 k2[4];
            unpack8(kw, k2);
#pragma unroll
            for (int hs = 0; hs < G; ++hs) {
                float2 t = ffma2(q2[hs][0], k2[0], make_float2(0.f, 0.f));
                t = ffma2(q2[hs][1], k2[1], t);
                t = ffma2(q2[hs][2], k2[2], t);
                t = ffma2(q2[hs][3], k2[3], t);
                acc[rp * G + hs] = t.x + t.y;
            }
        }
        // ---- reduce-scatter across the LPR lanes of a row group
#pragma unroll
        for (int s = 0; s < C::NSTEP; ++s) {
            const int half = (NV >> s) >> 1;
            const int m = LPR >> (s + 1);
#pragma unroll
            for (int i = 0; i < half; ++i) acc[i] += __shfl_xor_sync(kFull, acc[i + half], m);
        }
        // acc[e] (e < NVF) is now the full logit of tile row j_own*RPW+hr, head h0+e
        const int tok_own = pmask_r * RPW + hr;
        const bool own_valid = tok_own < nvalid;
        float xv[NVF];
#pragma unroll
        for (int e = 0; e < NVF; ++e) xv[e] = own_valid ? acc[e] : -INFINITY;
        if (a.write_logits && own_valid) {
            float* dst = a.logits + ((size_t)row * a.max_ctx + tok0 + tok_own) * G + h0;
            if constexpr (NVF == 2) {
                *reinterpret_cast<float2*>(dst) = make_float2(xv[0], xv[1]);
            } else {
#pragma unroll
                for (int e = 0; e < NVF; ++e) dst[e] = xv[e];
            }
        }
        // ---- online softmax: per-head tile max, rescale only when it grows
        float tmo[NVF], tmx[NVF];
#pragma unroll
        for (int e = 0; e < NVF; ++e) {
            float v = xv[e];
#pragma unroll
            for (int m = 2; m < 32; m <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
            tmo[e] = v;
            tmx[e] = __shfl_xor_sync(kFull, v, 1);
        }
        float m_new[G];
        bool grow = false;
#pragma unroll
        for (int e = 0; e < NVF; ++e) {
            m_new[e] = fmaxf(m_run[e], odd ? tmx[e] : tmo[e]);
            m_new[NVF + e] = fmaxf(m_run[NVF + e], odd ? tmo[e] : tmx[e]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) grow |= m_new[h] > m_run[h];
        if (grow) {
            float f[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                f[h] = fast_exp2(m_run[h] - m_new[h]);
                m_run[h] = m_new[h];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    o2[h][c].x *= f[h];
                    o2[h][c].y *= f[h];
                }
            }
#pragma unroll
            for (int e = 0; e < NVF; ++e) l_part[e] *= odd ? f[NVF + e] : f[e];
        }
        float p[NVF];
#pragma unroll
        for (int e = 0; e < NVF; ++e) {
            const float mh = odd ? m_run[NVF + e] : m_run[e];
            p[e] = fast_exp2(xv[e] - mh);
            l_part[e] += p[e];
        }
        // ---- p.v: every lane needs p for its rows and all G heads
#pragma unroll
        for (int j = 0; j < RPL; ++j) {
            const uint4 vw =
                *reinterpret_cast<const uint4*>(Vs + ((j * RPW + hr) * D + hl * 8) * 2);
            float2 v2[4];
            unpack8(vw, v2);
            if (nvalid < T && j * RPW + hr >= nvalid) {
#pragma unroll
                for (int c = 0; c < 4; ++c) v2[c] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const int vi = j * G + h;
                const float pp = __shfl_sync(kFull, p[vi & (NVF - 1)], hr * LPR + (vi >> C::LOG_NVF));
                const float2 pp2 = make_float2(pp, pp);
#pragma unroll
                for (int c = 0; c < 4; ++c) o2[h][c] = ffma2(pp2, v2[c], o2[h][c]);
            }
        }
        __syncwarp();
        if (lane == 0 && x + STAGES < x1) {
            fence_proxy_async();
            issue(x + STAGES, stage);
        }
    }
    if (!ok) {
        if (lane == 0) atomicOr(a.status, kStatusTimeout);
        // let the copies already issued land before the block exits
        for (int s = 0; s < STAGES; ++s) {
            const int64_t it2 = it + s;
            if (x0 + it2 < x1) mbar_wait(&bars[it2 % STAGES], (uint32_t)((it2 / STAGES) & 1));
        }
        return;
    }
    flush(cur_row);
}

template <int D, int G>
__global__ void __launch_bounds__(D) combine_kernel(const CombineArgs a) {
    griddep_wait();
    griddep_release();
    const int row = blockIdx.x, hh = blockIdx.y, d = threadIdx.x;
    const int64_t N = a.n_tiles_total;
    const int64_t W = a.total_warps;
    const int64_t first = (int64_t)row * a.tiles_per_row;
    const int64_t last = first + a.tiles_per_row - 1;
    // warp owning tile x: the largest w with floor(w*N/W) <= x
    const int w_lo = (int)(((first + 1) * W - 1) / N);
    const int w_hi = (int)(((last + 1) * W - 1) / N);
    float M = -INFINITY;
    for (int w = w_lo; w <= w_hi; ++w) {
        if ((int64_t)w * N / W == (int64_t)(w + 1) * N / W) continue;  // empty warp
        M = fmaxf(M, a.part_ml[(((int64_t)w + row) * G + hh) * 2]);
    }
    float lsum = 0.f, acc = 0.f;
    for (int w = w_lo; w <= w_hi; ++w) {
        if ((int64_t)w * N / W == (int64_t)(w + 1) * N / W) continue;
        const int64_t slot = (int64_t)w + row;
        const float f = fast_exp2(a.part_ml[(slot * G + hh) * 2] - M);
        lsum += a.part_ml[(slot * G + hh) * 2 + 1] * f;
        acc += a.part_o[(slot * G + hh) * D + d] * f;
    }
    const int g = row % a.n_kv;
    const int lb = row / a.n_kv;
    const int b = lb % a.batch, l = lb / a.batch;
    const int h = g * G + hh;
    a.out[(((size_t)b * a.n_layers + l) * a.n_q + h) * D + d] = acc / lsum;
    if (d == 0) a.lse2[(size_t)row * G + hh] = M + log2f(lsum);
}

constexpr int kStages = 2;
constexpr int kWarps = 4;

template <int D, int G>
cudaError_t launch_attn_t(const AttnArgs& a, int grid, cudaStream_t s) {
    using C = AttnCfg<D, G, kStages, kWarps>;
    auto kern = attn_splitk_kernel<D, G, kStages, kWarps>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kWarps * 32), C::SMEM, s, a);
}

template <int D, int G>
int ctas_per_sm_t() {
    using C = AttnCfg<D, G, kStages, kWarps>;
    auto kern = attn_splitk_kernel<D, G, kStages, kWarps>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kWarps * 32, C::SMEM) !=
        cudaSuccess)
        return 0;
    return n;
}

}  // namespace

int attn_warps_per_cta() { return kWarps; }

int attn_ctas_per_sm(int head_dim, int group) {
    if (group != 4) return 0;
    if (head_dim == 128) return ctas_per_sm_t<128, 4>();
    if (head_dim == 64) return ctas_per_sm_t<64, 4>();
    return 0;
}

size_t attn_smem_bytes(int head_dim, int group) {
    if (group != 4) return 0;
    if (head_dim == 128) return AttnCfg<128, 4, kStages, kWarps>::SMEM;
    if (head_dim == 64) return AttnCfg<64, 4, kStages, kWarps>::SMEM;
    return 0;
}

cudaError_t launch_attention(const AttnArgs& a, int head_dim, int group, int grid,
                             cudaStream_t s) {
    if (group == 4 && head_dim == 128) return launch_attn_t<128, 4>(a, grid, s);
    if (group == 4 && head_dim == 64) return launch_attn_t<64, 4>(a, grid, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_combine(const CombineArgs& a, int head_dim, int group, cudaStream_t s) {
    const dim3 grid(a.n_layers * a.batch * a.n_kv, group);
    if (group == 4 && head_dim == 128) return launch_pdl(combine_kernel<128, 4>, grid, dim3(128), 0, s, a);
    if (group == 4 && head_dim == 64) return launch_pdl(combine_kernel<64, 4>, grid, dim3(64), 0, s, a);
    return cudaErrorInvalidValue;
}

}  // namespace kvev
