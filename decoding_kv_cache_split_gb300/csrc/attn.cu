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
//  * Every warp owns an equal contiguous range of 16-token tiles of the
//    concatenated rows (no tail imbalance at any length) and streams them
//    through its own ring of stages in shared memory with 2-D TMA
//    (cp.async.bulk.tensor, boxes of 16 tokens x 64 dims, 128-byte swizzle,
//    completion on an mbarrier, L2 evict-first).  No block-level barrier
//    exists in the main loop.
//  * The op is a GEMV over bf16 K/V (4 flop per byte at GQA group 4), so the
//    goal is HBM bandwidth.  A first version on the FP32 pipes (packed
//    fma.rn.f32x2 and a shuffle reduce-scatter) was issue-bound at 6.1 TB/s
//    while a pure TMA stream of the same tiles reaches 7.4 TB/s; here the
//    two contractions of a tile run on mma.sync m16n8k16 (bf16 in, fp32
//    accumulate), which removes most of the per-token instructions.
//  * Softmax partials (running max, sum, output) of each warp's piece of a
//    row go to a slot, and the combine kernel below merges a row's slots on
//    every step into the output and the per-head log2-sum-exp the scoring
//    kernel needs.  Merging inside this kernel (last warp of a row) stalled
//    that warp's TMA pipeline and cost ~3% of the kernel.
//  * A warp whose bounded wait gives up flags the status word and writes
//    NaN as the running max of every slot it owns, so the combine turns the
//    rows it touched into NaN instead of merging stale partials.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <type_traits>

#include "kvev_internal.h"
#include "mma_ops.h"
#include "score_refresh.cuh"

namespace kvev {
namespace {

constexpr unsigned kFull = 0xffffffffu;

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
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_test(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}


// ---------------------------------------------------------------------------
// The two contractions of a 16-token tile on mma.sync m16n8k16 (bf16 in,
// fp32 accumulate):
//   S = Q K^T : A = Q (query heads of the group in rows 0..G-1, zero rows
//               above), B = the K tile; 2 token blocks x D/16 k-steps.
//   O += P V  : A = P from the S accumulators (the fragment layouts line up),
//               split into bf16 hi + lo so P keeps ~16 mantissa bits;
//               B = the V tile through ldmatrix.trans.
// K/V tiles arrive by 2-D TMA in boxes of 16 tokens x 64 dims with the
// 128-byte swizzle, so every ldmatrix is conflict-free.  Each thread owns
// one head g = lane/4 of the group (rows g >= G are padding), so the online
// softmax needs only 4-lane shuffles and no head selects.
template <int D, int G, int STAGES, int WARPS>
struct MmaCfg {
    static constexpr int T = kTile;                 // tokens per tile
    static constexpr int BOXES = D / 64;            // 64-dim (128-byte) boxes per tile
    static constexpr int BOX_BYTES = T * 128;       // one box: 16 rows x 128 B
    static constexpr int TILE_BYTES = BOXES * BOX_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K and V
    static constexpr int NB = D / 8;                // 8-dim output blocks
    static constexpr int KS = D / 16;               // k-steps of the QK contraction
    static constexpr size_t SMEM = 1024 + (size_t)WARPS * STAGES * STAGE_BYTES +
                                   (size_t)WARPS * STAGES * (sizeof(uint64_t) + 2 * sizeof(int));
    static_assert(G <= 8 && (D == 64 || D == 128), "mma tile shape");
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// shared-memory byte address of 16-byte chunk c (0 .. D/8-1) of tile row r
template <int D>
__device__ __forceinline__ uint32_t tile_chunk(uint32_t tile, int r, int c) {
    return tile + (c >> 3) * (kTile * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One warp's share of an attention launch (the kernel below, and the first
// phase of the fused step).  `smem` is the CTA's 1024-byte aligned dynamic
// shared memory.  Returns false when a bounded wait gave up (the status word
// is flagged and the warp's split slots poisoned).
template <int D, int G, int STAGES, int WARPS, bool PAGED, int ST>
__device__ __forceinline__ bool attn_warp(const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                          const AttnArgs& a, unsigned char* smem) {
    using C = MmaCfg<D, G, STAGES, WARPS>;
    constexpr int T = C::T, NB = C::NB, KS = C::KS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* wbuf = smem + (size_t)warp * STAGES * C::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)WARPS * STAGES * C::STAGE_BYTES) +
                     warp * STAGES;
    // valid tokens of the tile in each stage (written by lane 0 at issue)
    int* stage_nv = reinterpret_cast<int*>(reinterpret_cast<uint64_t*>(
                        smem + (size_t)WARPS * STAGES * C::STAGE_BYTES) + WARPS * STAGES) +
                    warp * STAGES;
    int* stage_pos = stage_nv + WARPS * STAGES;   // first token position of the tile (block mode)

    const int w = blockIdx.x * WARPS + warp;
    if (w >= a.total_warps) return true;   // the launch's last CTA may hold spare warps
    const int64_t N = a.n_tiles_total;
    const int64_t x0 = (int64_t)w * N / a.total_warps;
    const int64_t x1 = (int64_t)(w + 1) * N / a.total_warps;
    if (x0 >= x1) return true;

    if (lane == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t pol = evict_first_policy();
    const uint32_t wait_limit = a.wait_limit ? a.wait_limit : kWaitLimit;

    // tiles are walked with (row, tile-in-row) counters: no divisions in the loop
    const int tpr = a.tiles_per_row;
    // Block mode: the warp keeps 32 consecutive block-table entries of the row
    // it is issuing for (lane k holds tile tb_base + k), refreshed together when
    // the issue moves past them, so issuing a tile needs no dependent loads.
    int64_t tb_row = -1;
    int tb_base = 0, tb_y = 0, tb_nv = 0, tb_pos = 0;
    auto table_for = [&](int64_t row, int tile) {   // every lane of the warp
        if constexpr (PAGED) {
            if (row == tb_row && tile >= tb_base && tile < tb_base + 32) return;
            const int64_t arow = a.row0 + row;
            const int gk = (int)(arow % a.n_kv);
            const int64_t lb = arow / a.n_kv;
            const int b = (int)(lb % a.batch), l = (int)(lb / a.batch);
            const int tk = tile + lane;
            tb_y = 0;
            tb_nv = 0;
            tb_pos = tk * T;
            if (tk < a.n_blocks[b] && tk < a.tiles_per_row) {
                const int page = a.block_table[(size_t)b * a.pps + tk];
                tb_nv = a.blk_len[(size_t)b * a.pps + tk];
                tb_y = (int)((((int64_t)page * a.n_layers + l) * a.n_kv + gk) * T);
                if (a.blk_pos) tb_pos = a.blk_pos[(size_t)b * a.pps + tk];
            }
            tb_row = row;
            tb_base = tile;
        }
    };
    auto issue = [&](int64_t row, int tile, int stage) {   // every lane; lane 0 issues
        if constexpr (!PAGED) {
            if (lane != 0) return;
        }
        int y = 0, nv;
        if constexpr (PAGED) {
            table_for(row, tile);
            y = __shfl_sync(kFull, tb_y, tile - tb_base);
            nv = __shfl_sync(kFull, tb_nv, tile - tb_base);
            const int pos = __shfl_sync(kFull, tb_pos, tile - tb_base);
            if (lane == 0) stage_pos[stage] = pos;
        } else {
            y = (int)((a.row0 + row) * a.max_ctx + tile * T);
            nv = min(T, a.L - tile * T);
        }
        if (lane != 0) return;
        stage_nv[stage] = nv;
        if (nv == 0) {   // empty tile: complete the phase with no data
            mbar_arrive(&bars[stage]);
            return;
        }
        unsigned char* dst = wbuf + (size_t)stage * C::STAGE_BYTES;
        mbar_expect_tx(&bars[stage], C::STAGE_BYTES);
        // test-only: the tile's copies are never issued, so its wait runs out
        if (row * tpr + tile + 1 == a.fault_tile_p1) return;
#pragma unroll
        for (int bx = 0; bx < C::BOXES; ++bx) {
            tma_load_2d(dst + bx * C::BOX_BYTES, tmap_k, bx * 64, y, &bars[stage], pol);
            tma_load_2d(dst + C::TILE_BYTES + bx * C::BOX_BYTES, tmap_v, bx * 64, y,
                        &bars[stage], pol);
        }
    };
    int64_t prow = x0 / tpr;          // next tile to issue
    int ptile = (int)(x0 - prow * tpr);
    const int64_t n_issue0 = x1 - x0 < STAGES ? x1 - x0 : STAGES;
    for (int s = 0; s < n_issue0; ++s) {
        issue(prow, ptile, s);
        if (++ptile == tpr) { ptile = 0; ++prow; }
    }
    int64_t crow = x0 / tpr;          // tile being consumed
    int ctile = (int)(x0 - crow * tpr);

    const int g = lane >> 2, t = lane & 3;   // fragment row (query head) and column pair
    const bool real = g < G;
    uint32_t qa0[KS], qa2[KS];               // Q as the A operand, per k-step
    float o[NB][2];                          // O[g][8j + 2t .. 2t+1]
    float m_run = -INFINITY, l_run = 0.f;
    float e_run = 0.f;    // ST & kStatEntropy: sum of exp2(x - m_run) * x, this thread's tokens
    float vn_run = 0.f;   // ST & kStatVNorm: sum of the value norms of this lane's tokens
    int64_t cur_row = -1;

    auto flush = [&](int64_t row) {
        float l = l_run;
        l += __shfl_xor_sync(kFull, l, 1);
        l += __shfl_xor_sync(kFull, l, 2);
        const int64_t slot = (int64_t)w + row;
        if constexpr ((ST & kStatEntropy) != 0) {
            float e = e_run;
            e += __shfl_xor_sync(kFull, e, 1);
            e += __shfl_xor_sync(kFull, e, 2);
            if (real && t == 0) a.part_e[(size_t)slot * G + g] = e;
        }
        if constexpr ((ST & kStatVNorm) != 0) {
            float v = vn_run;
#pragma unroll
            for (int k = 16; k > 0; k >>= 1) v += __shfl_xor_sync(kFull, v, k);
            if (lane == 0) a.part_vn[slot] = v;
        }
        if (real) {
            float* po = a.part_o + ((size_t)slot * G + g) * D;
#pragma unroll
            for (int j = 0; j < NB; ++j)
                *reinterpret_cast<float2*>(po + 8 * j + 2 * t) = make_float2(o[j][0], o[j][1]);
            if (t == 0) {
                float* pml = a.part_ml + ((size_t)slot * G + g) * 2;
                pml[0] = m_run;
                pml[1] = l;
            }
        }
    };

    bool ok = true;
    int64_t it = 0;
    int stage = 0;
    uint32_t parity = 0;
    for (int64_t x = x0; x < x1; ++x, ++it) {
        const int64_t row = crow;
        const int tok0 = ctile * T;
        if (++ctile == tpr) { ctile = 0; ++crow; }

        if (row != cur_row) {
            if (cur_row >= 0) flush(cur_row);
            cur_row = row;
            const int gk = (int)((a.row0 + row) % a.n_kv);
            const int64_t lb = (a.row0 + row) / a.n_kv;
            const int b = (int)(lb % a.batch), l = (int)(lb / a.batch);
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                a.q + (((size_t)b * a.n_layers + l) * a.n_q + (size_t)gk * G + (real ? g : 0)) * D);
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                qa0[s] = real ? qrow[8 * s + t] : 0u;       // dims 16s + 2t, +1
                qa2[s] = real ? qrow[8 * s + 4 + t] : 0u;   // dims 16s + 8 + 2t, +1
            }
#pragma unroll
            for (int j = 0; j < NB; ++j) o[j][0] = o[j][1] = 0.f;
            m_run = -INFINITY;
            l_run = 0.f;
            e_run = 0.f;
            vn_run = 0.f;
        }

        if (!mbar_wait(&bars[stage], parity, wait_limit)) {
            ok = false;
            break;
        }
        const uint32_t ktile = smem_addr(wbuf + (size_t)stage * C::STAGE_BYTES);
        const uint32_t vtile = ktile + C::TILE_BYTES;
        const int nvalid = PAGED ? stage_nv[stage] : min(T, a.L - tok0);
        const int pos0 = PAGED ? stage_pos[stage] : tok0;   // position of the tile's first token
        if (PAGED && nvalid == 0) {   // past the sequence's live blocks: nothing to do
            __syncwarp();
            if (x + STAGES < x1) {
                issue(prow, ptile, stage);
                if (++ptile == tpr) { ptile = 0; ++prow; }
            }
            if (++stage == STAGES) { stage = 0; parity ^= 1u; }
            continue;
        }

        // ---- S = Q K^T for the two 8-token blocks (even and odd k-steps in
        //      separate accumulators: four independent MMA chains)
        float sc[2][2];
        {
            float acc[2][2][2] = {};
#pragma unroll
            for (int s = 0; s < KS; s += 2) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    uint32_t kb[4];   // b0, b1 of k-steps s and s+1
                    ldsm_x4(tile_chunk<D>(ktile, 8 * i + (lane & 7), 2 * s + (lane >> 3)), kb);
                    mma_rows8(acc[i][0][0], acc[i][0][1], qa0[s], qa2[s], kb[0], kb[1]);
                    mma_rows8(acc[i][1][0], acc[i][1][1], qa0[s + 1], qa2[s + 1], kb[2], kb[3]);
                }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                sc[i][0] = (acc[i][0][0] + acc[i][1][0]) * a.q_scale;
                sc[i][1] = (acc[i][0][1] + acc[i][1][1]) * a.q_scale;
            }
        }
        // tokens of this thread's four logits: 8i + 2t + e
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                if (!real || 8 * i + 2 * t + e >= nvalid) sc[i][e] = -INFINITY;
        if (a.write_logits && real) {
            float* lg = a.logits + ((size_t)(a.row0 + row) * a.logit_ld + pos0) * G + g;
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tok = 8 * i + 2 * t + e;
                    if (tok < nvalid) lg[tok * G] = sc[i][e];
                }
        }
        // ---- online softmax for head g
        float mt = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
        if (real && mt > m_run) {
            const float f = fast_exp2(m_run - mt);
            m_run = mt;
            l_run *= f;
            if constexpr ((ST & kStatEntropy) != 0) e_run *= f;
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                o[j][0] *= f;
                o[j][1] *= f;
            }
        }
        float p[2][2];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                p[i][e] = real ? fast_exp2(sc[i][e] - m_run) : 0.f;
                l_run += p[i][e];
                if constexpr ((ST & kStatEntropy) != 0)   // -inf logits (no token) add 0
                    e_run = fmaf(p[i][e], p[i][e] > 0.f ? sc[i][e] : 0.f, e_run);
            }
        if (PAGED && a.tile_stats && pos0 >= a.stats_base) {   // (running max, tile sum) per head
            float ts = (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
            ts += __shfl_xor_sync(kFull, ts, 1);
            ts += __shfl_xor_sync(kFull, ts, 2);
            if (real && t == 0)
                a.tile_stats[((size_t)(a.row0 + row) * a.stats_tiles +
                              (pos0 - a.stats_base) / T) * G + g] = make_float2(m_run, ts);
        }
        const uint32_t ph0 = pack_bf16x2(p[0][0], p[0][1]);   // tokens 2t, 2t+1
        const uint32_t ph2 = pack_bf16x2(p[1][0], p[1][1]);   // tokens 8+2t, 8+2t+1
        const uint32_t pl0 = pack_bf16x2(p[0][0] - bf16_lo(ph0), p[0][1] - bf16_hi(ph0));
        const uint32_t pl2 = pack_bf16x2(p[1][0] - bf16_lo(ph2), p[1][1] - bf16_hi(ph2));

        // rows past the end of the cache may hold anything: zero them in V
        if (nvalid < T) {
            unsigned char* vt = wbuf + (size_t)stage * C::STAGE_BYTES + C::TILE_BYTES;
            for (int u = lane; u < (T - nvalid) * (D / 8); u += 32) {
                const int r = nvalid + u / (D / 8), c = u % (D / 8);
                *reinterpret_cast<uint4*>(vt + (tile_chunk<D>(0, r, c))) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();   // ordered before the next TMA write to this stage
            __syncwarp();
        }
        if constexpr ((ST & kStatVNorm) != 0) {   // l2 norm of each token's value row
            constexpr int CPL = D / 16;            // 16-byte chunks per lane: two lanes a row
            const int r = lane & 15, hf = lane >> 4;
            float ss = 0.f;
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
                uint32_t u0, u1, u2, u3;
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(u0), "=r"(u1), "=r"(u2), "=r"(u3)
                             : "r"(tile_chunk<D>(vtile, r, hf * CPL + k)));
                const uint32_t uu[4] = {u0, u1, u2, u3};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float x0 = bf16_lo(uu[j]), x1 = bf16_hi(uu[j]);
                    ss = fmaf(x0, x0, ss);
                    ss = fmaf(x1, x1, ss);
                }
            }
            ss += __shfl_xor_sync(kFull, ss, 16);
            if (lane < 16 && r < nvalid) {
                const float nrm = sqrtf(ss);
                a.vnorm[(size_t)(a.row0 + row) * a.logit_ld + pos0 + r] = nrm;
                vn_run += nrm;
            }
        }
        // ---- O += P V, two 8-dim blocks per ldmatrix.x4.trans
#pragma unroll
        for (int jj = 0; jj < NB / 2; ++jj) {
            uint32_t vb[4];   // b0, b1 of dim blocks 2jj and 2jj+1
            const int mi = lane >> 3;
            ldsm_x4_t(tile_chunk<D>(vtile, (mi & 1) * 8 + (lane & 7), 2 * jj + (mi >> 1)), vb);
            mma_rows8(o[2 * jj][0], o[2 * jj][1], ph0, ph2, vb[0], vb[1]);
            mma_rows8(o[2 * jj][0], o[2 * jj][1], pl0, pl2, vb[0], vb[1]);
            mma_rows8(o[2 * jj + 1][0], o[2 * jj + 1][1], ph0, ph2, vb[2], vb[3]);
            mma_rows8(o[2 * jj + 1][0], o[2 * jj + 1][1], pl0, pl2, vb[2], vb[3]);
        }
        // Every ldmatrix of this stage fed an MMA issued above, so its read is
        // complete once the warp passes this point; only the zeroing stores of
        // a partial tile needed a proxy fence (done there).
        __syncwarp();
        if (x + STAGES < x1) {
            issue(prow, ptile, stage);
            if (++ptile == tpr) { ptile = 0; ++prow; }
        }
        if (++stage == STAGES) { stage = 0; parity ^= 1u; }
    }
    if (!ok) {
        if (lane == 0) atomicOr(a.status, kStatusTimeout);
        // poison every slot this warp owns: a NaN running max makes the
        // combine's merge of the row NaN (the slots may hold an earlier
        // launch's partials)
        for (int64_t r = x0 / tpr + (lane >> 2); r <= (x1 - 1) / tpr; r += 8)
            if ((lane & 3) < G)
                a.part_ml[((size_t)((int64_t)w + r) * G + (lane & 3)) * 2] = __int_as_float(0x7fc00000);
        if (G > 4)
            for (int64_t r = x0 / tpr + (lane >> 2); r <= (x1 - 1) / tpr; r += 8)
                if (4 + (lane & 3) < G)
                    a.part_ml[((size_t)((int64_t)w + r) * G + 4 + (lane & 3)) * 2] =
                        __int_as_float(0x7fc00000);
        // let the copies already issued land before the block exits (always
        // the full cap: a shortened test limit must not cut this wait; the
        // injected tile issued none)
        for (int s = 0; s < STAGES; ++s) {
            const int64_t it2 = it + s;
            if (x0 + it2 < x1 && x0 + it2 + 1 != a.fault_tile_p1)
                mbar_wait(&bars[it2 % STAGES], (uint32_t)((it2 / STAGES) & 1), kWaitLimit);
        }
        return false;
    }
    flush(cur_row);
    return true;
}

#ifndef KVEV_ATTN_MIN_CTAS
#define KVEV_ATTN_MIN_CTAS 1
#endif
template <int D, int G, int STAGES, int WARPS, bool PAGED, int ST>
__global__ void __launch_bounds__(WARPS * 32, KVEV_ATTN_MIN_CTAS)
    attn_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const AttnArgs a) {
    extern __shared__ unsigned char smem_raw[];
    griddep_wait();
    griddep_release();
    // 128-byte swizzled boxes want 1024-byte aligned destinations
    unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    attn_warp<D, G, STAGES, WARPS, PAGED, ST>(&tmap_k, &tmap_v, a, smem);
}

// Split combine: one warp per row of the launch (up to 8 rows per CTA); lane l
// owns output dims [V l, V l + V) of every head (V = D / 32, one vector
// load per head and segment).  The row's segments are merged with a running
// max, one at a time with the next one prefetched (KB = 1, rows split over
// few warps) or in batches of KB loaded before any merge (rows split over
// many warps).
constexpr int kCombineWarps = 8;

// Merge launch row r (one warp, lane = this thread's lane).
template <int D, int G, int KB>
__device__ __forceinline__ void combine_row(const CombineArgs& a, int64_t r, int lane) {
    constexpr int V = D / 32;   // dims per lane
    static_assert(V == 2 || V == 4, "head_dim 64 or 128");
    using VecT = typename std::conditional<V == 4, float4, float2>::type;
    float M[G], Ls[G], acc[G][V];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        M[h] = -INFINITY;
        Ls[h] = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) acc[h][v] = 0.f;
    }
    auto as_array = [](const VecT& x, float (&o)[V]) {
        const float* p = reinterpret_cast<const float*>(&x);
#pragma unroll
        for (int v = 0; v < V; ++v) o[v] = p[v];
    };
    for (int set = 0; set < 1 + a.has2; ++set) {
        const SplitPartials& sp = set ? a.sp2 : a.sp;
        int64_t lo, hi;
        split_warps_of_row(sp, r, &lo, &hi);
        // segment w of the row: (m, l) of every head and this lane's dims of o
        auto load = [&](int64_t w, float (&m)[G], float (&l)[G], VecT (&o)[G]) {
            const bool ok = w <= hi && split_warp_has_tiles(w, sp.n_tiles, sp.total_warps);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float* ml = sp.part_ml + ((w + r) * G + h) * 2;
                m[h] = ok ? __ldcg(ml) : -INFINITY;
                l[h] = ok ? __ldcg(ml + 1) : 0.f;
                o[h] = ok ? __ldcg(reinterpret_cast<const VecT*>(sp.part_o + ((w + r) * G + h) * D) + lane)
                          : VecT{};
            }
        };
        auto merge = [&](const float (&m)[G], const float (&l)[G], const VecT (&o)[G]) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                if (m[h] == -INFINITY) continue;
                const float mx = fmaxf(M[h], m[h]);
                const float fo = fast_exp2(M[h] - mx), fj = fast_exp2(m[h] - mx);
                float ov[V];
                as_array(o[h], ov);
                Ls[h] = Ls[h] * fo + l[h] * fj;
#pragma unroll
                for (int v = 0; v < V; ++v) acc[h][v] = acc[h][v] * fo + ov[v] * fj;
                M[h] = mx;
            }
        };
        if (KB == 1) {   // few segments per row: one at a time, the next one prefetched
            float mc[G], lc[G];
            VecT oc[G];
            load(lo, mc, lc, oc);
            for (int64_t w = lo; w <= hi; ++w) {
                float mn[G], ln[G];
                VecT on[G];
                if (w + 1 <= hi) load(w + 1, mn, ln, on);
                merge(mc, lc, oc);
                if (w + 1 <= hi) {
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        mc[h] = mn[h];
                        lc[h] = ln[h];
                        oc[h] = on[h];
                    }
                }
            }
        } else {         // many segments per row: batches of KB, all loads first
            for (int64_t w0 = lo; w0 <= hi; w0 += KB) {
                float m[KB][G], l[KB][G];
                VecT o[KB][G];
#pragma unroll
                for (int j = 0; j < KB; ++j) load(w0 + j, m[j], l[j], o[j]);
#pragma unroll
                for (int j = 0; j < KB; ++j) merge(m[j], l[j], o[j]);
            }
        }
    }
    const int64_t arow = a.sp.row0 + r;
    const int g = (int)(arow % a.n_kv);
    const int64_t lb = arow / a.n_kv;
    const int b = (int)(lb % a.batch), l = (int)(lb / a.batch);
    if ((a.part_e || a.part_vn) && lane == 0) {
        // weighting statistics: each head's sum of p * x over the row (its
        // segments rescaled to the merged max, like the softmax sums) and the
        // row's sum of value norms, in segment order
        int64_t lo, hi;
        split_warps_of_row(a.sp, r, &lo, &hi);
        float E[G], VS = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h) E[h] = 0.f;
        for (int64_t w = lo; w <= hi; ++w) {
            if (!split_warp_has_tiles(w, a.sp.n_tiles, a.sp.total_warps)) continue;
            if (a.part_e) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float m = __ldcg(a.sp.part_ml + ((w + r) * G + h) * 2);
                    if (m != -INFINITY)
                        E[h] += __ldcg(a.part_e + (w + r) * G + h) * fast_exp2(m - M[h]);
                }
            }
            if (a.part_vn) VS += __ldcg(a.part_vn + w + r);
        }
        const float n_tok = (float)a.n_tokens;
        if (a.ent) {   // entropy in bits = log2-sum-exp - E[p x]; over log2(tokens)
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float hb = M[h] + log2f(Ls[h]) - E[h] / Ls[h];
                a.ent[arow * G + h] = a.n_tokens > 1 ? hb / log2f(n_tok) : 1.0f;
            }
        }
        if (a.vmean) a.vmean[arow] = VS / n_tok;
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const float inv = 1.0f / Ls[h];
        VecT res;
        float* rp = reinterpret_cast<float*>(&res);
#pragma unroll
        for (int v = 0; v < V; ++v) rp[v] = acc[h][v] * inv;
        const size_t o0 = (((size_t)b * a.n_layers + l) * a.n_q + (size_t)g * G + h) * D;
        if (a.out_bf16) {   // the same fp32 values rounded to bf16
            uint32_t pk[V / 2];
#pragma unroll
            for (int v = 0; v < V / 2; ++v) pk[v] = pack_bf16x2(rp[2 * v], rp[2 * v + 1]);
            uint16_t* ob = static_cast<uint16_t*>(a.out) + o0 + (size_t)lane * V;
            if constexpr (V == 4)
                *reinterpret_cast<uint2*>(ob) = make_uint2(pk[0], pk[1]);
            else
                *reinterpret_cast<uint32_t*>(ob) = pk[0];
        } else {
            reinterpret_cast<VecT*>(static_cast<float*>(a.out) + o0)[lane] = res;
        }
        if (lane == 0) a.lse2[arow * G + h] = M[h] + log2f(Ls[h]);
    }
}

template <int D, int G, int KB>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineArgs a) {
    griddep_wait();
    griddep_release();
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);   // row of the launch
    if (r >= a.n_rows) return;
    combine_row<D, G, KB>(a, r, lane);
}


#ifndef KVEV_ATTN_STAGES
#define KVEV_ATTN_STAGES 2
#endif
#ifndef KVEV_ATTN_WARPS
#define KVEV_ATTN_WARPS 4
#endif
constexpr int kStages = KVEV_ATTN_STAGES;   // tiles in flight per warp
constexpr int kWarps = KVEV_ATTN_WARPS;     // warps per CTA

// ---------------------------------------------------------------------------
// The fused refresh step: one cooperative launch of the attention grid does
// the attention (phase A), then, behind a grid barrier, the split combine of
// every row (phase B: one warp per row), then, behind a second barrier, the
// scoring of every token block (phase C: the scorer's 128-thread body per
// 32 tokens, in the CTA's shared memory that the attention stages no longer
// use).  The work and its arithmetic are those of the three kernels it
// replaces, in the same order, so the results are the same bit for bit when
// the attention is split the same way; what goes is two kernel boundaries
// (their drain and launch) per step.
//
// Grid barrier: a count and a generation word in global memory.  Thread 0 of
// each CTA publishes its CTA's writes (fence), reads the generation and
// arrives; the last arrival zeroes the count and bumps the generation, the
// others spin on it with a bounded number of iterations (then they flag the
// status word and their CTA leaves).  The cooperative launch guarantees every
// CTA is resident, so the wait ends; the count is back to zero after every
// barrier, so the next barrier (and the next launch, graph replays included)
// starts from a clean state.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ bool grid_barrier(const FusedArgs& f, uint32_t* status) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        bool ok = true;
        const uint32_t gen = ld_acquire_gpu(f.bar + 1);
        __threadfence();   // this CTA's writes before its arrival
        if (f.skip_cta_p1 == (int)blockIdx.x + 1) {
            ok = false;   // test-only: this CTA never arrives
        } else if (atomicAdd(f.bar, 1u) == gridDim.x - 1) {
            f.bar[0] = 0;                 // reset for the next barrier
            __threadfence();
            atomicAdd(f.bar + 1, 1u);     // release the others
        } else {
            const uint32_t limit = f.wait_limit ? f.wait_limit : kWaitLimit;
            uint32_t i = 0;
            while (ld_acquire_gpu(f.bar + 1) == gen) {
                if (++i >= limit) {
                    ok = false;
                    atomicOr(status, kStatusTimeout | kStatusBarrier);
                    break;
                }
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

template <int D, int G, int NKV>
__global__ void __launch_bounds__(kWarps * 32)
    attn_fused_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const AttnArgs a,
                      const CombineArgs cb, const ScoreArgs sc, const FusedArgs f) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    __shared__ float s_c[kScoreSegs][32], s_tot[kScoreSegs][32];
    // phase A: attention, logits kept, split partials
    attn_warp<D, G, kStages, kWarps, false, 0>(&tmap_k, &tmap_v, a, smem);
    if (!grid_barrier(f, a.status)) return;
    // phase B: merge every row's split (output, per-head log2-sum-exp)
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const bool many = 1.0 + (double)cb.sp.total_warps / (cb.n_rows > 0 ? cb.n_rows : 1) >= 3.0;
    for (int64_t r = gw; r < cb.n_rows; r += nw) {
        if (many)
            combine_row<D, G, (G <= 4 ? 4 : 2)>(cb, r, lane);
        else
            combine_row<D, G, 1>(cb, r, lane);
    }
    if (!f.score) {   // the scorer runs as its own launch after this one
        griddep_release();
        return;
    }
    if (!grid_barrier(f, a.status)) return;
    // phase C: score every token block (the stage buffers hold the tables)
    float* tab = reinterpret_cast<float*>(smem);
    const int nblk = (sc.L + 31) / 32;
    for (int b = 0; b < sc.batch; ++b) {
        __syncthreads();   // the previous tables and chain are done
        score_tables<G, NKV, false>(sc, b, tab);
        for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
            __syncthreads();
            score_block<G, NKV, false, kScoreSegs, kWarps>(sc, b, blk, tab, s_c, s_tot);
        }
    }
    griddep_release();
}


// 2-D view of one cache buffer: rows x max_ctx tokens of D bf16; boxes of
// 16 tokens x 64 dims with the 128-byte swizzle.
bool encode_cache_map(CUtensorMap* map, const void* base, int64_t n_tokens, int D) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)n_tokens};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kTile};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G, bool PAGED, int ST = 0>
cudaError_t launch_attn_t(const AttnArgs& a, int grid, cudaStream_t s) {
    using C = MmaCfg<D, G, kStages, kWarps>;
    auto kern = attn_mma_kernel<D, G, kStages, kWarps, PAGED, ST>;
    CUtensorMap mk, mv;
    if (!encode_cache_map(&mk, a.k, a.view_tokens, D) || !encode_cache_map(&mv, a.v, a.view_tokens, D))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kWarps * 32), C::SMEM, s, mk, mv, a);
}

template <int D, int G>
int ctas_per_sm_t() {
    using C = MmaCfg<D, G, kStages, kWarps>;
    auto kern = attn_mma_kernel<D, G, kStages, kWarps, false, 0>;
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

// Instantiated shapes: head_dim 64 / 128, query heads per KV head 4 / 8.
int attn_ctas_per_sm(int head_dim, int group) {
    if (head_dim == 128 && group == 4) return ctas_per_sm_t<128, 4>();
    if (head_dim == 64 && group == 4) return ctas_per_sm_t<64, 4>();
    if (head_dim == 128 && group == 8) return ctas_per_sm_t<128, 8>();
    if (head_dim == 64 && group == 8) return ctas_per_sm_t<64, 8>();
    return 0;
}

size_t attn_smem_bytes(int head_dim, int group) {
    if (group != 4 && group != 8) return 0;
    if (head_dim == 128) return MmaCfg<128, 4, kStages, kWarps>::SMEM;
    if (head_dim == 64) return MmaCfg<64, 4, kStages, kWarps>::SMEM;
    return 0;
}

// The token-mode kernel with the weighting statistics `stats` (kStat* bits).
template <int D, int G>
cudaError_t launch_attn_stats(const AttnArgs& a, int grid, int stats, cudaStream_t s) {
    switch (stats) {
        case kStatEntropy: return launch_attn_t<D, G, false, kStatEntropy>(a, grid, s);
        case kStatVNorm: return launch_attn_t<D, G, false, kStatVNorm>(a, grid, s);
        case kStatEntropy | kStatVNorm:
            return launch_attn_t<D, G, false, kStatEntropy | kStatVNorm>(a, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attention(const AttnArgs& a, int head_dim, int group, int grid,
                             cudaStream_t s, int stats) {
    const bool paged = a.block_table != nullptr;
    if (stats != 0) {
        if (paged) return cudaErrorInvalidValue;
        if (group == 4 && head_dim == 128) return launch_attn_stats<128, 4>(a, grid, stats, s);
        if (group == 4 && head_dim == 64) return launch_attn_stats<64, 4>(a, grid, stats, s);
        if (group == 8 && head_dim == 128) return launch_attn_stats<128, 8>(a, grid, stats, s);
        if (group == 8 && head_dim == 64) return launch_attn_stats<64, 8>(a, grid, stats, s);
        return cudaErrorInvalidValue;
    }
    if (group == 4 && head_dim == 128)
        return paged ? launch_attn_t<128, 4, true>(a, grid, s) : launch_attn_t<128, 4, false>(a, grid, s);
    if (group == 4 && head_dim == 64)
        return paged ? launch_attn_t<64, 4, true>(a, grid, s) : launch_attn_t<64, 4, false>(a, grid, s);
    if (group == 8 && head_dim == 128)
        return paged ? launch_attn_t<128, 8, true>(a, grid, s) : launch_attn_t<128, 8, false>(a, grid, s);
    if (group == 8 && head_dim == 64)
        return paged ? launch_attn_t<64, 8, true>(a, grid, s) : launch_attn_t<64, 8, false>(a, grid, s);
    return cudaErrorInvalidValue;
}

template <int D, int G>
cudaError_t launch_combine_t(const CombineArgs& a, cudaStream_t s) {
    // warps a row's tiles are split over, on average
    const double per_row = 1.0 + (double)a.sp.total_warps / (a.n_rows > 0 ? a.n_rows : 1);
    if (per_row < 3.0) {
        const dim3 grid((a.n_rows + kCombineWarps - 1) / kCombineWarps), block(kCombineWarps * 32);
        return launch_pdl(combine_kernel<D, G, 1>, grid, block, 0, s, a);
    }
    // few rows, many segments each: one warp per CTA to spread the rows over the SMs
    return launch_pdl(combine_kernel<D, G, (G <= 4 ? 4 : 2)>, dim3(a.n_rows), dim3(32), 0, s, a);
}

template <int D, int G, int NKV>
int fused_ctas_per_sm_t() {
    using C = MmaCfg<D, G, kStages, kWarps>;
    auto kern = attn_fused_kernel<D, G, NKV>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kWarps * 32, C::SMEM) !=
        cudaSuccess)
        return 0;
    return n;
}

template <int D, int G, int NKV>
cudaError_t launch_fused_t(const AttnArgs& a, const CombineArgs& cb, const ScoreArgs& sc,
                           const FusedArgs& f, int grid, cudaStream_t s) {
    using C = MmaCfg<D, G, kStages, kWarps>;
    auto kern = attn_fused_kernel<D, G, NKV>;
    // the scorer's tables live in the stage buffers once the attention is done
    if ((size_t)sc.n_layers * (sc.n_q + 1 + sc.n_kv) * sizeof(float) >
        (size_t)kWarps * kStages * C::STAGE_BYTES)
        return cudaErrorInvalidValue;
    CUtensorMap mk, mv;
    if (!encode_cache_map(&mk, a.k, a.view_tokens, D) || !encode_cache_map(&mv, a.v, a.view_tokens, D))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: the barriers end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mk, mv, a, cb, sc, f);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& a, int head_dim, int group, cudaStream_t s) {
    if (group == 4 && head_dim == 128) return launch_combine_t<128, 4>(a, s);
    if (group == 4 && head_dim == 64) return launch_combine_t<64, 4>(a, s);
    if (group == 8 && head_dim == 128) return launch_combine_t<128, 8>(a, s);
    if (group == 8 && head_dim == 64) return launch_combine_t<64, 8>(a, s);
    return cudaErrorInvalidValue;
}

// Shapes with a fused step: head_dim 128 and 64, 4 or 8 query heads per KV
// head, and the KV-head counts of the workloads (8, 2, 1).
#define KVEV_FUSED_SHAPES(X) \
    X(128, 4, 8) X(128, 4, 2) X(128, 4, 1) X(64, 4, 2) X(128, 8, 2) X(64, 8, 2)

int attn_fused_ctas_per_sm(int head_dim, int group, int n_kv) {
#define KVEV_FUSED_OCC(D, G, N) \
    if (head_dim == D && group == G && n_kv == N) return fused_ctas_per_sm_t<D, G, N>();
    KVEV_FUSED_SHAPES(KVEV_FUSED_OCC)
#undef KVEV_FUSED_OCC
    return 0;
}

cudaError_t launch_attn_fused(const AttnArgs& a, const CombineArgs& cb, const ScoreArgs& sc,
                              const FusedArgs& f, int head_dim, int group, int grid,
                              cudaStream_t s) {
#define KVEV_FUSED_LAUNCH(D, G, N) \
    if (head_dim == D && group == G && sc.n_kv == N) return launch_fused_t<D, G, N>(a, cb, sc, f, grid, s);
    KVEV_FUSED_SHAPES(KVEV_FUSED_LAUNCH)
#undef KVEV_FUSED_LAUNCH
    return cudaErrorInvalidValue;
}

}  // namespace kvev
