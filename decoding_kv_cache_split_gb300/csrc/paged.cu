// Block-granular (paged) eviction with score persistence.
//
// The LRFU policy per (sequence, token block) of the kv-cache-docs figure
// "ema-eviction": a block's new score per layer is the max over its tokens
// of the head-summed attention probability, folded into the block's EMA in
// ascending layer order ("What Matters for Aggressive Decoding-Time KV
// Eviction?" Appendix E "Layer scoring"); priority (1 - score)(1 - exp(-beta
// age)); the budget counts blocks.  When a block is evicted its score is
// kept under (sequence, logical block) and restored when the block is
// re-admitted ("when block B is evicted its identity key and score persist
// and are restored on re-admission rather than reset").
//
// K/V never move: a sequence owns a fixed range of pages of the pool, its
// live blocks are a block table in slot order, eviction pushes the freed
// pages on the sequence's free stack and new blocks pop from it.  Every
// bookkeeping kernel runs one CTA per sequence, so page reuse is
// deterministic.
#include <math.h>

#include "kvev_internal.h"

namespace kvev {
namespace {

constexpr int kPagedThreads = 128;   // scorer: 8 blocks of 16 tokens per CTA
constexpr int kBookThreads = 1024;   // bookkeeping CTAs (one per sequence)

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t order_bits(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide sum (float), result valid in every thread.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];   // fixed order
    __syncthreads();
    return s;
}
__device__ __forceinline__ int block_sum_int(int v, int* red) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int s = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    __syncthreads();
    return s;
}
// Exclusive block scan (int).
__device__ __forceinline__ int block_scan_excl(int v, int* red, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, m);
        if (lane >= m) x += y;
    }
    if (lane == 31) red[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? red[lane] : 0;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, m);
            if (lane >= m) w += y;
        }
        red[lane] = w;
    }
    __syncthreads();
    const int before = (warp > 0 ? red[warp - 1] : 0) + x - v;
    *total = red[nw - 1];
    __syncthreads();
    return before;
}

// ---------------------------------------------------------------- begin
__global__ void __launch_bounds__(kBookThreads) paged_begin_kernel(const PagedArgs a, int n0) {
    griddep_wait();
    griddep_release();
    const int b = blockIdx.x, pps = a.c.pages_per_seq;
    const int nb0 = (n0 + a.page - 1) / a.page;   // the last prefill block may be partial
    const size_t base = (size_t)b * pps;
    for (int j = threadIdx.x; j < pps; j += blockDim.x) {
        a.c.block_table[base + j] = j < nb0 ? b * pps + j : -1;
        a.st.score[base + j] = 0.f;
        a.st.t_ins[base + j] = 0;
        a.st.t_ref[base + j] = 0;
        a.st.lid[base + j] = j < nb0 ? j : -1;
        a.st.len[base + j] = j < nb0 ? min(a.page, n0 - j * a.page) : 0;
        // free stack: popping from the top yields the lowest free page first
        if (j < pps - nb0) a.c.free_pages[base + j] = b * pps + (pps - 1 - j);
    }
    for (int j = threadIdx.x; j < a.st.table_len; j += blockDim.x)
        a.st.table[(size_t)b * a.st.table_len + j] = __int_as_float(0x7fc00000);   // NaN
    if (a.rp.memdecay) {   // prefill tokens: importance 0, clock at insertion (step 0)
        for (int i = threadIdx.x; i < nb0 * a.page; i += blockDim.x) {
            const size_t ti = ((size_t)b * pps) * a.page + i;   // page b*pps + i/P, token i%P
            a.st.tok_a[ti] = 0.f;
            a.st.tok_t_ref[ti] = 0;
        }
    }
    if (threadIdx.x == 0) {
        a.c.n_blocks[b] = nb0;
        a.c.n_free[b] = pps - nb0;
        a.c.next_lid[b] = nb0;
        a.tokens[b] = n0;
    }
}

// --------------------------------------------------------------- append
// New token of sequence b: into the last block while it has room, else into
// a newly opened block (a page popped from the free stack; its score is 0
// on refresh steps and the mean score of the live blocks otherwise).
__global__ void __launch_bounds__(256) paged_append_kernel(const PagedArgs a,
                                                           const uint16_t* k_new,
                                                           const uint16_t* v_new) {
    __shared__ float redf[32];
    __shared__ int redi[32];
    __shared__ int s_page, s_tok;
    griddep_wait();
    griddep_release();
    const int b = blockIdx.x, pps = a.c.pages_per_seq;
    const size_t base = (size_t)b * pps;
    const int nb = a.c.n_blocks[b];
    const bool open_new = nb == 0 || a.st.len[base + nb - 1] >= a.page;
    float msum = 0.f;
    if (open_new && !a.refresh)
        for (int j = threadIdx.x; j < nb; j += blockDim.x) msum += a.st.score[base + j];
    msum = block_sum(msum, redf);
    if (threadIdx.x == 0) {
        int j = nb - 1, page = -1;
        if (open_new) {
            const int nf = a.c.n_free[b];
            if (nf > 0) {
                page = a.c.free_pages[base + nf - 1];
                a.c.n_free[b] = nf - 1;
                j = nb;
                a.c.block_table[base + j] = page;
                a.st.len[base + j] = 0;
                a.st.score[base + j] = a.refresh || nb == 0 ? 0.f : msum / (float)nb;
                a.st.t_ins[base + j] = a.t;
                a.st.lid[base + j] = a.c.next_lid[b]++;
                a.c.n_blocks[b] = nb + 1;
            } else {
                atomicOr(a.status, kStatusNoPage);
            }
        } else {
            page = a.c.block_table[base + j];
        }
        if (page >= 0) {
            const int tok = a.st.len[base + j];
            a.st.len[base + j] = tok + 1;
            a.st.t_ref[base + j] = a.t;   // insertion counts as an access
            s_tok = tok;
            if (a.rp.on) {                // the new token's label and MemDecay state
                const size_t ti = (size_t)page * a.page + tok;
                a.st.region[ti] = (uint8_t)a.rp.decode_region;
                if (a.rp.memdecay) {
                    a.st.tok_a[ti] = 0.f;
                    a.st.tok_t_ref[ti] = a.t;
                }
            }
        }
        s_page = page;
    }
    __syncthreads();
    const int page = s_page;
    if (page >= 0) {   // copy the new K/V rows into the page, every layer and KV head
        const int lpr = a.head_dim / 8;
        const int rows = a.n_layers * a.n_kv;
        constexpr int kBatch = 8;   // loads in flight per thread before their stores
        for (int u0 = threadIdx.x; u0 < 2 * rows * lpr; u0 += kBatch * blockDim.x) {
            uint4 w[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int u = u0 + k * blockDim.x;
                if (u >= 2 * rows * lpr) break;
                const int kv = u / (rows * lpr), rest = u - kv * rows * lpr;
                w[k] = __ldg(reinterpret_cast<const uint4*>(kv ? v_new : k_new) +
                             ((size_t)b * rows * lpr + rest));
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int u = u0 + k * blockDim.x;
                if (u >= 2 * rows * lpr) break;
                const int kv = u / (rows * lpr), rest = u - kv * rows * lpr;
                const int r = rest / lpr, c = rest - r * lpr;   // r = l * n_kv + g
                const size_t dst = ((((size_t)page * rows) + r) * a.page + s_tok) * lpr + c;
                reinterpret_cast<uint4*>(kv ? a.c.v_pool : a.c.k_pool)[dst] = w[k];
            }
        }
    }
    int ntok = 0;
    const int nb2 = a.c.n_blocks[b];
    __syncthreads();
    for (int j = threadIdx.x; j < nb2; j += blockDim.x) ntok += a.st.len[base + j];
    ntok = block_sum_int(ntok, redi);
    if (threadIdx.x == 0) a.tokens[b] = ntok;
}

// --------------------------------------------------------------- scoring
// One thread per token slot (16 consecutive lanes = one block).  Per layer,
// the token's head sum, then the block max across the 16 lanes, folded into
// the block's EMA.  On non-refresh steps the state is frozen and only the
// priority is formed.
template <int G, int NKV>
__global__ void __launch_bounds__(kPagedThreads) score_paged_kernel(const ScoreArgs sc,
                                                                    const PagedArgs a) {
    constexpr int V4 = G / 4;
    extern __shared__ float s_lse[];   // [Ly][NKV * G]
    griddep_wait();
    griddep_release();
    const int b = blockIdx.y, pps = a.c.pages_per_seq;
    const size_t base = (size_t)b * pps;
    if (sc.refresh) {
        const int nlse = sc.n_layers * NKV * G;
        for (int k = threadIdx.x; k < nlse; k += blockDim.x) {
            const int l = k / (NKV * G), h = k % (NKV * G);
            s_lse[k] = sc.lse2[((size_t)l * sc.batch + b) * sc.n_q + h];
        }
    }
    __syncthreads();
    const int slot = blockIdx.x * kPagedThreads + threadIdx.x;
    const int j = slot / a.page, k = slot % a.page;
    const int nb = a.c.n_blocks[b];
    const bool blk_live = j < nb;
    const int len = blk_live ? a.st.len[base + j] : 0;
    const bool live = k < len;
    float m = blk_live ? a.st.score[base + j] : 0.f;
    bool acc_blk = false;
    if (sc.refresh) {
        const float thr = 2.0f * (float)(sc.n_q * sc.n_layers) / (float)a.tokens[b];
        const size_t head_stride = (size_t)sc.logit_ld * G;
        const size_t layer_stride = (size_t)sc.batch * NKV * head_stride;
        const float* lbase = sc.logits + ((size_t)b * NKV) * head_stride + (size_t)slot * G;
        const float oma = 1.0f - a.alpha, inv_hq = 1.0f / (float)sc.n_q;
        float tot = 0.f;
        // the next layer's loads are issued before this layer is used
        float4 nx[NKV][V4];
#pragma unroll
        for (int g = 0; g < NKV; ++g)
#pragma unroll
            for (int c = 0; c < V4; ++c)
                nx[g][c] = live ? __ldcs(reinterpret_cast<const float4*>(lbase + g * head_stride) + c)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int l = 0; l < sc.n_layers; ++l) {
            float4 xb[NKV][V4];
#pragma unroll
            for (int g = 0; g < NKV; ++g)
#pragma unroll
                for (int c = 0; c < V4; ++c) {
                    xb[g][c] = nx[g][c];
                    nx[g][c] = live && l + 1 < sc.n_layers
                                   ? __ldcs(reinterpret_cast<const float4*>(
                                         lbase + (size_t)(l + 1) * layer_stride + g * head_stride) + c)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            float s = 0.f;
            if (live) {
                const float4* lg = reinterpret_cast<const float4*>(s_lse + l * NKV * G);
#pragma unroll
                for (int g = 0; g < NKV; ++g)
#pragma unroll
                    for (int c = 0; c < V4; ++c) {
                        const float4 x = xb[g][c], e = lg[g * V4 + c];
                        const float p0 = fast_exp2(x.x - e.x), p1 = fast_exp2(x.y - e.y);
                        const float p2 = fast_exp2(x.z - e.z), p3 = fast_exp2(x.w - e.w);
                        if (sc.dbg_probs) {
                            float* dp = sc.dbg_probs +
                                        (((size_t)b * sc.n_layers + l) * sc.n_q + g * G + 4 * c) *
                                            sc.max_ctx + slot;
                            dp[0] = p0;
                            dp[(size_t)sc.max_ctx] = p1;
                            dp[2 * (size_t)sc.max_ctx] = p2;
                            dp[3 * (size_t)sc.max_ctx] = p3;
                        }
                        s += (p0 + p1) + (p2 + p3);
                    }
            }
            tot += s;
            float sb = s;   // block max over the 16 lanes of this block (probabilities >= 0)
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) sb = fmaxf(sb, __shfl_xor_sync(0xffffffffu, sb, o));
            m = fmaf(a.alpha, a.pool_mean ? sb * inv_hq : sb, oma * m);
        }
        const bool acc_tok = live && tot >= thr;
        const unsigned bal = __ballot_sync(0xffffffffu, acc_tok);
        acc_blk = ((bal >> (threadIdx.x & 16)) & 0xffffu) != 0;
    }
    bool pinned = false;
    if (a.rp.on) {   // a block holding a token of a pinned region is never evicted
        const int pg = blk_live ? a.c.block_table[base + j] : 0;
        const bool pin_tok = live && ((a.rp.pinned_mask >> a.st.region[(size_t)pg * a.page + k]) & 1u);
        const unsigned pb = __ballot_sync(0xffffffffu, pin_tok);
        pinned = ((pb >> (threadIdx.x & 16)) & 0xffffu) != 0;
    }
    if (k != 0 || !blk_live) return;
    int t_ref = a.st.t_ref[base + j];
    const int t_ins = a.st.t_ins[base + j];
    if (acc_blk) t_ref = a.t;
    const int age = a.t - (a.age_mode == KVEV_AGE_SINCE_ACCESS ? t_ref : t_ins);
    const float pr = age == 0 ? 0.0f : (1.0f - m) * -expm1f(-a.beta * (float)age);
    a.keys[base + j] = pinned ? 0u : order_bits(pr);
    a.m_s[base + j] = m;
    a.tref_s[base + j] = t_ref;
    a.tins_s[base + j] = t_ins;
    a.lid_s[base + j] = a.st.lid[base + j];
    a.len_s[base + j] = len;
    a.page_s[base + j] = a.c.block_table[base + j];
    if (a.dbg_prio) a.dbg_prio[base + j] = pr + 0.0f;
}

// --------------------------------------------------------------- compaction
// Kept blocks (ascending slots from the selection) move to slots 0..n-1;
// evicted blocks store their score under their logical id and return their
// pages to the free stack in slot order.
__global__ void __launch_bounds__(kBookThreads) paged_compact_kernel(const PagedArgs a) {
    __shared__ int red[32];
    extern __shared__ int s_kept[];    // [pps] flags
    griddep_wait();
    griddep_release();
    const int b = blockIdx.x, pps = a.c.pages_per_seq;
    const size_t base = (size_t)b * pps;
    const int nb = a.c.n_blocks[b];
    const int nk = a.n_sel[b];
    const int32_t* sel = a.sel + (size_t)b * a.sel_ld;
    for (int j = threadIdx.x; j < nb; j += blockDim.x) s_kept[j] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < nk; j += blockDim.x) s_kept[sel[j]] = 1;
    __syncthreads();
    for (int j = threadIdx.x; j < nk; j += blockDim.x) {
        const size_t src = base + sel[j], dst = base + j;
        a.c.block_table[dst] = a.page_s[src];
        a.st.score[dst] = a.m_s[src];
        a.st.t_ins[dst] = a.tins_s[src];
        a.st.t_ref[dst] = a.tref_s[src];
        a.st.lid[dst] = a.lid_s[src];
        a.st.len[dst] = a.len_s[src];
        a.retained_lid[(size_t)b * a.sel_ld + j] = a.lid_s[src];
    }
    int nf = a.c.n_free[b];
    for (int j0 = 0; j0 < nb; j0 += blockDim.x) {   // evicted: persist, free the page
        const int j = j0 + threadIdx.x;
        const bool ev = j < nb && !s_kept[j];
        int total;
        const int before = block_scan_excl(ev ? 1 : 0, red, &total);
        if (ev) {
            const int lid = a.lid_s[base + j];
            if (!a.rp.memdecay && lid >= 0 && lid < a.st.table_len)
                a.st.table[(size_t)b * a.st.table_len + lid] = a.m_s[base + j];
            a.c.free_pages[base + nf + before] = a.page_s[base + j];
        }
        nf += total;
    }
    if (threadIdx.x == 0) {
        a.c.n_free[b] = nf;
        a.c.n_blocks[b] = nk;
    }
}

// --------------------------------------------------------------- re-admission
// One CTA: if logical block `lid` of sequence `seq` is not resident, pop a
// free page, open a slot at the block's sorted place (shifting the later
// blocks up by one) and set its state; the page goes to readmit_page for the
// copy kernel (-1: nothing to copy).
__global__ void __launch_bounds__(kBookThreads) readmit_meta_kernel(const PagedArgs a, int seq,
                                                                    int lid, int persist) {
    __shared__ int red[32];
    griddep_wait();
    griddep_release();
    const int pps = a.c.pages_per_seq;
    const size_t base = (size_t)seq * pps;
    const int nb = a.c.n_blocks[seq];
    int found = 0, below = 0;
    for (int j = threadIdx.x; j < nb; j += blockDim.x) {
        const int x = a.st.lid[base + j];
        found += x == lid;
        below += x < lid;
    }
    found = block_sum_int(found, red);
    below = block_sum_int(below, red);
    const int nf = a.c.n_free[seq];
    if (found || nf == 0 || nb >= pps) {
        if (threadIdx.x == 0) {
            a.readmit_page[0] = -1;
            if (!found) atomicOr(a.status, kStatusNoPage);
        }
        return;
    }
    // shift slots [below, nb) up by one, top chunk first: a chunk is read in
    // full before it is written one slot higher, above the next chunk down
    for (int hi = nb; hi > below; hi -= blockDim.x) {
        const int lo = max(below, hi - (int)blockDim.x);
        const int j = lo + threadIdx.x;
        const bool mv = j < hi;
        int tb = 0, ti = 0, tr = 0, li = 0, ln = 0;
        float sc = 0.f;
        if (mv) {
            tb = a.c.block_table[base + j];
            sc = a.st.score[base + j];
            ti = a.st.t_ins[base + j];
            tr = a.st.t_ref[base + j];
            li = a.st.lid[base + j];
            ln = a.st.len[base + j];
        }
        __syncthreads();
        if (mv) {
            a.c.block_table[base + j + 1] = tb;
            a.st.score[base + j + 1] = sc;
            a.st.t_ins[base + j + 1] = ti;
            a.st.t_ref[base + j + 1] = tr;
            a.st.lid[base + j + 1] = li;
            a.st.len[base + j + 1] = ln;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const int page = a.c.free_pages[base + nf - 1];
        a.c.n_free[seq] = nf - 1;
        a.c.block_table[base + below] = page;
        const float stored = lid < a.st.table_len ? a.st.table[(size_t)seq * a.st.table_len + lid]
                                                  : __int_as_float(0x7fc00000);
        a.st.score[base + below] = persist && !isnan(stored) ? stored : 0.f;
        a.st.t_ins[base + below] = 0;
        a.st.t_ref[base + below] = a.t;
        a.st.lid[base + below] = lid;
        a.st.len[base + below] = a.page;
        a.c.n_blocks[seq] = nb + 1;
        a.readmit_page[0] = page;
    }
}

// Copies the backing-tier block (all layers and KV heads) into the page.
__global__ void readmit_copy_kernel(const PagedArgs a, int seq, int lid) {
    griddep_wait();
    griddep_release();
    const int page = a.readmit_page[0];
    if (page < 0) return;
    const size_t units = (size_t)a.n_layers * a.n_kv * a.page * a.head_dim / 8;   // 16 B
    const size_t src = ((size_t)seq * a.c.n_backing + lid) * units;
    const size_t dst = (size_t)page * units;
    for (size_t u = blockIdx.x * (size_t)blockDim.x + threadIdx.x; u < 2 * units;
         u += (size_t)gridDim.x * blockDim.x) {
        const bool v = u >= units;
        const size_t c = v ? u - units : u;
        const uint4 w = reinterpret_cast<const uint4*>(v ? a.c.backing_v : a.c.backing_k)[src + c];
        reinterpret_cast<uint4*>(v ? a.c.v_pool : a.c.k_pool)[dst + c] = w;
    }
}

// ---------------------------------------------------------- region-aware
// MemDecay scoring ("MemDecay: Region-Aware KV Cache Eviction ...", Sec.
// III-C/D): one thread per token slot, 16 lanes = one block.  On refresh
// (observation) steps the token's attention averaged over heads and layers
// updates its importance (Eq. (2)) and may reset its decay clock (Eq. (3));
// every step the token's retention score (Eq. (4)) is averaged over the
// block (Eq. (5)).  Per-token state is indexed by page, so it never moves.
// Key: 0 for a pinned block (always kept), else the order bits of -S_p
// (the selection keeps the smallest keys: the highest page scores).
template <int G, int NKV>
__global__ void __launch_bounds__(kPagedThreads) score_memdecay_kernel(const ScoreArgs sc,
                                                                       const PagedArgs a) {
    constexpr int V4 = G / 4;
    extern __shared__ float s_lse[];   // [Ly][NKV * G]
    griddep_wait();
    griddep_release();
    const int b = blockIdx.y, pps = a.c.pages_per_seq;
    const size_t base = (size_t)b * pps;
    if (sc.refresh) {
        const int nlse = sc.n_layers * NKV * G;
        for (int k = threadIdx.x; k < nlse; k += blockDim.x) {
            const int l = k / (NKV * G), h = k % (NKV * G);
            s_lse[k] = sc.lse2[((size_t)l * sc.batch + b) * sc.n_q + h];
        }
    }
    __syncthreads();
    const int slot = blockIdx.x * kPagedThreads + threadIdx.x;
    const int j = slot / a.page, k = slot % a.page;
    const int nb = a.c.n_blocks[b];
    const bool blk_live = j < nb;
    const int len = blk_live ? a.st.len[base + j] : 0;
    const bool live = k < len;
    float s = 0.f;
    bool pin = false;
    if (live) {
        const size_t ti = (size_t)a.c.block_table[base + j] * a.page + k;
        float av = a.st.tok_a[ti];
        int tref = a.st.tok_t_ref[ti];
        const int r = a.st.region[ti];
        if (sc.refresh) {
            const size_t head_stride = (size_t)sc.logit_ld * G;
            const size_t layer_stride = (size_t)sc.batch * NKV * head_stride;
            const float* lbase = sc.logits + ((size_t)b * NKV) * head_stride + (size_t)slot * G;
            float tot = 0.f;
            // the next layer's loads are issued before this layer is used
            float4 nx[NKV][V4];
#pragma unroll
            for (int g = 0; g < NKV; ++g)
#pragma unroll
                for (int c = 0; c < V4; ++c)
                    nx[g][c] = __ldcs(reinterpret_cast<const float4*>(lbase + g * head_stride) + c);
            for (int l = 0; l < sc.n_layers; ++l) {
                float4 xb[NKV][V4];
#pragma unroll
                for (int g = 0; g < NKV; ++g)
#pragma unroll
                    for (int c = 0; c < V4; ++c) {
                        xb[g][c] = nx[g][c];
                        if (l + 1 < sc.n_layers)
                            nx[g][c] = __ldcs(reinterpret_cast<const float4*>(
                                                  lbase + (size_t)(l + 1) * layer_stride +
                                                  g * head_stride) + c);
                    }
                const float4* lg = reinterpret_cast<const float4*>(s_lse + l * NKV * G);
                float sl = 0.f;
#pragma unroll
                for (int g = 0; g < NKV; ++g)
#pragma unroll
                    for (int c = 0; c < V4; ++c) {
                        const float4 x = xb[g][c], e = lg[g * V4 + c];
                        const float p0 = fast_exp2(x.x - e.x), p1 = fast_exp2(x.y - e.y);
                        const float p2 = fast_exp2(x.z - e.z), p3 = fast_exp2(x.w - e.w);
                        if (sc.dbg_probs) {
                            float* dp = sc.dbg_probs +
                                        (((size_t)b * sc.n_layers + l) * sc.n_q + g * G + 4 * c) *
                                            sc.max_ctx + slot;
                            dp[0] = p0;
                            dp[(size_t)sc.max_ctx] = p1;
                            dp[2 * (size_t)sc.max_ctx] = p2;
                            dp[3 * (size_t)sc.max_ctx] = p3;
                        }
                        sl += (p0 + p1) + (p2 + p3);
                    }
                tot += sl;
            }
            const float A = tot / (float)(sc.n_q * sc.n_layers);
            av = fmaf(a.rp.rho, av, (1.0f - a.rp.rho) * A);
            if (A >= a.rp.tau_scale / (float)a.tokens[b]) tref = a.t;
            a.st.tok_a[ti] = av;
            a.st.tok_t_ref[ti] = tref;
        }
        s = fmaf(a.rp.attn_w, av, a.rp.base[r] * expf(-a.rp.lam[r] * (float)(a.t - tref)));
        pin = (a.rp.pinned_mask >> r) & 1u;
    }
    float sum = s;   // block sum over the 16 lanes of this block
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const unsigned pb = __ballot_sync(0xffffffffu, pin);
    const bool pinned = ((pb >> (threadIdx.x & 16)) & 0xffffu) != 0;
    if (k != 0 || !blk_live) return;
    const float S = sum / (float)len;
    a.keys[base + j] = pinned ? 0u : max(order_bits(-S), 1u);
    a.m_s[base + j] = S;
    a.tref_s[base + j] = a.st.t_ref[base + j];
    a.tins_s[base + j] = a.st.t_ins[base + j];
    a.lid_s[base + j] = a.st.lid[base + j];
    a.len_s[base + j] = len;
    a.page_s[base + j] = a.c.block_table[base + j];
    if (a.dbg_prio) a.dbg_prio[base + j] = S;
}

// Blocks the selection keeps per sequence when a region table is set.
// LRFU: the budget, or every pinned block when they are more.  MemDecay:
// evicting the blocks of least S_p one by one until the tokens fit the
// budget removes the j largest keys, j the least count whose blocks hold at
// least the excess.  Every block but the last is full, so j is
// ceil(excess / P), plus one when the partial last block is among those and
// falls short.
__global__ void __launch_bounds__(256) block_budget_kernel(const PagedArgs a) {
    __shared__ int red[32];
    griddep_wait();
    griddep_release();
    const int b = blockIdx.x, pps = a.c.pages_per_seq;
    const size_t base = (size_t)b * pps;
    const int nb = a.c.n_blocks[b];
    if (!a.rp.memdecay) {
        int pinned = 0;
        for (int j = threadIdx.x; j < nb; j += blockDim.x) pinned += a.keys[base + j] == 0u;
        pinned = block_sum_int(pinned, red);
        if (threadIdx.x == 0) a.budgets[b] = max(a.budget, pinned);
        return;
    }
    const int excess = a.tokens[b] - a.rp.budget_tokens;
    if (excess <= 0 || nb == 0) {          // the same in every thread
        if (threadIdx.x == 0) a.budgets[b] = nb;
        return;
    }
    const int last = nb - 1;
    const uint32_t kl = a.keys[base + last];
    const int rl = a.len_s[base + last];
    int n_free = 0, ahead = 0;   // evictable blocks; blocks ranked before the last one
    for (int j = threadIdx.x; j < nb; j += blockDim.x) {
        const uint32_t kj = a.keys[base + j];
        n_free += kj != 0u;
        ahead += j < last && kj <= kl;
    }
    n_free = block_sum_int(n_free, red);
    ahead = block_sum_int(ahead, red);
    if (threadIdx.x == 0) {
        int j0 = min((excess + a.page - 1) / a.page, n_free);
        const bool last_goes = kl != 0u && ahead >= nb - j0;
        if (rl < a.page && last_goes && a.page * (j0 - 1) + rl < excess && j0 < n_free) ++j0;
        a.budgets[b] = nb - j0;
    }
}

template <int G>
void* memdecay_score_for(int nkv) {
    switch (nkv) {
        case 1: return (void*)score_memdecay_kernel<G, 1>;
        case 2: return (void*)score_memdecay_kernel<G, 2>;
        case 4: return (void*)score_memdecay_kernel<G, 4>;
        case 8: return (void*)score_memdecay_kernel<G, 8>;
        default: return nullptr;
    }
}

template <int G>
void* paged_score_for(int nkv) {
    switch (nkv) {
        case 1: return (void*)score_paged_kernel<G, 1>;
        case 2: return (void*)score_paged_kernel<G, 2>;
        case 4: return (void*)score_paged_kernel<G, 4>;
        case 8: return (void*)score_paged_kernel<G, 8>;
        default: return nullptr;
    }
}

}  // namespace

cudaError_t launch_paged_begin(const PagedArgs& a, int prefill_tokens, cudaStream_t s) {
    return launch_pdl(paged_begin_kernel, dim3(a.batch), dim3(kBookThreads), 0, s, a,
                      prefill_tokens);
}

cudaError_t launch_paged_append(const PagedArgs& a, const uint16_t* k_new, const uint16_t* v_new,
                                cudaStream_t s) {
    return launch_pdl(paged_append_kernel, dim3(a.batch), dim3(256), 0, s, a, k_new, v_new);
}

cudaError_t launch_paged_score(const ScoreArgs& sc, const PagedArgs& a, int group, int ub_blocks,
                               cudaStream_t s) {
    void* kern = group == 4 ? paged_score_for<4>(sc.n_kv) : group == 8 ? paged_score_for<8>(sc.n_kv)
                                                                       : nullptr;
    if (!kern || a.page != 16) return cudaErrorInvalidValue;
    const int slots = ub_blocks * a.page;
    const dim3 grid((slots + kPagedThreads - 1) / kPagedThreads, a.batch);
    const size_t smem = sizeof(float) * (size_t)sc.n_layers * sc.n_q;
    return launch_pdl(reinterpret_cast<void (*)(ScoreArgs, PagedArgs)>(kern), grid,
                      dim3(kPagedThreads), smem, s, sc, a);
}

cudaError_t launch_memdecay_score(const ScoreArgs& sc, const PagedArgs& a, int group,
                                  int ub_blocks, cudaStream_t s) {
    void* kern = group == 4 ? memdecay_score_for<4>(sc.n_kv)
                 : group == 8 ? memdecay_score_for<8>(sc.n_kv) : nullptr;
    if (!kern || a.page != 16) return cudaErrorInvalidValue;
    const int slots = ub_blocks * a.page;
    const dim3 grid((slots + kPagedThreads - 1) / kPagedThreads, a.batch);
    const size_t smem = sizeof(float) * (size_t)sc.n_layers * sc.n_q;
    return launch_pdl(reinterpret_cast<void (*)(ScoreArgs, PagedArgs)>(kern), grid,
                      dim3(kPagedThreads), smem, s, sc, a);
}

cudaError_t launch_block_budget(const PagedArgs& a, cudaStream_t s) {
    return launch_pdl(block_budget_kernel, dim3(a.batch), dim3(256), 0, s, a);
}

cudaError_t launch_paged_compact(const PagedArgs& a, cudaStream_t s) {
    return launch_pdl(paged_compact_kernel, dim3(a.batch), dim3(kBookThreads),
                      sizeof(int) * (size_t)a.c.pages_per_seq, s, a);
}

cudaError_t launch_readmit(const PagedArgs& a, int seq, int lid, int persist, cudaStream_t s) {
    cudaError_t e = launch_pdl(readmit_meta_kernel, dim3(1), dim3(kBookThreads), 0, s, a, seq,
                               lid, persist);
    if (e != cudaSuccess) return e;
    return launch_pdl(readmit_copy_kernel, dim3(256), dim3(256), 0, s, a, seq, lid);
}

}  // namespace kvev
