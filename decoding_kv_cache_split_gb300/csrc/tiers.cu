// Two-tier window routing with an INT2 tier ("QEvict: Recoverable Quantized
// KV Eviction for Attention-Drift-Robust Long-Context Decoding", review
// page Sec. 4): bookkeeping, window scores, routing, quantization.
//
// Positions [0, 5) are sinks, [5 + 128 j, 5 + 128 (j + 1)) window j; the
// bf16 pool holds 16-token pages aligned to that grid (page b*pps holds the
// sinks), so a window is 8 pages and its tiles are the 16-token tiles
// 8 j .. 8 j + 7 of the grid.  A sequence's bookkeeping runs in one CTA;
// the routing sorts the candidates in shared memory (bitonic), then
// quantization (first demotion only) and promotion (from the ledger) run as
// grid-stride kernels over (window, layer, KV head) items, and the pages the
// demoted and evicted windows held return to the free stack last, after the
// quantization has read them.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvev_internal.h"

namespace kvev {
namespace {

constexpr int kBook = 1024;

__device__ __forceinline__ uint32_t order_bits(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Exclusive block scan of one int per thread (blockDim.x = kBook); *total.
__device__ __forceinline__ int scan_excl(int v, int* red, int* total) {
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
// 16-byte asynchronous global -> shared copies: every copy of a stage is in
// flight at once (no register round trip), then one wait.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ bool is_bf16_tier(uint8_t t) {
    return t == KVEV_TIER_UNROUTED || t == KVEV_TIER_FULL;
}

// ---------------------------------------------------------------- begin
__global__ void __launch_bounds__(kBook) tier_begin_kernel(const TierArgs a, int n0) {
    griddep_wait();
    griddep_release();
    const int b = blockIdx.x, pps = a.c.pages_per_seq, MW = a.c.max_windows;
    const int base = b * pps;
    const int hist = n0 - kTierSinks;
    const int nw = hist / kTierW, tl = hist - nw * kTierW;
    const int n_tail_pages = (tl + kTile - 1) / kTile;
    const int used = 1 + nw * (kTierW / kTile) + n_tail_pages;
    for (int w = threadIdx.x; w < MW; w += blockDim.x) {
        const size_t wi = (size_t)b * MW + w;
        a.st.tier[wi] = w < nw ? KVEV_TIER_UNROUTED : KVEV_TIER_NONE;
        a.st.score[wi] = 0.f;
        a.st.has_codes[wi] = 0;
        for (int i = 0; i < kTierW / kTile; ++i)
            a.st.win_pages[wi * (kTierW / kTile) + i] = w < nw ? base + 1 + w * (kTierW / kTile) + i : -1;
    }
    for (int i = threadIdx.x; i < kTierW / kTile; i += blockDim.x)
        a.st.tail_pages[(size_t)b * (kTierW / kTile) + i] =
            i < n_tail_pages ? base + 1 + nw * (kTierW / kTile) + i : -1;
    const int avail = pps - a.scratch;   // the last `scratch` pages hold reconstructions
    for (int k = threadIdx.x; k < avail - used; k += blockDim.x)   // lowest free page on top
        a.c.free_pages[(size_t)base + k] = base + avail - 1 - k;
    if (a.rope) {   // no INT2 window yet: every reconstruction slot is free, lowest on top
        const int n_slots = a.scratch / (kTierW / kTile);
        for (int w = threadIdx.x; w < MW; w += blockDim.x) {
            a.rslot[(size_t)b * MW + w] = -1;
            if (w < n_slots) a.rfree[(size_t)b * MW + w] = n_slots - 1 - w;
        }
        if (threadIdx.x == 0) {
            a.n_rfree[b] = n_slots;
            a.n_rlist[b] = 0;
        }
    }
    if (threadIdx.x == 0) {
        a.c.n_free[b] = avail - used;
        a.st.n_windows[b] = nw;
        a.st.tail_len[b] = tl;
        a.seq_len[b] = n0;
    }
}

// --------------------------------------------------------------- append
// The new token joins the tail (a page popped when the tail needs one); a
// tail of 128 tokens becomes a new unrouted window.  Then the attention
// lists are rebuilt: bf16 blocks (sink page, the pages of unrouted and Full
// windows in window order, the tail pages) with their positions and
// lengths, and the INT2 windows in window order.
__global__ void __launch_bounds__(kBook) tier_append_kernel(const TierArgs a,
                                                            const uint16_t* k_new,
                                                            const uint16_t* v_new) {
    __shared__ int red[32];
    __shared__ int s_page, s_row, s_nw, s_tl;
    griddep_wait();
    griddep_release();
    const int b = blockIdx.x, pps = a.c.pages_per_seq, MW = a.c.max_windows;
    constexpr int PW = kTierW / kTile;   // pages per window
    int32_t* tail = a.st.tail_pages + (size_t)b * PW;
    if (threadIdx.x == 0) {
        int tl = a.st.tail_len[b];
        int page = -1;
        if (tl >= kTierW) {      // no window slot was left for a complete tail
            atomicOr(a.status, kStatusNoPage);
        } else if (tl % kTile == 0) {   // the tail needs a fresh page
            const int nf = a.c.n_free[b];
            if (nf > 0) {
                page = a.c.free_pages[(size_t)b * pps + nf - 1];
                a.c.n_free[b] = nf - 1;
                tail[tl / kTile] = page;
            } else {
                atomicOr(a.status, kStatusNoPage);
            }
        } else {
            page = tail[tl / kTile];
        }
        s_page = page;
        s_row = tl % kTile;
        int nw = a.st.n_windows[b];
        if (page >= 0) {
            ++tl;
            a.seq_len[b] += 1;
            if (tl == kTierW && nw < MW) {   // the tail completes window nw
                const size_t wi = (size_t)b * MW + nw;
                for (int i = 0; i < PW; ++i) {
                    a.st.win_pages[wi * PW + i] = tail[i];
                    tail[i] = -1;
                }
                a.st.tier[wi] = KVEV_TIER_UNROUTED;
                a.st.score[wi] = 0.f;
                a.st.has_codes[wi] = 0;
                ++nw;
                tl = 0;
            }
        }
        a.st.tail_len[b] = tl;
        a.st.n_windows[b] = nw;
        s_nw = nw;
        s_tl = tl;
    }
    __syncthreads();
    const int page = s_page;
    if (page >= 0) {   // K/V rows of the new token, every layer and KV head
        const int lpr = a.head_dim / 8;
        const int rows = a.n_layers * a.n_kv;
        constexpr int kBatch = 8;   // loads in flight per thread before their stores
        for (int u0 = threadIdx.x; u0 < 2 * rows * lpr; u0 += kBatch * blockDim.x) {
            uint4 v[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int u = u0 + k * blockDim.x;
                if (u >= 2 * rows * lpr) break;
                const int kv = u / (rows * lpr), rest = u - kv * rows * lpr;
                v[k] = __ldg(reinterpret_cast<const uint4*>(kv ? v_new : k_new) +
                             ((size_t)b * rows * lpr + rest));
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int u = u0 + k * blockDim.x;
                if (u >= 2 * rows * lpr) break;
                const int kv = u / (rows * lpr), rest = u - kv * rows * lpr;
                const int r = rest / lpr, c = rest - r * lpr;
                const size_t dst = (((size_t)page * rows + r) * kTile + s_row) * lpr + c;
                reinterpret_cast<uint4*>(kv ? a.c.v_pool : a.c.k_pool)[dst] = v[k];
            }
        }
    }
    // ---- attention lists
    const int nw = s_nw, tl = s_tl;
    int32_t* bt = a.bt + (size_t)b * a.bt_ld;
    int32_t* bpos = a.bpos + (size_t)b * a.bt_ld;
    int32_t* blen = a.blen + (size_t)b * a.bt_ld;
    if (threadIdx.x == 0) {
        bt[0] = b * pps;
        bpos[0] = 0;
        blen[0] = kTierSinks;
    }
    int n_bf = 0, n_q = 0;
    for (int w0 = 0; w0 < nw; w0 += blockDim.x) {
        const int w = w0 + threadIdx.x;
        const uint8_t tr = w < nw ? a.st.tier[(size_t)b * MW + w] : KVEV_TIER_NONE;
        int tot_bf, tot_q;
        const int off_bf = scan_excl(is_bf16_tier(tr) ? 1 : 0, red, &tot_bf);
        const int off_q = scan_excl(tr == KVEV_TIER_QUANT ? 1 : 0, red, &tot_q);
        if (is_bf16_tier(tr)) {
            const int j0 = 1 + (n_bf + off_bf) * PW;
            for (int i = 0; i < PW; ++i) {
                bt[j0 + i] = a.st.win_pages[((size_t)b * MW + w) * PW + i];
                bpos[j0 + i] = kTierSinks + w * kTierW + i * kTile;
                blen[j0 + i] = kTile;
            }
        }
        if (tr == KVEV_TIER_QUANT) a.qlist[(size_t)b * MW + n_q + off_q] = w;
        n_bf += tot_bf;
        n_q += tot_q;
    }
    const int j0 = 1 + n_bf * PW;
    const int n_tail = (tl + kTile - 1) / kTile;
    for (int i = threadIdx.x; i < n_tail; i += blockDim.x) {
        bt[j0 + i] = tail[i];
        bpos[j0 + i] = kTierSinks + nw * kTierW + i * kTile;
        blen[j0 + i] = min(kTile, tl - i * kTile);
    }
    int n_rec = 0;
    if (a.rope) {   // rotary mode: the INT2 windows' bf16 reconstructions
        __syncthreads();   // the INT2 list is complete
        const int n_slots = a.scratch / PW;
        int32_t* rslot = a.rslot + (size_t)b * MW;
        if (a.rebuild) {   // slot e for the e-th INT2 window; all of them to reconstruct
            for (int w = threadIdx.x; w < MW; w += blockDim.x) rslot[w] = -1;
            __syncthreads();
            for (int k = threadIdx.x; k < n_q; k += blockDim.x) {
                const int w = a.qlist[(size_t)b * MW + k];
                rslot[w] = k < n_slots ? k : -1;   // (k_q never exceeds the slots)
                a.rlist[(size_t)b * MW + k] = w;
            }
            for (int k = threadIdx.x; k < n_slots - n_q; k += blockDim.x)
                a.rfree[(size_t)b * MW + k] = n_slots - 1 - k;
            if (threadIdx.x == 0) {
                a.n_rfree[b] = max(n_slots - n_q, 0);
                a.n_rlist[b] = n_q;
            }
            __syncthreads();
        }
        const int jq = j0 + n_tail, sbase = b * pps + pps - a.scratch;
        for (int u = threadIdx.x; u < n_q * PW; u += blockDim.x) {
            const int k = u / PW, i = u % PW;
            const int w = a.qlist[(size_t)b * MW + k];
            const int slot = rslot[w];
            // a window without a slot (flagged by the routing) reads the sink page
            bt[jq + u] = slot >= 0 && slot < n_slots ? sbase + slot * PW + i : b * pps;
            bpos[jq + u] = kTierSinks + w * kTierW + i * kTile;
            blen[jq + u] = kTile;
        }
        n_rec = n_q * PW;
    }
    if (threadIdx.x == 0) {
        a.nblk[b] = j0 + n_tail + n_rec;
        a.nq[b] = n_q;
    }
}

// ---------------------------------------------------------- window score
// One warp per window: per layer, the head-averaged attention the window's
// 128 tokens received, from the tile statistics of the attention kernels
// (running max m, sum of exp2(x - m) per head and 16-token tile) and the
// combine's log2-sum-exp: sum exp2(m - lse) * sum; folded into the EMA
// layer after layer, or added to the score (the cumulative score of the
// review's Sec. 4.2 Eq. (1): alpha = oma = 1).
template <int G>
__global__ void __launch_bounds__(256) tier_score_kernel(const TierArgs a) {
    griddep_wait();
    griddep_release();
    const int b = blockIdx.y, MW = a.c.max_windows;
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (w >= a.st.n_windows[b]) return;
    const size_t wi = (size_t)b * MW + w;
    const uint8_t tr = a.st.tier[wi];
    if (!is_bf16_tier(tr) && tr != KVEV_TIER_QUANT) return;
    constexpr int PW = kTierW / kTile;
    float m = a.st.score[wi];
    const float inv_hq = 1.0f / (float)a.n_q, oma = a.oma;
    // the layers' masses in batches of 8 (their loads are independent), then
    // the EMA folded over them in layer order
    constexpr int kLB = 8;
    for (int l0 = 0; l0 < a.n_layers; l0 += kLB) {
        float sl[kLB];
#pragma unroll
        for (int u = 0; u < kLB; ++u) {
            const int l = l0 + u;
            float s = 0.f;
            if (l < a.n_layers) {
#pragma unroll 2
                for (int k = lane; k < PW * a.n_kv; k += 32) {   // (tile, KV head) pairs
                    const int i = k % PW, g = k / PW;
                    const size_t row = ((size_t)l * a.batch + b) * a.n_kv + g;
                    const float2* st = a.tile_stats + (row * a.stats_tiles + (size_t)w * PW + i) * G;
                    const float* lse = a.lse2 + ((size_t)l * a.batch + b) * a.n_q + g * G;
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float2 v = st[h];
                        s = fmaf(exp2_approx(v.x - lse[h]), v.y, s);
                    }
                }
            }
            sl[u] = s;
        }
#pragma unroll
        for (int u = 0; u < kLB; ++u) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sl[u] += __shfl_xor_sync(0xffffffffu, sl[u], o);
            if (l0 + u < a.n_layers) m = fmaf(a.alpha, sl[u] * inv_hq, oma * m);
        }
    }
    if (lane == 0) a.st.score[wi] = m;
}

// --------------------------------------------------------------- routing
// Candidates: Full and INT2 windows, and unrouted windows whose last token
// is older than the recent region.  Ranked by score (ties: lower index)
// with a bitonic sort of (order bits of -score, window) keys; the top K_f
// are Full, the next K_q INT2, the rest evicted.
__global__ void __launch_bounds__(kBook) tier_route_kernel(const TierArgs a) {
    __shared__ unsigned long long keys[kTierRouteCap];
    __shared__ uint8_t nt[kTierRouteCap];
    __shared__ uint8_t enters[kTierRouteCap];   // rotary mode: the window enters the INT2 tier
    __shared__ int red[32];
    griddep_wait();
    griddep_release();
    const int b = blockIdx.x, pps = a.c.pages_per_seq, MW = a.c.max_windows;
    constexpr int PW = kTierW / kTile;
    const int nw = a.st.n_windows[b];
    if (nw > kTierRouteCap) {
        if (threadIdx.x == 0) {
            atomicOr(a.status, kStatusRouteCap);
            a.n_quant[b] = a.n_prom[b] = a.n_freeing[b] = 0;
        }
        return;
    }
    int n = 1;
    while (n < nw) n <<= 1;
    const int horizon = a.seq_len[b] - kTierRecent;
    for (int w = threadIdx.x; w < n; w += blockDim.x) {
        unsigned long long key = ~0ull;
        if (w < nw) {
            const size_t wi = (size_t)b * MW + w;
            const uint8_t tr = a.st.tier[wi];
            nt[w] = tr;
            const bool cand = tr == KVEV_TIER_FULL || tr == KVEV_TIER_QUANT ||
                              (tr == KVEV_TIER_UNROUTED && kTierSinks + (w + 1) * kTierW <= horizon);
            if (cand) key = ((unsigned long long)order_bits(-a.st.score[wi]) << 32) | (unsigned)w;
        }
        keys[w] = key;
    }
    __syncthreads();
    for (int k = 2; k <= n; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int p = i ^ j;
                if (p > i) {
                    const unsigned long long x = keys[i], y = keys[p];
                    if ((x > y) == ((i & k) == 0)) {
                        keys[i] = y;
                        keys[p] = x;
                    }
                }
            }
            __syncthreads();
        }
    for (int r = threadIdx.x; r < n; r += blockDim.x) {
        const unsigned long long key = keys[r];
        if (key != ~0ull) {
            const int w = (int)(key & 0xffffffffu);
            nt[w] = r < a.k_full ? KVEV_TIER_FULL
                    : r < a.k_full + a.k_quant ? KVEV_TIER_QUANT : KVEV_TIER_EVICTED;
        }
    }
    __syncthreads();
    // transitions: lists for quantization, promotion and freeing; in rotary
    // mode the reconstruction slots of windows leaving the INT2 tier return
    // to their stack
    int nq = 0, np = 0, nf = 0, nl = 0;
    const int free0 = a.c.n_free[b];
    const int rfree0 = a.rope ? a.n_rfree[b] : 0;
    for (int w0 = 0; w0 < nw; w0 += blockDim.x) {
        const int w = w0 + threadIdx.x;
        uint8_t o = KVEV_TIER_NONE, t = KVEV_TIER_NONE;
        bool codes = false;
        if (w < nw) {
            o = a.st.tier[(size_t)b * MW + w];
            t = nt[w];
            codes = a.st.has_codes[(size_t)b * MW + w] != 0;
        }
        const bool quant = is_bf16_tier(o) && t == KVEV_TIER_QUANT && !codes;
        const bool prom = o == KVEV_TIER_QUANT && t == KVEV_TIER_FULL;
        const bool frees = is_bf16_tier(o) && (t == KVEV_TIER_QUANT || t == KVEV_TIER_EVICTED);
        const bool leaves = a.rope && o == KVEV_TIER_QUANT && t != KVEV_TIER_QUANT;
        int tq, tp, tf, tl;
        const int oq = scan_excl(quant ? 1 : 0, red, &tq);
        const int op = scan_excl(prom ? 1 : 0, red, &tp);
        const int of = scan_excl(frees ? 1 : 0, red, &tf);
        const int ol = a.rope ? scan_excl(leaves ? 1 : 0, red, &tl) : (tl = 0, 0);
        if (w < nw) {
            const size_t wi = (size_t)b * MW + w;
            if (a.rope) {
                enters[w] = o != KVEV_TIER_QUANT && t == KVEV_TIER_QUANT;
                if (leaves) {
                    if (rfree0 + nl + ol < MW) a.rfree[(size_t)b * MW + rfree0 + nl + ol] = a.rslot[wi];
                    a.rslot[wi] = -1;
                }
            }
            if (quant) a.quant_list[(size_t)b * MW + nq + oq] = w;
            if (frees) a.free_list[(size_t)b * MW + nf + of] = w;
            if (prom) {   // 8 pages from the top of the free stack (pages freed before this event)
                const int k = np + op;
                for (int i = 0; i < PW; ++i) {
                    const int top = free0 - 1 - k * PW - i;
                    a.st.win_pages[wi * PW + i] =
                        top >= 0 ? a.c.free_pages[(size_t)b * pps + top] : -1;
                }
                a.prom_list[(size_t)b * MW + k] = w;
            }
            if (quant) a.st.has_codes[wi] = 1;
            if (t == KVEV_TIER_EVICTED) a.st.has_codes[wi] = 0;
            a.st.tier[wi] = t;
        }
        nq += tq;
        np += tp;
        nf += tf;
        nl += tl;
    }
    if (a.rope) {   // entering windows pop slots (the top first) and are listed for reconstruction
        __syncthreads();
        const int top = rfree0 + nl;
        int ne = 0;
        for (int w0 = 0; w0 < nw; w0 += blockDim.x) {
            const int w = w0 + threadIdx.x;
            const bool e = w < nw && enters[w];
            int te;
            const int oe = scan_excl(e ? 1 : 0, red, &te);
            if (e) {
                const int k = ne + oe, at = top - 1 - k;
                // every INT2 window holds one slot and there are at least K_q:
                // the stack cannot run dry
                const bool ok = at >= 0 && at < MW;
                if (!ok) atomicOr(a.status, kStatusNoPage);
                a.rslot[(size_t)b * MW + w] = ok ? a.rfree[(size_t)b * MW + at] : -1;
                a.rlist[(size_t)b * MW + k] = w;
            }
            ne += te;
        }
        if (threadIdx.x == 0) {
            a.n_rfree[b] = max(top - ne, 0);
            a.n_rlist[b] = ne;
        }
    }
    if (threadIdx.x == 0) {
        a.n_quant[b] = nq;
        a.n_prom[b] = np;
        a.n_freeing[b] = nf;
        if (np * PW > free0) {
            atomicOr(a.status, kStatusNoPage);
            a.n_prom[b] = free0 / PW;
        }
        a.c.n_free[b] = free0 - min(np * PW, free0 / PW * PW);
    }
}

// Items of the quantize / promote kernels: (sequence, list entry, layer,
// KV head) over the lists' actual lengths, grid-stride.
__device__ __forceinline__ int64_t item_count(const int32_t* n, int batch, int LG) {
    int64_t c = 0;
    for (int b = 0; b < batch; ++b) c += (int64_t)n[b] * LG;
    return c;
}
__device__ __forceinline__ void item_at(const int32_t* n, int batch, int LG, int64_t it, int* b,
                                        int* e, int* lg) {
    int bb = 0;
    while (bb < batch - 1 && it >= (int64_t)n[bb] * LG) it -= (int64_t)n[bb++] * LG;
    *b = bb;
    *e = (int)(it / LG);
    *lg = (int)(it % LG);
}

// The code of x in a group with fp16 zero z and scale sc > 0: rint of the
// correctly rounded fp32 quotient y = (x - z) / sc, clamped to [0, 3], i.e.
// (y > 0.5) + (y >= 1.5) + (y > 2.5) (rint rounds ties to even).  The
// quotient is first taken as (x - z) * r with r = 1 / sc correctly rounded:
// the two roundings put it within 3 * 2^-24 relative of the exact quotient,
// so within 2^-19 of y while it is below 8 in magnitude; only within 2^-16
// of a threshold can it fall on the other side of one than y does, and there
// the quotient is divided out exactly (out of line: the rare path stays out
// of the unrolled loops).
__device__ __noinline__ float exact_quotient(float d, float sc) { return __fdiv_rn(d, sc); }
__device__ __forceinline__ float int2_quotient(float x, float z, float sc, float r) {
    const float d = __fsub_rn(x, z);
    const float y = __fmul_rn(d, r);
    const float dc = fabsf(y - 1.5f);
    return dc <= 0x1p-16f || fabsf(dc - 1.f) <= 0x1p-16f ? exact_quotient(d, sc) : y;
}
__device__ __forceinline__ uint32_t int2_code(float x, float z, float sc, float r) {
    const float y = int2_quotient(x, z, sc, r);
    return (uint32_t)(y > 0.5f) + (uint32_t)(y >= 1.5f) + (uint32_t)(y > 2.5f);
}

// Quantization of one half (keys or values) of a (window, layer, KV head)
// item: the window's 128 rows are staged in shared memory (rows padded by 16
// bytes so row-strided reads spread over the banks).  Keys: a thread per
// channel pair and 32-token group (min / max on bf16 pairs), the 8 threads
// whose codes share a ledger word in consecutive lanes; each places its
// codes in their fields and the 8 OR them together with three shuffles.
// Values: a thread per token and 32-channel group; each turns its codes into
// the sign / magnitude bits of their ledger registers, and the threads whose
// bits share a word OR them together with two shuffles.  One thread of a
// word stores it.  With rotary positions (ROPE) a key pair is first rotated
// back in fp32 with its partner pair, the table's cos / sin of 8 rows loaded
// together.
constexpr int kQuantThreads = 256;
constexpr int kRowPad = 8;     // bf16 elements of padding per staged row

template <int D, bool ROPE>
__device__ __forceinline__ void quantize_items(const TierArgs& a, int max_items) {
    using Lay = LedgerLayout<D>;
    static_assert(D == 128, "ledger registers are laid out for head_dim 128");
    constexpr int PW = kTierW / kTile, WPL = Lay::WORDS_PER_LANE;
    constexpr int XS = D + kRowPad;                 // staged row stride (elements)
    extern __shared__ __align__(16) unsigned char qsm[];
    __nv_bfloat16* xt = reinterpret_cast<__nv_bfloat16*>(qsm);            // [128][XS]
    (void)max_items;
    griddep_wait();
    griddep_release();
    const int LG = a.n_layers * a.n_kv, MW = a.c.max_windows;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t total = 2 * item_count(a.n_quant, a.batch, LG);
    for (int64_t it = blockIdx.x; it < total; it += gridDim.x) {
        const int kv = (int)(it & 1);
        int b, e, lg;
        item_at(a.n_quant, a.batch, LG, it >> 1, &b, &e, &lg);
        const int w = a.quant_list[(size_t)b * MW + e];
        const int l = lg / a.n_kv, g = lg % a.n_kv;
        const int32_t* pages = a.st.win_pages + ((size_t)b * MW + w) * PW;
        unsigned char* led = reinterpret_cast<unsigned char*>(a.c.ledger) +
                             ((((size_t)b * MW + w) * a.n_layers + l) * a.n_kv + g) * Lay::BYTES;
        // stage: page i holds tokens 16 i .. 16 i + 15 of the window, rows contiguous
        constexpr int kChunks = kTile * D / 8;   // 16-byte chunks per page row block
        const uint4* pool = reinterpret_cast<const uint4*>(kv ? a.c.v_pool : a.c.k_pool);
#pragma unroll
        for (int pi = 0; pi < PW; ++pi) {
            const uint4* src = pool + ((((size_t)pages[pi] * a.n_layers + l) * a.n_kv + g) * kTile) * D / 8;
#pragma unroll
            for (int k = 0; k < kChunks / kQuantThreads; ++k) {
                const int c = tid + k * kQuantThreads;
                cp_async16(reinterpret_cast<uint4*>(xt + (pi * kTile + c / (D / 8)) * XS) + c % (D / 8),
                           src + c);
            }
        }
        cp_async_wait_all();
        __syncthreads();
        uint32_t* words = reinterpret_cast<uint32_t*>(led + (kv ? Lay::VC : Lay::KC));
        if (kv == 0) {
            // keys: channels c = 16 s + 8 h + 2 t, c + 1 over group grp (tokens
            // 32 grp .. + 31); lane = 8 t + s, h = warp & 1, so the 8 threads of
            // a word (its 8 k-steps s) are consecutive lanes
            const int s8 = lane & 7, t = lane >> 3, h = warp & 1, grp = warp >> 1;
            const int p = 8 * s8 + 4 * h + t;   // channel pair 2p, 2p + 1
            const __nv_bfloat162* col =
                reinterpret_cast<const __nv_bfloat162*>(xt + grp * kQGroup * XS) + p;
            // the pair at `row` of the group as quantized: with rotary positions
            // rotated back by the row's position (the partner pair 2p +- D/2 is
            // lane ^ 4's), fp32 products and sums in the oracle's order
            const bool first_half = 2 * p < D / 2;
            const float4* cs_row = ROPE
                ? reinterpret_cast<const float4*>(a.rope) +
                      ((size_t)(kTierSinks + w * kTierW + grp * kQGroup) * (D / 2) +
                       ((2 * p) & (D / 2 - 1))) / 2
                : nullptr;
            // the (cos, sin) of channels j, j + 1 at 8 rows row0 + k step, loaded
            // together so that their latencies overlap
            auto load_cs = [&](float4 (&cs)[8], int row0, int step) {
#pragma unroll
                for (int k = 0; k < 8; ++k) cs[k] = __ldg(cs_row + (size_t)(row0 + k * step) * (D / 4));
            };
            auto key_at = [&](int row, const float4& cs) -> float2 {
                const float2 x = __bfloat1622float2(col[row * (XS / 2)]);
                if (!ROPE) return x;
                const float yx = __shfl_xor_sync(0xffffffffu, x.x, 4);
                const float yy = __shfl_xor_sync(0xffffffffu, x.y, 4);
                return first_half
                    ? make_float2(__fadd_rn(__fmul_rn(x.x, cs.x), __fmul_rn(yx, cs.y)),
                                  __fadd_rn(__fmul_rn(x.y, cs.z), __fmul_rn(yy, cs.w)))
                    : make_float2(__fsub_rn(__fmul_rn(x.x, cs.x), __fmul_rn(yx, cs.y)),
                                  __fsub_rn(__fmul_rn(x.y, cs.z), __fmul_rn(yy, cs.w)));
            };
            float4 cs[8];
            float2 mn, mx;
            if constexpr (ROPE) {
                mn = make_float2(INFINITY, INFINITY);
                mx = make_float2(-INFINITY, -INFINITY);
#pragma unroll
                for (int r0 = 0; r0 < kQGroup; r0 += 8) {
                    load_cs(cs, r0, 1);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float2 x = key_at(r0 + k, cs[k]);
                        mn = make_float2(fminf(mn.x, x.x), fminf(mn.y, x.y));
                        mx = make_float2(fmaxf(mx.x, x.x), fmaxf(mx.y, x.y));
                    }
                }
            } else {
                mn = key_at(0, cs[0]);
                mx = mn;
#pragma unroll
                for (int r = 1; r < kQGroup; ++r) {
                    const float2 x = key_at(r, cs[0]);
                    mn = make_float2(fminf(mn.x, x.x), fminf(mn.y, x.y));
                    mx = make_float2(fmaxf(mx.x, x.x), fmaxf(mx.y, x.y));
                }
            }
            const __half2 z16 = __floats2half2_rn(mn.x, mn.y);
            const __half2 s16 = __floats2half2_rn(__fdiv_rn(__fsub_rn(mx.x, mn.x), 3.0f),
                                                  __fdiv_rn(__fsub_rn(mx.y, mn.y), 3.0f));
            const float2 z = __half22float2(z16), sc = __half22float2(s16);
            const int k = Lay::key_scale_index(grp, 2 * p);
            reinterpret_cast<__half2*>(led + Lay::KS)[k / 2] = s16;
            reinterpret_cast<__half2*>(led + Lay::KZ)[k / 2] = z16;
            const float r0 = sc.x == 0.f ? 0.f : __frcp_rn(sc.x);
            const float r1 = sc.y == 0.f ? 0.f : __frcp_rn(sc.y);
            const int b0 = Lay::key_bit(Lay::key_field(s8), 0);   // field of k-step s8
            // token 8 i + gg of tile 2 grp + tt: word 2 i + h of lane 4 gg + t (with
            // rotary positions the 8 rows of one (tt, i) share a batch of loads)
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
#pragma unroll
                for (int io = 0; io < (ROPE ? 2 : 8); ++io) {
                    if constexpr (ROPE) load_cs(cs, 16 * tt + 8 * io, 1);
#pragma unroll
                    for (int ii = 0; ii < (ROPE ? 8 : 2); ++ii) {
                        const int gg = ROPE ? ii : io, i = ROPE ? io : ii;
                        const float2 x = key_at(16 * tt + 8 * i + gg, cs[ROPE ? ii : 0]);
                        const uint32_t c0 = sc.x == 0.f ? 0u : int2_code(x.x, z.x, sc.x, r0);
                        const uint32_t c1 = sc.y == 0.f ? 0u : int2_code(x.y, z.y, sc.y, r1);
                        uint32_t word = (c0 << b0) | (c1 << (b0 + 16));
                        word |= __shfl_xor_sync(0xffffffffu, word, 1);
                        word |= __shfl_xor_sync(0xffffffffu, word, 2);
                        word |= __shfl_xor_sync(0xffffffffu, word, 4);
                        if (s8 == 0)
                            words[(2 * grp + tt) * D + (4 * gg + t) * WPL + 2 * i + h] = word;
                    }
                }
        } else {
            // values: token tok over channel groups cg and cg + 2; the codes of
            // channel 8 j + gg sit in register 2 j + h of lane 4 gg + t, half e,
            // for token 2 t + 8 h + e of the tile: the lanes xor 1 and xor 8
            // (tokens e and h) fill one word's 8 slots with the 4 j of a group
            const int tok = tid & 127;
            const int e2 = tok & 1, t = (tok & 7) >> 1, hh = (tok >> 3) & 1, ti = tok >> 4;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int cg = (tid >> 7) + 2 * half;
                const __nv_bfloat162* row =
                    reinterpret_cast<const __nv_bfloat162*>(xt + tok * XS + cg * kQGroup);
                __nv_bfloat162 v2[kQGroup / 2];
#pragma unroll
                for (int k = 0; k < kQGroup / 8; ++k) {
                    const uint4 q4 = reinterpret_cast<const uint4*>(row)[k];
                    v2[4 * k] = *reinterpret_cast<const __nv_bfloat162*>(&q4.x);
                    v2[4 * k + 1] = *reinterpret_cast<const __nv_bfloat162*>(&q4.y);
                    v2[4 * k + 2] = *reinterpret_cast<const __nv_bfloat162*>(&q4.z);
                    v2[4 * k + 3] = *reinterpret_cast<const __nv_bfloat162*>(&q4.w);
                }
                __nv_bfloat162 mn2 = v2[0], mx2 = v2[0];
#pragma unroll
                for (int i = 1; i < kQGroup / 2; ++i) {
                    mn2 = __hmin2(mn2, v2[i]);
                    mx2 = __hmax2(mx2, v2[i]);
                }
                const float mnf = fminf(__low2float(mn2), __high2float(mn2));
                const float mxf = fmaxf(__low2float(mx2), __high2float(mx2));
                const __half z16 = __float2half_rn(mnf);
                const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mxf, mnf), 3.0f));
                const float z = __half2float(z16), sc = __half2float(s16);
                reinterpret_cast<__half*>(led + Lay::VS)[Lay::value_scale_index(tok, cg)] = s16;
                reinterpret_cast<__half*>(led + Lay::VZ)[Lay::value_scale_index(tok, cg)] = z16;
                const float r = sc == 0.f ? 0.f : __frcp_rn(sc);
                // channel 32 cg + 8 jj + gg -> register 2 (4 cg + jj) + hh: word cg,
                // slot 2 jj + hh, half e2: the code's sign bit (code <= 1, i.e. the
                // quotient y < 1.5) at 15 + 16 e2 + 2 slot and its magnitude bit
                // (code 0 or 3: y <= 0.5 or y > 2.5) 9 below, both mod 32; a zero
                // scale gives code 0
                uint32_t sbit[4], mbit[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    sbit[jj] = 1u << ((15 + 16 * e2 + 2 * (2 * jj + hh)) & 31);
                    mbit[jj] = 1u << ((6 + 16 * e2 + 2 * (2 * jj + hh)) & 31);
                }
#pragma unroll
                for (int gg = 0; gg < 8; ++gg) {
                    uint32_t word = 0;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int c = 8 * jj + gg;
                        const float x = (c & 1) ? __high2float(v2[c >> 1]) : __low2float(v2[c >> 1]);
                        const float y = sc == 0.f ? 0.f : int2_quotient(x, z, sc, r);
                        word |= (y < 1.5f ? sbit[jj] : 0u) | (y <= 0.5f || y > 2.5f ? mbit[jj] : 0u);
                    }
                    word |= __shfl_xor_sync(0xffffffffu, word, 1);
                    word |= __shfl_xor_sync(0xffffffffu, word, 8);
                    if ((lane & 9) == 0)
                        words[ti * D + (4 * gg + t) * WPL + cg] = word;
                }
            }
        }
        __syncthreads();
    }
}

// The plain quantizer at 4 CTAs per SM; the rotary one without a register cap
// (its batches of table loads want the registers).
template <int D>
__global__ void __launch_bounds__(kQuantThreads, 4) tier_quantize_kernel(const TierArgs a,
                                                                         int max_items) {
    quantize_items<D, false>(a, max_items);
}
template <int D>
__global__ void __launch_bounds__(kQuantThreads) tier_quantize_rope_kernel(const TierArgs a,
                                                                           int max_items) {
    quantize_items<D, true>(a, max_items);
}

// Promotion of one half (keys or values) of a (window, layer, KV head) item:
// the half's ledger codes and scales are staged in shared memory, then each
// thread walks the two pages of one channel pair and a quarter of the window
// (for keys a 32-token group, so one scale pair), reading each code (keys:
// from its field; values: a register's bf16 pair (2 c - 3) * 2^-128, exact
// subnormals, so c = v * 2^127 + 1.5 exactly in fp32) and writing
// code * scale + zero rounded to bf16 (warps store 128 contiguous bytes of a
// page row).
constexpr int kPromThreads = 256;

__device__ __forceinline__ float2 reg_codes(uint32_t x) {   // x rotated to slot 0
    const uint32_t r = (x & 0x80408040u) | 0x00200020u;
    return make_float2(fmaf(__uint_as_float(r << 16), 0x1p127f, 1.5f),
                       fmaf(__uint_as_float(r & 0xffff0000u), 0x1p127f, 1.5f));
}

template <int D>
__global__ void __launch_bounds__(kPromThreads, 4) tier_promote_kernel(const TierArgs a,
                                                                    int max_items) {
    using Lay = LedgerLayout<D>;
    static_assert(D == 128, "ledger registers are laid out for head_dim 128");
    constexpr int PW = kTierW / kTile, WPL = Lay::WORDS_PER_LANE;
    constexpr int HALF = Lay::VC;   // bytes of one half: codes, then scales, then zeros
    __shared__ __align__(16) unsigned char led_s[HALF];
    griddep_wait();
    griddep_release();
    (void)max_items;
    const int LG = a.n_layers * a.n_kv, MW = a.c.max_windows;
    // promotion: the routing event's promoted windows into their new pages;
    // reconstruction (rotary mode): the windows of rlist into the scratch
    // pages pps - scratch + slot PW .. + PW - 1 of their sequence
    const int32_t* counts = a.recon ? a.n_rlist : a.n_prom;
    const int32_t* list = a.recon ? a.rlist : a.prom_list;
    const int64_t total = 2 * item_count(counts, a.batch, LG);
    const int tid = threadIdx.x;
    const int n_slots = a.scratch / PW;
    for (int64_t it = blockIdx.x; it < total; it += gridDim.x) {
        const int kv = (int)(it & 1);
        int b, e, lg;
        item_at(counts, a.batch, LG, it >> 1, &b, &e, &lg);
        const int w = list[(size_t)b * MW + e];
        const int l = lg / a.n_kv, g = lg % a.n_kv;
        const int32_t* pages = a.st.win_pages + ((size_t)b * MW + w) * PW;
        const int slot = a.recon ? a.rslot[(size_t)b * MW + w] : 0;
        if (a.recon && (slot < 0 || slot >= n_slots)) continue;   // (flagged by the routing)
        const int rec0 = b * a.c.pages_per_seq + a.c.pages_per_seq - a.scratch + slot * PW;
        const uint4* led = reinterpret_cast<const uint4*>(
            reinterpret_cast<const unsigned char*>(a.c.ledger) +
            ((((size_t)b * MW + w) * a.n_layers + l) * a.n_kv + g) * Lay::BYTES +
            (kv ? Lay::VC : Lay::KC));
        for (int u = tid; u < HALF / 16; u += blockDim.x)
            cp_async16(reinterpret_cast<uint4*>(led_s) + u, led + u);
        cp_async_wait_all();
        __syncthreads();
        const uint32_t* cw = reinterpret_cast<const uint32_t*>(led_s);
        const __half2* sc2 = reinterpret_cast<const __half2*>(led_s + (Lay::KS - Lay::KC));
        const __half2* zc2 = reinterpret_cast<const __half2*>(led_s + (Lay::KZ - Lay::KC));
        uint32_t* pool = reinterpret_cast<uint32_t*>(kv ? a.c.v_pool : a.c.k_pool);
        const int p = tid & 63;   // channel pair 2p, 2p + 1
        const int q4 = tid >> 6;  // key group / quarter of the window: pages 2 q4, 2 q4 + 1
        auto page_of = [&](int i) { return a.recon ? rec0 + i : pages[i]; };
        auto row_ptr = [&](int page, int pair) {
            return pool + ((((int64_t)page * a.n_layers + l) * a.n_kv + g) * kTile) * D / 2 + pair;
        };
        // key channels 2 pp, 2 pp + 1 of token 16 ti + r (one field, halves 0 and 1)
        auto deq = [&](int pp, int ti, int r) -> float2 {
            const int k = Lay::key_scale_index(q4, 2 * pp);
            const float2 sf = __half22float2(sc2[k / 2]), zf = __half22float2(zc2[k / 2]);
            int word, field, half;
            Lay::key_place(16 * ti + r, 2 * pp, &word, &field, &half);
            const uint32_t wd = cw[word];
            const float c0 = (float)((wd >> Lay::key_bit(field, 0)) & 3u);
            const float c1 = (float)((wd >> Lay::key_bit(field, 1)) & 3u);
            return make_float2(fmaf(c0, sf.x, zf.x), fmaf(c1, sf.y, zf.y));
        };
        if (kv == 0 && a.rope) {
            // keys with rotary positions: thread (q4, p) takes page 2 q4 + p / 32
            // and the pairs pp = p mod 32 and pp + D/4 (channels j, j + 1 and
            // j + D/2, j + D/2 + 1 for j = 2 pp), which rotate together by the
            // token's position, fp32 products and sums in the oracle's order
            const int pp = p & (D / 4 - 1), ti = 2 * q4 + (p >> 5);
            const int page = page_of(ti);
            if (page >= 0) {
                uint32_t* dst = row_ptr(page, pp);
                const float4* cs_row = reinterpret_cast<const float4*>(a.rope) +
                                       ((size_t)(kTierSinks + w * kTierW + 16 * ti) * (D / 2) + 2 * pp) / 2;
#pragma unroll 4
                for (int r = 0; r < kTile; ++r) {
                    const float2 x = deq(pp, ti, r), y = deq(pp + D / 4, ti, r);
                    const float4 cs = __ldg(cs_row + (size_t)r * (D / 4));   // cos, sin of j, j + 1
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(
                        __fsub_rn(__fmul_rn(x.x, cs.x), __fmul_rn(y.x, cs.y)),
                        __fsub_rn(__fmul_rn(x.y, cs.z), __fmul_rn(y.y, cs.w)));
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(
                        __fadd_rn(__fmul_rn(y.x, cs.x), __fmul_rn(x.x, cs.y)),
                        __fadd_rn(__fmul_rn(y.y, cs.z), __fmul_rn(x.y, cs.w)));
                    dst[r * (D / 2)] = *reinterpret_cast<const uint32_t*>(&lo);
                    dst[r * (D / 2) + D / 4] = *reinterpret_cast<const uint32_t*>(&hi);
                }
            }
            __syncthreads();
            continue;
        }
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {
            const int page = page_of(2 * q4 + pg);
            if (page < 0) continue;   // no page could be taken for this promotion
            uint32_t* dst = row_ptr(page, p);
            const uint32_t* cwt = cw + (2 * q4 + pg) * D;   // code words of this 16-token tile
            if (kv == 0) {
                // keys: channels 2p, 2p + 1 of the tokens 16 (2 q4 + pg) + r,
                // read from their ledger fields
#pragma unroll
                for (int r = 0; r < kTile; ++r) {
                    const float2 x = deq(p, 2 * q4 + pg, r);
                    const __nv_bfloat162 bb = __floats2bfloat162_rn(x.x, x.y);
                    dst[r * (D / 2)] = *reinterpret_cast<const uint32_t*>(&bb);
                }
            } else {
                // values: channels c0 = 2p, 2p + 1 (lanes 4 gg + t, 4 (gg + 1) + t) of the
                // token pair 16 (2 q4 + pg) + 2 kk (+1): register 2 j + h, h = kk / 4, t = kk % 4
                const int c0 = 2 * p, j = c0 >> 3, gg = c0 & 7, cg = c0 / kQGroup;
                const uint32_t* cwl = cwt + 4 * gg * WPL + (j >> 2);
                const int rot0 = 2 * (2 * (j & 3));
#pragma unroll
                for (int kk = 0; kk < kTile / 2; ++kk) {
                    const int h = kk >> 2, t = kk & 3;
                    const uint32_t w0 = cwl[t * WPL];
                    const uint32_t w1 = cwl[(4 + t) * WPL];
                    const float2 ca = reg_codes(__funnelshift_r(w0, w0, rot0 + 2 * h));   // channel c0
                    const float2 cb = reg_codes(__funnelshift_r(w1, w1, rot0 + 2 * h));   // channel c0 + 1
                    const int kq = Lay::value_scale_index(16 * (2 * q4 + pg) + 2 * kk, cg);
                    const float2 sf = __half22float2(sc2[kq / 2]), zf = __half22float2(zc2[kq / 2]);
                    const __nv_bfloat162 r0 = __floats2bfloat162_rn(fmaf(ca.x, sf.x, zf.x),
                                                                    fmaf(cb.x, sf.x, zf.x));
                    const __nv_bfloat162 r1 = __floats2bfloat162_rn(fmaf(ca.y, sf.y, zf.y),
                                                                    fmaf(cb.y, sf.y, zf.y));
                    dst[(2 * kk) * (D / 2)] = *reinterpret_cast<const uint32_t*>(&r0);
                    dst[(2 * kk + 1) * (D / 2)] = *reinterpret_cast<const uint32_t*>(&r1);
                }
            }
        }
        __syncthreads();
    }
}

// The pages of windows that left the bf16 tier return to the free stack.
__global__ void __launch_bounds__(256) tier_finish_kernel(const TierArgs a) {
    griddep_wait();
    griddep_release();
    const int b = blockIdx.x, pps = a.c.pages_per_seq, MW = a.c.max_windows;
    constexpr int PW = kTierW / kTile;
    const int n = a.n_freeing[b], nf = a.c.n_free[b];
    for (int u = threadIdx.x; u < n * PW; u += blockDim.x) {
        const int k = u / PW, i = u % PW;
        const int w = a.free_list[(size_t)b * MW + k];
        int32_t* wp = a.st.win_pages + ((size_t)b * MW + w) * PW;
        a.c.free_pages[(size_t)b * pps + nf + u] = wp[i];
        wp[i] = -1;
    }
    __syncthreads();
    if (threadIdx.x == 0) a.c.n_free[b] = nf + n * PW;
}

// Global LIR bookkeeping after a routing event (the QEvict review, Sec. 3:
// how often a window inactive for a sustained period re-enters the
// full-precision set).  Per window of the sequence, routed ones only: Full
// -> a revival when it had been outside Full at `sustain` or more routing
// events in a row, then its streak restarts; INT2 or evicted -> the streak
// grows, and reaching `sustain` opens a sustained-inactive span.  One CTA
// per sequence; the counts are added in a fixed order (block reduction).
__global__ void __launch_bounds__(256) tier_lir_kernel(const TierArgs a) {
    __shared__ int red[2][8];
    griddep_wait();
    griddep_release();
    const int b = blockIdx.x, MW = a.c.max_windows;
    const int nw = a.st.n_windows[b];
    int rev = 0, span = 0;
    for (int w = threadIdx.x; w < nw; w += blockDim.x) {
        const size_t wi = (size_t)b * MW + w;
        const uint8_t tr = a.st.tier[wi];
        if (tr == KVEV_TIER_UNROUTED || tr == KVEV_TIER_NONE) continue;
        const int st = a.lir_streak[wi];
        if (tr == KVEV_TIER_FULL) {
            rev += st >= a.lir_sustain;
            a.lir_streak[wi] = 0;
        } else {
            a.lir_streak[wi] = st + 1;
            span += st + 1 == a.lir_sustain;
        }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        rev += __shfl_xor_sync(0xffffffffu, rev, m);
        span += __shfl_xor_sync(0xffffffffu, span, m);
    }
    if ((threadIdx.x & 31) == 0) {
        red[0][threadIdx.x >> 5] = rev;
        red[1][threadIdx.x >> 5] = span;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int r = 0, sp = 0;
        for (int k = 0; k < 8; ++k) {
            r += red[0][k];
            sp += red[1][k];
        }
        int32_t* c = a.lir_counters + (size_t)b * 3;
        c[0] += 1;
        c[1] += r;
        c[2] += sp;
    }
}

}  // namespace

cudaError_t launch_tier_lir(const TierArgs& a, cudaStream_t s) {
    return launch_pdl(tier_lir_kernel, dim3(a.batch), dim3(256), 0, s, a);
}

cudaError_t launch_tier_begin(const TierArgs& a, int prefill_tokens, cudaStream_t s) {
    return launch_pdl(tier_begin_kernel, dim3(a.batch), dim3(kBook), 0, s, a, prefill_tokens);
}

cudaError_t launch_tier_append(const TierArgs& a, const uint16_t* k_new, const uint16_t* v_new,
                               cudaStream_t s) {
    return launch_pdl(tier_append_kernel, dim3(a.batch), dim3(kBook), 0, s, a, k_new, v_new);
}

cudaError_t launch_tier_score(const TierArgs& a, int max_nw, int group, cudaStream_t s) {
    if (max_nw <= 0) return cudaSuccess;
    const dim3 grid((max_nw + 7) / 8, a.batch);
    if (group == 4) return launch_pdl(tier_score_kernel<4>, grid, dim3(256), 0, s, a);
    if (group == 8) return launch_pdl(tier_score_kernel<8>, grid, dim3(256), 0, s, a);
    return cudaErrorInvalidValue;
}

cudaError_t launch_tier_route(const TierArgs& a, cudaStream_t s) {
    return launch_pdl(tier_route_kernel, dim3(a.batch), dim3(kBook), 0, s, a);
}

cudaError_t launch_tier_quantize(const TierArgs& a, int max_items, int num_sms, cudaStream_t s) {
    if (max_items <= 0) return cudaSuccess;
    if (a.head_dim != 128) return cudaErrorInvalidValue;
    auto kern = a.rope ? tier_quantize_rope_kernel<128> : tier_quantize_kernel<128>;
    const int smem = kTierW * (128 + kRowPad) * 2;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t items = 2LL * a.batch * max_items * a.n_layers * a.n_kv;
    const int grid = (int)std::min<int64_t>(items, 4LL * num_sms);
    return launch_pdl(kern, dim3(grid), dim3(kQuantThreads), (size_t)smem, s, a, max_items);
}

cudaError_t launch_tier_promote(const TierArgs& a, int max_items, int num_sms, cudaStream_t s) {
    if (max_items <= 0) return cudaSuccess;
    if (a.head_dim != 128) return cudaErrorInvalidValue;
    const int64_t items = 2LL * a.batch * max_items * a.n_layers * a.n_kv;
    const int grid = (int)std::min<int64_t>(items, 4LL * num_sms);
    return launch_pdl(tier_promote_kernel<128>, dim3(grid), dim3(kPromThreads), 0, s, a,
                      max_items);
}

cudaError_t launch_tier_finish(const TierArgs& a, cudaStream_t s) {
    return launch_pdl(tier_finish_kernel, dim3(a.batch), dim3(256), 0, s, a);
}

}  // namespace kvev
