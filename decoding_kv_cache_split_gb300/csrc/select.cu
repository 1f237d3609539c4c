// Budgeted selection: keep the B tokens of lowest eviction priority, ties
// to the lower slot index, and list them in ascending slot order.
//
// "What Matters for Aggressive Decoding-Time KV Eviction?" Sec. 3.1: whenever
// the cache exceeds B, the lowest-utility tokens are evicted; with the LRFU
// priority of the kv-cache-docs "ema-eviction" figure a higher priority is
// evicted, so the B lowest priorities are retained.
//
// One thread-block cluster of kCl CTAs per sequence (one CTA when the
// sequence's keys fit its shared memory).  The keys are the
// order-preserving bits of the fp32 priorities; CTA r of the cluster stages
// the r-th contiguous chunk of a sequence's keys in shared memory.  A 4-pass
// radix select (8-bit digits) finds the B-th smallest key T: in every pass
// each CTA histograms its chunk, the CTAs read each other's histograms
// through distributed shared memory after a cluster barrier, and all of them
// take the same digit.  Then each CTA counts its keys below / equal to T,
// the counts are exchanged the same way, and each CTA writes its kept slots
// (all keys < T, and the first keys == T in slot order up to B) at its
// offset, ascending.  The cluster barriers are hardware barriers
// (barrier.cluster), there is no software spin-wait.
//
// Few evictions (L - B <= kFewEvict, the steady state of a decode, where one
// new token arrives and one leaves): the first CTA alone takes the L - B
// largest (key, slot) pairs by repeated block-wide maxima and keeps every
// other slot, which is the same set as the radix path's (the B smallest
// pairs, ties to the lower slot) at a fraction of its barriers.
#include "kvev_internal.h"

namespace kvev {
namespace {

constexpr int kCl = 8;                      // CTAs per sequence (portable cluster size)
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;

__device__ __forceinline__ uint32_t cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 32-bit load from the same shared-memory variable of CTA `rank` of the cluster
__device__ __forceinline__ uint32_t ld_remote(const void* local, uint32_t rank) {
    uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(local)), ra, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
    return v;
}

// Exclusive block scan of one int per thread; also returns the total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* red, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, m);
        if (lane >= m) x += y;
    }
    if (lane == 31) red[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kSelWarps ? red[lane] : 0;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, m);
            if (lane >= m) w += y;
        }
        red[lane] = w;   // inclusive prefix of warp totals
    }
    __syncthreads();
    const int before = (warp > 0 ? red[warp - 1] : 0) + x - v;
    *total = red[kSelWarps - 1];
    __syncthreads();
    return before;
}

// The L - B (<= kFewEvict) largest (key, slot) pairs leave, every other slot
// is kept in ascending order.  Pairs are distinct (the slot breaks ties), so
// each round's maximum below the previous round's is a new pair.
__device__ void select_few(const uint32_t* gkeys, int L, int B, int32_t* ret,
                           int32_t* n_retained, int32_t* first_moved, int32_t* evicted) {
    __shared__ unsigned long long wmax[kSelWarps];
    __shared__ int ev[kFewEvict];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = L - B;
    unsigned long long prev = ~0ull;
    for (int r = 0; r < E; ++r) {
        // a thread without candidates offers (0, 0), the least pair: B >= 1
        // leaves at least one candidate in every round, so the maximum is real
        unsigned long long best = 0;
        for (int i = tid; i < L; i += kSelThreads) {
            const unsigned long long c = ((unsigned long long)__ldcg(gkeys + i) << 32) | (uint32_t)i;
            if (c < prev && c > best) best = c;
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, m);
            best = o > best ? o : best;
        }
        if (lane == 0) wmax[warp] = best;
        __syncthreads();
        if (warp == 0) {
            static_assert(kSelWarps == 32, "one warp reduces the warps' maxima");
            unsigned long long v = wmax[lane];
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, m);
                v = o > v ? o : v;
            }
            if (lane == 0) {
                ev[r] = (int)(uint32_t)v;
                wmax[0] = v;
            }
        }
        __syncthreads();
        prev = wmax[0];
        __syncthreads();   // wmax is rewritten by the next round
    }
    // keep every slot but the E evicted ones, ascending
    int gone_slot[kFewEvict];
    int lowest = L;
#pragma unroll
    for (int k = 0; k < kFewEvict; ++k) {
        gone_slot[k] = k < E ? ev[k] : L;
        lowest = min(lowest, gone_slot[k]);
    }
    for (int i = tid; i < L; i += kSelThreads) {
        int below = 0;
        bool gone = false;
#pragma unroll
        for (int k = 0; k < kFewEvict; ++k) {
            below += gone_slot[k] < i;
            gone |= gone_slot[k] == i;
        }
        if (!gone) ret[i - below] = i;
    }
    if (evicted && tid < E) {   // ascending: thread k writes the k-th pick at its rank
        const int mine = ev[tid];   // (ev is only read after the last barrier)
        int rank = 0;
#pragma unroll
        for (int k = 0; k < kFewEvict; ++k) rank += gone_slot[k] < mine;
        evicted[rank] = mine;
    }
    if (tid == 0) {
        *n_retained = B;
        if (first_moved) *first_moved = lowest;
    }
}

template <int CL>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectArgs a) {
    extern __shared__ uint32_t s_keys[];             // this CTA's chunk (if it fits)
    __shared__ uint32_t hist[kSelWarps][256];
    __shared__ uint32_t local[2][256];               // this CTA's histogram, double-buffered
    __shared__ uint32_t counts[2];                   // keys < T, keys == T in this chunk
    __shared__ int red[32];
    __shared__ uint32_t s_digit, s_rank;

    griddep_wait();
    griddep_release();
    const uint32_t rank = cta_rank();
    const int b = blockIdx.x / CL;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = a.n_units ? min(a.n_units[blockIdx.x / CL], a.L) : a.L;
    const int B = a.budgets ? a.budgets[b] : a.budget;
    const uint32_t* gkeys = a.keys + (size_t)b * a.max_ctx;
    int32_t* ret = a.retained + (size_t)b * (a.ret_ld ? a.ret_ld : a.budget);

    if (!a.refresh && rank == 0 && tid == 0) {
        // new token's score: mean of the old tokens' scores (block sums in order)
        float s = 0.f;
        for (int k = 0; k < a.n_part; ++k) s += a.msum_part[(size_t)b * a.n_part + k];
        a.m_s[(size_t)b * a.max_ctx + L - 1] = L > 1 ? s / (float)(L - 1) : 0.f;
    }
    if (B <= 0) {   // keep nothing (the same for every CTA: no exchange)
        if (rank == 0 && tid == 0) a.n_retained[b] = 0;
        return;
    }
    if (L <= B) {   // nothing to evict: identity (the same for every CTA: no exchange)
        if (rank == 0) {
            for (int i = tid; i < L; i += kSelThreads) ret[i] = i;
            if (tid == 0) {
                a.n_retained[b] = L;
                if (a.first_moved) a.first_moved[b] = L;
            }
        }
        return;
    }
    if (L - B <= kFewEvict) {   // the same for every CTA of the cluster: no exchange
        if (rank == 0)
            select_few(gkeys, L, B, ret, a.n_retained + b,
                       a.first_moved ? a.first_moved + b : nullptr,
                       a.evicted ? a.evicted + (size_t)b * kFewEvict : nullptr);
        return;
    }
    const int chunk = select_chunk(L, CL);
    const int c0 = min(L, (int)rank * chunk), c1 = min(L, c0 + chunk);
    const int n = c1 - c0;
    const bool staged = a.staged != 0;   // chunk <= the launch's chunk: it fits
    if (staged) {
        for (int i = tid; i < n; i += kSelThreads) s_keys[i] = __ldcg(gkeys + c0 + i);
    }
    const uint32_t* keys = staged ? s_keys : gkeys + c0;

    uint32_t prefix = 0, pmask = 0, want = (uint32_t)B;   // want: 1-based rank within candidates
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int k = tid; k < kSelWarps * 256; k += kSelThreads) (&hist[0][0])[k] = 0;
        __syncthreads();
        for (int i0 = 0; i0 < n; i0 += kSelThreads) {   // every lane runs every round
            const int i = i0 + tid;
            const uint32_t u = i < n ? keys[i] : 0u;
            const bool act = i < n && (u & pmask) == prefix;
            const uint32_t digit = (u >> shift) & 255u;
            // equal priorities are common (every token accessed this step has
            // 0): lanes sharing the first active lane's digit add once
            const unsigned am = __ballot_sync(0xffffffffu, act);
            if (!am) continue;
            const int leader = __ffs(am) - 1;
            const uint32_t d0 = __shfl_sync(0xffffffffu, digit, leader);
            const unsigned same = __ballot_sync(0xffffffffu, act && digit == d0);
            if (lane == leader) atomicAdd(&hist[warp][d0], (uint32_t)__popc(same));
            else if (act && digit != d0) atomicAdd(&hist[warp][digit], 1u);
        }
        __syncthreads();
        uint32_t* mine = local[pass & 1];
        if (tid < 256) {
            uint32_t t = 0;
            for (int w = 0; w < kSelWarps; ++w) t += hist[w][tid];
            mine[tid] = t;
        }
        cluster_sync();   // every CTA's histogram of this pass is complete
        if (warp < 8) {   // sum over the cluster, then scan the 256 bins
            uint32_t t = 0;
#pragma unroll
            for (uint32_t r = 0; r < CL; ++r) t += ld_remote(&mine[tid], r);
            uint32_t x = t;
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, x, m);
                if (lane >= m) x += y;
            }
            if (lane == 31) red[warp] = (int)x;
            asm volatile("bar.sync 1, 256;" ::: "memory");
            uint32_t base = 0;
            for (int w = 0; w < warp; ++w) base += (uint32_t)red[w];
            const uint32_t incl = base + x, excl = incl - t;
            if (excl < want && want <= incl) {
                s_digit = (uint32_t)tid;
                s_rank = want - excl;
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        pmask |= 255u << shift;
        want = s_rank;
        __syncthreads();
    }
    const uint32_t T = prefix;        // the B-th smallest key
    const int keep_eq = (int)want;    // keys equal to T kept, lowest slots first

    // per-thread contiguous sub-chunks (odd length: conflict-free shared reads)
    int sub = (n + kSelThreads - 1) / kSelThreads;
    sub |= 1;
    const int i0 = min(n, tid * sub), i1 = min(n, i0 + sub);
    int n_lt = 0, n_eq = 0;
    for (int i = i0; i < i1; ++i) {
        const uint32_t u = keys[i];
        n_lt += u < T;
        n_eq += u == T;
    }
    int cta_eq, cta_lt;
    const int eq_before_t = block_exclusive_scan(n_eq, red, &cta_eq);
    block_exclusive_scan(n_lt, red, &cta_lt);
    if (tid == 0) {
        counts[0] = (uint32_t)cta_lt;
        counts[1] = (uint32_t)cta_eq;
    }
    cluster_sync();   // every CTA's counts are published
    int eq_before_c = 0, out_before_c = 0;
    for (uint32_t r = 0; r < rank; ++r) {   // CTAs before this one, in slot order
        const int lt_r = (int)ld_remote(&counts[0], r);
        const int eq_r = (int)ld_remote(&counts[1], r);
        out_before_c += lt_r + max(0, min(eq_r, keep_eq - eq_before_c));
        eq_before_c += eq_r;
    }
    const int eq_before = eq_before_c + eq_before_t;
    const int my_keep = n_lt + max(0, min(n_eq, keep_eq - eq_before));
    int cta_kept;
    const int out0 = out_before_c + block_exclusive_scan(my_keep, red, &cta_kept);
    int o = out0, eqr = eq_before;
    // the thread whose slots hold the first one not kept, with every slot
    // before them kept, records it (exactly one such thread: L > B)
    bool all_before = out0 == c0 + i0;
    for (int i = i0; i < i1; ++i) {
        const uint32_t u = keys[i];
        bool keep = u < T;
        if (u == T) {
            keep = eqr < keep_eq;
            ++eqr;
        }
        if (keep) {
            ret[o++] = c0 + i;
        } else if (all_before) {
            if (a.first_moved) a.first_moved[b] = c0 + i;
            all_before = false;
        }
    }
    if (rank == CL - 1 && tid == 0) a.n_retained[b] = out_before_c + cta_kept;
    cluster_sync();   // no CTA leaves while another may still read its shared memory
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, int batch, int num_sms, cudaStream_t s) {
    // Many sequences whose keys fit one CTA's shared memory, or steps that
    // evict few tokens (the maxima path runs on one CTA): one CTA each (no
    // cluster barriers or remote reads).  Otherwise a cluster of kCl CTAs each.
    const bool one = a.few || (a.L <= kSelChunkCap && batch * kCl > num_sms);
    const int cl = one ? 1 : kCl;
    SelectArgs args = a;
    args.staged = select_stages_keys(a.L, cl) ? 1 : 0;
    const size_t smem = select_smem_bytes(a.L, cl);
    auto kern = one ? select_kernel<1> : select_kernel<kCl>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(uint32_t) * kSelChunkCap));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl * batch);
    cfg.blockDim = dim3(kSelThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace kvev
