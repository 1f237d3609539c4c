// Budgeted selection: keep the B tokens of lowest eviction priority, ties
// to the lower slot index, and list them in ascending slot order.
//
// "What Matters for Aggressive Decoding-Time KV Eviction?" Sec. 3.1: whenever
// the cache exceeds B, the lowest-utility tokens are evicted; with the LRFU
// priority of the kv-cache-docs "ema-eviction" figure a higher priority is
// evicted, so the B lowest priorities are retained.
//
// One CTA per sequence.  The keys are the order-preserving bits of the fp32
// priorities; a 4-pass radix select (8-bit digits, per-warp shared-memory
// histograms) finds the B-th smallest key T and how many keys equal to T
// are kept; a final pass over contiguous per-thread chunks, with two block
// scans, emits the kept slots in ascending order.  When the sequence's keys
// fit in shared memory they are staged there on the first pass.
#include "kvev_internal.h"

namespace kvev {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSmemKeyCap = 40960;   // keys staged in shared memory up to this length

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

__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectArgs a) {
    extern __shared__ uint32_t s_keys[];
    __shared__ uint32_t hist[kSelWarps][256];
    __shared__ uint32_t tot[256];
    __shared__ int red[32];
    __shared__ uint32_t s_digit, s_rank;

    griddep_wait();
    griddep_release();
    const int b = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    (void)lane;
    const int L = a.L, B = a.budget;
    const uint32_t* gkeys = a.keys + (size_t)b * a.max_ctx;
    int32_t* ret = a.retained + (size_t)b * B;

    if (!a.refresh && tid == 0) {
        // new token's score: mean of the old tokens' scores (block sums in order)
        float s = 0.f;
        for (int k = 0; k < a.n_part; ++k) s += a.msum_part[(size_t)b * a.n_part + k];
        a.m_s[(size_t)b * a.max_ctx + L - 1] = L > 1 ? s / (float)(L - 1) : 0.f;
    }
    if (L <= B) {
        for (int i = tid; i < L; i += kSelThreads) ret[i] = i;
        if (tid == 0) a.n_retained[b] = L;
        return;
    }
    const bool staged = L <= kSmemKeyCap;
    if (staged) {   // stage the keys: a batch of loads in flight per thread
        constexpr int kBatch = 8;
        for (int i0 = 0; i0 < L; i0 += kSelThreads * kBatch) {
            uint32_t v[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int i = i0 + k * kSelThreads + tid;
                v[k] = i < L ? __ldcg(gkeys + i) : 0u;
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int i = i0 + k * kSelThreads + tid;
                if (i < L) s_keys[i] = v[k];
            }
        }
    }
    const uint32_t* keys = staged ? s_keys : gkeys;

    uint32_t prefix = 0, pmask = 0, rank = (uint32_t)B;   // rank: 1-based within candidates
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int k = tid; k < kSelWarps * 256; k += kSelThreads) (&hist[0][0])[k] = 0;
        __syncthreads();
        for (int i0 = 0; i0 < L; i0 += kSelThreads) {   // every lane runs every round
            const int i = i0 + tid;
            const uint32_t u = i < L ? keys[i] : 0u;
            const bool act = i < L && (u & pmask) == prefix;
            const uint32_t digit = (u >> shift) & 255u;
            // Equal priorities are common (e.g. every accessed token has 0): the
            // lanes sharing the first active lane's digit add with one atomic.
            const unsigned am = __ballot_sync(0xffffffffu, act);
            if (!am) continue;
            const int leader = __ffs(am) - 1;
            const uint32_t d0 = __shfl_sync(0xffffffffu, digit, leader);
            const unsigned same = __ballot_sync(0xffffffffu, act && digit == d0);
            if (lane == leader) atomicAdd(&hist[warp][d0], (uint32_t)__popc(same));
            else if (act && digit != d0) atomicAdd(&hist[warp][digit], 1u);
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t t = 0;
            for (int w = 0; w < kSelWarps; ++w) t += hist[w][tid];
            tot[tid] = t;
        }
        __syncthreads();
        if (warp < 8) {   // exclusive scan of the 256 bins by 8 warps
            const int lane = tid & 31;
            uint32_t x = tot[tid];
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, x, m);
                if (lane >= m) x += y;
            }
            if (lane == 31) red[warp] = (int)x;
            __syncwarp();
            asm volatile("bar.sync 1, 256;" ::: "memory");
            uint32_t base = 0;
            for (int w = 0; w < warp; ++w) base += (uint32_t)red[w];
            const uint32_t incl = base + x, excl = incl - tot[tid];
            if (excl < rank && rank <= incl) {
                s_digit = (uint32_t)tid;
                s_rank = rank - excl;
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        pmask |= 255u << shift;
        rank = s_rank;
        __syncthreads();
    }
    const uint32_t T = prefix;        // the B-th smallest key
    const int keep_eq = (int)rank;    // keys equal to T kept, lowest slots first

    // contiguous chunks; an odd chunk length keeps shared-memory reads conflict-free
    int chunk = (L + kSelThreads - 1) / kSelThreads;
    chunk |= 1;
    const int i0 = min(L, tid * chunk), i1 = min(L, i0 + chunk);
    int n_lt = 0, n_eq = 0;
    for (int i = i0; i < i1; ++i) {
        const uint32_t u = keys[i];
        n_lt += u < T;
        n_eq += u == T;
    }
    int total;
    const int eq_before = block_exclusive_scan(n_eq, red, &total);
    const int my_eq_keep = max(0, min(n_eq, keep_eq - eq_before));
    const int out0 = block_exclusive_scan(n_lt + my_eq_keep, red, &total);
    int o = out0, eqr = eq_before;
    for (int i = i0; i < i1; ++i) {
        const uint32_t u = keys[i];
        bool keep = u < T;
        if (u == T) {
            keep = eqr < keep_eq;
            ++eqr;
        }
        if (keep) ret[o++] = i;
    }
    if (tid == 0) a.n_retained[b] = total;
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, int batch, cudaStream_t s) {
    const size_t smem = a.L <= kSmemKeyCap ? sizeof(uint32_t) * (size_t)a.L : 0;
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(uint32_t) * kSmemKeyCap));
    if (e != cudaSuccess) return e;
    return launch_pdl(select_kernel, dim3(batch), dim3(kSelThreads), smem, s, a);
}

}  // namespace kvev
