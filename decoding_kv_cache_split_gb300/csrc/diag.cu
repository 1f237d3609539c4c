// Ranking diagnostics of the eviction pass, computed on the device from what
// the step already holds.
//
// "What Matters for Aggressive Decoding-Time KV Eviction?" Sec. 5.3 and
// Appendix I (Table 13) trace, per scoring step, the top-B set of the raw
// per-step score R_t (the attention summed over heads and layers, before any
// aggregation) against the retained set E_t: their Jaccard overlap, the
// churn of each between consecutive scoring steps, and the share of R_t
// evicted.  The scorer writes each token's raw score as a sortable key, the
// selection kernel picks R_t from it like the retained set (ties to the
// lower slot), and diag_kernel below counts the intersections exactly:
//   |R_t|, |E_t|, |R_t & E_t|, |R_t & R_prev| (tokens of the previous
//   scoring step's raw set still cached, tracked by a per-slot flag that
//   follows the compaction), |R_prev|, |E_t & E_(t-1)|.
// The host turns the counts into Jaccard indices and churn.
//
// missed_mass_kernel: the QEvict review's Future Missed Mass (Sec. 3): the
// share of a FullKV run's attention at a step that lands on positions a
// policy has already discarded, from the FullKV run's raw scores (by
// position) and the policy's cached positions.
#include "kvev_internal.h"

namespace kvev {
namespace {

constexpr int kDiagThreads = 1024;

// Deterministic block sum of one int per thread (warp shuffles, then the
// warps' totals in order).
__device__ __forceinline__ int block_sum(int v, int* red) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
    return t;
}

__device__ __forceinline__ float block_sum_f(float v, float* red) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
    return t;
}

__global__ void __launch_bounds__(kDiagThreads) diag_kernel(const DiagArgs a) {
    __shared__ int red[32];
    griddep_wait();
    griddep_release();
    const int b = blockIdx.x, tid = threadIdx.x;
    const int L = a.L;
    const int n_keep = a.n_retained[b];
    const int32_t* ret = a.retained + (size_t)b * a.budget;
    uint8_t* in_raw = a.in_raw + (size_t)b * a.max_ctx;
    const uint8_t* fin = a.flags_in + (size_t)b * a.max_ctx;
    uint8_t* fout = a.flags_out + (size_t)b * a.max_ctx;
    int n_raw = 0, c_re = 0, c_rr = 0;
    if (a.refresh) {
        for (int i = tid; i < L; i += kDiagThreads) in_raw[i] = 0;
        __syncthreads();
        n_raw = a.raw_n[b];
        for (int j = tid; j < n_raw; j += kDiagThreads) in_raw[a.raw_list[(size_t)b * a.budget + j]] = 1;
        __syncthreads();
        int x = 0;
        for (int j = tid; j < n_keep; j += kDiagThreads) x += in_raw[ret[j]];
        c_re = block_sum(x, red);
        x = 0;
        if (a.flags_valid)
            for (int i = tid; i < L - 1; i += kDiagThreads) x += in_raw[i] & fin[i];
        c_rr = block_sum(x, red);
    }
    // the flags of the cache after this step's compaction: in the raw set of
    // this scoring step, or carried from the last one (the new token: 0)
    for (int j = tid; j < n_keep; j += kDiagThreads) {
        const int s = ret[j];
        fout[j] = a.refresh ? in_raw[s] : (a.flags_valid && s < L - 1 ? fin[s] : 0);
    }
    if (tid == 0) {
        const int new_kept = n_keep > 0 && ret[n_keep - 1] == L - 1;
        int32_t* c = a.counters + (size_t)b * KVEV_DIAG_FIELDS;
        c[0] = a.t;
        c[1] = a.refresh;
        c[2] = n_raw;
        c[3] = n_keep;
        c[4] = c_re;
        c[5] = c_rr;
        c[6] = a.refresh && a.flags_valid ? a.prev_n[b] : 0;
        c[7] = n_keep - new_kept;
        if (a.refresh) a.prev_n[b] = n_raw;
    }
}

__global__ void __launch_bounds__(kDiagThreads) missed_mass_kernel(const MissedMassArgs a) {
    __shared__ float red[32];
    const int b = blockIdx.x, tid = threadIdx.x;
    const float* fs = a.full_score + (size_t)b * a.score_ld;
    const int32_t* pos = a.pos + (size_t)b * a.pos_ld;
    float tot = 0.f, held = 0.f;
    for (int p = tid; p < a.n_pos; p += kDiagThreads) tot += fs[p];
    for (int j = tid; j < a.n_cached; j += kDiagThreads) {
        const int p = pos[j];
        if (p >= 0 && p < a.n_pos - 1) held += fs[p];
    }
    tot = block_sum_f(tot, red);
    held = block_sum_f(held, red);
    if (tid == 0) a.out[b] = 1.0f - (held + fs[a.n_pos - 1]) / tot;
}

}  // namespace

cudaError_t launch_diag(const DiagArgs& a, int batch, cudaStream_t s) {
    return launch_pdl(diag_kernel, dim3(batch), dim3(kDiagThreads), 0, s, a);
}

cudaError_t launch_missed_mass(const MissedMassArgs& a, int batch, cudaStream_t s) {
    missed_mass_kernel<<<batch, kDiagThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kvev
