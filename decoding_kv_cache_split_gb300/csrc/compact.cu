// Cache maintenance kernels: append of the new token, prefill state, and
// the stable gather-compaction of the retained K/V rows and state.
//
// Compaction: retained slot retained[b][j] (ascending) moves to slot j, in
// every layer and KV head, out of place into the other ping-pong buffer, so
// no row is overwritten before it is read.  That buffer still holds the
// live rows below the first slot the previous compaction moved; rows below
// the smaller of that and this step's first moved slot are not copied again.
// One CTA moves a chunk of retained rows of one (K or V, layer, sequence,
// KV head) row of the cache with 16-byte loads and stores; a warp covers
// 32/(D/8) rows per instruction.
// The per-token state (score, clocks, position) is gathered from the
// scoring kernel's scratch copy by the CTAs of the first cache row.
#include "kvev_internal.h"

namespace kvev {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) compact_kernel(const CompactArgs a) {
    griddep_wait();
    griddep_release();
    const int lpr = a.head_dim / 8;                 // 16-byte units per row
    const int rows_per_pass = kCopyThreads / lpr;
    const int chunk = rows_per_pass * kCopyUnroll;  // retained rows per CTA
    const int j0 = blockIdx.x * chunk;
    const int r = blockIdx.y;                        // (layer, sequence, KV head)
    const int b = (r / a.n_kv) % a.batch;
    const int32_t* idx = a.retained + (size_t)b * a.budget;

    if (r == 0 && blockIdx.z == 0) {
        if (blockIdx.x == 0 && a.vp_out)   // next step's reused prefix
            for (int bb = threadIdx.x; bb < a.batch; bb += kCopyThreads)
                a.vp_out[bb] = a.identity ? a.vp_in[bb] : a.first_moved[bb];
        for (int e = threadIdx.x; e < chunk * a.batch; e += kCopyThreads) {
            const int j = j0 + e % chunk, bb = e / chunk;
            if (j >= a.n_keep) continue;
            const int src = a.identity ? j : a.retained[(size_t)bb * a.budget + j];
            const size_t si = (size_t)bb * a.max_ctx + src, di = (size_t)bb * a.max_ctx + j;
            a.st.score[di] = a.m_s[si];
            a.st.t_ins[di] = a.tins_s[si];
            a.st.t_ref[di] = a.tref_s[si];
            a.st.pos[di] = a.pos_s[si];
        }
    }
    if (a.identity) return;
    // rows the destination already holds (identity below first_moved)
    const int skip = a.vp_in ? min(a.vp_in[b], a.first_moved[b]) : 0;
    if (j0 + chunk <= skip) return;

    const uint4* src = reinterpret_cast<const uint4*>(blockIdx.z == 0 ? a.k_src : a.v_src) +
                       (size_t)r * a.max_ctx * lpr;
    uint4* dst = reinterpret_cast<uint4*>(blockIdx.z == 0 ? a.k_dst : a.v_dst) +
                 (size_t)r * a.max_ctx * lpr;
    const int c = threadIdx.x % lpr, jr = threadIdx.x / lpr;
    uint4 buf[kCopyUnroll];
    int jj[kCopyUnroll], from[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {       // every index load in flight first
        const int j = j0 + u * rows_per_pass + jr;
        jj[u] = j;
        from[u] = j < a.n_keep ? __ldg(idx + j) : 0;
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
        if (jj[u] < a.n_keep && jj[u] >= skip) buf[u] = __ldcs(src + (size_t)from[u] * lpr + c);
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
        if (jj[u] < a.n_keep && jj[u] >= skip) __stcs(dst + (size_t)jj[u] * lpr + c, buf[u]);
}

__global__ void append_kernel(const AppendArgs a) {
    // one CTA per (layer, sequence, KV head) row; threads copy 16-byte units
    griddep_wait();
    griddep_release();
    const int r = blockIdx.x;
    const int g = r % a.n_kv, lb = r / a.n_kv;
    const int b = lb % a.batch, l = lb / a.batch;
    const int lpr = a.head_dim / 8;
    const size_t src = (((size_t)b * a.n_layers + l) * a.n_kv + g) * lpr;
    const size_t dst = ((size_t)r * a.max_ctx + a.slot) * lpr;
    for (int u = threadIdx.x; u < 2 * lpr; u += blockDim.x) {
        const bool is_v = u >= lpr;
        const int c = is_v ? u - lpr : u;
        const uint4 w = reinterpret_cast<const uint4*>(is_v ? a.v_new : a.k_new)[src + c];
        reinterpret_cast<uint4*>(is_v ? a.v : a.k)[dst + c] = w;
    }
    if (l == 0 && g == 0 && threadIdx.x == 0) {
        const size_t si = (size_t)b * a.max_ctx + a.slot;
        a.st.score[si] = 0.f;   // momentum starts at 0; refreshed below or set to the mean
        a.st.t_ins[si] = a.t;
        a.st.t_ref[si] = a.t;   // insertion counts as an access
        a.st.pos[si] = a.pos;
    }
}

__global__ void init_state_kernel(kvev_state st, int batch, int max_ctx, int len, int32_t* vp) {
    griddep_wait();
    griddep_release();
    if (vp && blockIdx.x == 0)   // no reused rows yet
        for (int i = threadIdx.x; i < 2 * batch; i += blockDim.x) vp[i] = 0;
    const int64_t n = (int64_t)batch * len;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(e / len), i = (int)(e % len);
        const size_t si = (size_t)b * max_ctx + i;
        st.score[si] = 0.f;
        st.t_ins[si] = 0;
        st.t_ref[si] = 0;
        st.pos[si] = i;
    }
}

}  // namespace

cudaError_t launch_compact(const CompactArgs& a, int num_sms, cudaStream_t s) {
    (void)num_sms;
    const int lpr = a.head_dim / 8;
    const int chunk = (kCopyThreads / lpr) * kCopyUnroll;
    const dim3 grid((a.n_keep + chunk - 1) / chunk, a.identity ? 1 : a.rows, a.identity ? 1 : 2);
    return launch_pdl(compact_kernel, grid, dim3(kCopyThreads), 0, s, a);
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
    const int rows = a.n_layers * a.batch * a.n_kv;
    return launch_pdl(append_kernel, dim3(rows), dim3(32), 0, s, a);
}

cudaError_t launch_init_state(kvev_state st, int batch, int max_ctx, int len, int32_t* vp,
                              cudaStream_t s) {
    if (batch == 0 || (len == 0 && !vp)) return cudaSuccess;
    const int64_t n = (int64_t)batch * len;
    int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    if (blocks < 1) blocks = 1;
    return launch_pdl(init_state_kernel, dim3(blocks), dim3(256), 0, s, st, batch, max_ctx, len,
                      vp);
}

}  // namespace kvev
