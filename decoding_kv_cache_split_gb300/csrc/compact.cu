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
//
// Steps that evict few rows (at most kFewEvict: the steady state, one token
// in and one out) compact in place instead: only the rows at and after the
// first evicted slot move, each by the number of evicted slots below it.  One
// CTA walks one (K or V, layer, sequence, KV head) row of the cache upwards
// in chunks; slot j's source is never below j, so a chunk's stores land below
// the next chunk's sources, and the loads of chunk c + 1 are issued before the
// stores of chunk c.  A barrier after each chunk orders every load of the next
// chunk before any of its stores (another thread's store may hit a row this
// thread loaded).  The other ping-pong buffer is left as it is: its rows
// still equal the live ones below the first moved slot.
#include <climits>

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

constexpr int kInThreads = 256;
constexpr int kInUnroll = 4;

__global__ void __launch_bounds__(kInThreads, 4) compact_inplace_kernel(const CompactArgs a) {
    griddep_wait();
    griddep_release();
    const int nthreads = gridDim.x * gridDim.y * kInThreads;
    const int gtid = (blockIdx.y * gridDim.x + blockIdx.x) * kInThreads + threadIdx.x;
    // per-token state, gathered by every CTA's threads in turn
    for (int64_t e = gtid; e < (int64_t)a.batch * a.n_keep; e += nthreads) {
        const int bb = (int)(e / a.n_keep), j = (int)(e % a.n_keep);
        const int src = a.retained[(size_t)bb * a.budget + j];
        const size_t si = (size_t)bb * a.max_ctx + src, di = (size_t)bb * a.max_ctx + j;
        a.st.score[di] = a.m_s[si];
        a.st.t_ins[di] = a.tins_s[si];
        a.st.t_ref[di] = a.tref_s[si];
        a.st.pos[di] = a.pos_s[si];
    }
    if (gtid < a.batch && a.vp_out)   // the other buffer equals this one below both
        a.vp_out[gtid] = min(a.vp_in[gtid], a.first_moved[gtid]);

    const int r = blockIdx.x;                        // (layer, sequence, KV head)
    const int b = (r / a.n_kv) % a.batch;
    int f[kFewEvict];                                // e_i - i, ascending
#pragma unroll
    for (int i = 0; i < kFewEvict; ++i)
        f[i] = i < a.n_evict ? __ldg(a.evicted + (size_t)b * kFewEvict + i) - i : INT_MAX;
    const int lpr = a.head_dim / 8;
    const int rows_per_pass = kInThreads / lpr;
    const int chunk = rows_per_pass * kInUnroll;
    const int c = threadIdx.x % lpr, jr = threadIdx.x / lpr;
    uint4* rowp = reinterpret_cast<uint4*>(blockIdx.y == 0 ? a.k_dst : a.v_dst) +
                  (size_t)r * a.max_ctx * lpr;
    auto source = [&](int j) {
        int s = j;
#pragma unroll
        for (int i = 0; i < kFewEvict; ++i) s += f[i] <= j;
        return s;
    };
    uint4 cur[kInUnroll], nxt[kInUnroll] = {};
    auto load = [&](int j0, uint4* buf) {
#pragma unroll
        for (int u = 0; u < kInUnroll; ++u) {
            const int j = j0 + u * rows_per_pass + jr;
            if (j < a.n_keep) buf[u] = __ldcg(rowp + (size_t)source(j) * lpr + c);
        }
    };
    const int first = a.n_evict > 0 ? f[0] : a.n_keep;   // e_0: rows below stay
    load(first, cur);
    __syncthreads();
    for (int j0 = first; j0 < a.n_keep; j0 += chunk) {
        if (j0 + chunk < a.n_keep) load(j0 + chunk, nxt);
#pragma unroll
        for (int u = 0; u < kInUnroll; ++u) {
            const int j = j0 + u * rows_per_pass + jr;
            if (j < a.n_keep) __stcg(rowp + (size_t)j * lpr + c, cur[u]);
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kInUnroll; ++u) cur[u] = nxt[u];
    }
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
    if (a.in_place && !a.identity)
        return launch_pdl(compact_inplace_kernel, dim3(a.rows, 2), dim3(kInThreads), 0, s, a);
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
