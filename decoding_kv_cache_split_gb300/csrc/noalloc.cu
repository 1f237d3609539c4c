// kvev_attend_noalloc: the split-K attention of the eviction pass for
// callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: engines that hand all
// of the GPU's memory to their own allocator up front and forbid any other
// allocation, and latency-critical paths that cannot afford the implicit
// device synchronisation of cudaMalloc/cudaFree.  This entry point runs the
// same attention and split-combine kernels as kvev_step, but keeps the
// softmax partials of the split in a fixed-size array in device global
// memory that is part of the library image (kScratchBytes below), so it
// creates no context and allocates nothing.
//
// Set-up: the first call on each device, with that device current, looks up
// the array's device address with cudaGetSymbolAddress (host code cannot use
// the array's name as a device pointer).  Make that first call before any
// stream capture.
//
// Sharing: every call on a device uses the same array, which keeps the last
// call's contents.  Calls whose work overlaps on the GPU (different streams,
// or different host threads) race on it and give undefined results; order
// them on one stream.  The status word is cleared at the start of every call.
//
// A bounded device wait that gives up is not returned as a status (nothing
// reads the status word back, which would synchronise the stream): the warp
// that gave up writes NaN as the running max of its split slots, so the
// rows it touched come out NaN in `out` and `lse2` rather than merged from
// stale partials.
//
// The address looked up at set-up belongs to the device's current CUDA
// context: after cudaDeviceReset (or any teardown of the primary context)
// the library image is loaded again and the cached address is stale, so do
// not call this entry point after a reset in the same process.
#include <math.h>
#include <stdio.h>

#include <mutex>

#include "kvev_internal.h"

namespace kvev {
kvev_status report_error(kvev_status st, const char* msg);
int attn_warps_per_cta();
}  // namespace kvev

using namespace kvev;

namespace {

// 16 MiB: every GPU that loads the library holds this until the process exits.
constexpr size_t kScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once).
cudaError_t scratch_address(int dev, unsigned char** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *out = static_cast<unsigned char*>(g_addr[dev]);
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" kvev_status kvev_attend_noalloc(const kvev_layout* L, const void* q, const void* k,
                                           const void* v, int32_t len, float* out, float* lse2,
                                           void* stream) {
    if (!L || !q || !k || !v || !out || !lse2)
        return report_error(KVEV_EINVAL, "kvev_attend_noalloc: NULL argument");
    if (L->n_layers < 1 || L->batch < 1 || L->n_kv_heads < 1 || L->n_q_heads < 1 ||
        L->n_q_heads % L->n_kv_heads != 0)
        return report_error(KVEV_EINVAL, "kvev_attend_noalloc: bad head/layer/batch counts");
    const int G = L->n_q_heads / L->n_kv_heads;
    if ((L->head_dim != 64 && L->head_dim != 128) || (G != 4 && G != 8))
        return report_error(KVEV_EUNSUPPORTED,
                            "kvev_attend_noalloc: supports head_dim 64/128 with 4 or 8 query heads "
                            "per KV head");
    if (len < 1 || len > L->max_ctx)
        return report_error(KVEV_EINVAL, "kvev_attend_noalloc: len must be in [1, max_ctx]");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return report_error(KVEV_EINVAL, "kvev_attend_noalloc: q, k, v, out must be 16-byte aligned");

    // scratch: status word (256 B), then (warps + rows) softmax partial slots
    const int64_t rows = (int64_t)L->n_layers * L->batch * L->n_kv_heads;
    const size_t slot_bytes = (size_t)G * (L->head_dim + 2) * sizeof(float);
    const int64_t slot_cap = (int64_t)((kScratchBytes - 256) / slot_bytes);
    const int wpc = attn_warps_per_cta();
    if (rows + wpc > slot_cap) {
        char msg[192];
        snprintf(msg, sizeof msg,
                 "kvev_attend_noalloc: n_layers*batch*n_kv_heads = %lld exceeds %lld, the most "
                 "the 16 MiB static scratch holds at head_dim %d",
                 (long long)rows, (long long)(slot_cap - wpc), L->head_dim);
        return report_error(KVEV_EINVAL, msg);
    }

    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && (dev < 0 || dev >= kMaxDevices)) e = cudaErrorInvalidDevice;
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    unsigned char* base = nullptr;
    if (e == cudaSuccess) e = scratch_address(dev, &base);
    if (e != cudaSuccess) return report_error(KVEV_ECUDA, cudaGetErrorString(e));

    const int per_sm = attn_ctas_per_sm(L->head_dim, G);
    int64_t grid = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
    const int64_t grid_fit = (slot_cap - rows) / wpc;   // CTAs whose partials fit
    if (grid > grid_fit) grid = grid_fit;
    // one warp per 4 tiles at most, as kvev_step launches it (the same split,
    // so the same output bit for bit)
    const int tiles_per_row = (len + kTile - 1) / kTile;
    const int64_t n_tiles = rows * tiles_per_row;
    const int64_t want = (n_tiles + 3) / 4;
    const int64_t warps = want < grid * wpc ? (want > 0 ? want : 1) : grid * wpc;
    grid = (warps + wpc - 1) / wpc;

    cudaStream_t s = (cudaStream_t)stream;
    uint32_t* status = reinterpret_cast<uint32_t*>(base);
    float* part_ml = reinterpret_cast<float*>(base + 256);
    const int64_t slots = warps + rows;
    float* part_o = part_ml + slots * G * 2;
    e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return report_error(KVEV_ECUDA, cudaGetErrorString(e));

    AttnArgs at{};
    at.k = (const uint16_t*)k;
    at.v = (const uint16_t*)v;
    at.q = (const uint16_t*)q;
    at.logits = nullptr;
    at.part_o = part_o;
    at.part_ml = part_ml;
    at.status = status;
    at.n_tiles_total = n_tiles;
    at.tiles_per_row = tiles_per_row;
    at.L = len;
    at.max_ctx = L->max_ctx;
    at.n_layers = L->n_layers;
    at.batch = L->batch;
    at.n_kv = L->n_kv_heads;
    at.n_q = L->n_q_heads;
    at.total_warps = (int32_t)warps;
    at.write_logits = 0;
    at.q_scale = (float)(1.4426950408889634 / sqrt((double)L->head_dim));
    at.view_tokens = rows * L->max_ctx;
    e = launch_attention(at, L->head_dim, G, (int)grid, s);
    if (e != cudaSuccess) return report_error(KVEV_ECUDA, cudaGetErrorString(e));

    CombineArgs cb{};
    cb.sp.part_o = part_o;
    cb.sp.part_ml = part_ml;
    cb.sp.n_tiles = at.n_tiles_total;
    cb.sp.row0 = 0;
    cb.sp.total_warps = at.total_warps;
    cb.sp.tiles_per_row = tiles_per_row;
    cb.n_rows = (int32_t)rows;
    cb.out = out;
    cb.lse2 = lse2;
    cb.n_layers = L->n_layers;
    cb.batch = L->batch;
    cb.n_kv = L->n_kv_heads;
    cb.n_q = L->n_q_heads;
    e = launch_combine(cb, L->head_dim, G, s);
    if (e != cudaSuccess) return report_error(KVEV_ECUDA, cudaGetErrorString(e));
    return KVEV_OK;
}
