// C ABI of the eviction pass: argument checking, scratch ownership and the
// per-step launch sequence (append -> attention -> combine -> score ->
// select -> compact) on the caller's stream.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "kvev_internal.h"

namespace kvev {
int attn_warps_per_cta();
}

using namespace kvev;

namespace {

thread_local char g_err[512] = "no error";

kvev_status fail(kvev_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

kvev_status cuda_fail(cudaError_t e, const char* what) {
    return fail(KVEV_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// token stride of a logits row: whole 128-byte lines per row
int logit_ld(int max_ctx) { return (max_ctx + 7) / 8 * 8; }

enum {
    kProfAppend = 0, kProfAttn, kProfCombine, kProfScore, kProfSelect, kProfCompact, kProfInit,
    kProfReadmit
};

// An NVTX range around each step-level call (free when no tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

struct Workspace {
    float* logits = nullptr;
    float* part_o = nullptr;
    float* part_ml = nullptr;
    float* lse2 = nullptr;
    uint32_t* keys = nullptr;
    float* m_s = nullptr;
    int32_t* tref_s = nullptr;
    int32_t* tins_s = nullptr;
    int32_t* pos_s = nullptr;
    float* msum_part = nullptr;
    uint32_t* status = nullptr;
    uint32_t* gbar = nullptr;         // [2] grid barrier of the fused step (zero at rest)
    uint16_t* stg_q = nullptr;
    uint16_t* stg_k = nullptr;
    uint16_t* stg_v = nullptr;
    float* stg_out = nullptr;
    int32_t* stg_ret = nullptr;
    int32_t* stg_nret = nullptr;
    // block-granular mode: scratch copies of the block state, [batch][pps]
    int32_t* lid_s = nullptr;
    int32_t* len_s = nullptr;
    int32_t* page_s = nullptr;
    int32_t* tokens = nullptr;        // [batch] live tokens after the append
    int32_t* sel = nullptr;           // [batch][units] kept block slots
    int32_t* budgets = nullptr;       // [batch] blocks kept (region-aware selection)
    int32_t* readmit_page = nullptr;  // [1]
    int32_t* first_moved = nullptr;   // [batch] first slot not kept this step
    int32_t* vp = nullptr;            // [2][batch] reused-prefix rows, by step parity
    int32_t* evicted = nullptr;       // [batch][kFewEvict] slots a few-eviction step drops
    // two-tier mode (page_tokens = window)
    int32_t* t_bt = nullptr;          // [batch][bt_ld] attention block list
    int32_t* t_bpos = nullptr;
    int32_t* t_blen = nullptr;
    int32_t* t_nblk = nullptr;        // [batch]
    int32_t* t_qlist = nullptr;       // [batch][max_windows]
    int32_t* t_nq = nullptr;
    int32_t* t_seq_len = nullptr;
    int32_t* t_quant = nullptr;       // [batch][max_windows] routing lists + counts
    int32_t* t_nquant = nullptr;
    int32_t* t_prom = nullptr;
    int32_t* t_nprom = nullptr;
    int32_t* t_free = nullptr;
    int32_t* t_nfree = nullptr;
    float2* t_stats = nullptr;        // [rows][stats_tiles][G]
    float* part_o2 = nullptr;         // INT2 attention partials
    float* part_ml2 = nullptr;
    int32_t* lir_streak = nullptr;    // [batch][max_windows] Global LIR streaks
    int32_t* t_rslot = nullptr;       // rotary mode: [batch][max_windows] reconstruction slots,
    int32_t* t_rfree = nullptr;       // free-slot stacks and the windows to reconstruct
    int32_t* t_nrfree = nullptr;
    int32_t* t_rlist = nullptr;
    int32_t* t_nrlist = nullptr;
    // token mode, scorer weightings (VNorm, entropy)
    float* part_e = nullptr;          // [slots][G]
    float* part_vn = nullptr;         // [slots]
    float* vnorm = nullptr;           // [rows][logit_ld]
    float* ent = nullptr;             // [rows][G]
    float* vmean = nullptr;           // [rows]
    // token mode, ranking diagnostics
    uint32_t* raw_keys = nullptr;     // [batch][max_ctx]
    int32_t* raw_list = nullptr;      // [batch][budget]
    int32_t* raw_n = nullptr;         // [batch]
    uint8_t* in_raw = nullptr;        // [batch][max_ctx]
    uint8_t* raw_flags = nullptr;     // [2][batch][max_ctx], by step parity
    int32_t* raw_prev_n = nullptr;    // [batch]
    size_t bytes = 0;
    // a guard band of kGuardBytes follows every region: its offset and the
    // region's name (checked by kvev_check_scratch)
    static constexpr int kMaxRegions = 64;
    size_t guard_off[kMaxRegions] = {};
    const char* guard_name[kMaxRegions] = {};
    int n_guard = 0;
};
constexpr size_t kGuardBytes = 256;
constexpr unsigned char kGuardByte = 0xA5;

// Lays out (or, with base == nullptr, only sizes) the context's scratch.
int tier_max_windows(const kvev_layout& L) { return (L.max_ctx - kTierSinks) / kTierW; }
int tier_bt_ld(const kvev_layout& L) { return tier_max_windows(L) * (kTierW / kTile) + 10; }
int tier_stats_tiles(const kvev_layout& L) { return tier_max_windows(L) * (kTierW / kTile) + 8; }

// slots2: softmax partial slots of the INT2 attention (two-tier mode only).
Workspace carve(const kvev_layout& L, int64_t budget, int64_t slots, char* base,
                int64_t slots2 = 0) {
    Workspace w;
    size_t off = 0;
    auto take = [&](size_t bytes, const char* name) -> char* {
        char* p = base ? base + off : nullptr;
        off += align_up(bytes, 256);
        if (w.n_guard < Workspace::kMaxRegions) {
            w.guard_off[w.n_guard] = off;
            w.guard_name[w.n_guard++] = name;
        }
        off += kGuardBytes;
        return p;
    };
    const size_t rows = (size_t)L.n_layers * L.batch * L.n_kv_heads;
    const size_t G = (size_t)(L.n_q_heads / L.n_kv_heads);
    const size_t ctx = (size_t)L.batch * L.max_ctx;
    const size_t nblk = (size_t)((L.max_ctx + kScoreThreads - 1) / kScoreThreads);
    // two-tier mode scores windows from per-tile statistics: no logits
    if (L.page_tokens != kTierW)
        w.logits = (float*)take(rows * (size_t)logit_ld(L.max_ctx) * G * 4, "logits");
    w.part_o = (float*)take((size_t)slots * G * L.head_dim * 4, "part_o");
    w.part_ml = (float*)take((size_t)slots * G * 2 * 4, "part_ml");
    w.lse2 = (float*)take(rows * G * 4, "lse2");
    w.keys = (uint32_t*)take(ctx * 4, "keys");
    w.m_s = (float*)take(ctx * 4, "m_s");
    w.tref_s = (int32_t*)take(ctx * 4, "tref_s");
    w.tins_s = (int32_t*)take(ctx * 4, "tins_s");
    w.pos_s = (int32_t*)take(ctx * 4, "pos_s");
    w.msum_part = (float*)take((size_t)L.batch * nblk * 4, "msum_part");
    w.status = (uint32_t*)take(4, "status");
    w.gbar = (uint32_t*)take(8, "gbar");
    const size_t qn = (size_t)L.batch * L.n_layers * L.n_q_heads * L.head_dim;
    const size_t kn = (size_t)L.batch * L.n_layers * L.n_kv_heads * L.head_dim;
    w.stg_q = (uint16_t*)take(qn * 2, "stg_q");
    w.stg_k = (uint16_t*)take(kn * 2, "stg_k");
    w.stg_v = (uint16_t*)take(kn * 2, "stg_v");
    w.stg_out = (float*)take(qn * 4, "stg_out");
    w.stg_ret = (int32_t*)take((size_t)L.batch * budget * 4, "stg_ret");
    w.stg_nret = (int32_t*)take((size_t)L.batch * 4, "stg_nret");
    const size_t units = (size_t)L.batch * (L.max_ctx / L.page_tokens);
    w.lid_s = (int32_t*)take(units * 4, "lid_s");
    w.len_s = (int32_t*)take(units * 4, "len_s");
    w.page_s = (int32_t*)take(units * 4, "page_s");
    w.tokens = (int32_t*)take((size_t)L.batch * 4, "tokens");
    w.sel = (int32_t*)take(units * 4, "sel");
    w.budgets = (int32_t*)take((size_t)L.batch * 4, "budgets");
    w.readmit_page = (int32_t*)take(4, "readmit_page");
    w.first_moved = (int32_t*)take((size_t)L.batch * 4, "first_moved");
    w.vp = (int32_t*)take((size_t)L.batch * 8, "vp");
    w.evicted = (int32_t*)take((size_t)L.batch * kFewEvict * 4, "evicted");
    if (L.page_tokens == 1) {
        w.part_e = (float*)take((size_t)slots * G * 4, "part_e");
        w.part_vn = (float*)take((size_t)slots * 4, "part_vn");
        w.vnorm = (float*)take(rows * (size_t)logit_ld(L.max_ctx) * 4, "vnorm");
        w.ent = (float*)take(rows * G * 4, "ent");
        w.vmean = (float*)take(rows * 4, "vmean");
        w.raw_keys = (uint32_t*)take(ctx * 4, "raw_keys");
        w.raw_list = (int32_t*)take((size_t)L.batch * budget * 4, "raw_list");
        w.raw_n = (int32_t*)take((size_t)L.batch * 4, "raw_n");
        w.in_raw = (uint8_t*)take(ctx, "in_raw");
        w.raw_flags = (uint8_t*)take(2 * ctx, "raw_flags");
        w.raw_prev_n = (int32_t*)take((size_t)L.batch * 4, "raw_prev_n");
    }
    if (L.page_tokens == kTierW) {
        const size_t B = (size_t)L.batch, MW = (size_t)tier_max_windows(L);
        const size_t bt = B * tier_bt_ld(L);
        w.t_bt = (int32_t*)take(bt * 4, "t_bt");
        w.t_bpos = (int32_t*)take(bt * 4, "t_bpos");
        w.t_blen = (int32_t*)take(bt * 4, "t_blen");
        w.t_nblk = (int32_t*)take(B * 4, "t_nblk");
        w.t_qlist = (int32_t*)take(B * MW * 4, "t_qlist");
        w.t_nq = (int32_t*)take(B * 4, "t_nq");
        w.t_seq_len = (int32_t*)take(B * 4, "t_seq_len");
        w.t_quant = (int32_t*)take(B * MW * 4, "t_quant");
        w.t_nquant = (int32_t*)take(B * 4, "t_nquant");
        w.t_prom = (int32_t*)take(B * MW * 4, "t_prom");
        w.t_nprom = (int32_t*)take(B * 4, "t_nprom");
        w.t_free = (int32_t*)take(B * MW * 4, "t_free");
        w.t_nfree = (int32_t*)take(B * 4, "t_nfree");
        w.t_stats = (float2*)take(rows * (size_t)tier_stats_tiles(L) * G * sizeof(float2), "t_stats");
        w.part_o2 = (float*)take((size_t)slots2 * G * L.head_dim * 4, "part_o2");
        w.part_ml2 = (float*)take((size_t)slots2 * G * 2 * 4, "part_ml2");
        w.lir_streak = (int32_t*)take(B * MW * 4, "lir_streak");
        w.t_rslot = (int32_t*)take(B * MW * 4, "t_rslot");
        w.t_rfree = (int32_t*)take(B * MW * 4, "t_rfree");
        w.t_nrfree = (int32_t*)take(B * 4, "t_nrfree");
        w.t_rlist = (int32_t*)take(B * MW * 4, "t_rlist");
        w.t_nrlist = (int32_t*)take(B * 4, "t_nrlist");
    }
    w.bytes = off;
    return w;
}

// budget_tokens: the budget counts tokens even at block granularity
// (region-aware MemDecay selection).
kvev_status check_layout(const kvev_layout* L, int64_t budget, bool budget_tokens = false) {
    if (!L) return fail(KVEV_EINVAL, "layout is NULL");
    if (L->n_layers < 1 || L->n_q_heads < 1 || L->n_kv_heads < 1 || L->batch < 1)
        return fail(KVEV_EINVAL, "layout: n_layers, n_q_heads, n_kv_heads, batch must be >= 1");
    if (L->n_q_heads % L->n_kv_heads != 0)
        return fail(KVEV_EINVAL, "layout: n_q_heads (%d) must be a multiple of n_kv_heads (%d)",
                    L->n_q_heads, L->n_kv_heads);
    if (L->head_dim != 64 && L->head_dim != 128)
        return fail(KVEV_EUNSUPPORTED, "layout: head_dim %d (supported: 64, 128)", L->head_dim);
    if (L->n_q_heads / L->n_kv_heads != 4 && L->n_q_heads / L->n_kv_heads != 8)
        return fail(KVEV_EUNSUPPORTED, "layout: query heads per KV head %d (supported: 4, 8)",
                    L->n_q_heads / L->n_kv_heads);
    if (L->max_ctx < 2) return fail(KVEV_EINVAL, "layout: max_ctx must be >= 2");
    if (L->page_tokens != 1 && L->page_tokens != kTile && L->page_tokens != kTierW)
        return fail(KVEV_EUNSUPPORTED, "layout: page_tokens %d (supported: 1, %d, %d)",
                    L->page_tokens, kTile, kTierW);
    if (L->kv_dtype != KVEV_BF16) return fail(KVEV_EUNSUPPORTED, "layout: kv_dtype must be BF16");
    if (L->page_tokens == kTierW) {   // two-tier windows: budget = K_f windows
        if (L->head_dim != 128 || L->n_q_heads / L->n_kv_heads != 4)
            return fail(KVEV_EUNSUPPORTED, "two-tier windows: head_dim 128 and 4 query heads per "
                        "KV head only");
        const int mw = (L->max_ctx - kTierSinks) / kTierW;
        if (mw < 1 || mw > kTierRouteCap)
            return fail(KVEV_EINVAL, "layout: max_ctx %d gives %d windows (1 .. %d)", L->max_ctx,
                        mw, kTierRouteCap);
        if (budget < 0 || budget > mw)
            return fail(KVEV_EINVAL, "budget (K_f) %lld must be in [0, %d]", (long long)budget, mw);
        return KVEV_OK;
    }
    if (L->max_ctx % L->page_tokens != 0)
        return fail(KVEV_EINVAL, "layout: max_ctx %d must be a multiple of page_tokens %d",
                    L->max_ctx, L->page_tokens);
    const int64_t units = budget_tokens ? L->max_ctx : L->max_ctx / L->page_tokens;
    if (budget < 1 || budget >= units)
        return fail(KVEV_EINVAL, "budget %lld must be in [1, %lld)", (long long)budget,
                    (long long)units);
    return KVEV_OK;
}

int64_t attn_grid_for_device(int num_sms, const kvev_layout& L) {
    const int per_sm = attn_ctas_per_sm(L.head_dim, L.n_q_heads / L.n_kv_heads);
    return (int64_t)num_sms * (per_sm > 0 ? per_sm : 1);
}

// Warps of one attention launch over n_tiles tiles: all of them when every
// warp gets kMinTilesPerWarp tiles or more, else one per kMinTilesPerWarp
// tiles, so a short cache is not cut into many one-tile pieces (the combine
// walks a row's pieces one after another).  Sets *grid to the CTAs that hold
// them.
constexpr int kMinTilesPerWarp = 4;
int attn_launch_warps(int max_warps, int64_t n_tiles, int* grid) {
    const int64_t want = (n_tiles + kMinTilesPerWarp - 1) / kMinTilesPerWarp;
    const int w = want < (int64_t)max_warps ? (int)(want > 0 ? want : 1) : max_warps;
    const int wpc = attn_warps_per_cta();
    *grid = (w + wpc - 1) / wpc;
    return w;
}

int64_t int2_grid_for_device(int num_sms, const kvev_layout& L) {
    if (L.page_tokens != kTierW) return 0;
    const int per_sm = int2_ctas_per_sm(L.head_dim, L.n_q_heads / L.n_kv_heads);
    return (int64_t)num_sms * (per_sm > 0 ? per_sm : 1);
}

}  // namespace

namespace kvev {
// Lets other translation units of the library set the message that
// kvev_last_error returns.
kvev_status report_error(kvev_status st, const char* msg) { return fail(st, "%s", msg); }
}  // namespace kvev

struct kvev_ctx {
    kvev_layout lay{};
    int64_t budget = 0;
    float alpha = 0.f, beta = 0.f;
    int32_t refresh_mode = KVEV_REFRESH_FULL, refresh_period = 1;
    int32_t age_mode = KVEV_AGE_SINCE_INSERT, pool = KVEV_POOL_SUM;
    int32_t out_type = KVEV_OUT_F32;
    int32_t aggregation = KVEV_AGG_EMA, weighting = 0;
    int32_t group = 4;
    RegionParams rp{};
    std::vector<int32_t> pin_blocks;  // per sequence: prefill blocks holding a pinned token
    // two-tier mode: capacities, routing interval, INT2 attention grid, and the
    // host's exact copy of the window counts (the same for every sequence:
    // windows form by position and routing fills the tiers by capacity)
    int k_full = 0, k_quant = 0, omega = 8;
    int int2_grid = 0, int2_warps = 0;
    int t_nw = 0, t_tl = 0, t_first_u = 0, t_nf = 0, t_nq = 0;
    // rotary positions: the model's (cos, sin) table of the run (null: off)
    // and the one kvev_set_rope gave for the next run, the pages at the end
    // of each sequence's range that hold the INT2 windows' bf16
    // reconstructions, and whether the device's slot map is current (it is
    // not kept in a checkpoint: after an import the next step rebuilds it)
    const float* rope = nullptr;
    const float* rope_next = nullptr;
    int t_scratch = 0;
    bool t_recon_valid = false;
    int32_t len = 0, prefill_len = 0;
    std::vector<int32_t> ub_blocks;   // block mode: upper bound of each sequence's live blocks
    int64_t step = 0;
    bool begun = false;
    int device = 0, num_sms = 0;
    int attn_grid = 0, attn_warps = 0;
    int fused_grid = 0;                 // CTAs of the fused refresh step (0: no such shape)
    int32_t fused = 0;                  // KVEV_FUSED_* of refresh steps
    int32_t test_skip_cta = -1;         // test-only barrier timeout injection
    uint32_t test_bar_limit = 0;
    char* ws_base = nullptr;
    Workspace ws;
    float* dbg_probs = nullptr;
    float* dbg_prio = nullptr;
    int32_t* lir_counters = nullptr;    // Global LIR counts (two-tier mode)
    int32_t lir_sustain = 0;
    int32_t* diag_counters = nullptr;   // ranking diagnostics (token mode)
    float* diag_raw = nullptr;
    bool diag_flags_valid = false;      // the raw-set flags of the live cache are set
    bool prof = false;
    std::vector<cudaEvent_t> ev_pool;
    std::vector<int> ev_kind;   // kernel slot of each recorded start/end pair
    size_t ev_used = 0;
    float prof_ms[KVEV_PROFILE_SLOTS] = {};
    int64_t prof_n[KVEV_PROFILE_SLOTS] = {};
    int64_t launches = 0;
    int64_t test_fault_tile = -1;   // test-only timeout injection for the next step
    uint32_t test_wait_limit = 0;
};

namespace {

cudaEvent_t next_event(kvev_ctx* c) {
    if (c->ev_used == c->ev_pool.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        c->ev_pool.push_back(e);
    }
    return c->ev_pool[c->ev_used++];
}

kvev_status harvest_profile(kvev_ctx* c) {
    for (size_t k = 0; k + 1 < c->ev_used; k += 2) {
        cudaError_t e = cudaEventSynchronize(c->ev_pool[k + 1]);
        if (e != cudaSuccess) return cuda_fail(e, "profile event");
        float ms = 0.f;
        e = cudaEventElapsedTime(&ms, c->ev_pool[k], c->ev_pool[k + 1]);
        if (e != cudaSuccess) return cuda_fail(e, "profile elapsed");
        const int slot = c->ev_kind[k / 2];
        c->prof_ms[slot] += ms;
        c->prof_n[slot] += 1;
    }
    c->ev_used = 0;
    c->ev_kind.clear();
    return KVEV_OK;
}

// Launch helper: optional event pair around the launch, launch counting.
template <typename F>
kvev_status timed_launch(kvev_ctx* c, int slot, cudaStream_t s, const char* what, F&& f) {
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (c->prof) {
        if (c->ev_used + 2 > (1u << 16)) {
            kvev_status st = harvest_profile(c);
            if (st != KVEV_OK) return st;
        }
        e0 = next_event(c);
        e1 = next_event(c);
        if (!e0 || !e1) return fail(KVEV_ENOMEM, "cannot create profiling events");
        cudaEventRecord(e0, s);
    }
    cudaError_t e = f();
    c->launches += 1;
    if (e != cudaSuccess) {
        if (c->prof) c->ev_used -= 2;
        return cuda_fail(e, what);
    }
    if (c->prof) {
        cudaEventRecord(e1, s);
        c->ev_kind.push_back(slot);
    }
    return KVEV_OK;
}

kvev_status check_status_word(kvev_ctx* c, cudaStream_t s) {
    uint32_t host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, c->ws.status, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "device status");
    if (host != 0) {
        cudaMemsetAsync(c->ws.status, 0, 4, s);
        // a barrier that gave up may have left arrivals behind
        if (host & kStatusTimeout) cudaMemsetAsync(c->ws.gbar, 0, 8, s);
        cudaStreamSynchronize(s);
    }
    if (host & kStatusTimeout)
        return fail(KVEV_ETIMEOUT, "a device wait exceeded its iteration limit%s",
                    (host & kStatusBarrier) ? " (a grid barrier of the fused step)" : "");
    if (host & kStatusNoPage)
        return fail(KVEV_ESTATE, "a sequence had no free page for a new or re-admitted block");
    return KVEV_OK;
}

}  // namespace

extern "C" {

const char* kvev_last_error(const kvev_ctx*) { return g_err; }

kvev_status kvev_workspace_size(const kvev_layout* layout, int64_t budget, size_t* bytes) {
    kvev_status st = check_layout(layout, budget);
    if (st != KVEV_OK) return st;
    if (!bytes) return fail(KVEV_EINVAL, "bytes is NULL");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    const int64_t W = attn_grid_for_device(sms, *layout) * attn_warps_per_cta();
    const int64_t W2 = int2_grid_for_device(sms, *layout) * int2_warps_per_cta();
    const int64_t rows = (int64_t)layout->n_layers * layout->batch * layout->n_kv_heads;
    *bytes = carve(*layout, budget, W + rows, nullptr, W2 ? W2 + rows : 0).bytes;
    return KVEV_OK;
}

kvev_status kvev_create(const kvev_layout* layout, int64_t budget, int32_t granularity,
                        float alpha, float beta, const kvev_region_table* regions,
                        kvev_ctx** out) {
    if (!out) return fail(KVEV_EINVAL, "out is NULL");
    *out = nullptr;
    const bool memdecay = regions && regions->score_kind == KVEV_SCORE_MEMDECAY;
    kvev_status st = check_layout(layout, budget, memdecay);
    if (st != KVEV_OK) return st;
    if (granularity != layout->page_tokens)
        return fail(KVEV_EINVAL, "granularity %d != layout.page_tokens %d", granularity,
                    layout->page_tokens);
    if (!(alpha > 0.f && alpha <= 1.f)) return fail(KVEV_EINVAL, "alpha must be in (0, 1]");
    if (!(beta >= 0.f)) return fail(KVEV_EINVAL, "beta must be >= 0 (+inf allowed)");
    RegionParams rp{};
    if (regions) {
        const kvev_region_table& R = *regions;
        if (layout->page_tokens != kTile)
            return fail(KVEV_EUNSUPPORTED, "a region table needs %d-token blocks", kTile);
        if (R.n_regions < 1 || R.n_regions > KVEV_MAX_REGIONS)
            return fail(KVEV_EINVAL, "n_regions %d out of [1, %d]", R.n_regions, KVEV_MAX_REGIONS);
        if (R.score_kind != KVEV_SCORE_LRFU && R.score_kind != KVEV_SCORE_MEMDECAY)
            return fail(KVEV_EINVAL, "unknown score_kind %d", R.score_kind);
        if (R.decode_region < 0 || R.decode_region >= R.n_regions)
            return fail(KVEV_EINVAL, "decode_region %d out of range", R.decode_region);
        if (!(R.rho >= 0.f && R.rho < 1.f) || !(R.attn_weight >= 0.f) || !(R.tau_scale >= 0.f))
            return fail(KVEV_EINVAL, "rho must be in [0, 1), attn_weight and tau_scale >= 0");
        rp.on = 1;
        rp.memdecay = memdecay ? 1 : 0;
        rp.decode_region = R.decode_region;
        for (int r = 0; r < R.n_regions; ++r) {
            if (!(R.base_priority[r] >= 0.f) || !(R.decay_lambda[r] >= 0.f))
                return fail(KVEV_EINVAL, "region %d: base_priority and decay_lambda must be >= 0",
                            r);
            rp.base[r] = R.base_priority[r];
            rp.lam[r] = R.decay_lambda[r];
            if (R.pinned[r]) rp.pinned_mask |= 1u << r;
        }
        rp.rho = R.rho;
        rp.attn_w = R.attn_weight;
        rp.tau_scale = R.tau_scale;
        rp.budget_tokens = (int32_t)budget;
    }

    kvev_ctx* c = new (std::nothrow) kvev_ctx;
    if (!c) return fail(KVEV_ENOMEM, "host allocation failed");
    c->lay = *layout;
    c->budget = budget;
    c->alpha = alpha;
    c->beta = beta;
    c->group = layout->n_q_heads / layout->n_kv_heads;
    c->rp = rp;
    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) {
        delete c;
        return cuda_fail(e, "device query");
    }
    c->attn_grid = (int)attn_grid_for_device(c->num_sms, *layout);
    c->attn_warps = c->attn_grid * attn_warps_per_cta();
    if (layout->page_tokens == 1) {
        // at most the attention kernel's grid: the split partial slots are
        // sized for its warps, and with the same CTAs the two paths split the
        // tiles alike (the same outputs bit for bit)
        const int fg = c->num_sms * attn_fused_ctas_per_sm(layout->head_dim, c->group,
                                                           layout->n_kv_heads);
        c->fused_grid = fg < c->attn_grid ? fg : c->attn_grid;
    }
    c->int2_grid = (int)int2_grid_for_device(c->num_sms, *layout);
    c->int2_warps = c->int2_grid * int2_warps_per_cta();
    const int64_t rows = (int64_t)layout->n_layers * layout->batch * layout->n_kv_heads;
    const int64_t slots2 = c->int2_warps ? c->int2_warps + rows : 0;
    const size_t bytes = carve(*layout, budget, c->attn_warps + rows, nullptr, slots2).bytes;
    e = cudaMalloc(&c->ws_base, bytes);
    if (e != cudaSuccess) {
        delete c;
        cudaGetLastError();
        return fail(KVEV_ENOMEM, "cudaMalloc of %zu bytes of scratch failed", bytes);
    }
    c->ws = carve(*layout, budget, c->attn_warps + rows, c->ws_base, slots2);
    c->k_full = (int)budget;
    e = cudaMemset(c->ws_base, 0, bytes);   // row counters and status start at zero
    for (int i = 0; i < c->ws.n_guard && e == cudaSuccess; ++i)
        e = cudaMemset(c->ws_base + c->ws.guard_off[i], kGuardByte, kGuardBytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(c->ws_base);
        delete c;
        return cuda_fail(e, "scratch init");
    }
    *out = c;
    return KVEV_OK;
}

void kvev_destroy(kvev_ctx* c) {
    if (!c) return;
    for (cudaEvent_t e : c->ev_pool) cudaEventDestroy(e);
    if (c->ws_base) cudaFree(c->ws_base);
    delete c;
}

kvev_status kvev_refresh_mode(kvev_ctx* c, int32_t mode, int32_t period) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (mode != KVEV_REFRESH_FULL && mode != KVEV_REFRESH_LAZY && mode != KVEV_REFRESH_FROZEN)
        return fail(KVEV_EINVAL, "unknown refresh mode %d", mode);
    if (mode == KVEV_REFRESH_LAZY && period < 1)
        return fail(KVEV_EINVAL, "lazy refresh period must be >= 1");
    c->refresh_mode = mode;
    c->refresh_period = mode == KVEV_REFRESH_LAZY ? period : 1;
    return KVEV_OK;
}

kvev_status kvev_configure(kvev_ctx* c, int32_t age_mode, int32_t pool) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (age_mode != KVEV_AGE_SINCE_INSERT && age_mode != KVEV_AGE_SINCE_ACCESS)
        return fail(KVEV_EINVAL, "unknown age mode %d", age_mode);
    if (pool != KVEV_POOL_SUM && pool != KVEV_POOL_MEAN)
        return fail(KVEV_EINVAL, "unknown pooling %d", pool);
    c->age_mode = age_mode;
    c->pool = pool;
    return KVEV_OK;
}

kvev_status kvev_begin(kvev_ctx* c, int32_t prefill_len) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (c->lay.page_tokens != 1)
        return fail(KVEV_ESTATE, "a block-granular context starts with kvev_paged_begin");
    if (prefill_len < 0 || prefill_len >= c->lay.max_ctx)
        return fail(KVEV_EINVAL, "prefill_len %d must be in [0, max_ctx)", prefill_len);
    c->len = prefill_len;
    c->prefill_len = prefill_len;
    c->step = 0;
    c->begun = true;
    c->diag_flags_valid = false;
    return KVEV_OK;
}

kvev_status kvev_length(const kvev_ctx* c, int32_t* len) {
    if (!c || !len) return fail(KVEV_EINVAL, "NULL argument");
    *len = c->len;
    return KVEV_OK;
}

kvev_status kvev_init_state(kvev_ctx* c, const kvev_state* st, void* stream) {
    if (!c || !st) return fail(KVEV_EINVAL, "NULL argument");
    if (!st->score || !st->t_ins || !st->t_ref || !st->pos)
        return fail(KVEV_EINVAL, "state has a NULL array");
    if (!c->begun) return fail(KVEV_ESTATE, "kvev_begin must come first");
    cudaStream_t s = (cudaStream_t)stream;
    const int len = c->len;
    c->diag_flags_valid = false;
    return timed_launch(c, kProfInit, s, "init_state", [&] {
        return launch_init_state(*st, c->lay.batch, c->lay.max_ctx, len, c->ws.vp, s);
    });
}

kvev_status kvev_set_diagnostics(kvev_ctx* c, int32_t* counters, float* raw_score) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (c->lay.page_tokens != 1 && (counters || raw_score))
        return fail(KVEV_EUNSUPPORTED, "ranking diagnostics are built for token granularity");
    c->diag_counters = counters;
    c->diag_raw = raw_score;
    c->diag_flags_valid = false;
    return KVEV_OK;
}

kvev_status kvev_missed_mass(const float* full_score, int32_t score_ld, int32_t n_pos,
                             const int32_t* pos, int32_t pos_ld, int32_t n_cached,
                             int32_t batch, float* out, void* stream) {
    if (!full_score || !out || (n_cached > 0 && !pos))
        return fail(KVEV_EINVAL, "kvev_missed_mass: NULL argument");
    if (batch < 1 || n_pos < 1 || score_ld < n_pos || n_cached < 0 || pos_ld < n_cached)
        return fail(KVEV_EINVAL, "kvev_missed_mass: batch >= 1, 1 <= n_pos <= score_ld and "
                    "0 <= n_cached <= pos_ld needed");
    MissedMassArgs a{};
    a.full_score = full_score;
    a.pos = pos;
    a.out = out;
    a.score_ld = score_ld;
    a.n_pos = n_pos;
    a.pos_ld = pos_ld;
    a.n_cached = n_cached;
    cudaError_t e = launch_missed_mass(a, batch, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "missed mass");
    return KVEV_OK;
}

kvev_status kvev_set_debug(kvev_ctx* c, float* probs, float* priority) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    c->dbg_probs = probs;
    c->dbg_prio = priority;
    return KVEV_OK;
}

kvev_status kvev_set_scorer(kvev_ctx* c, int32_t aggregation, int32_t weighting) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (aggregation != KVEV_AGG_EMA && aggregation != KVEV_AGG_CUMULATIVE)
        return fail(KVEV_EINVAL, "unknown aggregation %d", aggregation);
    if (weighting & ~(KVEV_W_VNORM | KVEV_W_ENTROPY))
        return fail(KVEV_EINVAL, "unknown weighting bits 0x%x", weighting);
    if (c->lay.page_tokens != 1 && weighting != 0)
        return fail(KVEV_EUNSUPPORTED, "the weightings are built for token granularity");
    if (c->lay.page_tokens != 1 && c->lay.page_tokens != kTierW &&
        aggregation != KVEV_AGG_EMA)
        return fail(KVEV_EUNSUPPORTED, "cumulative aggregation is built for token "
                    "granularity and two-tier windows");
    c->aggregation = aggregation;
    c->weighting = weighting;
    return KVEV_OK;
}

kvev_status kvev_set_fused_step(kvev_ctx* c, int32_t mode) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (mode != KVEV_FUSED_OFF && mode != KVEV_FUSED_ALL && mode != KVEV_FUSED_ATTN_COMBINE)
        return fail(KVEV_EINVAL, "unknown fused-step mode %d", mode);
    if (mode != KVEV_FUSED_OFF && c->fused_grid <= 0)
        return fail(KVEV_EUNSUPPORTED, "no fused step for this layout (token granularity; "
                    "head_dim 64/128; 4 or 8 query heads per KV head; 1, 2 or 8 KV heads)");
    c->fused = mode;
    return KVEV_OK;
}

kvev_status kvev_set_output(kvev_ctx* c, int32_t out_type) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (out_type != KVEV_OUT_F32 && out_type != KVEV_OUT_BF16)
        return fail(KVEV_EINVAL, "unknown output type %d", out_type);
    c->out_type = out_type;
    return KVEV_OK;
}

kvev_status kvev_step(kvev_ctx* c, const void* q, const void* k_new, const void* v_new,
                      kvev_cache* cache, const kvev_state* st, int64_t step, void* out,
                      int32_t* retained_idx, int32_t* n_retained, void* stream) {
    const NvtxRange trace("kvev_step");
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (!q || !k_new || !v_new || !cache || !st || !out || !retained_idx || !n_retained)
        return fail(KVEV_EINVAL, "NULL argument");
    if (!cache->k[0] || !cache->k[1] || !cache->v[0] || !cache->v[1])
        return fail(KVEV_EINVAL, "cache has a NULL buffer");
    if (cache->cur != 0 && cache->cur != 1) return fail(KVEV_EINVAL, "cache.cur must be 0 or 1");
    if (!st->score || !st->t_ins || !st->t_ref || !st->pos)
        return fail(KVEV_EINVAL, "state has a NULL array");
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(cache->k[0]) ||
        !aligned16(cache->k[1]) || !aligned16(cache->v[0]) || !aligned16(cache->v[1]) ||
        !aligned16(out))
        return fail(KVEV_EINVAL, "q, k_new, v_new, out and the cache buffers must be 16-byte aligned");
    if (!c->begun) return fail(KVEV_ESTATE, "kvev_begin must come before the first step");
    if (c->lay.page_tokens != 1)
        return fail(KVEV_ESTATE, "a block-granular context steps with kvev_paged_step");
    if (step != c->step + 1)
        return fail(KVEV_ESTATE, "step %lld out of order (expected %lld)", (long long)step,
                    (long long)(c->step + 1));
    if (c->len + 1 > c->lay.max_ctx)
        return fail(KVEV_EINVAL, "cache full: %d live tokens, max_ctx %d", c->len, c->lay.max_ctx);

    cudaStream_t s = (cudaStream_t)stream;
    const kvev_layout& Ly = c->lay;
    const int G = c->group;
    const int t = (int)step;
    const int L = c->len + 1;
    const int cur = cache->cur;
    bool refresh = true;
    if (c->refresh_mode == KVEV_REFRESH_LAZY) refresh = (t - 1) % c->refresh_period == 0;
    if (c->refresh_mode == KVEV_REFRESH_FROZEN) refresh = t == 1;
    const int rows = Ly.n_layers * Ly.batch * Ly.n_kv_heads;
    const int tiles_per_row = (L + kTile - 1) / kTile;
    const int n_keep = L < c->budget ? L : (int)c->budget;
    const bool identity = L <= c->budget;
    kvev_status rc;

    AppendArgs ap{};
    ap.k = (uint16_t*)cache->k[cur];
    ap.v = (uint16_t*)cache->v[cur];
    ap.k_new = (const uint16_t*)k_new;
    ap.v_new = (const uint16_t*)v_new;
    ap.st = *st;
    ap.slot = c->len;
    ap.t = t;
    ap.pos = c->prefill_len + t - 1;
    ap.n_layers = Ly.n_layers;
    ap.batch = Ly.batch;
    ap.n_kv = Ly.n_kv_heads;
    ap.max_ctx = Ly.max_ctx;
    ap.head_dim = Ly.head_dim;
    rc = timed_launch(c, kProfAppend, s, "append", [&] { return launch_append(ap, s); });
    if (rc != KVEV_OK) return rc;

    AttnArgs at{};
    at.k = (const uint16_t*)cache->k[cur];
    at.v = (const uint16_t*)cache->v[cur];
    at.q = (const uint16_t*)q;
    at.logits = c->ws.logits;
    at.logit_ld = logit_ld(Ly.max_ctx);
    at.part_o = c->ws.part_o;
    at.part_ml = c->ws.part_ml;
    at.status = c->ws.status;
    at.tiles_per_row = tiles_per_row;
    at.L = L;
    at.max_ctx = Ly.max_ctx;
    at.n_layers = Ly.n_layers;
    at.batch = Ly.batch;
    at.n_kv = Ly.n_kv_heads;
    at.n_q = Ly.n_q_heads;
    at.write_logits = refresh ? 1 : 0;
    at.q_scale = (float)(1.4426950408889634 / sqrt((double)Ly.head_dim));
    at.view_tokens = (int64_t)Ly.n_layers * Ly.batch * Ly.n_kv_heads * Ly.max_ctx;
    at.fault_tile_p1 = c->test_fault_tile + 1;
    at.wait_limit = c->test_wait_limit;
    c->test_fault_tile = -1;
    c->test_wait_limit = 0;
    // the weightings' statistics, gathered by the attention on refresh steps
    const int stats = !refresh ? 0
                      : ((c->weighting & KVEV_W_ENTROPY) ? kStatEntropy : 0) |
                            ((c->weighting & KVEV_W_VNORM) ? kStatVNorm : 0);
    at.part_e = (stats & kStatEntropy) ? c->ws.part_e : nullptr;
    at.vnorm = (stats & kStatVNorm) ? c->ws.vnorm : nullptr;
    at.part_vn = (stats & kStatVNorm) ? c->ws.part_vn : nullptr;

    ScoreArgs sc{};
    sc.logits = c->ws.logits;
    sc.logit_ld = logit_ld(Ly.max_ctx);
    sc.lse2 = c->ws.lse2;
    sc.st = *st;
    sc.m_s = c->ws.m_s;
    sc.tref_s = c->ws.tref_s;
    sc.tins_s = c->ws.tins_s;
    sc.pos_s = c->ws.pos_s;
    sc.keys = c->ws.keys;
    sc.msum_part = c->ws.msum_part;
    sc.dbg_probs = refresh ? c->dbg_probs : nullptr;
    sc.dbg_prio = c->dbg_prio;
    sc.L = L;
    sc.max_ctx = Ly.max_ctx;
    sc.n_layers = Ly.n_layers;
    sc.batch = Ly.batch;
    sc.n_kv = Ly.n_kv_heads;
    sc.n_q = Ly.n_q_heads;
    sc.refresh = refresh ? 1 : 0;
    sc.age_mode = c->age_mode;
    sc.pool_mean = c->pool == KVEV_POOL_MEAN ? 1 : 0;
    sc.t = t;
    const bool cumulative = c->aggregation == KVEV_AGG_CUMULATIVE;
    sc.alpha = cumulative ? 1.0f : c->alpha;
    sc.oma = cumulative ? 1.0f : 1.0f - c->alpha;
    for (int k = 0; k < kScoreSegMax; ++k) {   // oma^(layers of scorer segment k), fp64
        const int n = k < kScoreSegs
                          ? (k + 1) * Ly.n_layers / kScoreSegs - k * Ly.n_layers / kScoreSegs
                          : 0;
        double d = 1.0;
        for (int i = 0; i < n; ++i) d *= (double)sc.oma;
        sc.seg_decay[k] = (float)d;
    }
    sc.ent = (stats & kStatEntropy) ? c->ws.ent : nullptr;
    sc.vnorm = (stats & kStatVNorm) ? c->ws.vnorm : nullptr;
    sc.vmean = (stats & kStatVNorm) ? c->ws.vmean : nullptr;
    sc.beta = c->beta;
    sc.access_thr = (float)(2.0 * Ly.n_q_heads * Ly.n_layers / (double)L);
    const bool diag = c->diag_counters != nullptr;
    sc.raw_keys = diag && refresh ? c->ws.raw_keys : nullptr;
    sc.dbg_raw = refresh ? c->diag_raw : nullptr;

    const int64_t rows_per_layer = (int64_t)Ly.batch * Ly.n_kv_heads;
    at.row0 = 0;
    at.n_tiles_total = (int64_t)Ly.n_layers * rows_per_layer * tiles_per_row;
    // the fused step: refresh steps without the weightings' statistics
    const bool fused = c->fused && refresh && stats == 0 && c->fused_grid > 0;
    int attn_grid = 0;
    at.total_warps = attn_launch_warps(fused ? c->fused_grid * attn_warps_per_cta()
                                             : c->attn_warps,
                                       at.n_tiles_total, &attn_grid);
    if (!fused) {
        rc = timed_launch(c, kProfAttn, s, "attention", [&] {
            return launch_attention(at, Ly.head_dim, G, attn_grid, s, stats);
        });
        if (rc != KVEV_OK) return rc;
    }
    CombineArgs cb{};   // merge the split: outputs and per-head log2-sum-exp
    cb.part_e = at.part_e;
    cb.ent = at.part_e ? c->ws.ent : nullptr;
    cb.part_vn = at.part_vn;
    cb.vmean = at.part_vn ? c->ws.vmean : nullptr;
    cb.n_tokens = L;
    cb.sp.part_o = c->ws.part_o;
    cb.sp.part_ml = c->ws.part_ml;
    cb.sp.n_tiles = at.n_tiles_total;
    cb.sp.row0 = 0;
    cb.sp.total_warps = at.total_warps;
    cb.sp.tiles_per_row = tiles_per_row;
    cb.n_rows = (int32_t)(Ly.n_layers * rows_per_layer);
    cb.out = out;
    cb.out_bf16 = c->out_type == KVEV_OUT_BF16 ? 1 : 0;
    cb.lse2 = c->ws.lse2;
    cb.n_layers = Ly.n_layers;
    cb.batch = Ly.batch;
    cb.n_kv = Ly.n_kv_heads;
    cb.n_q = Ly.n_q_heads;
    int n_part = 0;
    if (fused) {   // attention, combine and scoring in one cooperative launch
        FusedArgs fa{};
        fa.bar = c->ws.gbar;
        fa.wait_limit = c->test_bar_limit;
        fa.skip_cta_p1 = c->test_skip_cta + 1;
        fa.score = c->fused == KVEV_FUSED_ALL ? 1 : 0;
        c->test_skip_cta = -1;
        c->test_bar_limit = 0;
        n_part = (L + 31) / 32;   // (not read on refresh steps)
        rc = timed_launch(c, kProfAttn, s, "fused step", [&] {
            return launch_attn_fused(at, cb, sc, fa, Ly.head_dim, G, c->fused_grid, s);
        });
        if (rc != KVEV_OK) return rc;
        if (!fa.score) {
            rc = timed_launch(c, kProfScore, s, "score",
                              [&] { return launch_score(sc, G, &n_part, s); });
            if (rc != KVEV_OK) return rc;
        }
    } else {
        rc = timed_launch(c, kProfCombine, s, "combine",
                          [&] { return launch_combine(cb, Ly.head_dim, G, s); });
        if (rc != KVEV_OK) return rc;
        rc = timed_launch(c, kProfScore, s, "score",
                          [&] { return launch_score(sc, G, &n_part, s); });
        if (rc != KVEV_OK) return rc;
    }

    SelectArgs se{};
    se.keys = c->ws.keys;
    se.m_s = c->ws.m_s;
    se.msum_part = c->ws.msum_part;
    se.n_part = n_part;
    se.retained = retained_idx;
    se.n_retained = n_retained;
    se.L = L;
    se.max_ctx = Ly.max_ctx;
    se.budget = (int)c->budget;
    se.refresh = refresh ? 1 : 0;
    se.first_moved = c->ws.first_moved;
    // few evictions: the maxima path lists them and the compaction runs in place
    const bool in_place = !identity && L - n_keep <= kFewEvict;
    se.evicted = in_place ? c->ws.evicted : nullptr;
    se.few = in_place ? 1 : 0;
    rc = timed_launch(c, kProfSelect, s, "select",
                      [&] { return launch_select(se, Ly.batch, c->num_sms, s); });
    if (rc != KVEV_OK) return rc;
    if (diag) {   // ranking diagnostics: the raw top-B set, then the counts
        if (refresh) {
            SelectArgs sr = se;
            sr.keys = c->ws.raw_keys;
            sr.retained = c->ws.raw_list;
            sr.n_retained = c->ws.raw_n;
            sr.refresh = 1;          // no new-token score to set
            sr.first_moved = nullptr;
            sr.evicted = nullptr;    // (the compaction reads the step's own list)
            rc = timed_launch(c, kProfSelect, s, "raw select",
                              [&] { return launch_select(sr, Ly.batch, c->num_sms, s); });
            if (rc != KVEV_OK) return rc;
        }
        DiagArgs dg{};
        dg.retained = retained_idx;
        dg.n_retained = n_retained;
        dg.raw_list = c->ws.raw_list;
        dg.raw_n = c->ws.raw_n;
        dg.in_raw = c->ws.in_raw;
        const size_t cb_ctx = (size_t)Ly.batch * Ly.max_ctx;
        dg.flags_in = c->ws.raw_flags + (step & 1) * cb_ctx;
        dg.flags_out = c->ws.raw_flags + ((step + 1) & 1) * cb_ctx;
        dg.prev_n = c->ws.raw_prev_n;
        dg.counters = c->diag_counters;
        dg.L = L;
        dg.max_ctx = Ly.max_ctx;
        dg.budget = (int)c->budget;
        dg.t = t;
        dg.refresh = refresh ? 1 : 0;
        dg.flags_valid = c->diag_flags_valid ? 1 : 0;
        rc = timed_launch(c, kProfSelect, s, "diagnostics",
                          [&] { return launch_diag(dg, Ly.batch, s); });
        if (rc != KVEV_OK) return rc;
        c->diag_flags_valid = c->diag_flags_valid || refresh;
    }

    CompactArgs cp{};
    cp.first_moved = c->ws.first_moved;
    cp.vp_in = c->ws.vp + (step & 1) * Ly.batch;
    cp.vp_out = c->ws.vp + ((step + 1) & 1) * Ly.batch;
    const int dst = identity || in_place ? cur : cur ^ 1;   // the live buffer after the step
    cp.k_src = (const uint16_t*)cache->k[cur];
    cp.v_src = (const uint16_t*)cache->v[cur];
    cp.k_dst = (uint16_t*)cache->k[dst];
    cp.v_dst = (uint16_t*)cache->v[dst];
    cp.in_place = in_place ? 1 : 0;
    cp.n_evict = L - n_keep;
    cp.evicted = c->ws.evicted;
    cp.retained = retained_idx;
    cp.m_s = c->ws.m_s;
    cp.tref_s = c->ws.tref_s;
    cp.tins_s = c->ws.tins_s;
    cp.pos_s = c->ws.pos_s;
    cp.st = *st;
    cp.n_keep = n_keep;
    cp.identity = identity ? 1 : 0;
    cp.rows = rows;
    cp.batch = Ly.batch;
    cp.n_kv = Ly.n_kv_heads;
    cp.max_ctx = Ly.max_ctx;
    cp.budget = (int)c->budget;
    cp.head_dim = Ly.head_dim;
    rc = timed_launch(c, kProfCompact, s, "compact",
                      [&] { return launch_compact(cp, c->num_sms, s); });
    if (rc != KVEV_OK) return rc;

    cache->cur = dst;
    c->len = n_keep;
    c->step = step;
    return KVEV_OK;
}

kvev_status kvev_step_host(kvev_ctx* c, const void* q_host, const void* k_new_host,
                           const void* v_new_host, kvev_cache* cache, const kvev_state* st,
                           int64_t step, void* out_host, int32_t* retained_idx_host,
                           int32_t* n_retained_host, void* stream) {
    const NvtxRange trace("kvev_step_host");
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (!q_host || !k_new_host || !v_new_host || !out_host || !retained_idx_host ||
        !n_retained_host)
        return fail(KVEV_EINVAL, "NULL argument");
    cudaStream_t s = (cudaStream_t)stream;
    const kvev_layout& Ly = c->lay;
    const size_t qb = (size_t)Ly.batch * Ly.n_layers * Ly.n_q_heads * Ly.head_dim * 2;
    const size_t kb = (size_t)Ly.batch * Ly.n_layers * Ly.n_kv_heads * Ly.head_dim * 2;
    cudaError_t e = cudaMemcpyAsync(c->ws.stg_q, q_host, qb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->ws.stg_k, k_new_host, kb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->ws.stg_v, v_new_host, kb, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    kvev_status rc = kvev_step(c, c->ws.stg_q, c->ws.stg_k, c->ws.stg_v, cache, st, step,
                               c->ws.stg_out, c->ws.stg_ret, c->ws.stg_nret, stream);
    if (rc != KVEV_OK) return rc;
    // qb is the bf16 size of q, which has the output's shape
    e = cudaMemcpyAsync(out_host, c->ws.stg_out, c->out_type == KVEV_OUT_BF16 ? qb : qb * 2,
                        cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(retained_idx_host, c->ws.stg_ret, (size_t)Ly.batch * c->budget * 4,
                            cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(n_retained_host, c->ws.stg_nret, (size_t)Ly.batch * 4,
                            cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
    return check_status_word(c, s);
}

// ---- block-granular (paged) mode ------------------------------------------

}  // extern "C"

namespace {

kvev_status check_paged(kvev_ctx* c, const kvev_paged_cache* pc, const kvev_block_state* bs) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (c->lay.page_tokens == 1)
        return fail(KVEV_ESTATE, "a token-granular context: use kvev_begin / kvev_step");
    if (!pc || !bs) return fail(KVEV_EINVAL, "NULL argument");
    if (!pc->k_pool || !pc->v_pool || !pc->block_table || !pc->n_blocks || !pc->free_pages ||
        !pc->n_free || !pc->next_lid)
        return fail(KVEV_EINVAL, "paged cache has a NULL array");
    if (!aligned16(pc->k_pool) || !aligned16(pc->v_pool))
        return fail(KVEV_EINVAL, "the page pools must be 16-byte aligned");
    if (pc->pages_per_seq != c->lay.max_ctx / c->lay.page_tokens)
        return fail(KVEV_EINVAL, "pages_per_seq %d != max_ctx / page_tokens = %d", pc->pages_per_seq,
                    c->lay.max_ctx / c->lay.page_tokens);
    if (pc->n_backing < 0) return fail(KVEV_EINVAL, "n_backing must be >= 0");
    if (pc->n_backing > 0 && (!pc->backing_k || !pc->backing_v || !aligned16(pc->backing_k) ||
                              !aligned16(pc->backing_v)))
        return fail(KVEV_EINVAL, "backing tier: NULL or unaligned buffer");
    if (!bs->score || !bs->t_ins || !bs->t_ref || !bs->lid || !bs->len || !bs->table)
        return fail(KVEV_EINVAL, "block state has a NULL array");
    if (bs->table_len < pc->n_backing || bs->table_len < 1)
        return fail(KVEV_EINVAL, "table_len %d must be >= max(1, n_backing %d)", bs->table_len,
                    pc->n_backing);
    if (c->rp.on && !bs->region) return fail(KVEV_EINVAL, "a region table needs state.region");
    if (c->rp.memdecay && (!bs->tok_a || !bs->tok_t_ref))
        return fail(KVEV_EINVAL, "MemDecay scoring needs state.tok_a and state.tok_t_ref");
    return KVEV_OK;
}

PagedArgs paged_args(kvev_ctx* c, const kvev_paged_cache* pc, const kvev_block_state* bs, int t,
                     bool refresh) {
    PagedArgs a{};
    a.c = *pc;
    a.st = *bs;
    a.tokens = c->ws.tokens;
    a.m_s = c->ws.m_s;
    a.tref_s = c->ws.tref_s;
    a.tins_s = c->ws.tins_s;
    a.lid_s = c->ws.lid_s;
    a.len_s = c->ws.len_s;
    a.page_s = c->ws.page_s;
    a.keys = c->ws.keys;
    a.sel = c->ws.sel;
    a.readmit_page = c->ws.readmit_page;
    a.status = c->ws.status;
    a.batch = c->lay.batch;
    a.n_layers = c->lay.n_layers;
    a.n_kv = c->lay.n_kv_heads;
    a.n_q = c->lay.n_q_heads;
    a.head_dim = c->lay.head_dim;
    a.page = c->lay.page_tokens;
    a.budget = (int)c->budget;
    a.t = t;
    a.refresh = refresh ? 1 : 0;
    a.age_mode = c->age_mode;
    a.pool_mean = c->pool == KVEV_POOL_MEAN ? 1 : 0;
    a.alpha = c->alpha;
    a.beta = c->beta;
    a.dbg_prio = c->dbg_prio;
    a.sel_ld = c->rp.on ? pc->pages_per_seq : (int)c->budget;
    a.budgets = c->ws.budgets;
    a.rp = c->rp;
    return a;
}

}  // namespace

extern "C" {

kvev_status kvev_paged_begin(kvev_ctx* c, const kvev_paged_cache* pc, const kvev_block_state* bs,
                             int32_t prefill_tokens, void* stream) {
    kvev_status rc = check_paged(c, pc, bs);
    if (rc != KVEV_OK) return rc;
    const int P = c->lay.page_tokens, pps = pc->pages_per_seq;
    if (prefill_tokens <= 0)
        return fail(KVEV_EINVAL, "prefill_tokens %d must be > 0", prefill_tokens);
    if (!c->rp.memdecay && prefill_tokens % P != 0)
        return fail(KVEV_EINVAL, "prefill_tokens %d must be a multiple of %d", prefill_tokens, P);
    const int nb0 = (prefill_tokens + P - 1) / P;
    if (nb0 + 1 > pps)
        return fail(KVEV_EINVAL, "%d prefill blocks leave no free page (pages_per_seq %d)", nb0,
                    pps);
    cudaStream_t s = (cudaStream_t)stream;
    const PagedArgs a = paged_args(c, pc, bs, 0, true);
    rc = timed_launch(c, kProfInit, s, "paged begin",
                      [&] { return launch_paged_begin(a, prefill_tokens, s); });
    if (rc != KVEV_OK) return rc;
    c->pin_blocks.assign(c->lay.batch, 0);
    if (c->rp.on && c->rp.pinned_mask) {   // bound the blocks no eviction can remove
        std::vector<uint8_t> lab((size_t)c->lay.batch * pps * P);
        cudaError_t e = cudaMemcpyAsync(lab.data(), bs->region, lab.size(),
                                        cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "reading the prefill region labels");
        for (int b = 0; b < c->lay.batch; ++b) {
            const uint8_t* lb = lab.data() + (size_t)b * pps * P;
            int n = 0;
            for (int j = 0; j < nb0; ++j) {
                bool pin = false;
                for (int k = 0; k < P && j * P + k < prefill_tokens; ++k)
                    pin |= ((c->rp.pinned_mask >> lb[(size_t)j * P + k]) & 1u) != 0;
                n += pin;
            }
            c->pin_blocks[b] = n;
        }
    }
    c->len = prefill_tokens;
    c->prefill_len = prefill_tokens;
    c->ub_blocks.assign(c->lay.batch, nb0);
    c->step = 0;
    c->begun = true;
    return KVEV_OK;
}

kvev_status kvev_paged_step(kvev_ctx* c, const void* q, const void* k_new, const void* v_new,
                            const kvev_paged_cache* pc, const kvev_block_state* bs, int64_t step,
                            void* out, int32_t* retained_lid, int32_t* n_retained,
                            void* stream) {
    const NvtxRange trace("kvev_paged_step");
    kvev_status rc = check_paged(c, pc, bs);
    if (rc != KVEV_OK) return rc;
    if (!q || !k_new || !v_new || !out || !retained_lid || !n_retained)
        return fail(KVEV_EINVAL, "NULL argument");
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out))
        return fail(KVEV_EINVAL, "q, k_new, v_new and out must be 16-byte aligned");
    if (!c->begun) return fail(KVEV_ESTATE, "kvev_paged_begin must come before the first step");
    if (step != c->step + 1)
        return fail(KVEV_ESTATE, "step %lld out of order (expected %lld)", (long long)step,
                    (long long)(c->step + 1));
    const int pps = pc->pages_per_seq;
    int ub = 0;   // live blocks of any sequence after the append, at most
    for (int b = 0; b < c->lay.batch; ++b) {
        if (c->ub_blocks[b] + 1 > pps)
            return fail(KVEV_EINVAL, "sequence %d may hold %d blocks: no page left for a new one",
                        b, c->ub_blocks[b]);
        ub = c->ub_blocks[b] + 1 > ub ? c->ub_blocks[b] + 1 : ub;
    }

    cudaStream_t s = (cudaStream_t)stream;
    const kvev_layout& Ly = c->lay;
    const int G = c->group;
    const int t = (int)step;
    bool refresh = true;
    if (c->refresh_mode == KVEV_REFRESH_LAZY) refresh = (t - 1) % c->refresh_period == 0;
    if (c->refresh_mode == KVEV_REFRESH_FROZEN) refresh = t == 1;
    PagedArgs pa = paged_args(c, pc, bs, t, refresh);
    pa.sel = c->ws.sel;
    pa.n_sel = n_retained;
    pa.retained_lid = retained_lid;

    rc = timed_launch(c, kProfAppend, s, "paged append", [&] {
        return launch_paged_append(pa, (const uint16_t*)k_new, (const uint16_t*)v_new, s);
    });
    if (rc != KVEV_OK) return rc;

    const int64_t rows = (int64_t)Ly.n_layers * Ly.batch * Ly.n_kv_heads;
    AttnArgs at{};
    at.k = (const uint16_t*)pc->k_pool;
    at.v = (const uint16_t*)pc->v_pool;
    at.q = (const uint16_t*)q;
    at.logits = c->ws.logits;
    at.logit_ld = logit_ld(Ly.max_ctx);
    at.part_o = c->ws.part_o;
    at.part_ml = c->ws.part_ml;
    at.status = c->ws.status;
    at.row0 = 0;
    at.tiles_per_row = ub;
    at.n_tiles_total = rows * ub;
    at.L = ub * kTile;
    at.max_ctx = Ly.max_ctx;
    at.n_layers = Ly.n_layers;
    at.batch = Ly.batch;
    at.n_kv = Ly.n_kv_heads;
    at.n_q = Ly.n_q_heads;
    int attn_grid = 0;
    at.total_warps = attn_launch_warps(c->attn_warps, at.n_tiles_total, &attn_grid);
    at.write_logits = refresh ? 1 : 0;
    at.q_scale = (float)(1.4426950408889634 / sqrt((double)Ly.head_dim));
    at.view_tokens = (int64_t)Ly.batch * pps * Ly.n_layers * Ly.n_kv_heads * Ly.page_tokens;
    at.block_table = pc->block_table;
    at.n_blocks = pc->n_blocks;
    at.blk_len = bs->len;
    at.pps = pps;
    rc = timed_launch(c, kProfAttn, s, "attention",
                      [&] { return launch_attention(at, Ly.head_dim, G, attn_grid, s); });
    if (rc != KVEV_OK) return rc;
    CombineArgs cb{};
    cb.sp.part_o = c->ws.part_o;
    cb.sp.part_ml = c->ws.part_ml;
    cb.sp.n_tiles = at.n_tiles_total;
    cb.sp.row0 = 0;
    cb.sp.total_warps = at.total_warps;
    cb.sp.tiles_per_row = ub;
    cb.n_rows = (int32_t)rows;
    cb.out = out;
    cb.out_bf16 = c->out_type == KVEV_OUT_BF16 ? 1 : 0;
    cb.lse2 = c->ws.lse2;
    cb.n_layers = Ly.n_layers;
    cb.batch = Ly.batch;
    cb.n_kv = Ly.n_kv_heads;
    cb.n_q = Ly.n_q_heads;
    rc = timed_launch(c, kProfCombine, s, "combine",
                      [&] { return launch_combine(cb, Ly.head_dim, G, s); });
    if (rc != KVEV_OK) return rc;

    ScoreArgs sc{};
    sc.logits = c->ws.logits;
    sc.logit_ld = logit_ld(Ly.max_ctx);
    sc.lse2 = c->ws.lse2;
    sc.dbg_probs = refresh ? c->dbg_probs : nullptr;
    sc.max_ctx = Ly.max_ctx;
    sc.n_layers = Ly.n_layers;
    sc.batch = Ly.batch;
    sc.n_kv = Ly.n_kv_heads;
    sc.n_q = Ly.n_q_heads;
    sc.refresh = refresh ? 1 : 0;
    sc.alpha = c->alpha;
    if (c->rp.memdecay) {
        rc = timed_launch(c, kProfScore, s, "memdecay score",
                          [&] { return launch_memdecay_score(sc, pa, G, ub, s); });
    } else {
        rc = timed_launch(c, kProfScore, s, "paged score",
                          [&] { return launch_paged_score(sc, pa, G, ub, s); });
    }
    if (rc != KVEV_OK) return rc;
    if (c->rp.on) {
        rc = timed_launch(c, kProfSelect, s, "block budget",
                          [&] { return launch_block_budget(pa, s); });
        if (rc != KVEV_OK) return rc;
    }

    SelectArgs se{};
    se.n_units = pc->n_blocks;
    se.keys = c->ws.keys;
    se.retained = c->ws.sel;
    se.n_retained = n_retained;
    se.L = ub;
    se.max_ctx = pps;
    se.budget = c->rp.on ? pps : (int)c->budget;
    se.budgets = c->rp.on ? c->ws.budgets : nullptr;
    se.ret_ld = pa.sel_ld;
    se.refresh = 1;   // a new block's score was set by the append
    rc = timed_launch(c, kProfSelect, s, "select",
                      [&] { return launch_select(se, Ly.batch, c->num_sms, s); });
    if (rc != KVEV_OK) return rc;
    rc = timed_launch(c, kProfCompact, s, "paged compact",
                      [&] { return launch_paged_compact(pa, s); });
    if (rc != KVEV_OK) return rc;

    for (int b = 0; b < c->lay.batch; ++b) {
        int32_t& u = c->ub_blocks[b];
        // blocks kept at most: the budget, or (MemDecay) as many as hold the
        // budget's tokens with all but the last full; more only when pinned
        // blocks alone exceed it
        int cap = c->rp.memdecay ? (int)(c->budget / c->lay.page_tokens) + 1 : (int)c->budget;
        if (c->rp.on) {
            if ((c->rp.pinned_mask >> c->rp.decode_region) & 1u) cap = pps;
            else if (c->pin_blocks[b] > cap) cap = c->pin_blocks[b];
        }
        u = u + 1 < cap ? u + 1 : cap;
    }
    c->step = step;
    return KVEV_OK;
}

kvev_status kvev_readmit(kvev_ctx* c, const kvev_paged_cache* pc, const kvev_block_state* bs,
                         int32_t seq, int32_t lid, int32_t persist, void* stream) {
    const NvtxRange trace("kvev_readmit");
    kvev_status rc = check_paged(c, pc, bs);
    if (rc != KVEV_OK) return rc;
    if (!c->begun) return fail(KVEV_ESTATE, "kvev_paged_begin must come first");
    if (c->rp.on)
        return fail(KVEV_EUNSUPPORTED, "re-admission needs LRFU scoring without a region table "
                    "(the backing tier keeps no region labels)");
    if (seq < 0 || seq >= c->lay.batch)
        return fail(KVEV_EINVAL, "seq %d out of [0, %d)", seq, c->lay.batch);
    if (lid < 0 || lid >= pc->n_backing)
        return fail(KVEV_EINVAL, "lid %d is not a block of the backing tier [0, %d)", lid,
                    pc->n_backing);
    if (c->ub_blocks[seq] + 2 > pc->pages_per_seq)
        return fail(KVEV_EINVAL, "sequence %d may hold %d blocks: no page left for a re-admission "
                    "and the next step's new block", seq, c->ub_blocks[seq]);
    cudaStream_t s = (cudaStream_t)stream;
    const PagedArgs a = paged_args(c, pc, bs, (int)(c->step + 1), true);
    rc = timed_launch(c, kProfReadmit, s, "readmit",
                      [&] { return launch_readmit(a, seq, lid, persist != 0 ? 1 : 0, s); });
    if (rc != KVEV_OK) return rc;
    c->launches += 1;   // the copy kernel
    c->ub_blocks[seq] += 1;
    return KVEV_OK;
}

// ---- two-tier windows with an INT2 tier -----------------------------------

}  // extern "C"

namespace {

kvev_status check_tier(kvev_ctx* c, const kvev_tier_cache* tc, const kvev_tier_state* ts) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (c->lay.page_tokens != kTierW)
        return fail(KVEV_ESTATE, "not a two-tier context (layout.page_tokens must be %d)", kTierW);
    if (!tc || !ts) return fail(KVEV_EINVAL, "NULL argument");
    if (!tc->k_pool || !tc->v_pool || !tc->free_pages || !tc->n_free || !tc->ledger)
        return fail(KVEV_EINVAL, "tier cache has a NULL array");
    if (!aligned16(tc->k_pool) || !aligned16(tc->v_pool) || !aligned16(tc->ledger))
        return fail(KVEV_EINVAL, "pools and ledger must be 16-byte aligned");
    if (tc->max_windows != tier_max_windows(c->lay))
        return fail(KVEV_EINVAL, "max_windows %d != (max_ctx - 5) / 128 = %d", tc->max_windows,
                    tier_max_windows(c->lay));
    if (tc->pages_per_seq < 2) return fail(KVEV_EINVAL, "pages_per_seq must be >= 2");
    if (!ts->score || !ts->tier || !ts->has_codes || !ts->win_pages || !ts->n_windows ||
        !ts->tail_pages || !ts->tail_len)
        return fail(KVEV_EINVAL, "tier state has a NULL array");
    return KVEV_OK;
}

TierArgs tier_args(kvev_ctx* c, const kvev_tier_cache* tc, const kvev_tier_state* ts, int t) {
    TierArgs a{};
    a.c = *tc;
    a.st = *ts;
    a.bt = c->ws.t_bt;
    a.bpos = c->ws.t_bpos;
    a.blen = c->ws.t_blen;
    a.nblk = c->ws.t_nblk;
    a.bt_ld = tier_bt_ld(c->lay);
    a.qlist = c->ws.t_qlist;
    a.nq = c->ws.t_nq;
    a.seq_len = c->ws.t_seq_len;
    a.quant_list = c->ws.t_quant;
    a.n_quant = c->ws.t_nquant;
    a.prom_list = c->ws.t_prom;
    a.n_prom = c->ws.t_nprom;
    a.free_list = c->ws.t_free;
    a.n_freeing = c->ws.t_nfree;
    a.tile_stats = c->ws.t_stats;
    a.stats_tiles = tier_stats_tiles(c->lay);
    a.lse2 = c->ws.lse2;
    a.status = c->ws.status;
    a.batch = c->lay.batch;
    a.n_layers = c->lay.n_layers;
    a.n_kv = c->lay.n_kv_heads;
    a.n_q = c->lay.n_q_heads;
    a.head_dim = c->lay.head_dim;
    a.k_full = c->k_full;
    a.k_quant = c->k_quant;
    a.t = t;
    const bool cumulative = c->aggregation == KVEV_AGG_CUMULATIVE;
    a.alpha = cumulative ? 1.0f : c->alpha;
    a.oma = cumulative ? 1.0f : 1.0f - c->alpha;
    a.lir_streak = c->ws.lir_streak;
    a.lir_counters = c->lir_counters;
    a.lir_sustain = c->lir_sustain;
    a.rope = c->rope;
    a.scratch = c->t_scratch;
    a.rslot = c->ws.t_rslot;
    a.rfree = c->ws.t_rfree;
    a.n_rfree = c->ws.t_nrfree;
    a.rlist = c->ws.t_rlist;
    a.n_rlist = c->ws.t_nrlist;
    return a;
}

// bf16 pages a sequence holds (sink page, unrouted and Full windows, tail)
int tier_used_pages(const kvev_ctx* c) {
    const int n_u = c->t_nw - c->t_first_u;
    return 1 + (kTierW / kTile) * (n_u + c->t_nf) + (c->t_tl + kTile - 1) / kTile;
}

}  // namespace

extern "C" {

kvev_status kvev_tier_diagnostics(kvev_ctx* c, int32_t sustain, int32_t* counters,
                                  void* stream) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (c->lay.page_tokens != kTierW)
        return fail(KVEV_ESTATE, "not a two-tier context (layout.page_tokens must be %d)", kTierW);
    if (counters && sustain < 1) return fail(KVEV_EINVAL, "sustain must be >= 1");
    c->lir_counters = counters;
    c->lir_sustain = counters ? sustain : 0;
    if (!counters) return KVEV_OK;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(c->ws.lir_streak, 0,
                                    (size_t)c->lay.batch * tier_max_windows(c->lay) * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(counters, 0, (size_t)c->lay.batch * 3 * 4, s);
    if (e != cudaSuccess) return cuda_fail(e, "resetting the LIR counts");
    return KVEV_OK;
}

kvev_status kvev_set_tiers(kvev_ctx* c, int64_t k_full, int64_t k_quant, int32_t omega) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (c->lay.page_tokens != kTierW)
        return fail(KVEV_ESTATE, "not a two-tier context (layout.page_tokens must be %d)", kTierW);
    const int mw = tier_max_windows(c->lay);
    if (k_full < 0 || k_quant < 0 || k_full > mw || k_quant > mw || omega < 1)
        return fail(KVEV_EINVAL, "K_f, K_q must be in [0, %d] and omega >= 1", mw);
    if (c->rope && c->begun && (int)k_quant * (kTierW / kTile) > c->t_scratch)
        return fail(KVEV_ESTATE, "with rotary positions K_q cannot grow past %d after "
                    "kvev_tier_begin (its reconstruction pages are set aside there)",
                    c->t_scratch / (kTierW / kTile));
    c->k_full = (int)k_full;
    c->k_quant = (int)k_quant;
    c->omega = omega;
    return KVEV_OK;
}

kvev_status kvev_set_rope(kvev_ctx* c, const float* table, int32_t n_pos) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (c->lay.page_tokens != kTierW)
        return fail(KVEV_ESTATE, "not a two-tier context (layout.page_tokens must be %d)", kTierW);
    if (table) {
        if (c->lay.head_dim != 128) return fail(KVEV_EINVAL, "rotary mode needs head_dim 128");
        if (!aligned16(table)) return fail(KVEV_EINVAL, "the table must be 16-byte aligned");
        if (n_pos < c->lay.max_ctx)
            return fail(KVEV_EINVAL, "table of %d positions < max_ctx %d", n_pos,
                        c->lay.max_ctx);
    }
    c->rope_next = table;
    return KVEV_OK;
}

kvev_status kvev_tier_begin(kvev_ctx* c, const kvev_tier_cache* tc, const kvev_tier_state* ts,
                            int32_t prefill_tokens, void* stream) {
    kvev_status rc = check_tier(c, tc, ts);
    if (rc != KVEV_OK) return rc;
    if (prefill_tokens < kTierSinks || prefill_tokens >= c->lay.max_ctx)
        return fail(KVEV_EINVAL, "prefill_tokens %d must be in [%d, max_ctx)", prefill_tokens,
                    kTierSinks);
    const int hist = prefill_tokens - kTierSinks;
    const int used = 1 + (hist + kTile - 1) / kTile;
    const int scratch = c->rope_next ? c->k_quant * (kTierW / kTile) : 0;
    if (used + 1 > tc->pages_per_seq - scratch)
        return fail(KVEV_EINVAL, "pages_per_seq %d too small for a %d-token prefill%s",
                    tc->pages_per_seq, prefill_tokens,
                    scratch ? " and the INT2 windows' reconstruction pages" : "");
    cudaStream_t s = (cudaStream_t)stream;
    c->rope = c->rope_next;
    c->t_scratch = scratch;
    const TierArgs a = tier_args(c, tc, ts, 0);
    rc = timed_launch(c, kProfInit, s, "tier begin",
                      [&] { return launch_tier_begin(a, prefill_tokens, s); });
    if (rc != KVEV_OK) return rc;
    if (c->lir_counters) {   // Global LIR counts start over with the run
        cudaError_t e = cudaMemsetAsync(c->ws.lir_streak, 0,
                                        (size_t)c->lay.batch * tier_max_windows(c->lay) * 4, s);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(c->lir_counters, 0, (size_t)c->lay.batch * 3 * 4, s);
        if (e != cudaSuccess) return cuda_fail(e, "resetting the LIR counts");
    }
    c->t_nw = hist / kTierW;
    c->t_tl = hist % kTierW;
    c->t_first_u = 0;
    c->t_nf = c->t_nq = 0;
    c->t_recon_valid = true;   // the begin kernel frees every reconstruction slot
    c->len = prefill_tokens;
    c->prefill_len = prefill_tokens;
    c->step = 0;
    c->begun = true;
    return KVEV_OK;
}

kvev_status kvev_tier_step(kvev_ctx* c, const void* q, const void* k_new, const void* v_new,
                           const kvev_tier_cache* tc, const kvev_tier_state* ts, int64_t step,
                           void* out, void* stream) {
    const NvtxRange trace("kvev_tier_step");
    kvev_status rc = check_tier(c, tc, ts);
    if (rc != KVEV_OK) return rc;
    if (!q || !k_new || !v_new || !out) return fail(KVEV_EINVAL, "NULL argument");
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out))
        return fail(KVEV_EINVAL, "q, k_new, v_new and out must be 16-byte aligned");
    if (!c->begun) return fail(KVEV_ESTATE, "kvev_tier_begin must come before the first step");
    if (step != c->step + 1)
        return fail(KVEV_ESTATE, "step %lld out of order (expected %lld)", (long long)step,
                    (long long)(c->step + 1));
    if (c->len + 1 > c->lay.max_ctx)
        return fail(KVEV_EINVAL, "max_ctx %d positions reached", c->lay.max_ctx);
    const int pps = tc->pages_per_seq, PW = kTierW / kTile;
    const int t = (int)step;
    // host copy of the counts after the append
    int nw = c->t_nw, tl = c->t_tl + 1;
    if (tl == kTierW) {
        ++nw;
        tl = 0;
    }
    const int L = c->len + 1;
    const bool routing = t % c->omega == 0;
    int n_aged = 0, n_cand = 0, nf2 = c->t_nf, nq2 = c->t_nq;
    if (routing) {   // windows whose last token is below the recent region
        const int horizon = L - kTierRecent;
        const int aged_total = horizon >= kTierSinks + kTierW ? (horizon - kTierSinks) / kTierW : 0;
        n_aged = std::max(0, std::min(nw, aged_total) - c->t_first_u);
        n_cand = c->t_nf + c->t_nq + n_aged;
        nf2 = std::min(c->k_full, n_cand);
        nq2 = std::min(c->k_quant, n_cand - nf2);
    }
    {
        int saved_nw = c->t_nw, saved_tl = c->t_tl;
        c->t_nw = nw;
        c->t_tl = tl;
        const int used = tier_used_pages(c);
        c->t_nw = saved_nw;
        c->t_tl = saved_tl;
        const int prom = routing ? std::min(c->t_nq, nf2) : 0;
        if (used + PW * prom > pps - c->t_scratch)
            return fail(KVEV_EINVAL, "pages_per_seq %d too small: %d bf16 pages needed", pps,
                        used + PW * prom + c->t_scratch);
    }
    cudaStream_t s = (cudaStream_t)stream;
    const kvev_layout& Ly = c->lay;
    const int G = c->group;
    TierArgs ta = tier_args(c, tc, ts, t);
    // rotary positions: the INT2 windows are attended as bf16 reconstructions
    // (keys rotated forward), made when a window enters the tier; after an
    // import the append gives every INT2 window a slot and all are rebuilt
    const bool recon = c->rope != nullptr;
    const bool rebuild = recon && !c->t_recon_valid;
    TierArgs tb = ta;
    tb.rebuild = rebuild ? 1 : 0;
    rc = timed_launch(c, kProfAppend, s, "tier append", [&] {
        return launch_tier_append(tb, (const uint16_t*)k_new, (const uint16_t*)v_new, s);
    });
    if (rc != KVEV_OK) return rc;
    if (rebuild) {
        TierArgs ra = ta;
        ra.recon = 1;
        rc = timed_launch(c, kProfCompact, s, "reconstruct",
                          [&] { return launch_tier_promote(ra, c->t_nq, c->num_sms, s); });
        if (rc != KVEV_OK) return rc;
        c->t_recon_valid = true;
    }

    const int64_t rows = (int64_t)Ly.n_layers * Ly.batch * Ly.n_kv_heads;
    const int n_bf = 1 + PW * (nw - c->t_first_u + c->t_nf) + (tl + kTile - 1) / kTile +
                     (recon ? PW * c->t_nq : 0);
    AttnArgs at{};
    at.k = (const uint16_t*)tc->k_pool;
    at.v = (const uint16_t*)tc->v_pool;
    at.q = (const uint16_t*)q;
    at.part_o = c->ws.part_o;
    at.part_ml = c->ws.part_ml;
    at.status = c->ws.status;
    at.row0 = 0;
    at.tiles_per_row = n_bf;
    at.n_tiles_total = rows * n_bf;
    at.L = n_bf * kTile;
    at.max_ctx = Ly.max_ctx;
    at.n_layers = Ly.n_layers;
    at.batch = Ly.batch;
    at.n_kv = Ly.n_kv_heads;
    at.n_q = Ly.n_q_heads;
    int attn_grid = 0;
    at.total_warps = attn_launch_warps(c->attn_warps, at.n_tiles_total, &attn_grid);
    at.write_logits = 0;
    at.q_scale = (float)(1.4426950408889634 / sqrt((double)Ly.head_dim));
    at.view_tokens = (int64_t)Ly.batch * pps * Ly.n_layers * Ly.n_kv_heads * kTile;
    at.block_table = c->ws.t_bt;
    at.n_blocks = c->ws.t_nblk;
    at.blk_len = c->ws.t_blen;
    at.pps = tier_bt_ld(Ly);
    at.blk_pos = c->ws.t_bpos;
    at.tile_stats = c->ws.t_stats;
    at.stats_tiles = tier_stats_tiles(Ly);
    at.stats_base = kTierSinks;
    rc = timed_launch(c, kProfAttn, s, "attention",
                      [&] { return launch_attention(at, Ly.head_dim, G, attn_grid, s); });
    if (rc != KVEV_OK) return rc;
    CombineArgs cb{};
    cb.sp.part_o = c->ws.part_o;
    cb.sp.part_ml = c->ws.part_ml;
    cb.sp.n_tiles = at.n_tiles_total;
    cb.sp.row0 = 0;
    cb.sp.total_warps = at.total_warps;
    cb.sp.tiles_per_row = n_bf;
    if (c->t_nq > 0 && !recon) {
        Int2Args ia{};
        ia.ledger = (const unsigned char*)tc->ledger;
        ia.max_windows = tc->max_windows;
        ia.q_list = c->ws.t_qlist;
        ia.q_ld = tc->max_windows;
        ia.n_qwin = c->ws.t_nq;
        ia.q = (const uint16_t*)q;
        ia.part_o = c->ws.part_o2;
        ia.part_ml = c->ws.part_ml2;
        ia.tile_stats = c->ws.t_stats;
        ia.stats_tiles = tier_stats_tiles(Ly);
        ia.status = c->ws.status;
        ia.slots = c->t_nq;
        ia.n_units = rows * c->t_nq;
        ia.total_warps = c->int2_warps;
        ia.n_layers = Ly.n_layers;
        ia.batch = Ly.batch;
        ia.n_kv = Ly.n_kv_heads;
        ia.n_q = Ly.n_q_heads;
        ia.q_scale = at.q_scale;
        rc = timed_launch(c, kProfAttn, s, "int2 attention",
                          [&] { return launch_attn_int2(ia, Ly.head_dim, G, c->int2_grid, s); });
        if (rc != KVEV_OK) return rc;
        cb.has2 = 1;
        cb.sp2.part_o = c->ws.part_o2;
        cb.sp2.part_ml = c->ws.part_ml2;
        cb.sp2.n_tiles = ia.n_units;
        cb.sp2.row0 = 0;
        cb.sp2.total_warps = c->int2_warps;
        cb.sp2.tiles_per_row = c->t_nq;
    }
    cb.n_rows = (int32_t)rows;
    cb.out = out;
    cb.out_bf16 = c->out_type == KVEV_OUT_BF16 ? 1 : 0;
    cb.lse2 = c->ws.lse2;
    cb.n_layers = Ly.n_layers;
    cb.batch = Ly.batch;
    cb.n_kv = Ly.n_kv_heads;
    cb.n_q = Ly.n_q_heads;
    rc = timed_launch(c, kProfCombine, s, "combine",
                      [&] { return launch_combine(cb, Ly.head_dim, G, s); });
    if (rc != KVEV_OK) return rc;
    rc = timed_launch(c, kProfScore, s, "window score",
                      [&] { return launch_tier_score(ta, nw, G, s); });
    if (rc != KVEV_OK) return rc;
    if (routing) {
        const int n_quant_max = std::min(c->k_quant, n_cand);
        const int n_prom_max = std::min(c->t_nq, nf2);
        rc = timed_launch(c, kProfSelect, s, "route", [&] { return launch_tier_route(ta, s); });
        if (rc == KVEV_OK)
            rc = timed_launch(c, kProfCompact, s, "quantize", [&] {
                return launch_tier_quantize(ta, n_quant_max, c->num_sms, s);
            });
        if (rc == KVEV_OK)
            rc = timed_launch(c, kProfCompact, s, "promote", [&] {
                return launch_tier_promote(ta, n_prom_max, c->num_sms, s);
            });
        if (rc == KVEV_OK && recon) {   // the windows entering the INT2 tier (codes written)
            TierArgs ra = ta;
            ra.recon = 1;
            rc = timed_launch(c, kProfCompact, s, "reconstruct",
                              [&] { return launch_tier_promote(ra, nq2, c->num_sms, s); });
        }
        if (rc == KVEV_OK)
            rc = timed_launch(c, kProfCompact, s, "finish",
                              [&] { return launch_tier_finish(ta, s); });
        if (rc == KVEV_OK && c->lir_counters)
            rc = timed_launch(c, kProfSelect, s, "lir", [&] { return launch_tier_lir(ta, s); });
        if (rc != KVEV_OK) return rc;
        c->t_first_u += n_aged;
        c->t_nf = nf2;
        c->t_nq = nq2;
    }
    c->t_nw = nw;
    c->t_tl = tl;
    c->len = L;
    c->step = step;
    return KVEV_OK;
}

kvev_status kvev_profile(kvev_ctx* c, int32_t enable) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    c->prof = enable != 0;
    return KVEV_OK;
}

kvev_status kvev_profile_read(kvev_ctx* c, float* ms, int64_t* launches) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    kvev_status st = harvest_profile(c);
    if (st != KVEV_OK) return st;
    for (int k = 0; k < KVEV_PROFILE_SLOTS; ++k) {
        if (ms) ms[k] = c->prof_ms[k];
        if (launches) launches[k] = c->prof_n[k];
        c->prof_ms[k] = 0.f;
        c->prof_n[k] = 0;
    }
    return KVEV_OK;
}

kvev_status kvev_launch_count(const kvev_ctx* c, int64_t* launches) {
    if (!c || !launches) return fail(KVEV_EINVAL, "NULL argument");
    *launches = c->launches;
    return KVEV_OK;
}

// ---- checkpoint / resume ---------------------------------------------------

}  // extern "C"

namespace {

constexpr uint32_t kBlobMagic = 0x5645564bu;   // "KVEV"
constexpr uint32_t kBlobVersion = 3;

struct BlobHead {
    uint32_t magic, version;
    kvev_layout lay;
    int64_t budget;
    float alpha, beta;
    RegionParams rp;
    int32_t refresh_mode, refresh_period, age_mode, pool, out_type, aggregation, weighting;
    int32_t k_full, k_quant, omega;
    int32_t begun, len, prefill_len;
    int64_t step;
    int32_t t_nw, t_tl, t_first_u, t_nf, t_nq, t_scratch;
    int32_t n_ub, n_pin;          // then n_ub + n_pin int32 values
};

}  // namespace

extern "C" {

kvev_status kvev_export_state(const kvev_ctx* c, void* host, size_t* bytes) {
    if (!c || !bytes) return fail(KVEV_EINVAL, "NULL argument");
    const size_t need = sizeof(BlobHead) + 4 * (c->ub_blocks.size() + c->pin_blocks.size());
    if (!host) {
        *bytes = need;
        return KVEV_OK;
    }
    if (*bytes < need) return fail(KVEV_EINVAL, "buffer of %zu bytes, %zu needed", *bytes, need);
    BlobHead h;
    memset(&h, 0, sizeof h);   // no indeterminate padding in the blob
    h.magic = kBlobMagic;
    h.version = kBlobVersion;
    h.lay = c->lay;
    h.budget = c->budget;
    h.alpha = c->alpha;
    h.beta = c->beta;
    h.rp = c->rp;
    h.refresh_mode = c->refresh_mode;
    h.refresh_period = c->refresh_period;
    h.age_mode = c->age_mode;
    h.pool = c->pool;
    h.out_type = c->out_type;
    h.aggregation = c->aggregation;
    h.weighting = c->weighting;
    h.k_full = c->k_full;
    h.k_quant = c->k_quant;
    h.omega = c->omega;
    h.begun = c->begun ? 1 : 0;
    h.len = c->len;
    h.prefill_len = c->prefill_len;
    h.step = c->step;
    h.t_nw = c->t_nw;
    h.t_tl = c->t_tl;
    h.t_first_u = c->t_first_u;
    h.t_nf = c->t_nf;
    h.t_nq = c->t_nq;
    h.t_scratch = c->t_scratch;
    h.n_ub = (int32_t)c->ub_blocks.size();
    h.n_pin = (int32_t)c->pin_blocks.size();
    char* out = static_cast<char*>(host);
    memcpy(out, &h, sizeof h);
    memcpy(out + sizeof h, c->ub_blocks.data(), 4 * c->ub_blocks.size());
    memcpy(out + sizeof h + 4 * c->ub_blocks.size(), c->pin_blocks.data(),
           4 * c->pin_blocks.size());
    *bytes = need;
    return KVEV_OK;
}

kvev_status kvev_import_state(kvev_ctx* c, const void* host, size_t bytes, void* stream) {
    if (!c || !host) return fail(KVEV_EINVAL, "NULL argument");
    BlobHead h;
    if (bytes < sizeof h) return fail(KVEV_EINVAL, "blob of %zu bytes is too short", bytes);
    memcpy(&h, host, sizeof h);
    if (h.magic != kBlobMagic || h.version != kBlobVersion)
        return fail(KVEV_EINVAL, "not a kvev state blob (or another version)");
    if (memcmp(&h.lay, &c->lay, sizeof h.lay) != 0 || h.budget != c->budget ||
        h.alpha != c->alpha || !(h.beta == c->beta) || memcmp(&h.rp, &c->rp, sizeof h.rp) != 0)
        return fail(KVEV_EINVAL, "blob from a context with another layout, budget, alpha, beta "
                    "or region table");
    if (h.n_ub < 0 || h.n_pin < 0 || bytes < sizeof h + 4 * ((size_t)h.n_ub + h.n_pin))
        return fail(KVEV_EINVAL, "truncated blob");
    // Every blob this library exports satisfies these; a damaged one would
    // otherwise reach a division (the lazy period, the routing interval) or
    // size a launch.  Nothing of the context changes before they pass.
    const auto in_range = [](int64_t x, int64_t lo, int64_t hi) { return x >= lo && x <= hi; };
    const int32_t nb = c->lay.batch;
    bool sane = in_range(h.refresh_mode, KVEV_REFRESH_FULL, KVEV_REFRESH_FROZEN) &&
                h.refresh_period >= 1 && in_range(h.age_mode, 0, 1) && in_range(h.pool, 0, 1) &&
                in_range(h.out_type, KVEV_OUT_F32, KVEV_OUT_BF16) &&
                in_range(h.aggregation, KVEV_AGG_EMA, KVEV_AGG_CUMULATIVE) &&
                in_range(h.weighting, 0, KVEV_W_VNORM | KVEV_W_ENTROPY) &&
                h.omega >= 1 && h.step >= 0 && h.len >= 0 && h.prefill_len >= 0 &&
                (h.n_ub == 0 || h.n_ub == nb) && (h.n_pin == 0 || h.n_pin == nb);
    if (c->lay.page_tokens == kTierW) {
        const int mw = tier_max_windows(c->lay);
        sane = sane && in_range(h.k_full, 0, mw) && in_range(h.k_quant, 0, mw) &&
               in_range(h.t_nw, 0, mw) && in_range(h.t_first_u, 0, h.t_nw) &&
               in_range(h.t_tl, 0, kTierW - 1) && in_range(h.t_nf, 0, mw) &&
               in_range(h.t_nq, 0, mw);
        // rotary positions: the reconstruction pages set aside at the
        // exporter's kvev_tier_begin; a context without a table takes none
        constexpr int PW = kTierW / kTile;
        sane = sane && (c->rope_next ? in_range(h.t_scratch, PW * (int64_t)h.k_quant,
                                                PW * (int64_t)mw) && h.t_scratch % PW == 0
                                     : h.t_scratch == 0);
    } else {
        sane = sane && h.t_scratch == 0;
    }
    const char* in = static_cast<const char*>(host);
    for (int32_t i = 0; sane && i < h.n_ub + h.n_pin; ++i) {
        int32_t x;
        memcpy(&x, in + sizeof h + 4 * (size_t)i, 4);
        sane = x >= 0;
    }
    if (!sane) return fail(KVEV_EINVAL, "state blob with fields out of range (damaged?)");
    c->refresh_mode = h.refresh_mode;
    c->refresh_period = h.refresh_period;
    c->age_mode = h.age_mode;
    c->pool = h.pool;
    c->out_type = h.out_type;
    c->aggregation = h.aggregation;
    c->weighting = h.weighting;
    c->k_full = h.k_full;
    c->k_quant = h.k_quant;
    c->omega = h.omega;
    c->begun = h.begun != 0;
    c->len = h.len;
    c->prefill_len = h.prefill_len;
    c->step = h.step;
    c->t_nw = h.t_nw;
    c->t_tl = h.t_tl;
    c->t_first_u = h.t_first_u;
    c->t_nf = h.t_nf;
    c->t_nq = h.t_nq;
    c->rope = c->rope_next;
    c->t_scratch = h.t_scratch;
    c->t_recon_valid = false;   // reconstructions are rebuilt from the ledger
    c->ub_blocks.assign(h.n_ub, 0);
    c->pin_blocks.assign(h.n_pin, 0);
    c->diag_flags_valid = false;   // the raw-set flags are not part of a checkpoint
    memcpy(c->ub_blocks.data(), in + sizeof h, 4 * (size_t)h.n_ub);
    memcpy(c->pin_blocks.data(), in + sizeof h + 4 * (size_t)h.n_ub, 4 * (size_t)h.n_pin);
    {   // the caller's other cache buffer holds nothing the next step may reuse
        cudaStream_t s = (cudaStream_t)stream;
        cudaError_t e = cudaMemsetAsync(c->ws.vp, 0, (size_t)c->lay.batch * 8, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "resetting the reused-prefix counts");
    }
    if (c->lay.page_tokens == kTierW && c->begun) {   // positions so far, per sequence
        std::vector<int32_t> sl(c->lay.batch, c->len);
        cudaStream_t s = (cudaStream_t)stream;
        cudaError_t e = cudaMemcpyAsync(c->ws.t_seq_len, sl.data(), 4 * sl.size(),
                                        cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "restoring the sequence positions");
    }
    return KVEV_OK;
}

kvev_status kvev_test_wait_timeout(kvev_ctx* c, int64_t tile, uint32_t wait_limit) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (tile < 0 || wait_limit == 0) return fail(KVEV_EINVAL, "tile >= 0 and wait_limit >= 1");
    c->test_fault_tile = tile;
    c->test_wait_limit = wait_limit;
    return KVEV_OK;
}

kvev_status kvev_test_barrier_timeout(kvev_ctx* c, int32_t cta, uint32_t wait_limit) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    if (cta < 0 || wait_limit == 0) return fail(KVEV_EINVAL, "cta >= 0 and wait_limit >= 1");
    c->test_skip_cta = cta;
    c->test_bar_limit = wait_limit;
    return KVEV_OK;
}

kvev_status kvev_check_scratch(kvev_ctx* c, void* stream) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    cudaStream_t s = (cudaStream_t)stream;
    std::vector<unsigned char> band((size_t)c->ws.n_guard * kGuardBytes);
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < c->ws.n_guard && e == cudaSuccess; ++i)
        e = cudaMemcpyAsync(band.data() + (size_t)i * kGuardBytes, c->ws_base + c->ws.guard_off[i],
                            kGuardBytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the scratch guard bands");
    for (int i = 0; i < c->ws.n_guard; ++i)
        for (size_t k = 0; k < kGuardBytes; ++k)
            if (band[(size_t)i * kGuardBytes + k] != kGuardByte)
                return fail(KVEV_ESTATE, "scratch guard band after region %s overwritten at byte %zu",
                            c->ws.guard_name[i], k);
    return KVEV_OK;
}

kvev_status kvev_sync(kvev_ctx* c, void* stream) {
    if (!c) return fail(KVEV_EINVAL, "ctx is NULL");
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "pending CUDA error");
    return check_status_word(c, s);
}

}  // extern "C"
