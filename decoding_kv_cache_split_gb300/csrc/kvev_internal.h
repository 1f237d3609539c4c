// Internal declarations of the kvev CUDA library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvev.h"

namespace kvev {

constexpr uint32_t kWaitLimit = 1u << 22;   // iteration cap of every device spin-wait

// Device status word bits (ctx->status_word); read by kvev_sync / kvev_step_host.
enum : uint32_t { kStatusTimeout = 1u };

// Work decomposition of the split-K attention: every (layer, sequence, KV head)
// "row" of the cache is cut into tiles of kTile tokens; the tiles of all rows,
// in row order, are dealt out to the grid's warps in equal contiguous ranges
// (so every warp streams the same number of bytes).  Warp w's piece of row r
// writes its softmax partial to slot w + r.
constexpr int kTile = 16;

struct AttnArgs {
    const uint16_t* k;     // cache buffer [rows][max_ctx][D] (rows = Ly*b*Hkv)
    const uint16_t* v;
    const uint16_t* q;     // [b][Ly][Hq][D]
    float* logits;         // [rows][logit_ld][G] log2-domain scaled logits (refresh)
    int32_t logit_ld;      // token stride of a logits row: max_ctx rounded up to 8, so
                           // every 128-byte line holds 8 tokens of one row
    float* part_o;         // [slots][G][D]
    float* part_ml;        // [slots][G][2] running max (log2 domain), sum
    uint32_t* status;
    int64_t n_tiles_total; // rows of this launch * tiles_per_row
    int64_t row0;          // first (layer, sequence, KV head) row of this launch
    int32_t tiles_per_row;
    int32_t L;             // live tokens per row (after the append)
    int32_t max_ctx;
    int32_t n_layers, batch, n_kv, n_q;
    int32_t total_warps;
    int32_t write_logits;
    float q_scale;         // log2(e) / sqrt(D)
    int64_t view_tokens;   // rows of the 2-D (token x D) view of k / v for the tensor maps
    // Block-granular cache (block_table non-null): k / v are page pools
    // [pages][Ly][Hkv][kTile][D]; tile j of a row is the sequence's j-th live
    // block (tiles at or past n_blocks[b] are empty); L is unused.
    const int32_t* block_table;   // [batch][pps]
    const int32_t* n_blocks;      // [batch]
    const int32_t* blk_len;       // [batch][pps]
    int32_t pps;
    // Optional (block mode): position of each block's first token; the
    // logits of a block go to that position (else to tile index * kTile).
    const int32_t* blk_pos;       // [batch][pps] or null
    // Optional per-tile softmax statistics instead of logits: for every
    // tile at position p >= stats_base (p - stats_base a multiple of kTile),
    // (running max, sum of exp2(logit - running max)) per head at
    // tile_stats[((row * stats_tiles) + (p - stats_base) / kTile) * G + h].
    float2* tile_stats;
    int32_t stats_tiles, stats_base;
    // Test-only: bounded-wait iterations (0: kWaitLimit) and 1 + the tile of
    // the launch whose copies are not issued (0: none), to exercise the
    // timeout path without a fault.  Zero-initialised arguments inject nothing.
    uint32_t wait_limit;
    int64_t fault_tile_p1;
    // Optional statistics of the scorer's weightings (token mode, refresh
    // steps): part_e [slots][G] the split's sum of exp2(x - running max) * x
    // per head (x the log2-domain logit), merged like the softmax sum into
    // each head's entropy; vnorm [rows][logit_ld] the l2 norm of each
    // token's value row, and part_vn [slots] the split's sum of those norms.
    float* part_e;
    float* vnorm;
    float* part_vn;
};

// The fused refresh step (attention, split combine and scoring in one
// cooperative launch, phases separated by grid barriers).
struct FusedArgs {
    uint32_t* bar;          // [2] grid barrier: arrivals, generation (zero at rest)
    uint32_t wait_limit;    // bounded barrier wait (0: kWaitLimit)
    int32_t skip_cta_p1;    // test-only: 1 + a CTA that leaves without arriving (0: none)
    int32_t score;          // 1: the scoring phase too; 0: it stays a launch of its own
};

// Attention statistics the scorer's weightings need (template flags of the
// attention kernel; 0 = the plain kernel).
enum : int { kStatEntropy = 1, kStatVNorm = 2 };

// Where one attention launch left its split partials: warp w's piece of the
// launch's row r (rows counted from row0) is slot w + r.
struct SplitPartials {
    const float* part_o;   // [slots][G][D]
    const float* part_ml;  // [slots][G][2]
    int64_t n_tiles;       // tiles of the launch
    int64_t row0;
    int32_t total_warps;
    int32_t tiles_per_row;
};

// Warps of the split whose tile range is empty write no partial.
// floor(a / n) for 0 <= a < 2^62, 0 < n, when the quotient is below 2^22:
// a single-precision estimate (off by at most one there) fixed with exact
// 64-bit products, instead of a 64-bit integer division.
__device__ __forceinline__ int64_t small_quotient(int64_t a, int64_t n) {
    if (n <= 0) return 0;
    int64_t q = (int64_t)__fdividef((float)a, (float)n);
    if (q < 0) q = 0;
    while (q * n > a) --q;
    while ((q + 1) * n <= a) ++q;
    return q;
}
__device__ __forceinline__ bool split_warp_has_tiles(int64_t w, int64_t N, int64_t W) {
    return N >= W || w * N / W != (w + 1) * N / W;   // every warp has a tile when N >= W
}
// The warps whose tile ranges meet launch row r: [*lo, *hi] (some may be empty).
__device__ __forceinline__ void split_warps_of_row(const SplitPartials& p, int64_t r,
                                                   int64_t* lo, int64_t* hi) {
    const int64_t first = r * p.tiles_per_row, last = first + p.tiles_per_row - 1;
    const int64_t W = p.total_warps, N = p.n_tiles;
    *lo = small_quotient((first + 1) * W - 1, N);   // the largest w with floor(w N / W) <= tile
    *hi = small_quotient((last + 1) * W - 1, N);
}

struct CombineArgs {
    SplitPartials sp;      // the attention launch to merge (its rows from sp.row0)
    // Optional weighting statistics of sp (null: not gathered):
    const float* part_e;   // [slots][G] -> ent [rows][G]: each head's attention
    float* ent;            //   entropy over log2 of the row's tokens (1 if <= 1 token)
    const float* part_vn;  // [slots]    -> vmean [rows]: mean l2 norm of the
    float* vmean;          //   row's value rows
    int32_t n_tokens;      // live tokens of every row (token mode)
    SplitPartials sp2;     // a second launch over the same rows (has2), e.g. the INT2 tier
    int32_t has2;
    int32_t n_rows;        // rows of that launch
    void* out;             // [b][Ly][Hq][D], fp32 or (out_bf16) bf16
    int32_t out_bf16;      // 1: round the fp32 result to bf16 (nearest even)
    float* lse2;           // [rows][G] = [Ly][b][Hq]
    int32_t n_layers, batch, n_kv, n_q;
};


constexpr int kScoreSegs = 4;     // layer segments of the refresh scorer (a warp each)
constexpr int kScoreSegMax = 8;   // room for the scorer's layer segments
static_assert(kScoreSegs <= kScoreSegMax, "ScoreArgs holds one decay per segment");

struct ScoreArgs {
    const float* logits;   // [rows][logit_ld][G]
    int32_t logit_ld;
    // Aggregation and weightings ("What Matters..." Sec. 3.1 Eqs. (3)-(4),
    // Appendix E "Per-step scoring"): per layer m <- alpha s + oma m (EMA:
    // oma = 1 - alpha; cumulative: alpha = oma = 1); ent [rows][G] per-head
    // normalized entropies whose head mean weighs a layer (null: 1); vnorm /
    // vmean the VNorm factors of each (row, token) (null: 1).
    float oma;
    const float* ent;
    const float* vnorm;
    const float* vmean;
    const float* lse2;     // [Ly][b][Hq] log2-sum-exp from the split combine
    kvev_state st;         // caller's state (read)
    float* m_s;            // scratch [b][max_ctx] updated score
    int32_t* tref_s;       // scratch updated t_ref
    int32_t* tins_s;       // scratch copy of t_ins
    int32_t* pos_s;        // scratch copy of pos
    uint32_t* keys;        // scratch [b][max_ctx] order-preserving priority bits
    float* msum_part;      // [b][gridDim.x] partial sums of the old tokens' scores
    float* dbg_probs;      // [b][Ly][Hq][max_ctx] or null
    float* dbg_prio;       // [b][max_ctx] or null
    int32_t L, max_ctx, n_layers, batch, n_kv, n_q;
    int32_t refresh, age_mode, pool_mean;
    int32_t t;
    float alpha, beta, access_thr;   // access: sum over layers of head-summed p >= access_thr
    // ranking diagnostics (refresh steps): the raw per-step score (the
    // head-summed probability summed over layers) as a sortable key that
    // ranks the largest first, and optionally as a value
    uint32_t* raw_keys;    // [b][max_ctx] or null
    float* dbg_raw;        // [b][max_ctx] or null
    // oma^n for the layers n of each scorer segment 1.. (kScoreSegs segments
    // of the layers in order), formed in fp64 on the host and rounded once
    float seg_decay[kScoreSegMax];
};

// Ranking diagnostics of one token-mode step (diag.cu).
struct DiagArgs {
    const int32_t* retained;    // [b][budget] kept slots (ascending), n_retained [b]
    const int32_t* n_retained;
    const int32_t* raw_list;    // [b][budget] top-B slots of the raw score (refresh)
    const int32_t* raw_n;       // [b]
    uint8_t* in_raw;            // [b][max_ctx] scratch
    const uint8_t* flags_in;    // [b][max_ctx] slot in the last raw set (pre-step cache)
    uint8_t* flags_out;         // [b][max_ctx] the same after this step's compaction
    int32_t* prev_n;            // [b] size of the last raw set
    int32_t* counters;          // [b][KVEV_DIAG_FIELDS] user output
    int32_t L, max_ctx, budget, t, refresh, flags_valid;
};

struct MissedMassArgs {
    const float* full_score;    // [b][score_ld] FullKV raw score by position
    const int32_t* pos;         // [b][pos_ld] positions the policy holds
    float* out;                 // [b]
    int32_t score_ld, n_pos, pos_ld, n_cached;
};

struct SelectArgs {
    const int32_t* n_units;   // [b] units per sequence on the device (paged mode), or null: L
    const uint32_t* keys;
    float* m_s;
    const float* msum_part;
    int32_t n_part;
    int32_t* retained;     // [b][budget]
    int32_t* n_retained;   // [b]
    int32_t L, max_ctx, budget, refresh;   // L: upper bound of n_units when n_units is set
    const int32_t* budgets;   // [b] per-sequence kept count (null: budget)
    int32_t staged;           // 1: the launch reserved shared memory for the keys of
                              //    its longest chunk (select_stages_keys on the host)
    int32_t ret_ld;           // row stride of retained (0: budget)
    int32_t* first_moved;     // [b] first slot not kept (L when none), or null
    int32_t* evicted;         // [b][kFewEvict] evicted slots, ascending, when L - B
                              //    <= kFewEvict (the maxima path), or null
    int32_t few;              // 1: every sequence evicts at most kFewEvict (host-known):
                              //    one CTA per sequence, no cluster
};

struct CompactArgs {
    const uint16_t* k_src; const uint16_t* v_src;
    uint16_t* k_dst; uint16_t* v_dst;
    const int32_t* retained;   // [b][budget]
    const float* m_s; const int32_t* tref_s; const int32_t* tins_s; const int32_t* pos_s;
    kvev_state st;             // written
    int32_t n_keep;            // retained per sequence (min(L, budget))
    int32_t identity;          // 1: no eviction, state only
    int32_t rows, batch, n_kv, max_ctx, budget, head_dim;
    // Reused prefix: vp_in[b] leading rows of the destination buffer already
    // equal the source's (it was the source of an earlier step), so rows below
    // min(vp_in[b], first_moved[b]) are not copied; vp_out[b] is that count for
    // the next step's destination (this step's source).  Null: copy all.
    const int32_t* first_moved;
    const int32_t* vp_in;
    int32_t* vp_out;
    // In place (few evictions): the sources are the destinations' buffer and
    // slot j's source is j plus the number of evicted slots e_i with
    // e_i - i <= j (evicted: [b][kFewEvict], ascending, n_evict of them).
    int32_t in_place;
    int32_t n_evict;
    const int32_t* evicted;
};

struct AppendArgs {
    uint16_t* k; uint16_t* v;            // live buffer
    const uint16_t* k_new; const uint16_t* v_new;   // [b][Ly][Hkv][D]
    kvev_state st;
    int32_t slot, t, pos, n_layers, batch, n_kv, max_ctx, head_dim;
};

// Region table as the kernels take it (by value).
struct RegionParams {
    int32_t on;             // a region table is set
    int32_t memdecay;       // KVEV_SCORE_MEMDECAY
    int32_t decode_region;
    uint32_t pinned_mask;   // bit r: region r pinned
    float base[KVEV_MAX_REGIONS];
    float lam[KVEV_MAX_REGIONS];
    float rho, attn_w, tau_scale;
    int32_t budget_tokens;  // MemDecay budget in tokens
};

// Block-granular (paged) mode: the caller's structures plus this context's
// per-block scratch (slot-indexed [b][pps], written by the scorer).
struct PagedArgs {
    kvev_paged_cache c;
    kvev_block_state st;
    int32_t* tokens;       // [b] live tokens (for the access threshold)
    float* m_s;            // scratch copies of the block state after scoring
    int32_t* tref_s;
    int32_t* tins_s;
    int32_t* lid_s;
    int32_t* len_s;
    int32_t* page_s;
    uint32_t* keys;        // [b][pps]
    const int32_t* sel;    // [b][budget] kept slots from the selection
    const int32_t* n_sel;  // [b]
    int32_t* retained_lid; // [b][budget] user output
    int32_t* readmit_page; // [1] page chosen by the last re-admission (-1: none)
    uint32_t* status;
    int32_t batch, n_layers, n_kv, n_q, head_dim, page, budget;
    int32_t t, refresh, age_mode, pool_mean;
    float alpha, beta;
    float* dbg_prio;       // [b][pps] or null
    int32_t sel_ld;        // row stride of sel and retained_lid (budget, or pps)
    int32_t* budgets;      // [b] with a region table: blocks the selection keeps
    RegionParams rp;
};

// Two-tier (bf16 + INT2 windows) mode.
constexpr int kTierW = KVEV_TIER_WINDOW;    // tokens per window
constexpr int kTierSinks = KVEV_TIER_SINKS;
constexpr int kTierRecent = KVEV_TIER_RECENT;
constexpr int kQGroup = 32;                 // quantization group
constexpr int kTierRouteCap = 2048;         // windows per sequence the routing sort holds

// Byte layout of one (window, layer, KV head) ledger entry at head_dim D,
// arranged for the INT2 attention kernel's tensor-core fragments (m16n8k16,
// lane = 4 g + t): per 16-token tile ti, lane L's D/32 code words sit at
// words ti * D + L * (D / 32) .. + D / 32 - 1 of kc / vc, one 16-byte load.
//   kc: a key word has 8 fields f; a field holds two codes (half e) as plain
//       2-bit numbers at bits 2 f + 16 e, + 1.  Field f is an operand register
//       after a right shift by 6 (f / 3) and a mask to bits 2 (f % 3), + 1 of
//       each half: the bf16 pair c 2^(2 (f % 3)) 2^-133 (exact subnormals),
//       two shifts and eight masks per word.  Key code (token 16 ti + 8 i + g,
//       channel 16 s + 8 h + 2 t + e) sits in field 3 (s % 3) + s / 3 of word
//       2 i + h of lane 4 g + t, so the four registers of k-step s share the
//       scale class s / 3 that the A operand undoes (the B operand of
//       S = Q K^T);
//   vc: a value word carries 8 operand registers (slot 0..7) of two codes
//       each (half e); a register is the word rotated right by 2 slot, masked
//       to its sign bits 15, 31 and magnitude bits 6, 22, with bits 5, 21 set:
//       the bf16 pair (2 c - 3) * 2^-128 (exact subnormals; sign = c <= 1,
//       magnitude 3 for c = 0 or 3, else 1).  Value code (token 16 ti + 8 h +
//       2 t + e, channel 8 j + g) sits in register 2 j + h of lane 4 g + t (the
//       B operand of O += P V; centred codes keep the output sums, which run
//       over whole rows, near the size of the result);
//   ks, kz: fp16 key scale / zero of (group, channel 16 s + 8 h + 2 t + e) at
//       group * D + t * D / 4 + 4 s + 2 h + e (a lane's 32 channels together);
//   vs, vz: fp16 value scale / zero of (token 16 ti + 8 h + 2 t + e, channel
//       group cg) at ti * 16 G + t * 4 G + h * 2 G + 2 cg + e, G = D / 32.
template <int D>
struct LedgerLayout {
    static_assert(D == 128, "the key fields cover 8 k-steps");
    static constexpr int NG = D / kQGroup;   // channel groups of a value row
    static constexpr int KC = 0;
    static constexpr int KS = KC + kTierW * D / 4;
    static constexpr int KZ = KS + (kTierW / kQGroup) * D * 2;
    static constexpr int VC = KZ + (kTierW / kQGroup) * D * 2;
    static constexpr int VS = VC + kTierW * D / 4;
    static constexpr int VZ = VS + kTierW * NG * 2;
    static constexpr int BYTES = VZ + kTierW * NG * 2;
    static constexpr int WORDS_PER_LANE = D / 32;
    // key fields: k-step s -> field, and the low bit of a field's half e (the
    // code's high bit is the next)
    __host__ __device__ static constexpr int key_field(int s) { return 3 * (s % 3) + s / 3; }
    __host__ __device__ static constexpr int key_bit(int field, int e) { return 2 * field + 16 * e; }
    // value words: the bit of the sign (the magnitude bit is 9 below)
    __host__ __device__ static int code_word(int ti, int lane, int w) {
        return ti * D + lane * WORDS_PER_LANE + w;
    }
    __host__ __device__ static int sign_bit(int reg, int e) {
        return (15 + 16 * e + 2 * (reg & 7)) & 31;
    }
    __host__ __device__ static int mag_bit(int reg, int e) {
        return (6 + 16 * e + 2 * (reg & 7)) & 31;
    }
    // key code (token in window, channel) -> word, field, half
    __host__ __device__ static void key_place(int tok, int c, int* word, int* field, int* e) {
        const int ti = tok >> 4, i = (tok >> 3) & 1, g = tok & 7;
        const int s = c >> 4, h = (c >> 3) & 1, t = (c & 7) >> 1;
        *field = key_field(s);
        *e = c & 1;
        *word = code_word(ti, 4 * g + t, 2 * i + h);
    }
    // value code (token in window, channel) -> word, register, half
    __host__ __device__ static void value_place(int tok, int c, int* word, int* reg, int* e) {
        const int ti = tok >> 4, h = (tok >> 3) & 1, t = (tok & 7) >> 1;
        const int j = c >> 3, g = c & 7;
        *reg = 2 * j + h;
        *e = tok & 1;
        *word = code_word(ti, 4 * g + t, *reg >> 3);
    }
    __host__ __device__ static int key_scale_index(int grp, int c) {
        return grp * D + ((c & 7) >> 1) * (D / 4) + 4 * (c >> 4) + 2 * ((c >> 3) & 1) + (c & 1);
    }
    __host__ __device__ static int value_scale_index(int tok, int cg) {
        return (tok >> 4) * 16 * NG + ((tok & 7) >> 1) * 4 * NG + ((tok >> 3) & 1) * 2 * NG +
               2 * cg + (tok & 1);
    }
};
// (sign, magnitude) bits of a code and back
__host__ __device__ inline uint32_t code_sign(uint32_t c) { return c <= 1u; }
__host__ __device__ inline uint32_t code_mag(uint32_t c) { return c == 0u || c == 3u; }
__host__ __device__ inline uint32_t code_from_bits(uint32_t sign, uint32_t mag) {
    return sign ? (mag ? 0u : 1u) : (mag ? 3u : 2u);
}

struct Int2Args {
    const unsigned char* ledger;
    int32_t max_windows;
    const int32_t* q_list;   // [b][q_ld] INT2 windows, ascending
    int32_t q_ld;
    const int32_t* n_qwin;   // [b]
    const uint16_t* q;       // [b][Ly][Hq][D]
    float* part_o;           // [slots][G][D]
    float* part_ml;          // [slots][G][2]
    float2* tile_stats;      // as AttnArgs
    int32_t stats_tiles;
    uint32_t* status;
    int64_t n_units;         // rows * slots
    int32_t slots;           // units per row (INT2 windows per sequence, at most)
    int32_t total_warps;
    int32_t n_layers, batch, n_kv, n_q;
    float q_scale;
};

struct TierArgs {
    kvev_tier_cache c;
    kvev_tier_state st;
    int32_t* bt;             // [b][bt_ld] attention block list (pages), rebuilt every step
    int32_t* bpos;
    int32_t* blen;
    int32_t* nblk;           // [b]
    int32_t bt_ld;
    int32_t* qlist;          // [b][max_windows] INT2 windows, ascending
    int32_t* nq;             // [b]
    int32_t* seq_len;        // [b] positions so far
    int32_t* quant_list;     // [b][max_windows] routing event lists
    int32_t* n_quant;
    int32_t* prom_list;
    int32_t* n_prom;
    int32_t* free_list;
    int32_t* n_freeing;
    const float2* tile_stats;
    int32_t stats_tiles;
    const float* lse2;
    uint32_t* status;
    int32_t batch, n_layers, n_kv, n_q, head_dim;
    int32_t k_full, k_quant;
    int32_t t;
    float alpha;           // window score per layer: m <- alpha s + oma m (EMA:
    float oma;             //   oma = 1 - alpha; cumulative, Eq. (1): both 1)
    // Global LIR bookkeeping (null: off): routing events each window has
    // spent outside the Full tier in a row, and per sequence the counts
    // {routing events, revivals, sustained-inactive spans}
    int32_t* lir_streak;   // [b][max_windows]
    int32_t* lir_counters; // [b][3]
    int32_t lir_sustain;
    // Rotary positions ("QEvict" review Sec. 4.4): keys are quantized rotated
    // back by their positions and rotated forward again on promotion; the
    // INT2 windows are attended as bf16 reconstructions in the last
    // `scratch` pages of each sequence's range, PW pages per reconstruction
    // slot (null rope: off, scratch 0).  A window holds a slot while it is
    // INT2: routing frees the slots of windows leaving the tier and gives
    // the entering ones a slot and a reconstruction.
    const float* rope;     // [positions][D/2][2] fp32 (cos, sin)
    int32_t scratch;
    int32_t* rslot;        // [b][max_windows] reconstruction slot (-1: none)
    int32_t* rfree;        // [b][max_windows] free-slot stacks
    int32_t* n_rfree;      // [b]
    int32_t* rlist;        // [b][max_windows] windows to reconstruct + counts
    int32_t* n_rlist;
    int32_t recon;         // tier_promote_kernel: 1 = reconstruct the windows of rlist
    int32_t rebuild;       // tier_append_kernel: 1 = slots and rlist anew from the INT2 list
};

// ---- programmatic dependent launch ----------------------------------------
// Every kernel of the pass is launched with programmatic stream serialisation:
// it may be scheduled while its predecessor drains, and waits in
// griddep_wait() (before touching global memory) until the predecessor has
// completed and its writes are visible.  griddep_release() lets the next
// kernel start being scheduled.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_release() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ---- launchers (return cudaGetLastError of the launch) --------------------
int attn_ctas_per_sm(int head_dim, int group);
size_t attn_smem_bytes(int head_dim, int group);
cudaError_t launch_attention(const AttnArgs& a, int head_dim, int group, int grid,
                             cudaStream_t s, int stats = 0);
cudaError_t launch_combine(const CombineArgs& a, int head_dim, int group, cudaStream_t s);
// 0 when the shape has no fused step
int attn_fused_ctas_per_sm(int head_dim, int group, int n_kv);
cudaError_t launch_attn_fused(const AttnArgs& a, const CombineArgs& cb, const ScoreArgs& sc,
                              const FusedArgs& f, int head_dim, int group, int grid,
                              cudaStream_t s);
cudaError_t launch_score(const ScoreArgs& a, int group, int* n_blocks, cudaStream_t s);
cudaError_t launch_select(const SelectArgs& a, int batch, int num_sms, cudaStream_t s);
cudaError_t launch_diag(const DiagArgs& a, int batch, cudaStream_t s);
cudaError_t launch_missed_mass(const MissedMassArgs& a, int batch, cudaStream_t s);
cudaError_t launch_compact(const CompactArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);
cudaError_t launch_init_state(kvev_state st, int batch, int max_ctx, int len, int32_t* vp,
                              cudaStream_t s);
cudaError_t launch_paged_begin(const PagedArgs& a, int prefill_tokens, cudaStream_t s);
cudaError_t launch_paged_append(const PagedArgs& a, const uint16_t* k_new, const uint16_t* v_new,
                                cudaStream_t s);
cudaError_t launch_paged_score(const ScoreArgs& sc, const PagedArgs& a, int group, int ub_blocks,
                               cudaStream_t s);
cudaError_t launch_paged_compact(const PagedArgs& a, cudaStream_t s);
cudaError_t launch_readmit(const PagedArgs& a, int seq, int lid, int persist, cudaStream_t s);
cudaError_t launch_memdecay_score(const ScoreArgs& sc, const PagedArgs& a, int group,
                                  int ub_blocks, cudaStream_t s);
cudaError_t launch_block_budget(const PagedArgs& a, cudaStream_t s);
int int2_ctas_per_sm(int head_dim, int group);
int int2_warps_per_cta();
cudaError_t launch_attn_int2(const Int2Args& a, int head_dim, int group, int grid, cudaStream_t s);
cudaError_t launch_tier_begin(const TierArgs& a, int prefill_tokens, cudaStream_t s);
cudaError_t launch_tier_append(const TierArgs& a, const uint16_t* k_new, const uint16_t* v_new,
                               cudaStream_t s);
cudaError_t launch_tier_score(const TierArgs& a, int max_nw, int group, cudaStream_t s);
cudaError_t launch_tier_route(const TierArgs& a, cudaStream_t s);
cudaError_t launch_tier_quantize(const TierArgs& a, int max_items, int num_sms, cudaStream_t s);
cudaError_t launch_tier_promote(const TierArgs& a, int max_items, int num_sms, cudaStream_t s);
cudaError_t launch_tier_finish(const TierArgs& a, cudaStream_t s);
cudaError_t launch_tier_lir(const TierArgs& a, cudaStream_t s);

enum : uint32_t { kStatusNoPage = 2u };   // a sequence ran out of free pages
enum : uint32_t { kStatusRouteCap = 4u };  // more windows than the routing sort holds
enum : uint32_t { kStatusBarrier = 8u };   // with kStatusTimeout: a grid-barrier wait gave up

constexpr int kScoreThreads = 256;

// Selection: the keys of a sequence are cut into `cl` chunks (one per CTA of
// its cluster); a CTA stages its chunk in shared memory when the launch's
// longest chunk fits kSelChunkCap keys (the host then reserves that much
// dynamic shared memory).  A sequence shorter than the launch's longest
// (block mode: fewer live blocks) stages exactly when the launch did, so a
// kernel never stages into memory the launch did not reserve.
constexpr int kSelChunkCap = 10240;
// Steps evicting at most this many units select by block maxima and (token
// mode) compact in place.
constexpr int kFewEvict = 8;
__host__ __device__ inline int select_chunk(int n_keys, int cl) { return (n_keys + cl - 1) / cl; }
__host__ __device__ inline bool select_stages_keys(int launch_keys, int cl) {
    return select_chunk(launch_keys, cl) <= kSelChunkCap;
}
// dynamic shared memory a selection launch reserves per CTA
__host__ __device__ inline size_t select_smem_bytes(int launch_keys, int cl) {
    return select_stages_keys(launch_keys, cl) ? 4 * (size_t)select_chunk(launch_keys, cl) : 0;
}

}  // namespace kvev
