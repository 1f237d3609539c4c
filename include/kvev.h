/*
 * kvev.h -- C ABI of the GB300 decode-time KV-cache eviction pass.
 *
 * One call, kvev_step, runs the whole per-decode-step pass on one CUDA
 * stream:
 *   1. append the new token's K/V in every layer and KV head;
 *   2. single-query GQA attention over the live cache, every layer at once,
 *      producing the attention output and the per-token probabilities
 *      ("What Matters for Aggressive Decoding-Time KV Eviction?", Sec. 3.1
 *      Eq. (1) and Appendix E "Per-step scoring");
 *   3. head pooling of those probabilities and the EMA fold of the per-token
 *      state, layer by layer in ascending order, kept across steps
 *      (kv-cache-docs figure "ema-eviction", EMA table; the same paper's
 *      Appendix E "Layer scoring");
 *   4. the eviction priority (1 - score) * (1 - exp(-beta * age))
 *      ("ema-eviction" figure, priority and decision matrix);
 *   5. selection of the B lowest-priority tokens, ties to the lower slot
 *      index, whenever the cache exceeds the budget (Sec. 3.1: evict the
 *      lowest-utility tokens whenever |cache| > B);
 *   6. stable compaction of the retained K/V rows and per-token state.
 * Lazy refresh and Score-Free (Sec. 3.2, Eq. (6)) skip steps 2's
 * probability capture and 3 on non-refresh steps.
 *
 * Conventions, for every entry point:
 *   - Device pointers are CUDA device memory of the current device, owned by
 *     the caller, contiguous, in the layouts stated; host pointers are said
 *     to be host pointers.  The context owns only its own scratch.
 *   - Every call returns a kvev_status.  Argument errors are reported before
 *     anything is launched and leave every buffer untouched.  A CUDA error
 *     raised by a launch, or an asynchronous fault of an earlier launch,
 *     returns KVEV_ECUDA; after that the cache and state are undefined.
 *   - kvev_last_error(ctx) gives a message for the last failing call on this
 *     thread (ctx may be NULL, e.g. after a failed kvev_create).
 *   - Calls taking a stream enqueue work on it asynchronously (NULL = the
 *     legacy default stream).  A context is not thread-safe: one context per
 *     stream.
 *   - All floating-point arithmetic on the device is fp32; K/V are bf16.
 */
#ifndef KVEV_H
#define KVEV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVEV_OK = 0,
    KVEV_EINVAL = 1,       /* bad argument (null pointer, size, range) */
    KVEV_ENOMEM = 2,       /* device or host allocation failed */
    KVEV_ECUDA = 3,        /* a CUDA call failed or an earlier launch faulted */
    KVEV_ESTATE = 4,       /* call out of order (step numbering, begin missing) */
    KVEV_ETIMEOUT = 5,     /* a bounded device wait gave up */
    KVEV_EUNSUPPORTED = 6  /* valid but not implemented for this layout */
} kvev_status;

typedef enum {
    KVEV_REFRESH_FULL = 0,    /* score every step */
    KVEV_REFRESH_LAZY = 1,    /* score at steps t with (t - 1) mod period == 0 */
    KVEV_REFRESH_FROZEN = 2   /* Score-Free: score at step 1 only */
} kvev_refresh;

typedef enum {
    KVEV_AGE_SINCE_INSERT = 0, /* age = t - insertion step */
    KVEV_AGE_SINCE_ACCESS = 1  /* age = t - last access; an access is a
                                  refresh step on which the token's attention,
                                  averaged over heads and layers, is at least
                                  2/L (MemDecay Sec. III-C Eq. (3), tau scaled
                                  to the uniform level); insertion counts */
} kvev_age_mode;

typedef enum {
    KVEV_POOL_SUM = 0,   /* s = sum over query heads of the probabilities */
    KVEV_POOL_MEAN = 1   /* s = mean over query heads (Sec. 3.1 Eq. (1)) */
} kvev_pool;

enum { KVEV_BF16 = 0 };

typedef struct {
    int32_t n_layers;     /* Ly */
    int32_t n_q_heads;    /* Hq; a multiple of n_kv_heads */
    int32_t n_kv_heads;   /* Hkv; query head h reads KV head h / (Hq/Hkv) */
    int32_t head_dim;     /* d: 64 or 128 */
    int32_t batch;        /* b: independent sequences */
    int32_t max_ctx;      /* slots per (layer, sequence, KV head) */
    int32_t page_tokens;  /* 1 = token-granular eviction; 16 = paged blocks */
    int32_t kv_dtype;     /* KVEV_BF16 */
} kvev_layout;
/* Size limit: the kernels address a cache buffer (or a page pool) as rows of
 * head_dim elements with 32-bit TMA coordinates, so
 * n_layers * batch * n_kv_heads * max_ctx must stay below 2^31.  The library
 * does not check this, because such a cache needs at least 2 x 256 GiB of K/V,
 * more than one GPU holds. */

/* The KV cache: two ping-pong buffers.  Each of k[0], k[1], v[0], v[1] is
 * [n_layers][batch][n_kv_heads][max_ctx][head_dim] bf16, 16-byte aligned.
 * Slots [0, len) of buffer `cur` are live.  kvev_step reads buffer `cur` and
 * appends into it.  When it evicts more than 8 tokens per sequence it writes
 * the compacted cache into the other buffer and flips `cur`; when it evicts
 * 1 to 8 (the steady state: one token in, one out) it shifts the rows after
 * the first evicted slot down within buffer `cur`, which stays live.  The
 * other buffer is the library's between steps: its leading rows still equal
 * the live buffer's up to the first slot a compaction since has moved, and
 * the next out-of-place compaction does not copy them again, so the caller
 * must not write into it during a run (from kvev_init_state or
 * kvev_import_state on). */
typedef struct {
    void* k[2];
    void* v[2];
    int32_t cur;
} kvev_cache;

/* Per-token state, each [batch][max_ctx], slot-aligned with the cache. */
typedef struct {
    float* score;    /* EMA state m (fp32) */
    int32_t* t_ins;  /* step at which the token was inserted (prefill: 0) */
    int32_t* t_ref;  /* step of the token's last access (prefill: 0) */
    int32_t* pos;    /* logical position of the token in its sequence */
} kvev_state;

typedef struct kvev_ctx kvev_ctx;

/* Region table (block granularity only): every cached token carries a
 * region label (uint8, < n_regions) supplied by the caller for the prefill;
 * decoded tokens take `decode_region`.  A block holding a token of a pinned
 * region is never evicted ("MemDecay: Region-Aware KV Cache Eviction ...",
 * Sec. III-A and IV-A: pinning protects whole pages).
 *   score_kind KVEV_SCORE_LRFU: the LRFU block priority of kvev_paged_step,
 *     with pinning; base_priority, decay_lambda, rho, attn_weight, tau_scale
 *     are unused.
 *   score_kind KVEV_SCORE_MEMDECAY: the MemDecay policy replaces the block
 *     EMA and priority.  Per token, at refresh (observation) steps:
 *       a <- rho a + (1 - rho) A,  A = the token's attention averaged over
 *            heads and layers                                     (Eq. (2))
 *       t_ref <- t  when A >= tau_scale / |K_t|                   (Eq. (3))
 *     and every step, for block p of the cache:
 *       s = base_priority[r] exp(-decay_lambda[r] (t - t_ref)) + attn_weight a
 *                                                                  (Eq. (4))
 *       S_p = mean of s over the block's tokens                   (Eq. (5))
 *     and while the cache holds more than `budget` TOKENS, the non-pinned
 *     block of least S_p is evicted (Algorithm 1; equal S_p: the later slot
 *     goes first).  kvev_create's alpha and beta are unused. */
enum { KVEV_MAX_REGIONS = 16 };
typedef enum { KVEV_SCORE_LRFU = 0, KVEV_SCORE_MEMDECAY = 1 } kvev_score_kind;
typedef struct {
    int32_t n_regions;                        /* 1 .. KVEV_MAX_REGIONS */
    float base_priority[KVEV_MAX_REGIONS];    /* b_r >= 0 */
    float decay_lambda[KVEV_MAX_REGIONS];     /* lambda_r >= 0, per decode step */
    uint8_t pinned[KVEV_MAX_REGIONS];         /* != 0: never evicted */
    int32_t score_kind;                       /* kvev_score_kind */
    float rho;                                /* in [0, 1) */
    float attn_weight;                        /* alpha of Eq. (4), >= 0 */
    float tau_scale;                          /* tau = tau_scale / |K_t|, >= 0 */
    int32_t decode_region;                    /* label of decoded tokens */
} kvev_region_table;

/* Create a context for `layout` with a budget of `budget` retained tokens
 * per sequence (1 <= budget < max_ctx).  `granularity` must equal
 * layout->page_tokens (1, or 16 for block-granular eviction, where the budget
 * counts blocks, or tokens under KVEV_SCORE_MEMDECAY).  `alpha` in (0, 1]
 * weights the new observation in the EMA; `beta` >= 0 is the recency
 * coefficient (+INFINITY allowed: rank by score, newest token protected).
 * `regions` is a kvev_region_table (copied) or NULL; it needs block
 * granularity.  Allocates the context's device scratch on the current
 * device (kvev_workspace_size bytes).  Defaults: full refresh, age since
 * insertion, head-sum pooling. */
kvev_status kvev_create(const kvev_layout* layout, int64_t budget, int32_t granularity,
                        float alpha, float beta, const kvev_region_table* regions,
                        kvev_ctx** out);

/* Release the context and its scratch.  NULL is a no-op. */
void kvev_destroy(kvev_ctx* ctx);

/* Message for the last failing call on this thread (never NULL). */
const char* kvev_last_error(const kvev_ctx* ctx);

/* Device scratch bytes that kvev_create allocates for this layout. */
kvev_status kvev_workspace_size(const kvev_layout* layout, int64_t budget, size_t* bytes);

/* Refresh schedule (Sec. 3.2): KVEV_REFRESH_FULL, KVEV_REFRESH_LAZY with
 * `period` >= 1, or KVEV_REFRESH_FROZEN.  Takes effect from the next step. */
kvev_status kvev_refresh_mode(kvev_ctx* ctx, int32_t mode, int32_t period);

/* Age definition (kvev_age_mode) and head pooling (kvev_pool). */
kvev_status kvev_configure(kvev_ctx* ctx, int32_t age_mode, int32_t pool);

/* Element type of the attention output `out` of kvev_step, kvev_step_host,
 * kvev_paged_step and kvev_tier_step (from the next step on):
 *   KVEV_OUT_F32   fp32, the combine's result as computed (default: it keeps
 *                  the accumulation's precision; the attention tolerance of
 *                  2e-3 relative is below bf16's own unit roundoff 2^-8 =
 *                  3.9e-3, so a bf16 output could not be held to it);
 *   KVEV_OUT_BF16  the same fp32 values rounded to bf16 (nearest even), half
 *                  the bytes, for a caller that feeds the output to a bf16
 *                  projection.
 * The pages state no output type: the attention output is the input of the
 * next layer, which the eviction pass does not compute. */
typedef enum { KVEV_OUT_F32 = 0, KVEV_OUT_BF16 = 1 } kvev_out_type;
kvev_status kvev_set_output(kvev_ctx* ctx, int32_t out_type);

/* Score aggregation and weighting of token-granular contexts ("What Matters
 * for Aggressive Decoding-Time KV Eviction?", Sec. 3.1 Eqs. (2)-(4) and
 * Appendix E "Per-step scoring"); from the next step on.
 *   aggregation  KVEV_AGG_EMA (default): m <- alpha s_l + (1 - alpha) m per
 *                layer (alpha = 1 is the single-step rule, Eq. (2));
 *                KVEV_AGG_CUMULATIVE: m <- m + s_l per layer (Eq. (3), the
 *                H2O-style sum that never forgets; alpha is unused).
 *   weighting    bit mask, applied on refresh steps before the fold:
 *                KVEV_W_VNORM: each query head's probability of token i times
 *                ||v_i|| / (mean over the cached tokens of ||v_j||), the value
 *                rows of its KV head in that layer (factor 1 when every norm
 *                is 0); KVEV_W_ENTROPY: the layer's pooled score times the
 *                mean over query heads of H(p_h) / ln L (H the entropy of the
 *                head's attention over the L cached tokens; 1 when L = 1).
 *                The access clock keeps reading the plain attention.
 * The attention gathers the weightings' statistics (value norms from the
 * tiles it already holds, the entropy from its softmax sums), so neither
 * reads the cache again.  Block-granular and two-tier contexts take only
 * the defaults (KVEV_EUNSUPPORTED otherwise). */
/* Fused refresh step (token granularity; from the next step): on refresh
 * steps without a weighting, KVEV_FUSED_ALL runs the attention, the split
 * combine and the scoring as ONE cooperative launch, their phases separated
 * by grid barriers, instead of three launches; KVEV_FUSED_ATTN_COMBINE fuses
 * the attention and the combine only (the scorer keeps its own launch);
 * KVEV_FUSED_OFF (default) launches the three kernels.  The arithmetic is
 * the three kernels' own, in the same order; the outputs are the same bit
 * for bit whenever the attention splits its tiles over the same number of
 * warps (the same CTAs per SM).  Every barrier wait is bounded: one that
 * gives up reports KVEV_ETIMEOUT at the next kvev_sync.  No counterpart on
 * the pages (their implementation reads the attention weights through a
 * separate eager pass: "What Matters...", Appendix J).  KVEV_EUNSUPPORTED for
 * shapes without a fused kernel (head_dim 64 or 128, 4 or 8 query heads per
 * KV head, 1, 2 or 8 KV heads are built). */
enum { KVEV_FUSED_OFF = 0, KVEV_FUSED_ALL = 1, KVEV_FUSED_ATTN_COMBINE = 2 };
kvev_status kvev_set_fused_step(kvev_ctx* ctx, int32_t mode);

typedef enum { KVEV_AGG_EMA = 0, KVEV_AGG_CUMULATIVE = 1 } kvev_aggregation;
enum { KVEV_W_VNORM = 1, KVEV_W_ENTROPY = 2 };
kvev_status kvev_set_scorer(kvev_ctx* ctx, int32_t aggregation, int32_t weighting);

/* Start a decode run: every sequence holds `prefill_len` live tokens
 * (0 <= prefill_len < max_ctx) and the next step is step 1. */
kvev_status kvev_begin(kvev_ctx* ctx, int32_t prefill_len);

/* Live tokens per sequence after the last step (or kvev_begin). */
kvev_status kvev_length(const kvev_ctx* ctx, int32_t* len);

/* Write the prefill state on `stream`: for every sequence and slot i below
 * the prefill length, score = 0, t_ins = t_ref = 0, pos = i (Appendix E
 * "Momentum initialization": m0 = 0).  The next compaction copies every
 * retained row (nothing in the other cache buffer is reused). */
kvev_status kvev_init_state(kvev_ctx* ctx, const kvev_state* state, void* stream);

/* One decode step `step` (must be the previous step + 1; the first step
 * after kvev_begin is 1).  Device inputs:
 *   q      [batch][n_layers][n_q_heads][head_dim] bf16
 *   k_new  [batch][n_layers][n_kv_heads][head_dim] bf16
 *   v_new  [batch][n_layers][n_kv_heads][head_dim] bf16
 * Device outputs:
 *   out           [batch][n_layers][n_q_heads][head_dim] attention output of
 *                 this step (over the cache including the new token), fp32
 *                 or bf16 as kvev_set_output chose
 *   retained_idx  [batch][budget] int32: the retained slots of the cache as it
 *                 was after the append, ascending; after the call retained
 *                 slot retained_idx[b][j] lives at slot j.  When the cache
 *                 does not exceed the budget nothing is evicted and the list
 *                 is 0..len-1.
 *   n_retained    [batch] int32: entries written to retained_idx.
 * `cache` and `state` are read and updated (cache->cur flips when the step
 * evicts more than 8 tokens per sequence). */
kvev_status kvev_step(kvev_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                      kvev_cache* cache, const kvev_state* state, int64_t step, void* out,
                      int32_t* retained_idx, int32_t* n_retained, void* stream);

/* kvev_step with the per-step inputs and outputs in HOST memory (pinned
 * memory gives asynchronous copies; pageable memory works too): copies
 * q/k_new/v_new to the context's device staging, runs the step, copies
 * out/retained_idx/n_retained back and synchronizes `stream` before
 * returning.  Same layouts as kvev_step; the cache and state stay on the
 * device. */
kvev_status kvev_step_host(kvev_ctx* ctx, const void* q_host, const void* k_new_host,
                           const void* v_new_host, kvev_cache* cache, const kvev_state* state,
                           int64_t step, void* out_host, int32_t* retained_idx_host,
                           int32_t* n_retained_host, void* stream);

/* Ranking diagnostics of token-granular steps ("What Matters for
 * Aggressive Decoding-Time KV Eviction?", Sec. 5.3 and Appendix I, Table 13),
 * computed on the device by every later step (counters NULL disables them):
 *   counters   [batch][KVEV_DIAG_FIELDS] int32, per step and sequence:
 *              step t, refreshed (1 on scoring steps), |R| (the raw top-B
 *              set: the `budget` tokens of largest raw score, ties to the
 *              lower slot; 0 on non-scoring steps), |E| (the retained set),
 *              |R & E|, |R & R_prev| (tokens of the previous scoring step's
 *              raw set still cached), |R_prev| (0 before the second scoring
 *              step), |E & E_prev| (retained tokens held before this step);
 *              raw/EMA Jaccard = |R & E| / (|R| + |E| - |R & E|), raw churn =
 *              1 - |R & R_prev| / (|R| + |R_prev| - |R & R_prev|), EMA churn
 *              likewise from |E & E_prev|, raw-top evicted = 1 - |R & E|/|R|;
 *   raw_score  [batch][max_ctx] fp32 or NULL: each slot's raw score of
 *              scoring steps (the attention summed over query heads and
 *              layers, before any aggregation), slots of the cache after the
 *              append (before compaction).
 * The raw score is the scorer's own sum (no extra read of the cache); the
 * raw set costs one more selection launch and the counts one small kernel
 * per step.  Block-granular and two-tier contexts: KVEV_EUNSUPPORTED. */
enum { KVEV_DIAG_FIELDS = 8 };
kvev_status kvev_set_diagnostics(kvev_ctx* ctx, int32_t* counters, float* raw_score);

/* Future Missed Mass (QEvict review, Sec. 3 "Diagnosing the problem") of one
 * step of a compressed run against a FullKV run of the same inputs: per
 * sequence b,
 *   out[b] = 1 - (sum over the positions p the policy holds of F[b][p] +
 *                 F[b][n_pos - 1]) / (sum over p < n_pos of F[b][p])
 * with F the FullKV run's raw scores by position (e.g. the raw_score output
 * of a context whose budget is never reached, where slot = position) after
 * its step over n_pos positions, and pos[b][0 .. n_cached) the positions
 * the policy held before its own step over the same new token (its
 * kvev_state.pos and kvev_length then); the new token (position n_pos - 1)
 * counts as held and positions outside [0, n_pos - 1) are ignored.  No
 * context, no allocation; asynchronous on `stream`. */
kvev_status kvev_missed_mass(const float* full_score, int32_t score_ld, int32_t n_pos,
                             const int32_t* pos, int32_t pos_ld, int32_t n_cached,
                             int32_t batch, float* out, void* stream);

/* Optional diagnostic outputs written by later steps (NULL disables):
 *   probs     [batch][n_layers][n_q_heads][max_ctx] fp32, the attention
 *             probabilities of refresh steps over slots [0, L) of the cache
 *             after the append;
 *   priority  [batch][max_ctx] fp32, every step's eviction priority of slots
 *             [0, L), before compaction.
 * The pointers must stay valid while set. */
kvev_status kvev_set_debug(kvev_ctx* ctx, float* probs, float* priority);

/* Per-kernel timing with CUDA events on the step's stream.  Enable, run
 * steps, then kvev_profile_read fills `ms[i]` (accumulated milliseconds) and
 * `launches[i]` for kernel i in the order append, attention, combine, score,
 * select, compact, state set-up (kvev_init_state, kvev_paged_begin),
 * re-admission (KVEV_PROFILE_SLOTS entries each; pass NULL to skip) and
 * resets the accumulators.  kvev_profile_read synchronizes. */
enum { KVEV_PROFILE_SLOTS = 8 };
kvev_status kvev_profile(kvev_ctx* ctx, int32_t enable);
kvev_status kvev_profile_read(kvev_ctx* ctx, float* ms, int64_t* launches);

/* Total kernel launches this context has made (all entry points). */
kvev_status kvev_launch_count(const kvev_ctx* ctx, int64_t* launches);

/* Test-only failure injection: in the next kvev_step the attention kernel
 * arms tile `tile` of its launch but issues none of its copies, and every
 * bounded device wait gives up after `wait_limit` iterations; the warp that
 * waits on that tile gives up, records the timeout in the device status word
 * and returns after its other copies have landed, so kvev_sync (or
 * kvev_step_host) returns KVEV_ETIMEOUT and the context stays usable (the
 * step's outputs are undefined).  No counterpart on the pages. */
kvev_status kvev_test_wait_timeout(kvev_ctx* ctx, int64_t tile, uint32_t wait_limit);

/* Test-only failure injection for the fused step: in the next fused step CTA
 * `cta` leaves without arriving at the first grid barrier and every barrier
 * wait gives up after `wait_limit` iterations, so the other CTAs stop waiting,
 * flag the status word and leave; kvev_sync then returns KVEV_ETIMEOUT, the
 * barrier state is reset and the context stays usable (the step's outputs are
 * undefined).  No counterpart on the pages. */
kvev_status kvev_test_barrier_timeout(kvev_ctx* ctx, int32_t cta, uint32_t wait_limit);

/* Debugging aid: every region of the context's scratch is followed by a
 * 256-byte guard band filled at create; this call reads the bands back
 * (synchronising `stream`) and returns KVEV_ESTATE naming the first region
 * whose band was overwritten, KVEV_OK when all are intact. */
kvev_status kvev_check_scratch(kvev_ctx* ctx, void* stream);

/* Block until `stream`'s work is done; returns KVEV_ECUDA on a device fault. */
kvev_status kvev_sync(kvev_ctx* ctx, void* stream);

/* ---- Block-granular eviction with score persistence ----------------------
 * layout->page_tokens = P > 1 (16 in the paged workloads), budget = blocks.
 * The LRFU policy per (sequence, token block) of the kv-cache-docs figure
 * "ema-eviction": per layer a block's new score is the max over its tokens of
 * the head-summed probability, folded into the block's EMA (layers in
 * ascending order); the priority (1 - score)(1 - exp(-beta age)) is per
 * block; the B blocks of lowest priority are kept, ties to the lower slot.
 * When a block is evicted its score is stored under (sequence, logical
 * block) and restored when the block is re-admitted.  K/V rows never move:
 * eviction only frees pages.  Slot order is ascending logical block id
 * (prefill blocks 0.., then blocks opened by decoding); new tokens fill the
 * last block while it has room, else open a new one. */
typedef struct {
    void* k_pool;            /* [n_pages][n_layers][n_kv_heads][P][head_dim] bf16,
                                n_pages = batch * pages_per_seq, 16-byte aligned */
    void* v_pool;
    int32_t pages_per_seq;   /* sequence b owns pages [b*pps, (b+1)*pps) */
    int32_t* block_table;    /* [batch][pps] page of each live block, slot order */
    int32_t* n_blocks;       /* [batch] live blocks */
    int32_t* free_pages;     /* [batch][pps] stack of free pages */
    int32_t* n_free;         /* [batch] */
    int32_t* next_lid;       /* [batch] logical id of the next block decoding opens */
    const void* backing_k;   /* [batch][n_backing][n_layers][n_kv_heads][P][head_dim]
                                bf16: the prefill blocks, for re-admission (may be NULL) */
    const void* backing_v;
    int32_t n_backing;
} kvev_paged_cache;

/* Per live block, each [batch][pps], slot-aligned with block_table. */
typedef struct {
    float* score;            /* EMA state of the block */
    int32_t* t_ins;          /* step the block was opened (prefill: 0) */
    int32_t* t_ref;          /* step of its last access (insertion, re-admission,
                                or a token of it accessed: KVEV_AGE_SINCE_ACCESS) */
    int32_t* lid;            /* logical block id */
    int32_t* len;            /* tokens in the block (1..P) */
    float* table;            /* [batch][table_len] persisted score per logical block
                                (NaN = never stored) */
    int32_t table_len;       /* > every logical id used */
    /* Per token, indexed [page][P] (pages never move), with a region table: */
    uint8_t* region;         /* region label; the caller writes the prefill's */
    float* tok_a;            /* KVEV_SCORE_MEMDECAY: importance a */
    int32_t* tok_t_ref;      /* KVEV_SCORE_MEMDECAY: decay clock t_ref */
} kvev_block_state;

/* Start a paged run.  `prefill_tokens` (> 0) per sequence are already in
 * the pool: block j of sequence b at page b*pps + j, the last one partial
 * when P does not divide prefill_tokens.  Sets the block tables, free lists,
 * per-block state (score 0, t_ins = t_ref = 0, lid j), empties the persisted
 * table, and with KVEV_SCORE_MEMDECAY sets tok_a = 0, tok_t_ref = 0 for the
 * prefill tokens; the next step is 1.  With a region table it reads the
 * prefill labels back to the host (to bound the pinned blocks) and
 * synchronizes `stream`. */
kvev_status kvev_paged_begin(kvev_ctx* ctx, const kvev_paged_cache* cache,
                             const kvev_block_state* state, int32_t prefill_tokens, void* stream);

/* One paged decode step `step` (previous + 1).  q, k_new, v_new, out as in
 * kvev_step.  retained_lid [batch][budget] int32 (device; [batch][pps] with a
 * region table): logical ids of the kept blocks in slot order; n_retained
 * [batch] int32 (device).  With a region table and LRFU scoring, every
 * pinned block is kept even when they outnumber the budget.  Launches
 * append, attention, combine, block scoring, selection and compaction.  The
 * host keeps an upper bound of each sequence's live blocks; a step whose
 * new block could find no free page returns KVEV_EINVAL before launching.
 * Debug outputs (kvev_set_debug) are indexed by block slot: probabilities
 * [batch][n_layers][n_q_heads][max_ctx] at slot j*P + k for token k of
 * block j, priorities [batch][pps] (the page score S_p under
 * KVEV_SCORE_MEMDECAY). */
kvev_status kvev_paged_step(kvev_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                            const kvev_paged_cache* cache, const kvev_block_state* state,
                            int64_t step, void* out, int32_t* retained_lid,
                            int32_t* n_retained, void* stream);

/* Re-admit prefill block `lid` (0 <= lid < n_backing, a full block) of
 * sequence `seq` (LRFU scoring without a region table, else
 * KVEV_EUNSUPPORTED: the backing tier keeps no region labels)
 * before the next step (a no-op when it is resident): a free page receives
 * the block's K/V from the backing tier, the block returns to its slot
 * (ascending logical id), its score is the persisted one (persist != 0 and
 * one was stored) or 0, its insertion step 0 and its access time the next
 * step.  Rejected (KVEV_EINVAL) when the sequence could be left without a
 * page for the next step's new block; KVEV_ESTATE at the next kvev_sync if
 * no page was free on the device. */
kvev_status kvev_readmit(kvev_ctx* ctx, const kvev_paged_cache* cache,
                         const kvev_block_state* state, int32_t seq, int32_t lid,
                         int32_t persist, void* stream);

/* ---- Two-tier window routing with an INT2 tier ---------------------------
 * "QEvict: Recoverable Quantized KV Eviction for Attention-Drift-Robust
 * Long-Context Decoding" (review page, Sec. 4): layout->page_tokens = 128
 * (the window W), budget = K_f.  Tokens [0, 5) are sinks; windows are
 * [5 + 128 j, 5 + 128 (j + 1)); the tokens after the last complete window
 * (the tail) and the sinks stay in bf16 and are always attended.  Every step
 * each live window's score folds the attention its tokens receive, averaged
 * over query heads, into an EMA (weight alpha on the new value) layer after
 * layer; every `omega` steps (at the end of steps t with t mod omega = 0)
 * the candidates (Full and INT2 windows, and new windows whose last token is
 * older than the 32 most recent) are ranked by score, ties to the lower
 * index: the top K_f are Full (bf16), the next K_q INT2, the rest evicted for
 * good (Eqs. (4)-(5)).  A window is quantized on its first demotion and its
 * codes are kept in a ledger and reused on every later demotion; a promoted
 * window is dequantized from the ledger into bf16 pages.  Attention runs over
 * the bf16 pages and, dequantizing in the kernel, the INT2 windows.
 * INT2 codec: keys per channel over 32-token groups, values per token over
 * 32-channel groups; zero = fp16(min), scale = fp16((max - min) / 3) in fp32,
 * code = clamp(rint((x - zero) / scale), 0, 3) in fp32 (0 when scale = 0);
 * value = code * scale + zero in fp32; a promoted copy rounds it to bf16.
 * Supported: head_dim 128, 4 query heads per KV head. */
enum { KVEV_TIER_NONE = 0, KVEV_TIER_UNROUTED = 1, KVEV_TIER_FULL = 2, KVEV_TIER_QUANT = 3,
       KVEV_TIER_EVICTED = 4 };
enum { KVEV_TIER_SINKS = 5, KVEV_TIER_RECENT = 32, KVEV_TIER_WINDOW = 128 };
typedef struct {
    void* k_pool;            /* [batch * pps][n_layers][n_kv_heads][16][head_dim] bf16 pages */
    void* v_pool;
    int32_t pages_per_seq;   /* pps: sequence b owns pages [b*pps, (b+1)*pps) */
    int32_t* free_pages;     /* [batch][pps] free-page stacks */
    int32_t* n_free;         /* [batch] */
    void* ledger;            /* [batch][max_windows][n_layers][n_kv_heads][12288 B] INT2
                                codes + fp16 scale/zero of each quantized window */
    int32_t max_windows;     /* (layout->max_ctx - 5) / 128 */
} kvev_tier_cache;

typedef struct {
    float* score;            /* [batch][max_windows] window EMA */
    uint8_t* tier;           /* [batch][max_windows] KVEV_TIER_* */
    uint8_t* has_codes;      /* [batch][max_windows] ledger entry valid */
    int32_t* win_pages;      /* [batch][max_windows][8] bf16 pages of a Full or unrouted window */
    int32_t* n_windows;      /* [batch] complete windows so far */
    int32_t* tail_pages;     /* [batch][8] bf16 pages of the tail */
    int32_t* tail_len;       /* [batch] tokens after the last complete window */
} kvev_tier_state;

/* Tier capacities K_f (Full windows), K_q (INT2 windows) and the routing
 * interval omega >= 1 (Eq. (3) gives K_f, K_q from a byte budget).  The
 * window score is the EMA above by default; kvev_set_scorer with
 * KVEV_AGG_CUMULATIVE makes it Sec. 4.2 Eq. (1)'s cumulative score: the
 * head-averaged window attention added up over steps and layers, never
 * decaying. */
kvev_status kvev_set_tiers(kvev_ctx* ctx, int64_t k_full, int64_t k_quant, int32_t omega);

/* Global LIR (Long-term Importance Revival, the QEvict review's Sec. 3
 * "Diagnosing the problem"): how often a window that stayed out of the Full
 * tier for a sustained period re-enters it.  With `counters` set
 * ([batch][3] int32, device), every later routing event adds per sequence
 * {1 routing event, revivals, sustained-inactive spans}: a routed window
 * outside Full (INT2 or evicted) at `sustain` routing events in a row opens
 * a span; such a window routed to Full counts a revival and its count
 * restarts.  Windows not yet routed do not count.  LIR = revivals / spans.
 * This call and kvev_tier_begin zero the counts (enqueued on `stream`);
 * counters = NULL turns the bookkeeping off. */
kvev_status kvev_tier_diagnostics(kvev_ctx* ctx, int32_t sustain, int32_t* counters,
                                  void* stream);

/* Rotary positions (the QEvict review, Sec. 4.4 "Positional handling for
 * promoted keys"): the cached keys are the model's rotated keys, and
 * `table` ([n_pos][head_dim/2][2] fp32 (cos, sin) of position p and
 * frequency j, device, 16-byte aligned, n_pos >= layout->max_ctx; the
 * caller keeps it alive while the context steps) is the model's own
 * rotation.  A window is quantized in the pre-rotation domain: each key of
 * position p is rotated back by p before the codec, channel pairs
 * (j, j + 64), every product and sum rounded to fp32:
 *     x_j = y_j cos + y_{j+64} sin,  x_{j+64} = y_{j+64} cos - y_j sin;
 * every use of an INT2 window rotates the dequantized key forward again
 * (y_j = x_j cos - x_{j+64} sin, y_{j+64} = x_{j+64} cos + x_j sin):
 * a promoted window's bf16 key is that value rounded to bf16, and the INT2
 * windows are attended as bf16 reconstructions (keys rotated, keys and
 * values rounded to bf16).  These live in the last 8 K_q pages of each
 * sequence's range, which kvev_tier_begin sets aside (pages_per_seq must
 * hold them too; K_q cannot grow past that value later): 8 pages per INT2
 * window, written at the routing event where the window enters the INT2
 * tier and kept while it stays there; the first step after
 * kvev_import_state writes them all again.
 * table = NULL turns the mode off.  Two-tier contexts with head_dim 128
 * only; takes effect at the next kvev_tier_begin or kvev_import_state (a
 * blob imports only into a context whose table is set as the exporter's
 * was, else KVEV_EINVAL). */
kvev_status kvev_set_rope(kvev_ctx* ctx, const float* table, int32_t n_pos);

/* Start a tiered run over a prefill of `prefill_tokens` (>= 5) tokens that
 * the caller wrote into the pool: tokens 0..4 in rows 0..4 of page b*pps,
 * token 5 + 16 i + r in row r of page b*pps + 1 + i.  All complete windows
 * start unrouted (bf16) with score 0; the next step is 1. */
kvev_status kvev_tier_begin(kvev_ctx* ctx, const kvev_tier_cache* cache,
                            const kvev_tier_state* state, int32_t prefill_tokens, void* stream);

/* One tiered decode step `step` (previous + 1): q, k_new, v_new, out as in
 * kvev_step; afterwards state->tier holds every window's tier (a routing
 * event at the end of this step included). */
kvev_status kvev_tier_step(kvev_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                           const kvev_tier_cache* cache, const kvev_tier_state* state,
                           int64_t step, void* out, void* stream);

/* ---- Checkpoint / resume -------------------------------------------------
 * A context's own state: the run's position (step, live length, the host's
 * per-sequence block bounds and tier counts) and its configuration (refresh
 * schedule, age and pooling modes, tier capacities).  Everything else a
 * checkpoint needs is in the caller's device buffers (cache, per-token or
 * per-block state, block tables, score table, ledger), which the caller
 * saves and restores itself; no counterpart on the pages beyond the
 * persistence of scores across eviction.
 * kvev_export_state: host memory; with host == NULL only *bytes is set to the
 * size; otherwise *bytes must be at least that size and is set to it.
 * kvev_import_state: a blob exported by a context created with the same
 * layout, budget, alpha, beta and region table (else KVEV_EINVAL); the next
 * step is the exported step + 1.  Enqueued on `stream` (two-tier contexts
 * restore a small device counter). */
kvev_status kvev_export_state(const kvev_ctx* ctx, void* host, size_t* bytes);
kvev_status kvev_import_state(kvev_ctx* ctx, const void* host, size_t bytes, void* stream);

/* Attention of the pass without allocating: no counterpart on the pages;
 * it exists for callers that cannot call cudaMalloc (engines whose allocator
 * owns all device memory, latency-critical paths that cannot take the
 * implicit synchronisation of cudaMalloc/cudaFree).  Runs the split-K
 * attention and split combine of kvev_step, with no context, keeping the
 * split partials in a 16 MiB array in device memory that belongs to the
 * library image (every GPU that loads the library holds it until exit).
 * With the same layout and cache it splits the work as kvev_step does, so
 * `out` equals kvev_step's fp32 output bit for bit.
 *   q      [batch][n_layers][n_q_heads][head_dim] bf16 (device)
 *   k, v   ONE cache buffer, [n_layers][batch][n_kv_heads][max_ctx][head_dim]
 *          bf16 (device); slots [0, len) are attended, 1 <= len <= max_ctx
 *   out    [batch][n_layers][n_q_heads][head_dim] fp32 (device)
 *   lse2   [n_layers][batch][n_q_heads] fp32 (device): log2 of the softmax
 *          normaliser, i.e. ln(sum_i exp(q.k_i/sqrt(d))) / ln 2
 * Limits: head_dim 64 or 128, 4 or 8 query heads per KV head, and
 * n_layers*batch*n_kv_heads at most floor((16 MiB - 256) / (4 G (head_dim +
 * 2))) minus the attention warps per CTA (4 in the default build), G the
 * query heads per KV head: 8061 at head_dim 128 and 15883 at 64 with G = 4;
 * larger layouts return KVEV_EINVAL, with the limit in the message, before
 * anything is launched.  layout->page_tokens and kv_dtype are ignored (bf16
 * tokens).  The first call on a device looks up the array's address (make
 * it before any stream capture); the address is kept for the life of the
 * process, so the entry point must not be called after cudaDeviceReset.
 * All calls share the array: calls that overlap on the GPU race; order them
 * on one stream.  Asynchronous on `stream`.  A device wait that gives up is
 * not reported by this call: the rows it touched come out NaN in `out` and
 * `lse2`. */
kvev_status kvev_attend_noalloc(const kvev_layout* layout, const void* q, const void* k,
                                const void* v, int32_t len, float* out, float* lse2,
                                void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVEV_H */
