/*
 * kvev_oracle.c -- plain, slow fp64 CPU oracle for the decode-time KV-cache
 * eviction pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference leg call this code.  It shares nothing
 * with the CUDA path: no headers, no helpers, no tables.
 *
 * Every function below is the plain definition from the pages, written out
 * with no blocking, no online softmax, no radix select:
 *
 *   attention   "What Matters for Aggressive Decoding-Time KV Eviction?" (p1),
 *               Sec. 3.1 Eq. (1) and Appendix E "Per-step scoring": last-query
 *               attention weights of every head over every cached position;
 *               with GQA each KV head serves its query-head group.
 *   pooling     p1 Eq. (1) (head mean) / the head sum used by the eviction
 *               configurations; selected by `pool_mean`.
 *   weighting   p1 Appendix E "Per-step scoring", optional: VNorm multiplies
 *               each head's attention to token i by the l2 norm of token i's
 *               value state (its KV head) over the mean of those norms across
 *               the cached tokens, before pooling; entropy weighting
 *               multiplies the layer's pooled score by the normalized entropy
 *               of its attention distributions (their entropy over ln L,
 *               averaged over the query heads).
 *   EMA         "ema-eviction" figure (kv-cache-docs, ch07), worked EMA
 *               table: score = alpha*new + (1-alpha)*score.  Applied once per
 *               layer in ascending layer order, the state carried across
 *               steps: p1 Appendix E "Layer scoring".
 *   cumulative  p1 Sec. 3.1 Eq. (3), the aggregation that never forgets:
 *               score = score + new, per layer in the same order.  (Eq. (2),
 *               single-step, is the EMA with alpha = 1.)
 *   refresh     p1 Sec. 3.2 Eq. (6) (lazy refresh) and "Score-Free
 *               decoding"; new tokens on non-refresh steps take the mean
 *               momentum of the existing tokens (p1 Appendix E "New token
 *               insertion during non-refresh steps"); momentum starts at 0
 *               (p1 Appendix E "Momentum initialization").
 *   access      MemDecay (arXiv 2607.10582) Sec. III-C Eq. (3): the clock
 *               resets when the token's head/layer-averaged attention reaches
 *               tau = 2/|K_t| (the scaled threshold of its Sec. IV).
 *   priority    "ema-eviction" figure: priority = (1 - score) * (1 -
 *               exp(-beta * steps)); a higher priority is evicted.
 *   selection   p1 Sec. 3.1 ("evict the tokens with the lowest m" whenever
 *               the cache exceeds B): keep the B smallest priorities, ties to
 *               the lower slot index; pinned slots are forced in (MemDecay
 *               Sec. III-A Eq. (1)).
 *   compaction  the retained slots, in ascending slot order, become slots
 *               0..B-1.
 *
 * Parity pins for each function live in tests/test_oracle_pins.py.
 *
 * Threads: the query heads of one layer's attention are independent and may
 * run on several host threads (OpenMP, kvo_set_threads); each head's
 * arithmetic and its order are the same on any number of threads, so the
 * results are identical bit for bit.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Host threads for the attention's query heads (1 = single thread).
 * Returns the count in effect (1 when built without OpenMP). */
int kvo_set_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Exact widening of a bf16 bit pattern. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ EMA */
/* "ema-eviction" figure: score = alpha * new_score + (1 - alpha) * score. */
double kvo_ema(double score, double new_score, double alpha) {
    return alpha * new_score + (1.0 - alpha) * score;
}

/* ------------------------------------------------------------- priority */
/* "ema-eviction" figure: priority = (1 - score) * recency_decay with
 * recency_decay = 1 - e^(-beta * steps).  At steps == 0 the decay is 0 for
 * every beta, which also fixes the beta = +inf case (0 * inf). */
double kvo_priority(double score, int64_t steps, double beta) {
    double decay = (steps == 0) ? 0.0 : 1.0 - exp(-beta * (double)steps);
    return (1.0 - score) * decay;
}

/* ------------------------------------------------------------ attention */
/* One layer of one sequence.  Query head h reads KV head g = h*Hkv/Hq (the
 * query-head groups are contiguous).  Logits q.k/sqrt(d), a two-pass
 * softmax over all L positions, output sum_i p_i v_i.
 *   q      [Hq][d]              bf16 bits
 *   k, v   row (g, i) at (g*ld + i)*d, bf16 bits
 *   probs  [Hq][L]  out
 *   out    [Hq][d]  out                                                    */
void kvo_attention(int Hq, int Hkv, int d, int64_t L, const uint16_t* q,
                   const uint16_t* k, const uint16_t* v, int64_t ld,
                   double* probs, double* out) {
    double scale = 1.0 / sqrt((double)d);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int h = 0; h < Hq; ++h) {
        int g = h * Hkv / Hq;
        double* p = probs + (int64_t)h * L;
        for (int64_t i = 0; i < L; ++i) {
            const uint16_t* kr = k + ((int64_t)g * ld + i) * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += bf16_to_double(q[h * d + c]) * bf16_to_double(kr[c]);
            p[i] = dot * scale;
        }
        double mx = -INFINITY;
        for (int64_t i = 0; i < L; ++i)
            if (p[i] > mx) mx = p[i];
        double sum = 0.0;
        for (int64_t i = 0; i < L; ++i) {
            p[i] = exp(p[i] - mx);
            sum += p[i];
        }
        for (int64_t i = 0; i < L; ++i) p[i] /= sum;
        /* out[h][c] = sum_i p_i v_i[c], accumulated in ascending i for every c */
        for (int c = 0; c < d; ++c) out[h * d + c] = 0.0;
        for (int64_t i = 0; i < L; ++i) {
            const uint16_t* vr = v + ((int64_t)g * ld + i) * d;
            for (int c = 0; c < d; ++c) out[h * d + c] += p[i] * bf16_to_double(vr[c]);
        }
    }
}

/* ------------------------------------------------------------ selection */
typedef struct {
    double pr;
    int64_t idx;
} kvo_key;

static int kvo_key_cmp(const void* a, const void* b) {
    const kvo_key* x = (const kvo_key*)a;
    const kvo_key* y = (const kvo_key*)b;
    if (x->pr < y->pr) return -1;
    if (x->pr > y->pr) return 1;
    return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

static int kvo_idx_cmp(const void* a, const void* b) {
    int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
    return (x < y) ? -1 : (x > y);
}

/* Keep the B units of lowest priority (ties to the lower index), pinned
 * units first; write the kept indices in ascending order.  Returns the
 * number kept (min(L, max(B, #pinned))). */
int64_t kvo_select(int64_t L, const double* pr, const uint8_t* pinned, int64_t B,
                   int64_t* kept) {
    kvo_key* keys = (kvo_key*)malloc(sizeof(kvo_key) * (size_t)(L > 0 ? L : 1));
    for (int64_t i = 0; i < L; ++i) {
        keys[i].pr = (pinned && pinned[i]) ? -INFINITY : pr[i];
        keys[i].idx = i;
    }
    qsort(keys, (size_t)L, sizeof(kvo_key), kvo_key_cmp);
    int64_t n = B < L ? B : L;
    if (pinned) {
        int64_t np = 0;
        for (int64_t i = 0; i < L; ++i) np += pinned[i] ? 1 : 0;
        if (np > n) n = np;
    }
    for (int64_t j = 0; j < n; ++j) kept[j] = keys[j].idx;
    qsort(kept, (size_t)n, sizeof(int64_t), kvo_idx_cmp);
    free(keys);
    return n;
}

/* ---------------------------------------------------------------- step */
typedef struct {
    int32_t n_layers, n_q_heads, n_kv_heads, head_dim;
    int64_t cap;           /* slots per (layer, KV head) */
    int64_t layer_stride;  /* elements between consecutive layers of K/V */
    int64_t budget;        /* B, in tokens */
    double alpha;          /* EMA weight of the new observation */
    double beta;           /* recency coefficient (may be +inf) */
    int32_t age_mode;      /* 0: steps since insertion, 1: since last access */
    int32_t pool_mean;     /* 0: sum over query heads, 1: mean */
    int32_t aggregation;   /* 0: EMA, 1: cumulative */
    int32_t weighting;     /* bit 0: VNorm, bit 1: entropy */
} kvo_params;

enum { KVO_AGG_EMA = 0, KVO_AGG_CUMULATIVE = 1 };
enum { KVO_W_VNORM = 1, KVO_W_ENTROPY = 2 };

/* VNorm factors of one layer: for KV head g and token i, the l2 norm of
 * v_{g,i} over the mean of the norms of the L cached tokens of head g (1
 * where every norm is 0).  v rows as in kvo_attention; w [Hkv][L] out. */
void kvo_vnorm(int Hkv, int d, int64_t L, const uint16_t* v, int64_t ld, double* w) {
    for (int g = 0; g < Hkv; ++g) {
        double* wg = w + (int64_t)g * L;
        double mean = 0.0;
        for (int64_t i = 0; i < L; ++i) {
            const uint16_t* vr = v + ((int64_t)g * ld + i) * d;
            double ss = 0.0;
            for (int c = 0; c < d; ++c) ss += bf16_to_double(vr[c]) * bf16_to_double(vr[c]);
            wg[i] = sqrt(ss);
            mean += wg[i];
        }
        mean /= (double)L;
        for (int64_t i = 0; i < L; ++i) wg[i] = mean > 0.0 ? wg[i] / mean : 1.0;
    }
}

/* Entropy weight of one layer: the entropy -sum_i p_i ln p_i of each query
 * head's attention distribution over ln L (1 for a uniform distribution, 0
 * for a one-hot one), averaged over the Hq heads; 1 when L = 1.
 * probs [Hq][L]. */
double kvo_layer_entropy(int Hq, int64_t L, const double* probs) {
    if (L <= 1) return 1.0;
    double acc = 0.0;
    for (int h = 0; h < Hq; ++h) {
        double hh = 0.0;
        for (int64_t i = 0; i < L; ++i) {
            double pi = probs[(int64_t)h * L + i];
            if (pi > 0.0) hh -= pi * log(pi);
        }
        acc += hh / log((double)L);
    }
    return acc / (double)Hq;
}

/* One decode step of one sequence, token granularity.
 *
 * In/out (appended in place at slot L_prev):
 *   K, V            [Ly] blocks at K + l*layer_stride, each [Hkv][cap][d]
 *   m, t_ins, t_ref, pos     [cap]
 * In:
 *   q [Ly][Hq][d], k_new/v_new [Ly][Hkv][d] (bf16 bits), new_pos
 *   forced_access   [L] or NULL; -1 = decide, 0/1 = take this decision
 * Out:
 *   out [Ly][Hq][d]; probs [Ly][Hq][L] or NULL; score_sum [L] or NULL
 *   (sum over layers of the head-summed probability); m_upd [L] (state
 *   after the EMA, before compaction); priority [L]; accessed [L] or NULL;
 *   retained [min(B,L)] ascending; compacted copies in *_out (same layout).
 * Returns the number retained.                                            */
int64_t kvo_step(const kvo_params* P, int64_t t, int refresh, int64_t L_prev,
                 uint16_t* K, uint16_t* V, double* m, int64_t* t_ins, int64_t* t_ref,
                 int64_t* pos, int64_t new_pos, const uint16_t* q,
                 const uint16_t* k_new, const uint16_t* v_new,
                 const int8_t* forced_access, double* out, double* probs,
                 double* score_sum, double* m_upd, double* priority, uint8_t* accessed,
                 int64_t* retained, uint16_t* K_out, uint16_t* V_out, double* m_out,
                 int64_t* t_ins_out, int64_t* t_ref_out, int64_t* pos_out) {
    const int Ly = P->n_layers, Hq = P->n_q_heads, Hkv = P->n_kv_heads, d = P->head_dim;
    const int64_t L = L_prev + 1;

    /* 1. append the new token in every layer and KV head */
    for (int l = 0; l < Ly; ++l)
        for (int g = 0; g < Hkv; ++g) {
            int64_t dst = l * P->layer_stride + ((int64_t)g * P->cap + L_prev) * d;
            memcpy(K + dst, k_new + ((int64_t)l * Hkv + g) * d, sizeof(uint16_t) * d);
            memcpy(V + dst, v_new + ((int64_t)l * Hkv + g) * d, sizeof(uint16_t) * d);
        }
    double new_m = 0.0;                      /* m0 = 0 on refresh steps */
    if (!refresh && L_prev > 0) {            /* mean momentum otherwise */
        double acc = 0.0;
        for (int64_t i = 0; i < L_prev; ++i) acc += m[i];
        new_m = acc / (double)L_prev;
    }
    m[L_prev] = new_m;
    t_ins[L_prev] = t;
    t_ref[L_prev] = t;
    pos[L_prev] = new_pos;

    /* 2. attention per layer; 3. head pooling and EMA, layers in order */
    double* p = (double*)malloc(sizeof(double) * (size_t)Hq * (size_t)L);
    double* ssum = (double*)calloc((size_t)L, sizeof(double));
    double* vw = (double*)malloc(sizeof(double) * (size_t)Hkv * (size_t)L);
    for (int64_t i = 0; i < L; ++i) m_upd[i] = m[i];
    for (int l = 0; l < Ly; ++l) {
        kvo_attention(Hq, Hkv, d, L, q + (int64_t)l * Hq * d, K + l * P->layer_stride,
                      V + l * P->layer_stride, P->cap, p, out + (int64_t)l * Hq * d);
        if (probs) memcpy(probs + (int64_t)l * Hq * L, p, sizeof(double) * (size_t)Hq * L);
        if (!refresh) continue;
        const int vnorm = (P->weighting & KVO_W_VNORM) != 0;
        if (vnorm) kvo_vnorm(Hkv, d, L, V + l * P->layer_stride, P->cap, vw);
        const double lw = (P->weighting & KVO_W_ENTROPY) ? kvo_layer_entropy(Hq, L, p) : 1.0;
        for (int64_t i = 0; i < L; ++i) {
            double s = 0.0, sw = 0.0;
            for (int h = 0; h < Hq; ++h) {
                s += p[(int64_t)h * L + i];
                if (vnorm) sw += p[(int64_t)h * L + i] * vw[(int64_t)(h * Hkv / Hq) * L + i];
            }
            ssum[i] += s;          /* the access test reads the plain attention */
            if (vnorm) s = sw;
            if (P->pool_mean) s /= (double)Hq;
            s *= lw;
            m_upd[i] = P->aggregation == KVO_AGG_CUMULATIVE ? m_upd[i] + s
                                                            : kvo_ema(m_upd[i], s, P->alpha);
        }
    }

    /* 4. access clock: head- and layer-averaged attention >= 2/L */
    for (int64_t i = 0; i < L; ++i) {
        int acc = 0;
        if (refresh) {
            double mean_attn = ssum[i] / ((double)Ly * (double)Hq);
            acc = mean_attn >= 2.0 / (double)L;
            if (forced_access && forced_access[i] >= 0) acc = forced_access[i];
        }
        if (accessed) accessed[i] = (uint8_t)acc;
        if (acc) t_ref[i] = t;
        if (score_sum) score_sum[i] = ssum[i];
    }

    /* 5. priority */
    for (int64_t i = 0; i < L; ++i) {
        int64_t age = t - (P->age_mode ? t_ref[i] : t_ins[i]);
        priority[i] = kvo_priority(m_upd[i], age, P->beta);
    }

    /* 6. selection, 7. compaction */
    int64_t n = kvo_select(L, priority, NULL, P->budget, retained);
    for (int l = 0; l < Ly; ++l)
        for (int g = 0; g < Hkv; ++g)
            for (int64_t j = 0; j < n; ++j) {
                int64_t src = l * P->layer_stride + ((int64_t)g * P->cap + retained[j]) * d;
                int64_t dst = l * P->layer_stride + ((int64_t)g * P->cap + j) * d;
                memcpy(K_out + dst, K + src, sizeof(uint16_t) * d);
                memcpy(V_out + dst, V + src, sizeof(uint16_t) * d);
            }
    for (int64_t j = 0; j < n; ++j) {
        m_out[j] = m_upd[retained[j]];
        t_ins_out[j] = t_ins[retained[j]];
        t_ref_out[j] = t_ref[retained[j]];
        pos_out[j] = pos[retained[j]];
    }
    free(p);
    free(ssum);
    free(vw);
    return n;
}
