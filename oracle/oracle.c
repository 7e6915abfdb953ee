/*
 * oracle.c -- plain float64 CPU oracle for the speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library. The product
 * path (libspecverify.so and its Python binding) never calls it, and this
 * file shares no code, header, table or constant with the CUDA path.
 *
 * Every function follows the pages' statement of the method step by step, in
 * float64, with plain sequential loops in index order. No blocking, fusion or
 * reordering beyond what the method states. Sources (page title, section):
 *
 *   [P1] "Speculative decoding" (mhtirogla.ai, ml-training encyclopaedia
 *        entry): "How it works" steps 1-5, the "Code" section's verify and
 *        sample routines (read for what they compute), "Implementation notes".
 *   [P3] "Speculative decoding: the secretary who types ahead of the boss"
 *        (blog.lo0.es): "The bare mechanism", step 3.
 *   [P4] "Speculative decoding" (inference.tusharamrit.in module): modified
 *        rejection sampling, the residual p'(z) and its normaliser identity.
 *   [P5] "Speculative Decoding" (tokentrails.org): "One round" and the greedy
 *        round in its "Code" section.
 *   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *        Easy as 1, 2, 3", SC'11, section on the Philox S-box and key schedule.
 *
 * Readings where the pages are silent or ambiguous:
 *   - uniforms come from Philox4x32-10 keyed by the 64-bit seed with counter
 *     (position, sequence, round lo, round hi); word 0 -> u_acc, word 1 ->
 *     u_smp, each (w >> 8) * 2^-24, the pages' 24-bit resolution ([P1] Code);
 *   - accept iff u * q(x) < p(x), strict ([P1] Code, division-free form);
 *   - inverse CDF: first index whose running sum exceeds u * total, in index
 *     order ([P1] Code, sample); if rounding leaves none, the last index with
 *     positive mass (the page returns the last index even if it has no mass);
 *   - residual normaliser Z == 0 at a rejection: sample from p_i instead;
 *   - greedy argmax: first index of the maximum raw logit, NaN read as -inf;
 *   - top-k (an option of the library, applied to both models' rows alike as
 *     [P1] Implementation notes asks of any logits processing): keep every
 *     column whose value is at least the row's k-th largest (NaN ranks as
 *     -inf; ties at the threshold all stay), renormalise over the kept ones;
 *   - top-p (the same note): the nucleus of the top-k-renormalised
 *     distribution (see orc_topp_threshold), or of the whole row when top-k
 *     is off.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

/* per-sequence status words (values mirror the library's documented codes) */
#define ORC_SEQ_OK 0
#define ORC_SEQ_BAD_TOKEN 1
#define ORC_SEQ_BAD_KV 2
#define ORC_SEQ_BAD_ROW 3
#define ORC_SEQ_BAD_LAYOUT 4
#define ORC_SEQ_BAD_TEMP 5
#define ORC_SEQ_UNSUPPORTED 7 /* tree verification: a visited node with too many candidates */

/* ------------------------------------------------------------------ */
/* Element access: bf16 is the top half of an IEEE binary32, so widening */
/* the 16 bits to 32 and reading them as float is exact.                 */
/* ------------------------------------------------------------------ */
double orc_value(const void* base, int32_t dtype, int64_t idx) {
    float f;
    if (dtype == ORC_F32) {
        memcpy(&f, (const char*)base + 4 * idx, 4);
    } else {
        uint16_t h;
        memcpy(&h, (const char*)base + 2 * idx, 2);
        uint32_t w = ((uint32_t)h) << 16;
        memcpy(&f, &w, 4);
    }
    return (double)f;
}

static const void* row_ptr(const void* base, int32_t dtype, int64_t row, int64_t V) {
    int64_t esz = (dtype == ORC_F32) ? 4 : 2;
    return (const char*)base + row * V * esz;
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (SC'11). One round: two 32x32->64 products of counter */
/* words 0 and 2 with the round multipliers; the new counter is        */
/* (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0). The key is bumped by the   */
/* Weyl constants between rounds.                                       */
/* ------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* u in [0,1) on the 24-bit grid, from the top 24 bits of a 32-bit word. */
double orc_u24(uint32_t w) { return (double)(w >> 8) * (1.0 / 16777216.0); }

/* (u_acc, u_smp) for global sequence `seq`, position `pos` of round `round`. */
void orc_uniform_pair(uint64_t seed, uint64_t round, uint32_t seq, uint32_t pos,
                      double* u_acc, double* u_smp) {
    uint32_t ctr[4] = {pos, seq, (uint32_t)(round & 0xffffffffu), (uint32_t)(round >> 32)};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    *u_acc = orc_u24(w[0]);
    *u_smp = orc_u24(w[1]);
}

/* ------------------------------------------------------------------ */
/* Distributions.                                                      */
/* ------------------------------------------------------------------ */

/* p = softmax(l / T) over the whole row ([P1] How it works, step 2; the same
 * temperature on both models, [P1] Implementation notes). Returns a status. */
int32_t orc_softmax_row(const void* row, int32_t dtype, int64_t V, double T, double* p) {
    if (!(T > 0.0) || !isfinite(T)) return ORC_SEQ_BAD_TEMP;
    double m = -INFINITY;
    int has_nan = 0;
    for (int64_t j = 0; j < V; ++j) {
        double x = orc_value(row, dtype, j) / T;
        if (isnan(x))
            has_nan = 1;
        else if (x > m)
            m = x;
    }
    if (has_nan || !isfinite(m)) return ORC_SEQ_BAD_ROW;
    double s = 0.0;
    for (int64_t j = 0; j < V; ++j) {
        p[j] = exp(orc_value(row, dtype, j) / T - m);
        s += p[j];
    }
    if (!(s > 0.0) || !isfinite(s)) return ORC_SEQ_BAD_ROW;
    for (int64_t j = 0; j < V; ++j) p[j] /= s;
    return ORC_SEQ_OK;
}

/* A probability row given directly is used after dividing by its own sum
 * (the page's sampler tolerates unnormalised input, [P1] Code). */
int32_t orc_normalize_row(const void* row, int32_t dtype, int64_t V, double* q) {
    double s = 0.0;
    int has_nan = 0;
    for (int64_t j = 0; j < V; ++j) {
        q[j] = orc_value(row, dtype, j);
        if (isnan(q[j])) has_nan = 1;
        s += q[j];
    }
    if (has_nan || !(s > 0.0) || !isfinite(s)) return ORC_SEQ_BAD_ROW;
    for (int64_t j = 0; j < V; ++j) q[j] /= s;
    return ORC_SEQ_OK;
}

/* Top-k truncation, applied the same way to the target's and the draft's row
 * ([P1] Implementation notes: both models' logits go through the same
 * processing). The threshold is the k-th largest value of the row, NaN read
 * as -inf; every column whose value is at least that large is kept (ties at
 * the threshold all stay). k <= 0 or k >= V keeps the whole row: the returned
 * threshold is then -inf. Plain: copy, sort in decreasing order, index. */
static int cmp_desc(const void* x, const void* y) {
    const double a = *(const double*)x, b = *(const double*)y;
    return (a < b) - (a > b);
}

double orc_topk_threshold(const void* row, int32_t dtype, int64_t V, int64_t k) {
    if (k < 1 || k >= V) return -INFINITY;
    double* v = (double*)malloc(sizeof(double) * (size_t)V);
    for (int64_t j = 0; j < V; ++j) {
        const double x = orc_value(row, dtype, j);
        v[j] = isnan(x) ? -INFINITY : x;
    }
    qsort(v, (size_t)V, sizeof(double), cmp_desc);
    const double t = v[k - 1];
    free(v);
    return t;
}

/* p = softmax(l / T) restricted to the columns with l >= tau (the others get
 * probability 0); tau = -inf keeps every column. The same checks as
 * orc_softmax_row over the whole row. */
int32_t orc_softmax_row_topk(const void* row, int32_t dtype, int64_t V, double T, double tau, double* p) {
    if (!(T > 0.0) || !isfinite(T)) return ORC_SEQ_BAD_TEMP;
    double m = -INFINITY;
    int has_nan = 0;
    for (int64_t j = 0; j < V; ++j) {
        double x = orc_value(row, dtype, j) / T;
        if (isnan(x))
            has_nan = 1;
        else if (x > m)
            m = x;
    }
    if (has_nan || !isfinite(m)) return ORC_SEQ_BAD_ROW;
    double s = 0.0;
    for (int64_t j = 0; j < V; ++j) {
        const double l = orc_value(row, dtype, j);
        p[j] = (l >= tau) ? exp(l / T - m) : 0.0;
        s += p[j];
    }
    if (!(s > 0.0) || !isfinite(s)) return ORC_SEQ_BAD_ROW;
    for (int64_t j = 0; j < V; ++j) p[j] /= s;
    return ORC_SEQ_OK;
}

/* A probability row restricted to the columns with value >= tau, divided by
 * the kept columns' sum. */
int32_t orc_normalize_row_topk(const void* row, int32_t dtype, int64_t V, double tau, double* q) {
    double s = 0.0;
    int has_nan = 0;
    for (int64_t j = 0; j < V; ++j) {
        const double v = orc_value(row, dtype, j);
        if (isnan(v)) has_nan = 1;
        q[j] = (v >= tau) ? v : 0.0;
        s += q[j];
    }
    if (has_nan || !(s > 0.0) || !isfinite(s)) return ORC_SEQ_BAD_ROW;
    for (int64_t j = 0; j < V; ++j) q[j] /= s;
    return ORC_SEQ_OK;
}

/* Top-p (nucleus) truncation after top-k, on both models' rows alike ([P1]
 * Implementation notes: the same temperature, top-k and top-p processing).
 * Reading: over the columns top-k kept (value >= tau_k) with weights
 * w = exp(l/T - max(l/T)) (a probabilities row: its values), taken in
 * decreasing value, the threshold is the value of the first group of equal
 * values at which the cumulative weight reaches top_p times the kept total;
 * every column at least that large stays (the whole group). Active for
 * 0 < top_p < 1; otherwise (and for NaN) off, so that a zeroed parameter
 * means no top-p: the function then returns tau_k. Plain: copy, sort, walk. */
typedef struct {
    double v, w;
} orc_vw_t;

static int cmp_vw_desc(const void* x, const void* y) {
    const double a = ((const orc_vw_t*)x)->v, b = ((const orc_vw_t*)y)->v;
    return (a < b) - (a > b);
}

double orc_topp_threshold(const void* row, int32_t dtype, int64_t V, double T, int32_t probs, double tau_k,
                          double top_p) {
    if (!(top_p > 0.0 && top_p < 1.0)) return tau_k; /* off (and NaN) */
    orc_vw_t* e = (orc_vw_t*)malloc(sizeof(orc_vw_t) * (size_t)(V > 0 ? V : 1));
    int64_t n = 0;
    double m = -INFINITY;
    for (int64_t j = 0; j < V; ++j) {
        const double l = orc_value(row, dtype, j);
        if (l >= tau_k) {
            e[n].v = l;
            ++n;
            if (!probs && l / T > m) m = l / T;
        }
    }
    if (n == 0) {
        free(e);
        return tau_k;
    }
    qsort(e, (size_t)n, sizeof(orc_vw_t), cmp_vw_desc);
    double S = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        e[i].w = probs ? e[i].v : exp(e[i].v / T - m);
        S += e[i].w;
    }
    const double target = top_p * S;
    double cum = 0.0, tau = e[n - 1].v;
    for (int64_t i = 0; i < n;) {
        int64_t k = i;
        while (k < n && e[k].v == e[i].v) cum += e[k++].w;
        if (cum >= target) {
            tau = e[i].v;
            break;
        }
        i = k;
    }
    free(e);
    return tau;
}

/* r = max(0, p - q) elementwise; returns Z = sum r ([P1] How it works step 3;
 * [P4] residual p'(z)). */
double orc_residual(const double* p, const double* q, int64_t V, double* r) {
    double Z = 0.0;
    for (int64_t j = 0; j < V; ++j) {
        double d = p[j] - q[j];
        r[j] = d > 0.0 ? d : 0.0;
        Z += r[j];
    }
    return Z;
}

/* First index whose running sum exceeds u * total, total = sum w in index
 * order ([P1] Code, sample). Fallback: last index with positive mass. */
int64_t orc_inverse_cdf(const double* w, int64_t V, double u) {
    double total = 0.0;
    for (int64_t j = 0; j < V; ++j) total += w[j];
    double t = u * total;
    double c = 0.0;
    for (int64_t j = 0; j < V; ++j) {
        c += w[j];
        if (c > t) return j;
    }
    for (int64_t j = V - 1; j >= 0; --j)
        if (w[j] > 0.0) return j;
    return -1;
}

/* Normalised CDF edges (C_{j-1}, C_j) of index j under weights w. */
void orc_cdf_edges(const double* w, int64_t V, int64_t j, double* lo, double* hi) {
    double total = 0.0;
    for (int64_t k = 0; k < V; ++k) total += w[k];
    double c = 0.0;
    for (int64_t k = 0; k < j; ++k) c += w[k];
    *lo = c / total;
    *hi = (c + w[j]) / total;
}

/* First index of the largest logit; NaN counts as -inf ([P5] Code, argmax). */
int64_t orc_argmax_row(const void* row, int32_t dtype, int64_t V) {
    double best = -INFINITY;
    int64_t idx = 0;
    for (int64_t j = 0; j < V; ++j) {
        double v = orc_value(row, dtype, j);
        if (isnan(v)) v = -INFINITY;
        if (v > best) {
            best = v;
            idx = j;
        }
    }
    return idx;
}

/* ------------------------------------------------------------------ */
/* Batched verify.                                                     */
/* ------------------------------------------------------------------ */
typedef struct {
    int32_t batch, vocab, gamma_max;
    int64_t rows_target, rows_draft;
    const int64_t* target_row_off; /* [B+1] or NULL: b*(gamma_max+1) */
    const int64_t* draft_row_off;  /* [B+1] or NULL: b*gamma_max */
    const void* target;            /* [rows_target, V] */
    int32_t target_dtype;
    const void* draft; /* [rows_draft, V] */
    int32_t draft_dtype;
    int32_t draft_is_probs;
    const int32_t* draft_tokens; /* [rows_draft] */
    const float* temperatures;   /* [B] or NULL */
    float temperature;
    uint64_t seed, round;
    uint32_t seq_offset;
    const float* uniforms; /* [rows_target, 2] or NULL */
    const int32_t* kv_in;  /* [B] or NULL */
    int32_t block_size;    /* 0: no block count */
    int32_t* out_tokens;   /* [rows_target] */
    int32_t* out_accepted; /* [B] */
    int32_t* kv_out;       /* [B] or NULL */
    int32_t* out_blocks;   /* [B] or NULL */
    int32_t* seq_status;   /* [B] or NULL */
    /* diagnostics, each [B] or NULL */
    double* diag_acc_margin; /* min over accept tests done of |u_acc - p(x)/q(x)| */
    double* diag_u_smp;      /* the u used for the final sample */
    double* diag_cdf_lo;     /* normalised CDF edges of the emitted token */
    double* diag_cdf_hi;
    double* diag_z; /* residual normaliser at the rejection, -1 for a bonus */
    /* top-k truncation of every row of a sequence (sampling only): k_b =
     * top_ks[b] if top_ks, else top_k; k_b <= 0 or k_b >= V keeps every column */
    int32_t top_k;
    const int32_t* top_ks;
    /* top-p (inside the top-k set when top-k is on, else over the whole
     * row): p_b = top_ps[b] if top_ps, else top_p; active when 0 < p_b < 1 */
    float top_p;
    const float* top_ps;
} orc_args_t;

typedef struct {
    const orc_args_t* a;
    int greedy;
    int tid, nthreads;
} orc_job_t;

static int64_t toff(const orc_args_t* a, int64_t b) {
    return a->target_row_off ? a->target_row_off[b] : b * (int64_t)(a->gamma_max + 1);
}
static int64_t doff(const orc_args_t* a, int64_t b) {
    return a->draft_row_off ? a->draft_row_off[b] : b * (int64_t)a->gamma_max;
}

/* Checks that do not depend on the logits, in a fixed order: layout,
 * temperature (sampling only), draft tokens, KV length. */
static int64_t top_k_of(const orc_args_t* a, int64_t b) { return a->top_ks ? a->top_ks[b] : a->top_k; }
static double top_p_of(const orc_args_t* a, int64_t b) {
    return a->top_ps ? (double)a->top_ps[b] : (double)a->top_p;
}

static int32_t precheck(const orc_args_t* a, int64_t b, int greedy, int64_t* g_out, double* T_out) {
    int64_t t0 = toff(a, b), t1 = toff(a, b + 1), d0 = doff(a, b), d1 = doff(a, b + 1);
    int64_t g = d1 - d0;
    *g_out = g;
    if (g < 0 || g > a->gamma_max || t1 - t0 != g + 1 || t0 < 0 || t1 > a->rows_target ||
        d0 < 0 || d1 > a->rows_draft)
        return ORC_SEQ_BAD_LAYOUT;
    double T = a->temperatures ? (double)a->temperatures[b] : (double)a->temperature;
    *T_out = T;
    if (!greedy && (!(T > 0.0) || !isfinite(T))) return ORC_SEQ_BAD_TEMP;
    for (int64_t i = 0; i < g; ++i) {
        int32_t x = a->draft_tokens[d0 + i];
        if (x < 0 || x >= a->vocab) return ORC_SEQ_BAD_TOKEN;
    }
    if (a->kv_in && a->kv_in[b] < g) return ORC_SEQ_BAD_KV;
    return ORC_SEQ_OK;
}

static void write_error(const orc_args_t* a, int64_t b, int32_t st) {
    a->out_accepted[b] = 0;
    if (st != ORC_SEQ_BAD_LAYOUT) {
        for (int64_t k = toff(a, b); k < toff(a, b + 1); ++k) a->out_tokens[k] = -1;
    }
    if (a->kv_out) a->kv_out[b] = a->kv_in ? a->kv_in[b] : 0;
    if (a->out_blocks) {
        int32_t kv = a->kv_in ? a->kv_in[b] : 0;
        a->out_blocks[b] = a->block_size > 0 ? (kv + a->block_size - 1) / a->block_size : 0;
    }
    if (a->seq_status) a->seq_status[b] = st;
}

static void write_result(const orc_args_t* a, int64_t b, int64_t g, int64_t acc) {
    a->out_accepted[b] = (int32_t)acc;
    if (a->kv_out || a->out_blocks) {
        /* drop the KV entries of the rejected drafts ([P1] How it works step 5) */
        int32_t kv = a->kv_in ? a->kv_in[b] : 0;
        int32_t kv2 = a->kv_in ? kv - (int32_t)(g - acc) : 0;
        if (a->kv_out) a->kv_out[b] = kv2;
        if (a->out_blocks)
            a->out_blocks[b] = a->block_size > 0 ? (kv2 + a->block_size - 1) / a->block_size : 0;
    }
    if (a->seq_status) a->seq_status[b] = ORC_SEQ_OK;
}

static void uniforms_for(const orc_args_t* a, int64_t b, int64_t i, double* ua, double* us) {
    if (a->uniforms) {
        int64_t row = toff(a, b) + i;
        *ua = (double)a->uniforms[2 * row];
        *us = (double)a->uniforms[2 * row + 1];
    } else {
        orc_uniform_pair(a->seed, a->round, (uint32_t)(a->seq_offset + b), (uint32_t)i, ua, us);
    }
}


/* p_i of sequence b from target row trow: softmax(l / T) over the row's
 * top-k columns (every column when top-k is off). */
static int32_t target_dist(const orc_args_t* a, int64_t b, int64_t trow, double T, double* p) {
    const void* rp = row_ptr(a->target, a->target_dtype, trow, a->vocab);
    double tau = orc_topk_threshold(rp, a->target_dtype, a->vocab, top_k_of(a, b));
    tau = orc_topp_threshold(rp, a->target_dtype, a->vocab, T, 0, tau, top_p_of(a, b));
    return orc_softmax_row_topk(rp, a->target_dtype, a->vocab, T, tau, p);
}

/* q_i of sequence b from draft row drow, truncated the same way. */
static int32_t draft_dist(const orc_args_t* a, int64_t b, int64_t drow, double T, double* q) {
    const void* rp = row_ptr(a->draft, a->draft_dtype, drow, a->vocab);
    double tau = orc_topk_threshold(rp, a->draft_dtype, a->vocab, top_k_of(a, b));
    tau = orc_topp_threshold(rp, a->draft_dtype, a->vocab, T, a->draft_is_probs, tau, top_p_of(a, b));
    if (a->draft_is_probs) return orc_normalize_row_topk(rp, a->draft_dtype, a->vocab, tau, q);
    return orc_softmax_row_topk(rp, a->draft_dtype, a->vocab, T, tau, q);
}

/* One sequence of the sampling verify ([P1] How it works steps 3-5;
 * [P3] The bare mechanism step 3; [P4] accept/residual rule). */
static void verify_sample_one(const orc_args_t* a, int64_t b, double* p, double* q, double* r) {
    int64_t g;
    double T;
    int32_t st = precheck(a, b, 0, &g, &T);
    if (st) {
        write_error(a, b, st);
        return;
    }
    const int64_t V = a->vocab, t0 = toff(a, b), d0 = doff(a, b);
    double margin = INFINITY;
    for (int64_t i = 0; i < g; ++i) {
        st = target_dist(a, b, t0 + i, T, p);
        if (st) { write_error(a, b, st); return; }
        st = draft_dist(a, b, d0 + i, T, q);
        if (st) { write_error(a, b, st); return; }
        int32_t x = a->draft_tokens[d0 + i];
        double ua, us;
        uniforms_for(a, b, i, &ua, &us);
        if (q[x] > 0.0) {
            double dm = fabs(ua - p[x] / q[x]);
            if (dm < margin) margin = dm;
        }
        if (ua * q[x] < p[x]) { /* accept x_i: u < p/q without dividing */
            a->out_tokens[t0 + i] = x;
            continue;
        }
        /* first rejection: draw from norm(max(0, p - q)) and stop */
        double Z = orc_residual(p, q, V, r);
        const double* w = (Z > 0.0) ? r : p;
        int64_t tok = orc_inverse_cdf(w, V, us);
        a->out_tokens[t0 + i] = (int32_t)tok;
        for (int64_t k = i + 1; k <= g; ++k) a->out_tokens[t0 + k] = -1;
        if (a->diag_acc_margin) a->diag_acc_margin[b] = margin;
        if (a->diag_u_smp) a->diag_u_smp[b] = us;
        if (a->diag_z) a->diag_z[b] = Z;
        if (a->diag_cdf_lo && a->diag_cdf_hi) orc_cdf_edges(w, V, tok, &a->diag_cdf_lo[b], &a->diag_cdf_hi[b]);
        write_result(a, b, g, i);
        return;
    }
    /* all gamma accepted: bonus token from p_{gamma+1} ([P1] step 4) */
    st = target_dist(a, b, t0 + g, T, p);
    if (st) { write_error(a, b, st); return; }
    double ua, us;
    uniforms_for(a, b, g, &ua, &us);
    int64_t tok = orc_inverse_cdf(p, V, us);
    a->out_tokens[t0 + g] = (int32_t)tok;
    if (a->diag_acc_margin) a->diag_acc_margin[b] = margin;
    if (a->diag_u_smp) a->diag_u_smp[b] = us;
    if (a->diag_z) a->diag_z[b] = -1.0;
    if (a->diag_cdf_lo && a->diag_cdf_hi) orc_cdf_edges(p, V, tok, &a->diag_cdf_lo[b], &a->diag_cdf_hi[b]);
    write_result(a, b, g, g);
}

/* One sequence of the greedy verify: accept while the draft token equals the
 * target's argmax, then append the target's own pick ([P1] How it works,
 * greedy remark; [P5] One round and its greedy Code). */
static void verify_greedy_one(const orc_args_t* a, int64_t b) {
    int64_t g;
    double T;
    int32_t st = precheck(a, b, 1, &g, &T);
    if (st) {
        write_error(a, b, st);
        return;
    }
    const int64_t V = a->vocab, t0 = toff(a, b), d0 = doff(a, b);
    int64_t n = 0;
    for (;;) {
        int64_t pick = orc_argmax_row(row_ptr(a->target, a->target_dtype, t0 + n, V), a->target_dtype, V);
        a->out_tokens[t0 + n] = (int32_t)pick;
        if (n < g && a->draft_tokens[d0 + n] == pick) {
            ++n;
            continue;
        }
        break;
    }
    for (int64_t k = n + 1; k <= g; ++k) a->out_tokens[t0 + k] = -1;
    write_result(a, b, g, n);
}

static void* worker(void* arg) {
    const orc_job_t* job = (const orc_job_t*)arg;
    const orc_args_t* a = job->a;
    double *p = NULL, *q = NULL, *r = NULL;
    if (!job->greedy) {
        p = (double*)malloc(sizeof(double) * (size_t)a->vocab);
        q = (double*)malloc(sizeof(double) * (size_t)a->vocab);
        r = (double*)malloc(sizeof(double) * (size_t)a->vocab);
    }
    for (int64_t b = job->tid; b < a->batch; b += job->nthreads) {
        if (job->greedy)
            verify_greedy_one(a, b);
        else
            verify_sample_one(a, b, p, q, r);
    }
    free(p);
    free(q);
    free(r);
    return NULL;
}

static int run(const orc_args_t* a, int greedy, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > a->batch) nthreads = a->batch > 0 ? a->batch : 1;
    pthread_t th[256];
    orc_job_t jobs[256];
    if (nthreads > 256) nthreads = 256;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].a = a;
        jobs[t].greedy = greedy;
        jobs[t].tid = t;
        jobs[t].nthreads = nthreads;
    }
    if (nthreads == 1) {
        worker(&jobs[0]);
        return 0;
    }
    for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, worker, &jobs[t]);
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    return 0;
}

int orc_verify_sample(const orc_args_t* a, int32_t nthreads) { return run(a, 0, nthreads); }
int orc_verify_greedy(const orc_args_t* a, int32_t nthreads) { return run(a, 1, nthreads); }

/* Length truncate by the rejected-draft count ([P1] How it works step 5,
 * Implementation notes on paged KV). */
void orc_kv_rollback(const int32_t* kv_in, int32_t* kv_out, const int32_t* accepted,
                     const int32_t* gammas, int32_t gamma_max, int32_t batch, int32_t block_size,
                     int32_t* out_blocks, int32_t* seq_status) {
    for (int32_t b = 0; b < batch; ++b) {
        int32_t g = gammas ? gammas[b] : gamma_max;
        int32_t acc = accepted[b];
        int32_t st = ORC_SEQ_OK;
        int32_t kv = kv_in[b];
        if (g < 0 || acc < 0 || acc > g)
            st = ORC_SEQ_BAD_LAYOUT;
        else if (kv < g)
            st = ORC_SEQ_BAD_KV;
        int32_t kv2 = st ? kv : kv - (g - acc);
        kv_out[b] = kv2;
        if (out_blocks) out_blocks[b] = block_size > 0 ? (kv2 + block_size - 1) / block_size : 0;
        if (seq_status) seq_status[b] = st;
    }
}

/* ------------------------------------------------------------------ */
/* Per-sequence views used by the parity tests.                        */
/* ------------------------------------------------------------------ */

/* p_i(x_i) and q_i(x_i) of sequence b at draft position i. Status return. */
int32_t orc_accept_terms(const orc_args_t* a, int64_t b, int64_t i, double* p_x, double* q_x) {
    const int64_t V = a->vocab;
    double T = a->temperatures ? (double)a->temperatures[b] : (double)a->temperature;
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    int32_t st = target_dist(a, b, toff(a, b) + i, T, p);
    if (!st) st = draft_dist(a, b, doff(a, b) + i, T, q);
    if (!st) {
        int32_t x = a->draft_tokens[doff(a, b) + i];
        *p_x = p[x];
        *q_x = q[x];
    }
    free(p);
    free(q);
    return st;
}

/* The rows the method uses at position i of sequence b: p_i, q_i (zeros for
 * the bonus position) and the sampling weights w (r = max(0, p - q) at a
 * draft position, p at the bonus position, p again if Z == 0). Returns a
 * status; *z_out receives Z (or -1 at the bonus position). */
int32_t orc_position_rows(const orc_args_t* a, int64_t b, int64_t i, double* p, double* q, double* w,
                          double* z_out) {
    const int64_t V = a->vocab;
    double T = a->temperatures ? (double)a->temperatures[b] : (double)a->temperature;
    int64_t g = doff(a, b + 1) - doff(a, b);
    int32_t st = target_dist(a, b, toff(a, b) + i, T, p);
    if (st) return st;
    if (i >= g) {
        for (int64_t j = 0; j < V; ++j) {
            q[j] = 0.0;
            w[j] = p[j];
        }
        *z_out = -1.0;
        return ORC_SEQ_OK;
    }
    st = draft_dist(a, b, doff(a, b) + i, T, q);
    if (st) return st;
    double Z = orc_residual(p, q, V, w);
    *z_out = Z;
    if (!(Z > 0.0))
        for (int64_t j = 0; j < V; ++j) w[j] = p[j];
    return ORC_SEQ_OK;
}

/* ------------------------------------------------------------ adaptive gamma
 * Under continuous batching gamma is chosen per request from its running
 * acceptance, and speculation is switched off once the batch is large enough
 * to be compute-bound ("Speculative decoding" (mhtirogla.ai), Implementation
 * notes and Efficiency, adaptive gamma). The pages give the cost model
 * (expected tokens per pass E = (1 - a^(g+1)) / (1 - a), wall-clock speedup
 * E / (1 + g c); "Speculative decoding" (inference.tusharamrit.in), the
 * actual speedup and its worked cases) but no estimator and no switch rule;
 * the readings:
 *   - a round of sequence b performed t_b accept tests (a_b + 1 when a draft
 *     was rejected, else gamma_b) of which a_b passed; its running acceptance
 *     is an exponential moving average of a_b / t_b over its rounds, state in
 *     float32: ema += lambda * (a_b / t_b - ema), in that order, each
 *     operation rounded to float32. Rounds with t_b = 0 (gamma_b = 0) or a
 *     sequence status other than OK leave it unchanged;
 *   - gamma_b for the next round is the smallest g in [0, gamma_max] with the
 *     largest E(a, g) / (1 + g c), a = the running acceptance clamped to
 *     [0, 1] (NaN read as 0), in float32 with every operation rounded in a
 *     fixed order: E(a, g) = 1 + a + ... + a^g (the same quantity as the
 *     pages' closed form, summed term by term: no cancellation near a = 1),
 *     the powers by repeated multiplication;
 *   - if max_positions > 0 and the verify positions sum_b (gamma_b + 1)
 *     exceed it, every gamma_b is 0 (speculation off for the batch). */
void orc_acceptance_ema(const int32_t* accepted, const int32_t* gammas, int32_t gamma_max, int64_t B,
                        const int32_t* status, float lambda, const float* ema_in, float* ema_out) {
    for (int64_t b = 0; b < B; ++b) {
        const int32_t g = gammas ? gammas[b] : gamma_max;
        const int32_t a = accepted[b];
        float e = ema_in[b];
        if ((!status || status[b] == 0) && g > 0 && a >= 0 && a <= g) {
            const int32_t t = a < g ? a + 1 : g;
            const float x = (float)a / (float)t;
            const float d = x - e;
            const float s = lambda * d;
            e = e + s;
        }
        ema_out[b] = e;
    }
}

/* E(a, g) / (1 + g c) for g = 0..gamma_max into sp[] (float32 arithmetic). */
void orc_speedups(float a, int32_t gamma_max, float c, float* sp) {
    if (!(a >= 0.0f)) a = 0.0f; /* NaN and negatives */
    if (a > 1.0f) a = 1.0f;
    float pw = 1.0f, E = 1.0f; /* a^g and 1 + a + ... + a^g */
    for (int32_t g = 0; g <= gamma_max; ++g) {
        if (g > 0) {
            pw = pw * a;
            E = E + pw;
        }
        const float den = 1.0f + (float)g * c;
        sp[g] = E / den;
    }
}

int32_t orc_best_gamma(float ema, int32_t gamma_max, float c) {
    float sp[65];
    if (gamma_max > 64) gamma_max = 64;
    if (gamma_max < 0) gamma_max = 0;
    orc_speedups(ema, gamma_max, c, sp);
    int32_t best = 0;
    for (int32_t g = 1; g <= gamma_max; ++g)
        if (sp[g] > sp[best]) best = g;
    return best;
}

/* Returns the verify positions sum_b (gamma_b + 1) of the chosen gammas,
 * before the switch (the quantity compared with max_positions). */
int64_t orc_adapt_gamma(const float* ema, int64_t B, int32_t gamma_max, float c, int64_t max_positions,
                        int32_t* gammas_out) {
    int64_t total = 0;
    for (int64_t b = 0; b < B; ++b) {
        gammas_out[b] = orc_best_gamma(ema[b], gamma_max, c);
        total += gammas_out[b] + 1;
    }
    if (max_positions > 0 && total > max_positions)
        for (int64_t b = 0; b < B; ++b) gammas_out[b] = 0;
    return total;
}

/* ------------------------------------------------------------ n-gram drafter
 * Prompt lookup / n-gram drafting ("Speculative decoding" (mhtirogla.ai),
 * Implementation notes: copy the continuation of the last matching n-gram;
 * "Speculative decoding" (inference.tusharamrit.in), n-gram / prompt lookup:
 * search the existing context for the current suffix and propose what
 * followed it last time). Readings where the pages stop short:
 *   - the search covers the whole context of the sequence (prompt and the
 *     tokens generated so far), ctx[0 .. L);
 *   - the suffix is the last n tokens; a match is an earlier start j
 *     (0 <= j <= L - n - 1, so at least one token follows it) with
 *     ctx[j .. j+n) equal to the suffix; the match taken is the latest such
 *     j (what followed "last time"); it may overlap the suffix;
 *   - n runs from n_max down to n_min and the first n with a match is used;
 *   - the draft is ctx[j+n .. min(j+n+gamma, L)), fewer than gamma tokens
 *     when the context ends first; no match gives no draft.
 * Outputs per sequence b: draft[b*gamma .. +gamma) (-1 after the drafted
 * tokens), n_draft[b], match_pos[b] (j, or -1), match_n[b] (n, or 0). */
void orc_ngram_draft(const int32_t* ctx, const int64_t* ctx_off, int64_t B, int32_t n_max, int32_t n_min,
                     int32_t gamma, int32_t* draft, int32_t* n_draft, int64_t* match_pos, int32_t* match_n) {
    for (int64_t b = 0; b < B; ++b) {
        const int32_t* c = ctx + ctx_off[b];
        const int64_t L = ctx_off[b + 1] - ctx_off[b];
        int64_t jbest = -1;
        int32_t nbest = 0;
        for (int32_t n = n_max; n >= n_min && n >= 1 && jbest < 0; --n) {
            if (L < (int64_t)n + 1) continue;
            for (int64_t j = L - n - 1; j >= 0; --j) {
                int32_t k = 0;
                while (k < n && c[j + k] == c[L - n + k]) ++k;
                if (k == n) {
                    jbest = j;
                    nbest = n;
                    break;
                }
            }
        }
        int32_t cnt = 0;
        for (int32_t i = 0; i < gamma; ++i) {
            const int64_t src = jbest + nbest + i;
            const int has = jbest >= 0 && src < L;
            draft[b * gamma + i] = has ? c[src] : -1;
            cnt += has;
        }
        n_draft[b] = cnt;
        if (match_pos) match_pos[b] = jbest;
        if (match_n) match_n[b] = nbest;
    }
}

/* ------------------------------------------------------------ tree verify
 * Verification of a token tree in one pass: several candidate continuations
 * per node ("Speculative decoding" (mhtirogla.ai), Levers and Implementation
 * notes: tree speculation, verify several candidates with a tree attention
 * mask; "Speculative decoding" (inference.tusharamrit.in), tree attention).
 * The pages give no multi-candidate acceptance rule; the reading (the
 * residual taken per node, the pages' single-draft rule applied to each
 * candidate in turn):
 *   - sequence b's tree has nodes 0..N_b-1, node 0 the root (the last
 *     context token), every other node a drafted token whose parent has a
 *     smaller index; the children of a node, in index order, are its
 *     candidates, drawn from q_u, the draft distribution at that node; p_u is
 *     the target's distribution after the path to node u (one target row and
 *     one draft row per node);
 *   - at node u with candidates c_1..c_m: r = p_u; candidate j with token x
 *     passes if u_acc(u, j) * q_u(x) < r(x), and the walk moves to c_j; else
 *     r becomes max(0, r - q_u) / Z (kept as it is if Z = 0) and the next
 *     candidate is tried. If all fail, the token is drawn from r with
 *     u_smp(u) (inverse CDF in index order, as the chain); at a node without
 *     children, from p_u (the bonus);
 *   - uniforms: u_acc(u, j) = word 0 of Philox4x32-10 at counter
 *     (u + j * 65536, seq_offset + b, round lo, round hi), u_smp(u) = word 1
 *     at counter (u, ...): a chain (one child per node) draws exactly what
 *     the chain verify draws;
 *   - greedy: the walk moves to the first child whose token is the target's
 *     argmax at the node (first index, NaN read as -inf), else emits that
 *     argmax and stops.
 * Outputs per sequence: out_tokens[off .. off + a] the a accepted tokens
 * then the emitted one, -1 after (up to N_b slots); out_path[off .. off+a)
 * the accepted nodes, -1 after; out_accepted[b] = a. Statuses as the chain:
 * layout (node offsets within [0, nodes], N_b >= 1, parents), temperature,
 * tokens, rows. The boundary keeps at most ORC_TREE_MAX_CAND candidates per
 * node for the sampling walk: a visited node with more gives the sequence
 * ORC_SEQ_UNSUPPORTED (checked on arrival, before the node's rows). */
#define ORC_TREE_MAX_CAND 64
typedef struct {
    int32_t batch, vocab, greedy;
    int64_t nodes; /* rows of parent / tokens / target / draft */
    const int64_t* node_off;
    const int32_t* parent;
    const int32_t* tokens;
    const void* target;
    int32_t target_dtype;
    const void* draft;
    int32_t draft_dtype, draft_is_probs;
    const float* temperatures;
    float temperature;
    uint64_t seed, round;
    uint32_t seq_offset;
    int32_t* out_tokens;
    int32_t* out_accepted;
    int32_t* out_path;
    int32_t* seq_status;
    double* diag_acc_margin; /* per sequence: min |u_acc - r(x)/q(x)| over the tests made */
    double* diag_u_smp;      /* u of the final draw */
    double* diag_cdf_lo;     /* normalised CDF edges of the emitted token */
    double* diag_cdf_hi;
} orc_tree_args_t;

static void tree_uniforms(const orc_tree_args_t* a, int64_t b, int64_t u, int64_t j, double* ua, double* us) {
    double x, y;
    orc_uniform_pair(a->seed, a->round, (uint32_t)(a->seq_offset + b), (uint32_t)(u + j * 65536), &x, &y);
    *ua = x;
    if (us) *us = y;
}

static void tree_write_error(const orc_tree_args_t* a, int64_t b, int32_t st) {
    const int64_t o = a->node_off[b], n = a->node_off[b + 1] - o;
    if (st != ORC_SEQ_BAD_LAYOUT)
        for (int64_t k = 0; k < n; ++k) {
            a->out_tokens[o + k] = -1;
            if (a->out_path) a->out_path[o + k] = -1;
        }
    a->out_accepted[b] = 0;
    if (a->seq_status) a->seq_status[b] = st;
}

static void tree_one(const orc_tree_args_t* a, int64_t b, double* p, double* q, double* r, double* t) {
    const int64_t V = a->vocab, o = a->node_off[b], N = a->node_off[b + 1] - o;
    if (N < 1 || o < 0 || o + N > a->nodes || a->parent[o] != -1) { tree_write_error(a, b, ORC_SEQ_BAD_LAYOUT); return; }
    for (int64_t v = 1; v < N; ++v)
        if (a->parent[o + v] < 0 || a->parent[o + v] >= v) { tree_write_error(a, b, ORC_SEQ_BAD_LAYOUT); return; }
    const double T = a->temperatures ? (double)a->temperatures[b] : (double)a->temperature;
    if (!a->greedy && (!(T > 0.0) || !isfinite(T))) { tree_write_error(a, b, ORC_SEQ_BAD_TEMP); return; }
    for (int64_t v = 1; v < N; ++v)
        if (a->tokens[o + v] < 0 || a->tokens[o + v] >= V) { tree_write_error(a, b, ORC_SEQ_BAD_TOKEN); return; }
    int64_t u = 0, acc = 0;
    double margin = INFINITY;
    for (;;) {
        const void* trow = row_ptr(a->target, a->target_dtype, o + u, V);
        if (a->greedy) {
            const int64_t g = orc_argmax_row(trow, a->target_dtype, V);
            int64_t next = -1;
            for (int64_t v = u + 1; v < N && next < 0; ++v)
                if (a->parent[o + v] == u && a->tokens[o + v] == g) next = v;
            if (next < 0) { a->out_tokens[o + acc] = (int32_t)g; break; }
            a->out_tokens[o + acc] = (int32_t)g;
            if (a->out_path) a->out_path[o + acc] = (int32_t)next;
            ++acc;
            u = next;
            continue;
        }
        int64_t n_child = 0;
        for (int64_t v = u + 1; v < N; ++v) n_child += a->parent[o + v] == u;
        if (n_child > ORC_TREE_MAX_CAND) { tree_write_error(a, b, ORC_SEQ_UNSUPPORTED); return; }
        int32_t st = orc_softmax_row(trow, a->target_dtype, V, T, p);
        if (st) { tree_write_error(a, b, st); return; }
        const int has_child = n_child > 0;
        double us;
        if (!has_child) { /* the bonus token from p_u */
            double ua;
            tree_uniforms(a, b, u, 0, &ua, &us);
            const int64_t tok = orc_inverse_cdf(p, V, us);
            a->out_tokens[o + acc] = (int32_t)tok;
            if (a->diag_u_smp) a->diag_u_smp[b] = us;
            if (a->diag_cdf_lo && a->diag_cdf_hi) orc_cdf_edges(p, V, tok, &a->diag_cdf_lo[b], &a->diag_cdf_hi[b]);
            break;
        }
        const void* drow = row_ptr(a->draft, a->draft_dtype, o + u, V);
        st = a->draft_is_probs ? orc_normalize_row(drow, a->draft_dtype, V, q)
                               : orc_softmax_row(drow, a->draft_dtype, V, T, q);
        if (st) { tree_write_error(a, b, st); return; }
        for (int64_t k = 0; k < V; ++k) r[k] = p[k];
        int64_t next = -1, j = 0;
        for (int64_t v = u + 1; v < N && next < 0; ++v) {
            if (a->parent[o + v] != u) continue;
            const int32_t x = a->tokens[o + v];
            double ua;
            tree_uniforms(a, b, u, j, &ua, NULL);
            if (q[x] > 0.0) {
                const double dm = fabs(ua - r[x] / q[x]);
                if (dm < margin) margin = dm;
            }
            if (ua * q[x] < r[x]) {
                next = v;
                break;
            }
            const double Z = orc_residual(r, q, V, t);
            if (Z > 0.0)
                for (int64_t k = 0; k < V; ++k) r[k] = t[k] / Z;
            ++j;
        }
        if (next >= 0) {
            a->out_tokens[o + acc] = a->tokens[o + next];
            if (a->out_path) a->out_path[o + acc] = (int32_t)next;
            ++acc;
            u = next;
            continue;
        }
        double ua0;
        tree_uniforms(a, b, u, 0, &ua0, &us);
        const int64_t tok = orc_inverse_cdf(r, V, us);
        a->out_tokens[o + acc] = (int32_t)tok;
        if (a->diag_u_smp) a->diag_u_smp[b] = us;
        if (a->diag_cdf_lo && a->diag_cdf_hi) orc_cdf_edges(r, V, tok, &a->diag_cdf_lo[b], &a->diag_cdf_hi[b]);
        break;
    }
    for (int64_t k = acc + 1; k < N; ++k) a->out_tokens[o + k] = -1;
    if (a->out_path)
        for (int64_t k = acc; k < N; ++k) a->out_path[o + k] = -1;
    a->out_accepted[b] = (int32_t)acc;
    if (a->diag_acc_margin) a->diag_acc_margin[b] = margin;
    if (a->seq_status) a->seq_status[b] = ORC_SEQ_OK;
}

void orc_tree_verify(const orc_tree_args_t* a) {
    const int64_t V = a->vocab;
    double* p = (double*)malloc(sizeof(double) * (size_t)V * 4);
    for (int64_t b = 0; b < a->batch; ++b) tree_one(a, b, p, p + V, p + 2 * V, p + 3 * V);
    free(p);
}
