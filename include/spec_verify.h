/*
 * spec_verify.h -- C ABI of libspecverify.so, the batched verify step of
 * speculative decoding on one GB300 (sm_103a).
 *
 * The operation (sources: page title, section):
 *   "Speculative decoding" (mhtirogla.ai), How it works, steps 2-5: the target
 *   returns p_1..p_{gamma+1} over the whole vocabulary; for i = 1..gamma accept
 *   x_i if u < p_i(x_i)/q_i(x_i); at the first rejection draw one token from
 *   norm(max(0, p_i - q_i)) and stop; if all gamma are accepted draw a bonus
 *   token from p_{gamma+1}; roll back the KV entries of the rejected drafts.
 *   Its "Code" section states the result: the accepted tokens plus exactly one
 *   corrected or bonus token. Greedy decoding reduces to "accept while the
 *   draft token equals the target's argmax" (same page, How it works; and
 *   "Speculative Decoding" (tokentrails.org), One round).
 *
 * Conventions for every entry point:
 *   - Pointers named *device* point to device memory owned by the caller; the
 *     library never frees or retains them after the call returns.
 *   - Every call is asynchronous on the given stream (NULL = legacy default
 *     stream) and never synchronises the host with the device.
 *   - The library allocates no device memory. Scratch space is the caller's
 *     workspace (see spec_verify_workspace_size / spec_workspace_init).
 *   - Host-detectable errors (NULL pointer, bad size, misaligned pointer, short
 *     workspace) return a non-zero spec_status_t synchronously and launch
 *     nothing. A failed launch returns SPEC_ERR_CUDA.
 *   - Data-dependent errors are reported per sequence in seq_status (one of
 *     SPEC_SEQ_*), never by a device trap or assert. An errored sequence gets
 *     accepted = 0, all of its token slots = -1 (not written for
 *     SPEC_SEQ_BAD_LAYOUT), and its KV length unchanged.
 *   - Two calls that share a workspace must not overlap on the device.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

/* Same type as cudaStream_t; declared here so plain C callers need no CUDA header. */
typedef struct CUstream_st* spec_stream_t;

#define SPEC_ABI_VERSION 5

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1, /* NULL where required, size out of range, bad enum */
    SPEC_ERR_ALIGNMENT = 2,   /* a pointer not aligned to its element type */
    SPEC_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned (256 B) or too small */
    SPEC_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
    SPEC_ERR_UNSUPPORTED = 5  /* a combination this build does not implement */
} spec_status_t;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

/* Per-sequence status words written to seq_status[b]. Checked in this order. */
enum {
    SPEC_SEQ_OK = 0,
    SPEC_SEQ_BAD_TOKEN = 1,  /* a draft token outside [0, V) */
    SPEC_SEQ_BAD_KV = 2,     /* kv_lens_in[b] < gamma_b */
    SPEC_SEQ_BAD_ROW = 3,    /* a row the decision needed has a NaN, +inf, no finite
                                logit, or (probs mode) a sum that is not > 0 */
    SPEC_SEQ_BAD_LAYOUT = 4, /* offsets of sequence b inconsistent or out of range */
    SPEC_SEQ_BAD_TEMP = 5,   /* temperature of sequence b not finite and > 0 */
    SPEC_SEQ_TIMEOUT = 6,    /* a bounded on-device wait for a copy gave up (the draw
                                is left at -1); never expected on a healthy GPU */
    SPEC_SEQ_UNSUPPORTED = 7 /* spec_tree_verify: a visited node with more than
                                SPEC_TREE_MAX_CANDIDATES children */
};
/* Precedence when several apply (the verify calls): LAYOUT, TEMP (sampling
 * only), TOKEN, KV, then ROW for the first bad row met while scanning
 * positions left to right. */

/*
 * Arguments of one batched verify call.
 *
 * Layout (row-major, V elements per row, rows packed contiguously):
 *   target_logits [rows_target, V]: sequence b owns rows target_row_off[b] ..
 *     target_row_off[b] + gamma_b, i.e. gamma_b + 1 rows, the last one being the
 *     bonus position (the target's distribution after x_gamma).
 *   draft [rows_draft, V]: sequence b owns rows draft_row_off[b] .. + gamma_b - 1,
 *     the drafter's logits (draft_is_probs = 0) or probabilities (= 1) at the
 *     positions where x_1..x_gamma were drawn.
 *   draft_tokens [rows_draft]: x_i of sequence b at draft_row_off[b] + i.
 *   out_tokens [rows_target]: slot target_row_off[b] + k, k = 0..gamma_b; slots
 *     0..accepted-1 hold the accepted drafts, slot `accepted` the corrected or
 *     bonus token, the rest -1.
 * With both offset pointers NULL every gamma_b = gamma_max and the offsets are
 * b*(gamma_max+1) and b*gamma_max. gamma_b is draft_row_off[b+1] -
 * draft_row_off[b] and must satisfy target_row_off[b+1] - target_row_off[b] ==
 * gamma_b + 1 and 0 <= gamma_b <= gamma_max (else SPEC_SEQ_BAD_LAYOUT). The
 * offsets must be non-decreasing from 0 to rows_target / rows_draft: the work
 * split relies on it, and a call that breaks it leaves undefined tokens
 * (but stays inside the buffers) and needs spec_workspace_init again.
 *
 * Temperature: both p and q are softmax(logits / T_b) with the same T_b
 * ("Speculative decoding" (mhtirogla.ai), Implementation notes: both models'
 * logits go through the same processing). A probabilities draft is used after
 * dividing each row by its own sum.
 *
 * Uniforms: with uniforms == NULL each draw comes from Philox4x32-10 (Salmon et
 * al., SC'11) keyed by seed, counter (position i, seq_offset + b, round lo 32,
 * round hi 32); word 0 gives u_acc, word 1 u_smp, each (w >> 8) * 2^-24, the
 * 24-bit uniforms of the page's Code section. Position i = 0..gamma_b - 1 is
 * draft x_{i+1}; i = gamma_b is the bonus position. With uniforms != NULL,
 * uniforms[2 * (target_row_off[b] + i) + {0, 1}] = (u_acc, u_smp) in [0, 1).
 * seq_offset lets a shard of a larger batch reproduce the whole batch's draws.
 */
typedef struct {
    uint32_t struct_size; /* sizeof(spec_verify_args_t), for ABI checks */
    int32_t batch;        /* 1 <= B <= 65536 */
    int32_t vocab;        /* 1 <= V <= 2097152 (larger: SPEC_ERR_UNSUPPORTED) */
    int32_t gamma_max;    /* 0 <= gamma_max <= 64 (larger: SPEC_ERR_UNSUPPORTED) */
    int64_t rows_target;  /* sum_b (gamma_b + 1) */
    int64_t rows_draft;   /* sum_b gamma_b */

    const int64_t* target_row_off; /* device [B+1] or NULL */
    const int64_t* draft_row_off;  /* device [B+1] or NULL (both or neither) */

    const void* target_logits; /* device [rows_target, V] */
    int32_t target_dtype;      /* spec_dtype_t */
    const void* draft;         /* device [rows_draft, V]; unused by greedy */
    int32_t draft_dtype;       /* spec_dtype_t */
    int32_t draft_is_probs;    /* 0: logits, 1: probabilities */
    const int32_t* draft_tokens; /* device [rows_draft] */

    const float* temperatures; /* device [B] or NULL; unused by greedy */
    float temperature;         /* used when temperatures == NULL; > 0 */

    uint64_t seed;       /* Philox key */
    uint64_t round;      /* Philox counter words 2-3 */
    uint32_t seq_offset; /* added to b in the Philox counter */
    const float* uniforms; /* device [rows_target, 2] or NULL */

    const int32_t* kv_lens_in; /* device [B] or NULL: target KV length incl. the gamma_b drafts */
    int32_t* kv_lens_out;      /* device [B] or NULL: kv - (gamma_b - accepted); may alias kv_lens_in */
    int32_t block_size;        /* > 0: also write ceil(kv_out / block_size) to out_num_blocks */
    int32_t* out_num_blocks;   /* device [B] or NULL */

    int32_t* out_tokens;   /* device [rows_target], required */
    int32_t* out_accepted; /* device [B], required */
    int32_t* seq_status;   /* device [B] or NULL */

    void* workspace;        /* device, 256-byte aligned, caller-owned */
    size_t workspace_bytes; /* >= spec_verify_workspace_size(this, mode) */

    /* Top-k truncation (sampling only; greedy ignores both): sequence b uses
     * k_b = top_ks[b] if top_ks != NULL, else top_k. With 0 < k_b < V every
     * target and draft row of b keeps the columns whose value is at least the
     * row's k_b-th largest value (NaN ranks as -inf; all ties at that value
     * stay) and p, q are renormalised over the kept columns; k_b <= 0 or
     * k_b >= V keeps the whole row. Both models' rows are processed alike
     * ("Speculative decoding" (mhtirogla.ai), Implementation notes). A draft
     * token outside its draft row's kept set has q = 0 (accepted iff p > 0).
     * Zero-initialise both for plain sampling. */
    int32_t top_k;
    const int32_t* top_ks; /* device [B] or NULL */

    /* Running acceptance per request, for adaptive gamma ("Speculative
     * decoding" (mhtirogla.ai), Implementation notes: gamma from running
     * acceptance). When accept_ema != NULL, every sequence with status OK and
     * gamma_b > 0 updates accept_ema[b] (float32, in place) by
     *   x = a_b / t_b,  accept_ema[b] += ema_lambda * (x - accept_ema[b]),
     * each operation rounded to float32 in that order, where a_b is the
     * accepted count and t_b = a_b + 1 if a draft was rejected, else gamma_b
     * (the accept tests the round performed). Other sequences keep their
     * value. Both verify calls update it. Zero-initialise both to skip it. */
    float* accept_ema; /* device [B] or NULL */
    float ema_lambda;

    /* Top-p (nucleus), after top-k or alone (sampling only; greedy ignores
     * it): sequence b uses p_b = top_ps[b] if top_ps != NULL, else top_p;
     * active for 0 < p_b < 1 (otherwise, and for NaN, off). Over the columns
     * top-k kept (every column when top-k is off for the sequence), each row
     * keeps the columns whose value is at least the value of the first group
     * of equal values, in decreasing order, at which the cumulative
     * probability reaches p_b (the whole group stays), on target and draft
     * rows alike ("Speculative decoding" (mhtirogla.ai), Implementation
     * notes: the same temperature, top-k and top-p processing). The masses
     * are double-float. Without top-k, one CTA per row takes the nucleus of
     * the whole row. A float histogram pass guesses the boundary; it bins only
     * values above 2^-16 of the row's largest and runs again over every value
     * when the guessed bin may hold one of the rest. f32 rows take a second
     * histogram pass. Double-float passes then check the guess and decide:
     * two reads of a bf16 row, four of an f32 row. A guess that fails the
     * check costs a full double-float bisection (8 more passes for bf16, 16
     * for f32), with the same result. Zero-initialise both for no top-p. */
    float top_p;
    const float* top_ps; /* device [B] or NULL */
} spec_verify_args_t;

/* ABI version of the loaded library (SPEC_ABI_VERSION at build time). */
SPEC_API int32_t spec_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
SPEC_API const char* spec_status_string(spec_status_t status);

/* Workspace bytes a call with these arguments needs (greedy != 0 for
 * spec_verify_greedy). Reads only the host fields batch, vocab, gamma_max,
 * rows_target, rows_draft, top_p and top_ps (a call that may ask for top-p
 * needs 4 KB more per row); pure host arithmetic, no CUDA call. Returns 0 if
 * those fields are out of range. */
SPEC_API size_t spec_verify_workspace_size(const spec_verify_args_t* args, int32_t greedy);

/* Zero the workspace's arrival counters (a stream-ordered memset of its
 * header). Call once after allocating a workspace, before its first use; the
 * kernels reset the counters themselves afterwards. */
SPEC_API spec_status_t spec_workspace_init(void* workspace, size_t workspace_bytes, spec_stream_t stream);

/* Sampling verify ("Speculative decoding" (mhtirogla.ai), How it works steps
 * 2-5 and Code; "Speculative decoding" (inference.tusharamrit.in), modified
 * rejection sampling). For each sequence: p_i = softmax(target row i / T_b),
 * q_i likewise for the draft row (or its normalised probabilities); accept x_i
 * while u_acc_i * q_i(x_i) < p_i(x_i); at the first rejection i emit the first
 * j with sum_{k<=j} max(0, p_i - q_i)_k > u_smp_i * Z, Z = sum max(0, p_i - q_i)
 * (if Z == 0, the same rule on p_i); if all gamma_b are accepted emit the bonus
 * from p_{gamma_b+1} by the same rule with u_smp at position gamma_b. Writes
 * out_tokens, out_accepted, kv_lens_out, out_num_blocks, seq_status. */
SPEC_API spec_status_t spec_verify_sample(const spec_verify_args_t* args, spec_stream_t stream);

/* Greedy verify ("Speculative decoding" (mhtirogla.ai), How it works;
 * "Speculative Decoding" (tokentrails.org), One round and Code): g_i = first
 * index of the largest raw target logit of row i (NaN read as -inf, -0 == +0);
 * accepted = number of leading i with x_i == g_i; emits x_1..x_accepted then
 * g_{accepted+1}. Ignores draft, draft_dtype, draft_is_probs, temperatures,
 * temperature, seed, round, seq_offset and uniforms. */
SPEC_API spec_status_t spec_verify_greedy(const spec_verify_args_t* args, spec_stream_t stream);

/* Largest scratch spec_verify_sample_static may use (bytes). */
#define SPEC_STATIC_SCRATCH_BYTES ((size_t)8 << 20)

/* spec_verify_sample on scratch the library owns, for callers that cannot
 * hand it device memory: a plain C caller with no device allocator of its
 * own, or an engine whose memory pool has already reserved the free HBM (for
 * its KV cache) and may not grow. Same arguments, results and errors as
 * spec_verify_sample except that workspace and workspace_bytes are ignored.
 * The source pages have no counterpart: this is a library convenience.
 *   - Scratch: a fixed device array of SPEC_STATIC_SCRATCH_BYTES (8 MiB) per
 *     device, part of the library's module; the call allocates nothing. A call
 *     with spec_verify_workspace_size(args, 0) > SPEC_STATIC_SCRATCH_BYTES
 *     returns SPEC_ERR_WORKSPACE before any CUDA call.
 *   - Set-up: the first call on a device (that device current) looks up the
 *     array's device address with cudaGetSymbolAddress; make that first call
 *     before any stream capture. The address is kept for the life of the
 *     process: it does not survive cudaDeviceReset (or any other teardown of
 *     the device's primary context), after which this entry point must not be
 *     called on that device again in the same process.
 *   - Every call clears the scratch's arrival counters and error word with a
 *     stream-ordered memset before its kernels; no spec_workspace_init needed.
 *   - There is one scratch per device: calls that overlap on the GPU (other
 *     streams, other host threads) race on it. Serialise them. */
SPEC_API spec_status_t spec_verify_sample_static(const spec_verify_args_t* args, spec_stream_t stream);

/* Adaptive gamma for the next round ("Speculative decoding" (mhtirogla.ai),
 * Implementation notes and Efficiency: gamma adaptive per request from
 * running acceptance, speculation off once the batch is compute-bound;
 * "Speculative decoding" (inference.tusharamrit.in), actual speedup
 * E / (1 + gamma c)). For each request b, with a = accept_ema[b] clamped to
 * [0, 1] (NaN read as 0), gammas_out[b] = the smallest g in [0, gamma_max]
 * with the largest E(a, g) / (1 + g c), E(a, g) = 1 + a + ... + a^g (the
 * pages' (1 - a^(g+1)) / (1 - a), summed term by term), c = draft_cost,
 * evaluated in float32 with correctly rounded operations in a fixed order
 * (the powers by repeated multiplication), so the result does not depend on
 * the device. If max_positions > 0 and the verify positions
 * P = sum_b (gammas_out[b] + 1) exceed it, every gammas_out[b] is 0.
 * total_positions_out (device int64, may be NULL) receives P, the positions
 * of the chosen gammas before that switch. accept_ema and gammas_out are
 * device [batch]; 1 <= batch <= 65536, 0 <= gamma_max <= 64, draft_cost >= 0
 * and finite. A batch above 1024 with max_positions > 0 needs
 * total_positions_out (the switch reads the sum from it); otherwise
 * SPEC_ERR_INVALID_ARG. */
SPEC_API spec_status_t spec_adapt_gamma(const float* accept_ema, int32_t batch, int32_t gamma_max, float draft_cost,
                                        int64_t max_positions, int32_t* gammas_out, int64_t* total_positions_out,
                                        spec_stream_t stream);

/* N-gram (prompt lookup) drafter: draft tokens at no model cost ("Speculative
 * decoding" (mhtirogla.ai), Implementation notes: copy the continuation of
 * the last matching n-gram; "Speculative decoding" (inference.tusharamrit.in),
 * n-gram / prompt lookup: search the context for the current suffix and
 * propose what followed it last time). Sequence b's context is
 * ctx[ctx_off[b] .. ctx_off[b+1]) (prompt and generated tokens, L_b of
 * them). For n = n_max down to n_min, the first n for which the last n
 * tokens occur earlier at a start j <= L_b - n - 1 (so a token follows; the
 * occurrence may overlap the suffix) gives the match: the latest such j.
 * Outputs: draft_out[b*gamma .. +gamma) = ctx[j+n ..] up to gamma tokens and
 * the end of the context, -1 after them; n_draft_out[b] = their number (0
 * without a match); match_pos_out[b] = j or -1 and match_n_out[b] = n or 0
 * (both may be NULL). All arrays are device memory; ctx_off is int64
 * [batch+1], non-decreasing. 1 <= batch <= 65536,
 * 1 <= n_min <= n_max <= 16, 0 <= gamma <= 64. The drafts feed either
 * verify: greedy as draft_tokens, sampling as draft_tokens with one-hot
 * probability rows. */
SPEC_API spec_status_t spec_ngram_draft(const int32_t* ctx, const int64_t* ctx_off, int32_t batch, int32_t n_max,
                                        int32_t n_min, int32_t gamma, int32_t* draft_out, int32_t* n_draft_out,
                                        int64_t* match_pos_out, int32_t* match_n_out, spec_stream_t stream);

/* Tree verification: several candidate continuations per position checked
 * in one target pass ("Speculative decoding" (mhtirogla.ai), Levers and
 * Implementation notes: tree speculation with a tree attention mask;
 * "Speculative decoding" (inference.tusharamrit.in), tree attention). The
 * pages give no rule for several candidates; this library takes the pages'
 * single-draft rule at every candidate in turn, with the residual carried
 * over:
 *   - sequence b owns nodes node_off[b] .. node_off[b+1) (N_b of them);
 *     local node 0 is the root (the last context token, parent -1), every
 *     other node v holds a drafted token tokens[v] and a parent in [0, v)
 *     (local indices); a node's children, in index order, are its
 *     candidates, drawn from the draft distribution q_u at that node;
 *   - target row o+u holds the target's logits after the path to node u
 *     (p_u), draft row o+u the draft's (q_u; probabilities if draft_is_probs);
 *   - sampling, at node u: r = p_u; candidate j (token x) passes if
 *     u_acc(u, j) * q_u(x) < r(x) and the walk moves to it; else r becomes
 *     max(0, r - q_u) / Z (left as it is if Z = 0) and the next candidate
 *     is tried; if none passes, the emitted token is drawn from r with
 *     u_smp(u) by inverse CDF in index order; a node without children emits
 *     the bonus token drawn from p_u. u_acc(u, j) = word 0 of Philox4x32-10
 *     at counter (u + 65536 j, seq_offset + b, round lo, round hi), u_smp(u) =
 *     word 1 at counter (u, ...), each (w >> 8) 2^-24: a chain-shaped tree
 *     draws what spec_verify_sample draws for the same chain;
 *   - greedy: the walk moves to the first child whose token is the target's
 *     argmax at the node (first index, NaN read as -inf), else emits it.
 * Outputs (device): out_tokens[node_off[b] + i] = the accepted tokens, then
 * the emitted one, -1 after (N_b slots); out_path (may be NULL) the accepted
 * nodes' local indices, -1 after; out_accepted[b] = their number;
 * seq_status[b] (may be NULL). Statuses, in this order: LAYOUT (N_b < 1,
 * offsets outside [0, nodes], a bad parent; the sequence's slots are not
 * written), TEMP (sampling), TOKEN (a node token outside [0, V)), then,
 * walking (sampling): UNSUPPORTED (a visited node with more than
 * SPEC_TREE_MAX_CANDIDATES children), ROW (the visited node's target row,
 * then its draft row if it has children). */
#define SPEC_TREE_MAX_CANDIDATES 64
typedef struct {
    uint32_t struct_size;        /* sizeof(spec_tree_args_t), for ABI checks */
    int32_t batch;               /* 1 <= batch <= 65536 */
    int32_t vocab;               /* 1 <= V <= 2097152 */
    int64_t nodes;               /* rows of parent, tokens, target, draft; <= 2^31 - 1 */
    const int64_t* node_off;     /* device [batch + 1] */
    const int32_t* parent;       /* device [nodes] */
    const int32_t* tokens;       /* device [nodes] (the root's entry is not read) */
    const void* target;          /* device [nodes, V], target_dtype */
    int32_t target_dtype;        /* spec_dtype_t */
    const void* draft;           /* device [nodes, V], draft_dtype (sampling; may be NULL for greedy) */
    int32_t draft_dtype;
    int32_t draft_is_probs;      /* 1: draft rows are probabilities, used divided by their sum */
    const float* temperatures;   /* device [batch] or NULL: then temperature */
    float temperature;
    uint64_t seed, round;
    uint32_t seq_offset;
    int32_t* out_tokens;         /* device [nodes] */
    int32_t* out_accepted;       /* device [batch] */
    int32_t* out_path;           /* device [nodes] or NULL */
    int32_t* seq_status;         /* device [batch] or NULL */
} spec_tree_args_t;

/* One launch, no workspace; greedy != 0 selects the greedy walk. Pointers
 * must be aligned to their element types (target/draft rows to their dtype). */
SPEC_API spec_status_t spec_tree_verify(const spec_tree_args_t* args, int32_t greedy, spec_stream_t stream);

/* KV-length rollback alone, e.g. for the draft model's cache ("Speculative
 * decoding" (mhtirogla.ai), How it works step 5: truncate the length in both
 * models; Implementation notes: paged KV makes this a length truncate).
 * kv_out[b] = kv_in[b] - (gamma_b - accepted[b]) with gamma_b = gammas[b] (or
 * gamma_max if gammas == NULL); out_num_blocks[b] = ceil(kv_out[b] / block_size)
 * if block_size > 0 and out_num_blocks != NULL. A sequence with accepted outside
 * [0, gamma_b] gets SPEC_SEQ_BAD_LAYOUT, one with kv_in < gamma_b SPEC_SEQ_BAD_KV;
 * both keep kv_out = kv_in. All arrays are device [batch]; kv_out may alias
 * kv_in; gammas, out_num_blocks, seq_status may be NULL. */
SPEC_API spec_status_t spec_kv_rollback(const int32_t* kv_in, int32_t* kv_out, const int32_t* accepted,
                                        const int32_t* gammas, int32_t gamma_max, int32_t batch,
                                        int32_t block_size, int32_t* out_num_blocks, int32_t* seq_status,
                                        spec_stream_t stream);

/* ---------------------------------------------------------------------------
 * Test hooks. Same conventions; they expose intermediate values of the last
 * spec_verify_sample / spec_verify_greedy call made with the same arguments
 * and workspace (stream-ordered after it).
 * ------------------------------------------------------------------------- */

/* The uniforms the sampling path draws: out[(b * npos + i) * 2 + {0,1}] =
 * (u_acc, u_smp) of sequence seq_offset + b at position i, i < npos.
 * out is device [batch * npos * 2]. */
SPEC_API spec_status_t spec_debug_philox(uint64_t seed, uint64_t round, uint32_t seq_offset, int32_t batch,
                                         int32_t npos, float* out, spec_stream_t stream);

/* Merged statistics of every row of the last call, in its row order (target
 * rows, then draft rows for sampling). Sampling: out_a[r] = m_r = max_j l_j
 * (the raw logit), out_b[r] = s_r = sum_j 2^(l_j k - fl(m_r k)), k = log2(e)/T
 * (probabilities rows: m_r = 0, s_r = sum_j q_j); greedy: out_a[r] = the
 * largest logit, out_idx[r] = its first index. Device arrays of
 * rows_target + rows_draft (greedy: rows_target) entries; any may be NULL. */
SPEC_API spec_status_t spec_debug_row_stats(const spec_verify_args_t* args, int32_t greedy, float* out_a,
                                            float* out_b, int32_t* out_idx, spec_stream_t stream);

/* The distributions the sampling path uses at position pos of sequence seq,
 * recomputed with the sampler's own arithmetic from the row statistics of the
 * last sampling call: out_p[V] = p_pos, out_q[V] = q_pos (zeros at the bonus
 * position), out_w[V] = the normalised sampling weights (max(0, p - q) / Z, or
 * p_pos at the bonus position or when Z == 0), out_scalars[4] = (p(x), q(x),
 * Z, 0) with x the draft token at pos and p(x), q(x) the values the accept
 * test used (0 at the bonus position; Z = -1 there). Device arrays; any may be
 * NULL. */
SPEC_API spec_status_t spec_debug_probs(const spec_verify_args_t* args, int32_t seq, int32_t pos, float* out_p,
                                        float* out_q, float* out_w, float* out_scalars, spec_stream_t stream);

/* The sampler's 2^x for light weights (exponents x <= -13) as its sums see
 * them: (y[2i], y[2i+1]) = (the SFU's 2^x[i], the correction that removes the
 * SFU's measured mean error when such weights are summed). x: device array of
 * n floats; y: device array of 2n floats. */
SPEC_API spec_status_t spec_debug_light_exp2(const float* x, float* y, int64_t n, spec_stream_t stream);

/* Profiling hook for the calling thread: when both are non-NULL, the next
 * spec_verify_sample / spec_verify_greedy call made by this thread records
 * start_event (a cudaEvent_t) on its stream just before its dominant kernel
 * (the fused verify kernel where a sampling call takes it, else the
 * streaming pass) and stop_event just after it, then clears the hook. Lets a
 * caller time that kernel with its own CUDA events. NULL, NULL clears it. */
SPEC_API spec_status_t spec_debug_time_next_stats(void* start_event, void* stop_event);

/* Test hook, process-wide: which kernels spec_verify_sample runs. path 0: the
 * default choice (the separate kernels: streaming pass, finalize, tile pass,
 * draw); 1: the separate kernels; 2: the fused verify kernel (one cooperative
 * launch that streams the sequences in waves and runs each sequence's
 * decision, tile pass and draw while later rows stream) wherever it applies:
 * sampling without top-k / top-p, rows on 16-byte boundaries, V <= 262144.
 * Both follow the same rules; the hook lets tests check each. Other values:
 * SPEC_ERR_INVALID_ARG. */
SPEC_API spec_status_t spec_debug_set_path(int32_t path);

/* Test hook for failure detection without a fault: one warp waits on the
 * device word *flag with the bounded wait the fused verify kernel uses for
 * its hand-offs between CTAs (poll with a growing sleep; give up after
 * limit_ns of the GPU's global timer or 2^26 polls), then writes out[0] =
 * the value it saw (0 if it gave up) and out[1] = 1 if it gave up, else 0.
 * flag and out: device pointers, 4-byte aligned (out holds two words).
 * limit_ns at most 10^10 (ten seconds). Asynchronous on `stream`; nothing
 * else is touched, and the context stays usable whichever way the wait ends.
 * Errors: SPEC_ERR_INVALID_ARG (null, misaligned or too long a limit),
 * SPEC_ERR_CUDA (the launch failed). No counterpart on the pages: it tests
 * the library's own bounded waits. */
SPEC_API spec_status_t spec_debug_wait_probe(const uint32_t* flag, uint64_t limit_ns, uint32_t* out,
                                             spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
