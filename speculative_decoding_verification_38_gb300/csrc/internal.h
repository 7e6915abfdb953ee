// internal.h -- kernel parameter blocks, workspace layout and launch entry
// points shared by the translation units of libspecverify.so. Not installed.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#define SPECV_F32 0
#define SPECV_BF16 1

namespace specv {

constexpr int kStatsThreads = 512;    // threads per CTA of the streaming pass (plain-load variant)
#ifndef SPECV_WS_WARPS
#define SPECV_WS_WARPS 16
#endif
#ifndef SPECV_WS_STAGES
#define SPECV_WS_STAGES 2
#endif
#ifndef SPECV_WS_STAGE_BYTES
#define SPECV_WS_STAGE_BYTES 6144
#endif
constexpr int kTmaConsumerWarps = SPECV_WS_WARPS;  // streaming pass, TMA variant: warps per CTA
constexpr int kTmaThreads = kTmaConsumerWarps * 32;
constexpr int kTmaStages = SPECV_WS_STAGES;          // stages in each warp's shared-memory ring
constexpr uint32_t kTmaStageBytes = SPECV_WS_STAGE_BYTES;  // bytes per stage (a multiple of 512)
static_assert(kTmaConsumerWarps * kTmaStages * kTmaStageBytes <= 200 * 1024, "warp rings exceed shared memory");
constexpr int kSampThreads = 256;     // threads per CTA of the residual sampler (one tile item per warp)
constexpr int kTile = 1024;           // sampler tile: 32 lanes x 32 contiguous columns
constexpr int kOpenCap = 32;           // open columns a sampler tile lists for the draw (more: the tile is summed again)
constexpr int64_t kChunkAlign = 64;   // elements; keeps 16-byte alignment for both dtypes
constexpr int64_t kMinChunk = 1024;   // smallest slice one CTA streams
constexpr int kGridCap = 4096;        // most CTAs of one streaming pass
constexpr int kMaxBatch = 65536;      // per-sequence words in the workspace header
// Workspace header, zeroed once by spec_workspace_init; every word returns
// to zero by the end of each call that uses it:
//   [0, 4B)     per-sequence arrival counters (both streaming passes)
//   [4B, 8B)    per-sequence tile items done (fused verify kernel)
//   [8B, 12B)   fused verify kernel: sequences in the order they were
//               finalized, as b + 1 (0: not yet)
//   then 256 bytes of words: the device error flags, the fused kernel's
//   ready-list length, its exit counter and its count of tile items handed out.
constexpr size_t kTilesDoneOffset = (size_t)kMaxBatch * 4;
constexpr size_t kReadyOffset = (size_t)kMaxBatch * 8;
constexpr size_t kErrWordOffset = (size_t)kMaxBatch * 12;       // device error flags (bit 0: a wait timed out)
constexpr size_t kReadyTailOffset = kErrWordOffset + 4;
constexpr size_t kExitCountOffset = kErrWordOffset + 8;
constexpr size_t kClaimOffset = kErrWordOffset + 12;              // fused kernel: tile items handed out
constexpr size_t kHeaderBytes = kErrWordOffset + 256;

constexpr int kSeqTimeout = 6;                                   // per-sequence status after a timed-out wait
constexpr int kSeqUnsupported = 7;                               // per-sequence status: a tree node with too many candidates
constexpr int kKeepCap = 1024;  // top-k-kept values stored per row for the nucleus (top-p) kernel
constexpr int64_t kMaxVocab = 2097152;                            // largest vocabulary (2^21 columns)

enum TaskMode : int32_t { kTaskNone = 0, kTaskResidual = 1, kTaskBonus = 2 };

// What the finalize step hands to the residual sampler, one per sequence.
struct __align__(16) SampleTask {
    int32_t mode;      // TaskMode
    int32_t probs;     // draft row holds probabilities
    int64_t trow;      // target row (index into target logits)
    int64_t drow;      // draft row (residual only), else -1
    int64_t out_slot;  // index into out_tokens
    float u;           // u_smp of the sampled position
    float k_hi, k_lo;  // log2(e) / T as a float pair
    float mt, md;      // raw maxima of the target / draft row
    float it_apx, id_apx;  // 1 / row normaliser of the target / draft row from the streaming pass (~1e-6)
    float z_hi, z_lo;  // written by the sampler: the Z it used
    float tau_t, tau_d;  // top-k thresholds of the two rows: columns below weigh 0 (-inf: no truncation)
    int32_t pad;
};
static_assert(sizeof(SampleTask) == 80, "task layout");

// Table 2^(i/64), i = 0..63, as float pairs (value = hi + lo).
struct Exp2Pairs {
    float hi[64], lo[64];
};

// Everything one streaming pass (and its finalize tail) needs.
struct StatsParams {
    const void* tgt;
    const void* dft;
    int32_t tdt, ddt, probs, greedy;
    int64_t V, rows_t, rows_d, N, chunk;
    int32_t S;   // partial slots (CTA pieces) per row
    int32_t pw;  // partials per slot (1: one per CTA piece; kTmaConsumerWarps: one per consumer warp)
    int32_t tma; // 1: TMA-pipelined variant (finalize runs as its own kernel)
    int32_t B, gmax, grid;
    const int64_t* tro;
    const int64_t* dro;
    const float* temps;
    float temperature;
    const int32_t* tokens;
    uint64_t seed, round;
    uint32_t seq_offset;
    const float* uniforms;
    const int32_t* kv_in;
    int32_t* kv_out;
    int32_t block_size;
    int32_t* out_blocks;
    int32_t* out_tokens;
    int32_t* out_accepted;
    int32_t* seq_status;
    // workspace views
    uint32_t* counters;  // [B] self-resetting arrival counters
    uint32_t* err;       // device error word (bit 0: a bounded wait gave up; bit 1: the fused kernel saw more
                         // finished sequences than the batch holds, i.e. offsets that break the work split)
    float2* partials;    // [rows_total * S * pw]
    float2* row_stats;   // [rows_total] merged per-row statistics
    float2* pq;          // [rows_d] (p(x), q(x))
    SampleTask* tasks;   // [B]
    // top-k truncation (sampling only): sequence b keeps the columns of each
    // of its rows whose value is at least the row's k_b-th largest, k_b =
    // top_ks[b] if top_ks, else top_k; k_b <= 0 or k_b >= V keeps every column
    const int32_t* top_ks;
    int32_t top_k;
    int32_t direct;      // 1: row_stats were written whole by the top-k pass; finalize reads them
    float* tau;          // [rows_total] threshold of every row (-inf: whole row), or null without top-k
    float* ema;          // [B] running acceptance (float32, updated in place), or null
    float ema_lambda;
    // top-p after top-k (sampling only): sequence b's p_b = top_ps[b] if
    // top_ps, else top_p; active for 0 < p_b < 1 (inside the top-k set, or over the whole row without top-k)
    const float* top_ps;
    float top_p;
    Exp2Pairs tab;       // 2^(i/64) for the double-float weights of the nucleus
    uint32_t* keep;      // [rows_total * kKeepCap] keys of each top-p row's top-k-kept values, or null
    int32_t* keep_n;     // [rows_total] their number (-1: more than kKeepCap; the row is read instead)
};


// One 1024-column tile of a sequence's task rows, as the sampler's first
// phase leaves it. Values are float pairs (double-float: value = [0] + [1]).
struct __align__(16) TileRec {
    float a[2], b[2];      // target / draft weight sums over the columns certainly in max(0, p - q)'s support
    float st[2], sd[2];    // target / draft weight sums over every column of the tile
    float uwt[2], uwd[2];  // the weights of the one column whose membership stayed open
    int32_t nu;            // such columns (more than one: see SampleParams::open)
    int32_t pad[3];
};
static_assert(sizeof(TileRec) == 64, "tile record layout");

struct SampleParams {
    const void* tgt;
    const void* dft;
    int32_t tdt, ddt;
    int64_t V;
    int32_t B;
    int32_t ntile;         // kTile-column tiles per row
    const SampleTask* tasks_in;
    SampleTask* tasks;
    TileRec* recs;         // [B * ntile]
    uint16_t* open;        // [B * ntile * kOpenCap]: a tile's open columns (first kOpenCap; more: summed again)
    int32_t* out_tokens;
    int32_t* seq_status;   // may be null
    uint32_t* err;         // workspace error word
    Exp2Pairs tab;         // 2^(i/64), i = 0..63
};

struct Layout {
    int64_t rows_total, N, chunk;
    int32_t S, grid;
    size_t off_partials, off_rowstats, off_pq, off_tasks, off_recs, off_open, off_tau, off_keep, off_keepn, off_spart,
        total;
};

// The fused sampling verify (one cooperative launch): the streaming pass,
// each sequence's accept scan as soon as its rows are folded, and the tile
// pass and draw of each finished sequence while other rows still stream.
struct VerifyParams {
    StatsParams s;          // streaming pass and decision (s.tma layout: one partial per warp)
    SampleParams t;         // tile pass and draw
    float2* spart;          // [rows_total * S] one merged partial per (row, CTA slice)
    uint32_t* tiles_done;   // header: [B] tile items finished
    uint32_t* ready;        // header: [B] finalized sequences in order, b + 1
    uint32_t* ready_tail;   // header word: entries in `ready`
    uint32_t* exit_count;   // header word: CTAs that finished
    uint32_t* claim;        // header word: tile items handed out
    uint64_t wait_ns;       // a wait on another CTA gives up after this long
    int32_t waves;          // sequence groups streamed one after another (1..kVerifyMaxWaves)
};
constexpr int kVerifyMaxLocalRows = 256;  // rows one CTA's slices of the fused kernel may touch
constexpr int kVerifyMaxWaves = 16;
constexpr int kVerifyMaxTiles = 256;      // fused kernel: V <= 256 * kTile
// Launch the fused kernel (cooperative); cudaErrorNotSupported-like errors
// leave the caller to use the separate kernels.
cudaError_t launch_verify(const VerifyParams& p, cudaStream_t s);
int verify_resident_ctas(int device);  // CTAs of the fused kernel one device holds at once (0: unknown)
// Test hook: one warp's bounded wait on *flag (the verify kernel's wait),
// recording the value seen (out[0]) and whether the wait gave up (out[1]).
cudaError_t launch_wait_probe(const uint32_t* flag, uint64_t limit_ns, uint32_t* out, cudaStream_t s);

// Work split and workspace layout for a given problem. grid_cap bounds the
// number of streaming CTAs (the launch uses the device's resident capacity).
// topp: the call may ask for top-p (the kept-value arrays are laid out).
Layout make_layout(int64_t B, int64_t V, int64_t rows_t, int64_t rows_d, int greedy, int64_t grid_cap, int pw,
                   bool topp = false);

cudaError_t launch_stats(const StatsParams& p, cudaStream_t s);
// TMA variant only: the per-sequence finalize (one warp each), chained to the
// streaming pass by programmatic launch.
cudaError_t launch_finalize(const StatsParams& p, cudaStream_t s);
int stats_resident_ctas(int device, int greedy);  // CTAs that fit at once on the device (plain-load variant)
// Top-k pass: for every row (one CTA each) its threshold into p.tau and its
// statistics over the kept columns into p.row_stats; replaces the streaming
// pass when any sequence truncates (finalize then runs with p.direct = 1).
cudaError_t launch_topk(const StatsParams& p, cudaStream_t s);
// Top-p: each top-p row's nucleus inside its top-k set (one warp per row),
// rewriting p.tau and the row sums; chained between launch_topk and
// launch_finalize by programmatic launch.
cudaError_t launch_nucleus(const StatsParams& p, cudaStream_t s);
// Rows with top-p and no top-k, f32 or probability rows (bf16 logits rows go
// to launch_whole): the nucleus of the whole row, one CTA per row; chained
// after launch_topk (programmatic launch).
cudaError_t launch_alone(const StatsParams& p, cudaStream_t s);
// Top-p without top-k on bf16 logits rows: each such row's maximum, nucleus
// and sum over the nucleus, whole (the top-k pass and alone_kernel leave these
// rows). One CTA per SM up to sms. after_topk: chained after launch_topk
// (programmatic launch); else launched as the step's first kernel.
cudaError_t launch_whole(const StatsParams& p, int sms, bool after_topk, cudaStream_t s);
cudaError_t launch_sampler(const SampleParams& p, cudaStream_t s, bool pdl);
void exp2_pairs(Exp2Pairs& t);  // host: fills the table
cudaError_t launch_kv_rollback(const int32_t* kv_in, int32_t* kv_out, const int32_t* accepted,
                               const int32_t* gammas, int32_t gmax, int32_t B, int32_t block_size,
                               int32_t* out_blocks, int32_t* seq_status, cudaStream_t s);
constexpr int kNgMaxN = 16;  // longest n-gram the drafter matches
cudaError_t launch_ngram(const int32_t* ctx, const int64_t* off, int32_t B, int32_t nmax, int32_t nmin, int32_t gamma,
                         int32_t* draft, int32_t* n_draft, int64_t* match_pos, int32_t* match_n, cudaStream_t s);
// Tree verification: one CTA per sequence walks its token tree.
struct TreeParams {
    int32_t B, greedy;
    int64_t V, nodes;
    const int64_t* node_off;  // [B+1]
    const int32_t* parent;    // [nodes] local parent index, -1 for a root
    const int32_t* tokens;    // [nodes]
    const void* tgt;          // [nodes, V]
    const void* dft;          // [nodes, V] (sampling)
    int32_t tdt, ddt, probs;
    const float* temps;
    float temperature;
    uint64_t seed, round;
    uint32_t seq_offset;
    int32_t* out_tokens;      // [nodes]
    int32_t* out_accepted;    // [B]
    int32_t* out_path;        // [nodes] or null
    int32_t* seq_status;      // [B] or null
    Exp2Pairs tab;
};
cudaError_t launch_tree(const TreeParams& p, cudaStream_t s);
cudaError_t launch_adapt_gamma(const float* ema, int32_t B, int32_t gmax, float c, int64_t max_positions,
                               int32_t* gammas, int64_t* total, cudaStream_t s);
cudaError_t launch_debug_philox(uint64_t seed, uint64_t round, uint32_t seq_offset, int32_t B, int32_t npos,
                                float* out, cudaStream_t s);
cudaError_t launch_debug_probs(const StatsParams& p, int32_t seq, int32_t pos, float* out_p, float* out_q,
                               float* out_w, float* out_scalars, cudaStream_t s);
cudaError_t launch_debug_light_exp2(const float* x, float* y, int64_t n, cudaStream_t s);
cudaError_t launch_debug_rowstats(const float2* row_stats, int64_t rows, int greedy, float* out_a, float* out_b,
                                  int32_t* out_idx, cudaStream_t s);

}  // namespace specv
