// api.cu -- the extern "C" entry points of libspecverify.so: argument
// validation, the workspace layout, and the launches. Nothing here computes
// part of the verify step on the host; every step runs in the kernels.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"
#include "spec_verify.h"

using namespace specv;

namespace {

constexpr int kMaxGammaApi = 64;  // finalize keeps per-position state in shared memory

struct DeviceInfo {
    bool ready = false;
    int resident_sample = 0;
    int resident_greedy = 0;
    int resident_verify = 0;  // CTAs of the fused verify kernel resident at once
    int sms = 0;
};
std::mutex g_mu;
DeviceInfo g_dev[64];

bool device_info(int& dev, DeviceInfo& out) {
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        d.resident_sample = stats_resident_ctas(dev, 0);
        d.resident_greedy = stats_resident_ctas(dev, 1);
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        d.resident_verify = verify_resident_ctas(dev);
        if (d.resident_sample <= 0 || d.resident_greedy <= 0) return false;
        d.ready = true;
    }
    out = d;
    return true;
}

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// 2^(i/64) as float pairs for the sampler's double-float exp2, computed once.
const Exp2Pairs& exp2_table() {
    static const Exp2Pairs t = [] {
        Exp2Pairs x;
        exp2_pairs(x);
        return x;
    }();
    return t;
}

thread_local cudaEvent_t t_ev_start = nullptr, t_ev_stop = nullptr;

// Launch the streaming pass (bracketed by the caller's events if the
// profiling hook is armed; the hook is consumed by this call) and, for the
// TMA variant, its finalize kernel.
cudaError_t stats_with_hook(const StatsParams& p, cudaStream_t s) {
    cudaEvent_t e0 = t_ev_start, e1 = t_ev_stop;
    t_ev_start = t_ev_stop = nullptr;
    if (e0 && e1 && cudaEventRecord(e0, s) != cudaSuccess) return cudaErrorUnknown;
    cudaError_t e = launch_stats(p, s);
    if (e != cudaSuccess) return e;
    if (e0 && e1 && cudaEventRecord(e1, s) != cudaSuccess) return cudaErrorUnknown;
    if (p.tma) {
        e = launch_finalize(p, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
// Whether whole_nucleus_kernel takes every row of the step: one top-p for
// all sequences, top-k off, bf16 logits on both sides and no row offsets (so
// no rows outside the sequences).
bool whole_only(const StatsParams& p) {
    return p.keep && !p.top_ks && !(p.top_k >= 1 && p.top_k < p.V) && !p.top_ps && p.top_p > 0.f &&
           p.top_p < 1.f && p.tdt == SPEC_BF16 && (p.rows_d == 0 || (p.ddt == SPEC_BF16 && !p.probs)) && !p.tro;
}
// The top-k pass, the whole-row nucleus kernels and the finalize kernel
// reading their rows. The hook brackets the top-k pass, or the whole-row
// kernel when that one takes every row (the top-k pass then does not run).
cudaError_t topk_with_hook(const StatsParams& p, int sms, cudaStream_t s) {
    cudaEvent_t e0 = t_ev_start, e1 = t_ev_stop;
    t_ev_start = t_ev_stop = nullptr;
    cudaError_t e;
    if (whole_only(p)) {
        if (e0 && e1 && cudaEventRecord(e0, s) != cudaSuccess) return cudaErrorUnknown;
        if ((e = launch_whole(p, sms, false, s)) != cudaSuccess) return e;
        if (e0 && e1 && cudaEventRecord(e1, s) != cudaSuccess) return cudaErrorUnknown;
        return launch_finalize(p, s);
    }
    if (e0 && e1 && cudaEventRecord(e0, s) != cudaSuccess) return cudaErrorUnknown;
    if ((e = launch_topk(p, s)) != cudaSuccess) return e;
    if (e0 && e1 && cudaEventRecord(e1, s) != cudaSuccess) return cudaErrorUnknown;
    if (p.keep && (e = launch_whole(p, sms, true, s)) != cudaSuccess) return e;
    if (p.keep && (e = launch_alone(p, s)) != cudaSuccess) return e;
    if (p.keep && (e = launch_nucleus(p, s)) != cudaSuccess) return e;
    return launch_finalize(p, s);
}
inline size_t esize(int32_t dt) { return dt == SPEC_F32 ? 4 : 2; }

// Host fields only; no CUDA call.
spec_status_t check_shape(const spec_verify_args_t* a) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->struct_size != sizeof(spec_verify_args_t)) return SPEC_ERR_INVALID_ARG;
    if (a->batch < 1 || a->batch > kMaxBatch) return SPEC_ERR_INVALID_ARG;
    if (a->vocab < 1) return SPEC_ERR_INVALID_ARG;
    if ((int64_t)a->vocab > kMaxVocab) return SPEC_ERR_UNSUPPORTED;
    if (a->gamma_max < 0) return SPEC_ERR_INVALID_ARG;
    if (a->gamma_max > kMaxGammaApi) return SPEC_ERR_UNSUPPORTED;
    if (a->rows_target < a->batch || a->rows_draft < 0) return SPEC_ERR_INVALID_ARG;
    if ((a->target_row_off == nullptr) != (a->draft_row_off == nullptr)) return SPEC_ERR_INVALID_ARG;
    if (!a->target_row_off) {
        if (a->rows_target != (int64_t)a->batch * (a->gamma_max + 1)) return SPEC_ERR_INVALID_ARG;
        if (a->rows_draft != (int64_t)a->batch * a->gamma_max) return SPEC_ERR_INVALID_ARG;
    }
    if (a->rows_target > (int64_t)a->batch * (a->gamma_max + 1)) return SPEC_ERR_INVALID_ARG;
    if (a->rows_draft > (int64_t)a->batch * a->gamma_max) return SPEC_ERR_INVALID_ARG;
    return SPEC_OK;
}

spec_status_t check_call(const spec_verify_args_t* a, int greedy) {
    spec_status_t st = check_shape(a);
    if (st) return st;
    if (a->target_dtype != SPEC_F32 && a->target_dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (!a->target_logits || !a->out_tokens || !a->out_accepted) return SPEC_ERR_INVALID_ARG;
    if (a->rows_draft > 0 && !a->draft_tokens) return SPEC_ERR_INVALID_ARG;
    if (!aligned(a->target_logits, esize(a->target_dtype))) return SPEC_ERR_ALIGNMENT;
    if (!greedy) {
        if (a->draft_dtype != SPEC_F32 && a->draft_dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
        if (a->draft_is_probs != 0 && a->draft_is_probs != 1) return SPEC_ERR_INVALID_ARG;
        if (a->rows_draft > 0 && !a->draft) return SPEC_ERR_INVALID_ARG;
        if (a->draft && !aligned(a->draft, esize(a->draft_dtype))) return SPEC_ERR_ALIGNMENT;
        if (!a->temperatures && !(a->temperature > 0.f && a->temperature < 3.0e38f)) return SPEC_ERR_INVALID_ARG;
        if (a->temperatures && !aligned(a->temperatures, 4)) return SPEC_ERR_ALIGNMENT;
        if (a->uniforms && !aligned(a->uniforms, 8)) return SPEC_ERR_ALIGNMENT;
        if (a->top_ks && !aligned(a->top_ks, 4)) return SPEC_ERR_ALIGNMENT;
        if (a->top_ps && !aligned(a->top_ps, 4)) return SPEC_ERR_ALIGNMENT;
    }
    if (a->accept_ema && !aligned(a->accept_ema, 4)) return SPEC_ERR_ALIGNMENT;
    if (a->accept_ema && !(a->ema_lambda >= 0.f && a->ema_lambda <= 1.f)) return SPEC_ERR_INVALID_ARG;
    if (a->block_size < 0) return SPEC_ERR_INVALID_ARG;
    if ((a->kv_lens_out || a->out_num_blocks) && !a->kv_lens_in) return SPEC_ERR_INVALID_ARG;
    if (a->out_num_blocks && a->block_size == 0) return SPEC_ERR_INVALID_ARG;
    const void* i32s[] = {a->draft_tokens, a->kv_lens_in, a->kv_lens_out, a->out_num_blocks,
                          a->out_tokens, a->out_accepted, a->seq_status};
    for (const void* p : i32s)
        if (p && !aligned(p, 4)) return SPEC_ERR_ALIGNMENT;
    if (a->target_row_off && (!aligned(a->target_row_off, 8) || !aligned(a->draft_row_off, 8)))
        return SPEC_ERR_ALIGNMENT;
    if (!a->workspace || !aligned(a->workspace, 256)) return SPEC_ERR_WORKSPACE;
    return SPEC_OK;
}

#ifndef SPECV_STREAM_TMA
#define SPECV_STREAM_TMA 1  // build-time choice: 0 always runs the plain-load streaming pass
#endif

// The TMA-pipelined streaming pass needs every row to start on a 16-byte
// boundary (bulk copies); otherwise the plain-load variant runs.
bool tma_ok(const spec_verify_args_t* a, int greedy) {
    const size_t V = (size_t)a->vocab;
    if (!aligned(a->target_logits, 16) || (V * esize(a->target_dtype)) % 16 != 0) return false;
    if (!greedy && a->rows_draft > 0 && (!aligned(a->draft, 16) || (V * esize(a->draft_dtype)) % 16 != 0))
        return false;
    return true;
}

// Whether any sequence of a sampling call truncates its rows (top-k or
// top-p; host fields only: a per-sequence array counts as truncating).
bool topp_possible(const spec_verify_args_t* a, int greedy) {
    return !greedy && (a->top_ps != nullptr || (a->top_p > 0.f && a->top_p < 1.f));
}

bool truncation_on(const spec_verify_args_t* a, int greedy) {
    if (greedy) return false;
    return a->top_ks != nullptr || (a->top_k > 0 && a->top_k < a->vocab) || a->top_ps != nullptr ||
           (a->top_p > 0.f && a->top_p < 1.f);
}

bool build_params(const spec_verify_args_t* a, int greedy, int grid_cap, int tma, StatsParams& p, Layout& L) {
    const int pw = tma ? kTmaConsumerWarps : 1;
    L = make_layout(a->batch, a->vocab, a->rows_target, a->rows_draft, greedy, grid_cap, pw, topp_possible(a, greedy));
    if (a->workspace_bytes < L.total) return false;
    char* ws = (char*)a->workspace;
    p.tgt = a->target_logits;
    p.dft = greedy ? nullptr : a->draft;
    p.tdt = a->target_dtype;
    p.ddt = greedy ? SPEC_F32 : a->draft_dtype;
    p.probs = greedy ? 0 : a->draft_is_probs;
    p.greedy = greedy;
    p.V = a->vocab;
    p.rows_t = a->rows_target;
    p.rows_d = a->rows_draft;
    p.N = L.N;
    p.chunk = L.chunk;
    p.S = L.S;
    p.pw = pw;
    p.tma = tma;
    p.B = a->batch;
    p.gmax = a->gamma_max;
    p.grid = L.grid;
    p.tro = a->target_row_off;
    p.dro = a->draft_row_off;
    p.temps = greedy ? nullptr : a->temperatures;
    p.temperature = greedy ? 1.f : a->temperature;
    p.tokens = a->draft_tokens;
    p.seed = a->seed;
    p.round = a->round;
    p.seq_offset = a->seq_offset;
    p.uniforms = greedy ? nullptr : a->uniforms;
    p.kv_in = a->kv_lens_in;
    p.kv_out = a->kv_lens_out;
    p.block_size = a->block_size;
    p.out_blocks = a->out_num_blocks;
    p.out_tokens = a->out_tokens;
    p.out_accepted = a->out_accepted;
    p.seq_status = a->seq_status;
    p.counters = (uint32_t*)ws;
    p.err = (uint32_t*)(ws + kErrWordOffset);
    p.partials = (float2*)(ws + L.off_partials);
    p.row_stats = (float2*)(ws + L.off_rowstats);
    p.pq = (float2*)(ws + L.off_pq);
    p.tasks = (SampleTask*)(ws + L.off_tasks);
    const bool tk = truncation_on(a, greedy);
    p.top_ks = tk ? a->top_ks : nullptr;
    p.top_k = tk ? a->top_k : 0;
    p.top_ps = tk ? a->top_ps : nullptr;
    p.top_p = tk ? a->top_p : 0.f;
    const bool tp = tk && topp_possible(a, greedy);
    if (tp) p.tab = exp2_table();
    p.keep = tp ? (uint32_t*)(ws + L.off_keep) : nullptr;
    p.keep_n = tp ? (int32_t*)(ws + L.off_keepn) : nullptr;
    p.direct = tk ? 1 : 0;
    p.tau = tk ? (float*)(ws + L.off_tau) : nullptr;
    p.ema = a->accept_ema;
    p.ema_lambda = a->ema_lambda;
    return true;
}

// Which kernels a sampling call takes (spec_debug_set_path): 0 the default
// choice, 1 the separate kernels, 2 the fused kernel wherever it applies.
std::atomic<int> g_path{0};
// The default: the separate kernels. The fused kernel is correct on every
// case it takes but does not yet beat them on the benchmarked workload.
constexpr bool kFusedByDefault = false;

spec_status_t prepare(const spec_verify_args_t* a, int greedy, StatsParams& p, Layout& L, int& dev,
                      DeviceInfo* info = nullptr) {
    spec_status_t st = check_call(a, greedy);
    if (st) return st;
    DeviceInfo di;
    if (!device_info(dev, di)) return SPEC_ERR_CUDA;
    if (info) *info = di;
    const int tma = (SPECV_STREAM_TMA && tma_ok(a, greedy)) ? 1 : 0;
    int cap = tma ? di.sms : (greedy ? di.resident_greedy : di.resident_sample);
    if (cap > kGridCap) cap = kGridCap;
    if (!build_params(a, greedy, cap, tma, p, L)) return SPEC_ERR_WORKSPACE;
    return SPEC_OK;
}

// ------------------------------------------------ library-owned scratch
// spec_verify_sample_static runs on this fixed device array instead of a
// caller workspace. Its device address is looked up once per device, with
// that device current, on the first call made there.
constexpr size_t kStaticScratchBytes = SPEC_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
static_assert(kStaticScratchBytes >= kHeaderBytes, "static scratch holds at least the header");
std::mutex g_scratch_mu;
void* g_scratch_ptr[64];

spec_status_t static_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
    if (dev < 0 || dev >= 64) return SPEC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return SPEC_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return SPEC_OK;
}

}  // namespace

extern "C" {

SPEC_API int32_t spec_abi_version(void) { return SPEC_ABI_VERSION; }

SPEC_API const char* spec_status_string(spec_status_t s) {
    switch (s) {
        case SPEC_OK: return "SPEC_OK";
        case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
        case SPEC_ERR_ALIGNMENT: return "SPEC_ERR_ALIGNMENT";
        case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE";
        case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
        case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
    }
    return "SPEC_ERR_UNKNOWN";
}

SPEC_API size_t spec_verify_workspace_size(const spec_verify_args_t* a, int32_t greedy) {
    if (check_shape(a) != SPEC_OK) return 0;
    // the smallest slice any launch uses gives the most partial slots
    Layout L = make_layout(a->batch, a->vocab, a->rows_target, a->rows_draft, greedy ? 1 : 0, kGridCap,
                           kTmaConsumerWarps, topp_possible(a, greedy ? 1 : 0));
    return L.total;
}

SPEC_API spec_status_t spec_workspace_init(void* workspace, size_t workspace_bytes, spec_stream_t stream) {
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < kHeaderBytes) return SPEC_ERR_WORKSPACE;
    if (cudaMemsetAsync(workspace, 0, kHeaderBytes, (cudaStream_t)stream) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_verify_sample(const spec_verify_args_t* a, spec_stream_t stream) {
    StatsParams p;
    Layout L;
    int dev = 0;
    DeviceInfo di;
    spec_status_t st = prepare(a, 0, p, L, dev, &di);
    if (st) return st;
    cudaStream_t s = (cudaStream_t)stream;
    // The fused kernel: rows on 16-byte boundaries, no truncation, V within
    // its tile limit, few enough rows per CTA, and the whole grid resident at
    // once. Its grid is one CTA per SM (fewer for small problems); the
    // sequences stream in W waves of about sixteen sequences each.
    const int32_t ntile = (int32_t)((p.V + kTile - 1) / kTile);
    const int64_t G = std::min<int64_t>(std::min(di.sms, di.resident_verify),
                                        std::max<int64_t>(1, (p.N + kMinChunk - 1) / kMinChunk));
    const int64_t chunk1 = std::max<int64_t>(kMinChunk, ((p.N + G - 1) / G + kChunkAlign - 1) / kChunkAlign * kChunkAlign);
    const int path = g_path.load();
    const bool want_fused = path == 2 || (path == 0 && kFusedByDefault);
    if (want_fused && p.tma && !p.direct && ntile <= kVerifyMaxTiles && G >= 1 &&
        2 * (chunk1 / p.V + 2) <= kVerifyMaxLocalRows) {
        const int32_t W = std::max(1, std::min(kVerifyMaxWaves, (p.B + 15) / 16));
        // partial slots as for the shortest slice any wave split can give
        StatsParams q;
        Layout Lf;
        if (!build_params(a, 0, (int)(W * G), 1, q, Lf)) return SPEC_ERR_WORKSPACE;
        q.grid = (int32_t)G;
        VerifyParams vp;
        vp.s = q;
        SampleParams& sp = vp.t;
        sp.tgt = q.tgt;
        sp.dft = q.dft;
        sp.tdt = q.tdt;
        sp.ddt = q.ddt;
        sp.V = q.V;
        sp.B = q.B;
        sp.ntile = ntile;
        sp.tasks_in = q.tasks;
        sp.tasks = q.tasks;
        char* ws = (char*)a->workspace;
        sp.recs = (TileRec*)(ws + Lf.off_recs);
        sp.open = (uint16_t*)(ws + Lf.off_open);
        sp.out_tokens = q.out_tokens;
        sp.seq_status = q.seq_status;
        sp.err = q.err;
        sp.tab = exp2_table();
        vp.spart = (float2*)(ws + Lf.off_spart);
        vp.tiles_done = (uint32_t*)(ws + kTilesDoneOffset);
        vp.ready = (uint32_t*)(ws + kReadyOffset);
        vp.ready_tail = (uint32_t*)(ws + kReadyTailOffset);
        vp.exit_count = (uint32_t*)(ws + kExitCountOffset);
        vp.claim = (uint32_t*)(ws + kClaimOffset);
        // a wait on another CTA gives up after 2 s plus the time to read the
        // rows at 100 GB/s
        const double bytes = (double)q.N * (q.tdt == SPEC_F32 ? 4.0 : 2.0);
        vp.wait_ns = (uint64_t)(2e9 + bytes / 100.0);
        vp.waves = W;
        cudaEvent_t e0 = t_ev_start, e1 = t_ev_stop;
        t_ev_start = t_ev_stop = nullptr;
        if (e0 && e1 && cudaEventRecord(e0, s) != cudaSuccess) return SPEC_ERR_CUDA;
        if (launch_verify(vp, s) != cudaSuccess) return SPEC_ERR_CUDA;
        if (e0 && e1 && cudaEventRecord(e1, s) != cudaSuccess) return SPEC_ERR_CUDA;
        return SPEC_OK;
    }
    if (p.direct) {
        // top-k: thresholds and truncated row statistics in one pass, then finalize
        if (topk_with_hook(p, di.sms, s) != cudaSuccess) return SPEC_ERR_CUDA;
    } else if (stats_with_hook(p, s) != cudaSuccess) {
        return SPEC_ERR_CUDA;
    }
    SampleParams sp;
    sp.tgt = p.tgt;
    sp.dft = p.dft;
    sp.tdt = p.tdt;
    sp.ddt = p.ddt;
    sp.V = p.V;
    sp.B = p.B;
    sp.ntile = (int32_t)((p.V + kTile - 1) / kTile);
    sp.tasks_in = p.tasks;
    sp.tasks = p.tasks;
    sp.recs = (TileRec*)((char*)a->workspace + L.off_recs);
    sp.open = (uint16_t*)((char*)a->workspace + L.off_open);
    sp.out_tokens = p.out_tokens;
    sp.seq_status = p.seq_status;
    sp.err = (uint32_t*)((char*)a->workspace + kErrWordOffset);
    sp.tab = exp2_table();
    if (launch_sampler(sp, s, true) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_verify_greedy(const spec_verify_args_t* a, spec_stream_t stream) {
    StatsParams p;
    Layout L;
    int dev = 0;
    spec_status_t st = prepare(a, 1, p, L, dev);
    if (st) return st;
    if (stats_with_hook(p, (cudaStream_t)stream) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_kv_rollback(const int32_t* kv_in, int32_t* kv_out, const int32_t* accepted,
                                        const int32_t* gammas, int32_t gamma_max, int32_t batch,
                                        int32_t block_size, int32_t* out_num_blocks, int32_t* seq_status,
                                        spec_stream_t stream) {
    if (!kv_in || !kv_out || !accepted || batch < 1 || gamma_max < 0 || block_size < 0) return SPEC_ERR_INVALID_ARG;
    if (out_num_blocks && block_size == 0) return SPEC_ERR_INVALID_ARG;
    const void* ps[] = {kv_in, kv_out, accepted, gammas, out_num_blocks, seq_status};
    for (const void* p : ps)
        if (p && !aligned(p, 4)) return SPEC_ERR_ALIGNMENT;
    if (launch_kv_rollback(kv_in, kv_out, accepted, gammas, gamma_max, batch, block_size, out_num_blocks,
                           seq_status, (cudaStream_t)stream) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_adapt_gamma(const float* accept_ema, int32_t batch, int32_t gamma_max, float draft_cost,
                                        int64_t max_positions, int32_t* gammas_out, int64_t* total_positions_out,
                                        spec_stream_t stream) {
    if (!accept_ema || !gammas_out || batch < 1 || batch > kMaxBatch) return SPEC_ERR_INVALID_ARG;
    if (gamma_max < 0 || gamma_max > kMaxGammaApi) return SPEC_ERR_INVALID_ARG;
    if (!(draft_cost >= 0.f && draft_cost < 3.0e38f)) return SPEC_ERR_INVALID_ARG;
    if (!aligned(accept_ema, 4) || !aligned(gammas_out, 4)) return SPEC_ERR_ALIGNMENT;
    if (total_positions_out && !aligned(total_positions_out, 8)) return SPEC_ERR_ALIGNMENT;
    if (max_positions > 0 && batch > 1024 && !total_positions_out) return SPEC_ERR_INVALID_ARG;
    if (launch_adapt_gamma(accept_ema, batch, gamma_max, draft_cost, max_positions, gammas_out, total_positions_out,
                           (cudaStream_t)stream) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_ngram_draft(const int32_t* ctx, const int64_t* ctx_off, int32_t batch, int32_t n_max,
                                        int32_t n_min, int32_t gamma, int32_t* draft_out, int32_t* n_draft_out,
                                        int64_t* match_pos_out, int32_t* match_n_out, spec_stream_t stream) {
    if (!ctx_off || !draft_out || !n_draft_out || batch < 1 || batch > kMaxBatch) return SPEC_ERR_INVALID_ARG;
    if (n_min < 1 || n_max < n_min || n_max > kNgMaxN || gamma < 0 || gamma > kMaxGammaApi) return SPEC_ERR_INVALID_ARG;
    if ((ctx && !aligned(ctx, 4)) || !aligned(ctx_off, 8) || !aligned(draft_out, 4) || !aligned(n_draft_out, 4))
        return SPEC_ERR_ALIGNMENT;
    if ((match_pos_out && !aligned(match_pos_out, 8)) || (match_n_out && !aligned(match_n_out, 4)))
        return SPEC_ERR_ALIGNMENT;
    if (launch_ngram(ctx, ctx_off, batch, n_max, n_min, gamma, draft_out, n_draft_out, match_pos_out, match_n_out,
                     (cudaStream_t)stream) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_tree_verify(const spec_tree_args_t* a, int32_t greedy, spec_stream_t stream) {
    if (!a || a->struct_size != sizeof(spec_tree_args_t)) return SPEC_ERR_INVALID_ARG;
    if (a->batch < 1 || a->batch > kMaxBatch || a->vocab < 1) return SPEC_ERR_INVALID_ARG;
    if ((int64_t)a->vocab > kMaxVocab) return SPEC_ERR_UNSUPPORTED;
    if (a->nodes < a->batch || a->nodes > INT32_MAX) return SPEC_ERR_INVALID_ARG;
    if (!a->node_off || !a->parent || !a->tokens || !a->target || !a->out_tokens || !a->out_accepted)
        return SPEC_ERR_INVALID_ARG;
    if (a->target_dtype != SPEC_F32 && a->target_dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (!aligned(a->node_off, 8) || !aligned(a->parent, 4) || !aligned(a->tokens, 4) ||
        !aligned(a->target, esize(a->target_dtype)) || !aligned(a->out_tokens, 4) || !aligned(a->out_accepted, 4))
        return SPEC_ERR_ALIGNMENT;
    if ((a->out_path && !aligned(a->out_path, 4)) || (a->seq_status && !aligned(a->seq_status, 4)))
        return SPEC_ERR_ALIGNMENT;
    if (!greedy) {
        if (!a->draft || (a->draft_dtype != SPEC_F32 && a->draft_dtype != SPEC_BF16)) return SPEC_ERR_INVALID_ARG;
        if (a->draft_is_probs != 0 && a->draft_is_probs != 1) return SPEC_ERR_INVALID_ARG;
        if (!aligned(a->draft, esize(a->draft_dtype))) return SPEC_ERR_ALIGNMENT;
        if (a->temperatures && !aligned(a->temperatures, 4)) return SPEC_ERR_ALIGNMENT;
    }
    TreeParams p{};
    p.B = a->batch;
    p.greedy = greedy ? 1 : 0;
    p.V = a->vocab;
    p.nodes = a->nodes;
    p.node_off = a->node_off;
    p.parent = a->parent;
    p.tokens = a->tokens;
    p.tgt = a->target;
    p.dft = greedy ? nullptr : a->draft;
    p.tdt = a->target_dtype;
    p.ddt = a->draft_dtype;
    p.probs = a->draft_is_probs;
    p.temps = a->temperatures;
    p.temperature = a->temperature;
    p.seed = a->seed;
    p.round = a->round;
    p.seq_offset = a->seq_offset;
    p.out_tokens = a->out_tokens;
    p.out_accepted = a->out_accepted;
    p.out_path = a->out_path;
    p.seq_status = a->seq_status;
    p.tab = exp2_table();
    if (launch_tree(p, (cudaStream_t)stream) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_debug_philox(uint64_t seed, uint64_t round, uint32_t seq_offset, int32_t batch,
                                         int32_t npos, float* out, spec_stream_t stream) {
    if (!out || batch < 1 || npos < 1 || !aligned(out, 4)) return SPEC_ERR_INVALID_ARG;
    if (launch_debug_philox(seed, round, seq_offset, batch, npos, out, (cudaStream_t)stream) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_debug_row_stats(const spec_verify_args_t* a, int32_t greedy, float* out_a,
                                            float* out_b, int32_t* out_idx, spec_stream_t stream) {
    StatsParams p;
    Layout L;
    int dev = 0;
    spec_status_t st = prepare(a, greedy ? 1 : 0, p, L, dev);
    if (st) return st;
    if (launch_debug_rowstats(p.row_stats, L.rows_total, greedy ? 1 : 0, out_a, out_b, out_idx,
                              (cudaStream_t)stream) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_debug_probs(const spec_verify_args_t* a, int32_t seq, int32_t pos, float* out_p,
                                        float* out_q, float* out_w, float* out_scalars, spec_stream_t stream) {
    StatsParams p;
    Layout L;
    int dev = 0;
    spec_status_t st = prepare(a, 0, p, L, dev);
    if (st) return st;
    if (seq < 0 || seq >= a->batch || pos < 0 || pos > a->gamma_max) return SPEC_ERR_INVALID_ARG;
    if (launch_debug_probs(p, seq, pos, out_p, out_q, out_w, out_scalars, (cudaStream_t)stream) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_debug_light_exp2(const float* x, float* y, int64_t n, spec_stream_t stream) {
    if (!x || !y || n < 1 || !aligned(x, 4) || !aligned(y, 4)) return SPEC_ERR_INVALID_ARG;
    if (launch_debug_light_exp2(x, y, n, (cudaStream_t)stream) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_debug_wait_probe(const uint32_t* flag, uint64_t limit_ns, uint32_t* out,
                                             spec_stream_t stream) {
    if (!flag || !out || !aligned(flag, 4) || !aligned(out, 4)) return SPEC_ERR_INVALID_ARG;
    if (limit_ns > 10000000000ull) return SPEC_ERR_INVALID_ARG;  // at most ten seconds
    if (launch_wait_probe(flag, limit_ns, out, (cudaStream_t)stream) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_debug_set_path(int32_t path) {
    if (path < 0 || path > 2) return SPEC_ERR_INVALID_ARG;
    g_path.store(path);
    return SPEC_OK;
}

SPEC_API spec_status_t spec_debug_time_next_stats(void* start_event, void* stop_event) {
    t_ev_start = (cudaEvent_t)start_event;
    t_ev_stop = (cudaEvent_t)stop_event;
    return SPEC_OK;
}

SPEC_API spec_status_t spec_verify_sample_static(const spec_verify_args_t* a, spec_stream_t stream) {
    // host checks first: nothing is looked up or launched for a rejected call
    spec_status_t st = check_shape(a);
    if (st) return st;
    if (spec_verify_workspace_size(a, 0) > kStaticScratchBytes) return SPEC_ERR_WORKSPACE;
    void* ws = nullptr;
    st = static_scratch(&ws);
    if (st) return st;
    spec_verify_args_t b = *a;
    b.workspace = ws;
    b.workspace_bytes = kStaticScratchBytes;
    // the call's own checks before the header is touched (spec_verify_sample
    // prepares the launch itself)
    st = check_call(&b, 0);
    if (st) return st;
    // arrival counters and error word start at zero on every call
    if (cudaMemsetAsync(ws, 0, kHeaderBytes, (cudaStream_t)stream) != cudaSuccess) return SPEC_ERR_CUDA;
    return spec_verify_sample(&b, stream);
}

}  // extern "C"
