// verify.cu -- the sampling verify step as one cooperative kernel.
//
// The separate kernels (stats.cu, sampler.cu) run the step as four launches:
// the streaming pass over every row, then each sequence's accept scan, the
// tile pass over the row pair its draw needs, and the draw. Every sequence's
// statistics are complete only when the whole stream is, so the last three
// run after the stream, on an idle memory system. Here one grid of one CTA
// per SM does all of it, and a sequence's tail runs while later rows stream:
//
//   Waves. The sequences are cut into W groups of consecutive sequences
//     (group w: sequences w B / W .. (w + 1) B / W - 1, by their offsets).
//     Every CTA streams its slice of group 0's rows, then its slice of group
//     1's, and so on, so group w's rows are all folded at about (w + 1) / W of
//     the stream.
//   Streaming warps (0..15) fold their CTA's slices through per-warp rings of
//     shared-memory stages filled by 1-D bulk copies, into per-warp partial
//     (max, sum) states ("Speculative decoding" (mhtirogla.ai), How it works,
//     steps 1-2: p and q over the whole vocabulary). A shared-memory counter
//     per row tells the last warp to leave a row; it merges the slice's warp
//     partials into one and counts the slice for the row's sequence. The warp
//     that completes a sequence's count takes its decision at once: the
//     strict accept scan u * q(x) < p(x) to the first rejection (same page,
//     step 3 and Code), the KV rollback (step 5) and the draw's task, which it
//     appends to a ready list. A streaming warp with no units left joins the
//     tail warps.
//   Tail warps (16..23) take tile items in ready-list order from a counter
//     (item k: list entry k / ntile, tile k % ntile): the double-float weight
//     sums of one 1024-column tile of the task's row pair (tile.cuh). The warp
//     that finishes a sequence's last tile draws its token: the residual
//     max(0, p - q) normalised by Z, or p for a bonus, by inverse CDF in index
//     order (step 4; "Speculative decoding" (inference.tusharamrit.in), the
//     residual p'(z) and its normaliser).
//
// Cross-CTA hand-offs are counters and one list in the workspace header. The
// only waits on other CTAs are waits for list entries, each bounded in time
// (on expiry the warp sets the workspace error word and stops; the draws it
// would have made stay at -1). The launch is cooperative, so every CTA is
// resident while others wait on it. Every counter and list entry is back at
// zero when the grid ends.
#include "stream.cuh"
#include "tile.cuh"

namespace specv {

namespace {

constexpr int kVStreamWarps = kTmaConsumerWarps;
constexpr int kVTailWarps = 8;
constexpr int kVThreads = (kVStreamWarps + kVTailWarps) * 32;
constexpr int kVRing = kTmaStages * (int)kTmaStageBytes;  // bytes of one streaming warp's ring
constexpr int kVMaxSegs = 2 * kVerifyMaxWaves;           // a CTA's slice of a wave: a target part and a draft part
constexpr int kVClosers = 2;                              // tail warps that close the CTA's rows

// One contiguous flat range of the CTA's work (flat element e: row e / V of
// the target rows, then of the draft rows, as in the streaming pass).
struct VSeg {
    int64_t f0, f1;  // elements [f0, f1)
    int64_t r0;      // row of f0
    int32_t u0;      // first unit of the segment in the CTA's numbering
    int32_t lbase;   // index of row r0 among the rows of the CTA (row counters)
    int32_t esz;     // element size of the segment's rows
    int32_t pad;
};

// A warp's shared memory while it works on tile items and draws.
struct VScratch {
    int32_t q[kQCap];  // heavy-column queue
    int32_t nu;        // open columns of the current tile
    float uw[4];       // the first one's weights
    float w_hi[kVerifyMaxTiles], w_lo[kVerifyMaxTiles];  // a draw's tile sums
};
static_assert(sizeof(VScratch) <= (size_t)kVRing, "a finished streaming warp's ring holds its scratch");

struct VSmem {
    uint64_t full[kVStreamWarps][kTmaStages];
    int64_t unit_of[kVStreamWarps][kTmaStages];
    int next_unit, failed;
    int nseg, nunits, nwaves;
    int64_t chunk;
    int64_t tw[kVerifyMaxWaves + 1], dw[kVerifyMaxWaves + 1];  // wave boundaries: target rows, draft rows
    VSeg seg[kVMaxSegs];
    uint32_t rowcnt[kVerifyMaxLocalRows];  // streaming warps that have left each row of the CTA
    Exp2Table tab;
    VScratch ts[kVTailWarps];
};

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Atomic adds that order this thread's earlier writes before the add
// (release) and its later reads after it (acquire), at CTA or GPU scope:
// the hand-offs between warps need no separate fence.
__device__ __forceinline__ uint32_t add_acq_rel_gpu(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ uint32_t add_acq_rel_cta_smem(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v) : "memory");
    return old;
}

constexpr uint32_t kPollCap = 1u << 26;  // polls of one wait, whatever the clock says

// Lane 0 polls *w until it is non-zero; the warp gets the value (0 if the
// wait gave up after limit_ns or kPollCap polls).
__device__ uint32_t warp_wait_nonzero(const uint32_t* w, uint64_t limit_ns) {
    uint32_t v = 0;
    if ((threadIdx.x & 31) == 0) {
        v = ld_acquire(w);
        if (!v) {
            const uint64_t t0 = global_ns();
            unsigned ns = 64;
            for (uint32_t it = 0; it < kPollCap; ++it) {
                __nanosleep(ns);
                if (ns < 2048) ns <<= 1;
                v = ld_acquire(w);
                if (v || global_ns() - t0 > limit_ns) break;
            }
        }
    }
    return __shfl_sync(0xffffffffu, v, 0);
}

__device__ __forceinline__ float2 v_ident(const StatsParams& p, int64_t r) {
    if (r >= p.rows_t && p.probs) return make_float2(0.f, 0.f);
    return make_float2(-INFINITY, 0.f);
}

__device__ __forceinline__ float2 v_merge(float2 a, float2 b, bool probs_row, float k) {
    return probs_row ? make_float2(0.f, a.y + b.y) : ms_merge(a, b, k);
}

// ------------------------------------------------------------ geometry
// The wave boundaries, the common slice length and this CTA's segments,
// computed by thread 0 from the offsets (the same values in every CTA).
// Wave w holds target rows [tw[w], tw[w+1]) and draft rows [dw[w], dw[w+1]);
// its rows form the virtual range target part then draft part, cut into one
// slice of `chunk` elements per CTA. Offsets that break the documented order
// still give a partition of the rows (boundaries clamped and made monotone).
__device__ void plan_waves(const VerifyParams& vp, VSmem& sm) {
    const StatsParams& p = vp.s;
    const int64_t V = p.V, G = gridDim.x;
    const int tesz = p.tdt == SPECV_F32 ? 4 : 2, desz = p.ddt == SPECV_F32 ? 4 : 2;
    int W = max(1, min(vp.waves, kVerifyMaxWaves));
    auto set_waves = [&](int w_count) {
        W = w_count;
        sm.tw[0] = sm.dw[0] = 0;
        for (int w = 1; w < W; ++w) {
            const int64_t b = (int64_t)w * p.B / W;
            const int64_t t = min(p.rows_t, max((int64_t)0, tro_at(p, b)));
            const int64_t d = min(p.rows_d, max((int64_t)0, dro_at(p, b)));
            sm.tw[w] = max(sm.tw[w - 1], t);
            sm.dw[w] = max(sm.dw[w - 1], d);
        }
        sm.tw[W] = p.rows_t;
        sm.dw[W] = p.rows_d;
        int64_t mx = 0;
        for (int w = 0; w < W; ++w) mx = max(mx, (sm.tw[w + 1] - sm.tw[w] + sm.dw[w + 1] - sm.dw[w]) * V);
        int64_t c = (mx + G - 1) / G;
        c = (c + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
        sm.chunk = max(c, kMinChunk);
    };
    set_waves(W);
    // rows a CTA may touch: per wave, each part spans at most chunk / V + 2 rows
    if ((int64_t)W * 2 * (sm.chunk / V + 2) > kVerifyMaxLocalRows) set_waves(1);
    sm.nwaves = W;
    int ns = 0, lrows = 0;
    int64_t units = 0;
    const int64_t c = blockIdx.x;
    auto add = [&](int64_t f0, int64_t f1, int esz) {
        VSeg& g = sm.seg[ns++];
        g.f0 = f0;
        g.f1 = f1;
        g.r0 = f0 / V;
        g.u0 = (int32_t)units;
        g.lbase = lrows;
        g.esz = esz;
        g.pad = 0;
        const int64_t ue = kTmaStageBytes / esz;
        units += (f1 - f0 + ue - 1) / ue;
        lrows += (int32_t)((f1 - 1) / V - g.r0 + 1);
    };
    for (int w = 0; w < W; ++w) {
        const int64_t nt = (sm.tw[w + 1] - sm.tw[w]) * V, n = nt + (sm.dw[w + 1] - sm.dw[w]) * V;
        const int64_t s0 = c * sm.chunk, s1 = min(n, s0 + sm.chunk);
        if (s0 >= s1) continue;
        if (s0 < nt) add(sm.tw[w] * V + s0, sm.tw[w] * V + min(s1, nt), tesz);
        if (s1 > nt) add((p.rows_t + sm.dw[w]) * V + (max(s0, nt) - nt), (p.rows_t + sm.dw[w]) * V + (s1 - nt), desz);
    }
    sm.nseg = ns;
    sm.nunits = (int)units;
}

// Where row r sits in its wave's virtual range: the first CTA slice it
// touches and how many slices it spans.
struct RowGeom {
    int64_t c_first;
    uint32_t nseg;
};
__device__ __forceinline__ RowGeom row_geom(const StatsParams& p, const VSmem& sm, int64_t r) {
    int64_t x;
    const int W = sm.nwaves;
    if (r < p.rows_t) {
        int w = 0;
        while (w + 1 < W && sm.tw[w + 1] <= r) ++w;
        x = (r - sm.tw[w]) * p.V;
    } else {
        const int64_t d = r - p.rows_t;
        int w = 0;
        while (w + 1 < W && sm.dw[w + 1] <= d) ++w;
        x = (sm.tw[w + 1] - sm.tw[w] + d - sm.dw[w]) * p.V;
    }
    RowGeom g;
    g.c_first = x / sm.chunk;
    g.nseg = (uint32_t)((x + p.V - 1) / sm.chunk - g.c_first + 1);
    return g;
}

// Slices of the rows of sequence b (the rows its offsets give, clamped to the
// tensors): the count of slice arrivals that completes b. Whole warp.
__device__ uint32_t expected_slices(const StatsParams& p, const VSmem& sm, int32_t b) {
    const int lane = threadIdx.x & 31;
    const int64_t t0 = max((int64_t)0, tro_at(p, b)), t1 = min(p.rows_t, tro_at(p, b + 1));
    const int64_t d0 = max((int64_t)0, dro_at(p, b)), d1 = min(p.rows_d, dro_at(p, b + 1));
    const int64_t nt = max((int64_t)0, t1 - t0), nd = max((int64_t)0, d1 - d0);
    uint32_t n = 0;
    for (int64_t j = lane; j < nt + nd; j += 32) n += row_geom(p, sm, j < nt ? t0 + j : p.rows_t + d0 + (j - nt)).nseg;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    return n;
}

// Merged statistics of row r from its slice partials (one lane).
__device__ float2 row_from_slices(const VerifyParams& vp, const VSmem& sm, int64_t r, bool probs_row, float k) {
    const StatsParams& p = vp.s;
    const uint32_t ns = row_geom(p, sm, r).nseg;
    const float2* src = vp.spart + r * p.S;
    float2 acc = probs_row ? make_float2(0.f, 0.f) : make_float2(-INFINITY, 0.f);
    uint32_t s = 0;
    for (; s + 4 <= ns; s += 4) {
        const float2 a = __ldcg(src + s), b = __ldcg(src + s + 1), c = __ldcg(src + s + 2), d = __ldcg(src + s + 3);
        acc = v_merge(acc, v_merge(v_merge(a, b, probs_row, k), v_merge(c, d, probs_row, k), probs_row, k),
                      probs_row, k);
    }
    for (; s < ns; ++s) acc = v_merge(acc, __ldcg(src + s), probs_row, k);
    return acc;
}

// Register slot h of lane l holds position l + 32 h; the value of position i
// (i uniform over the warp).
template <int N>
__device__ __forceinline__ float2 pick_pos(const float2 (&v)[N], int i) {
    float2 x = v[0];
#pragma unroll
    for (int h = 1; h < N; ++h)
        if ((i >> 5) == h) x = v[h];
    return make_float2(__shfl_sync(0xffffffffu, x.x, i & 31), __shfl_sync(0xffffffffu, x.y, i & 31));
}

// The decision of sequence b, once every slice of its rows is in: the checks
// in their documented order, the row statistics, p(x) and q(x) of every
// draft, the strict accept scan to the first rejection, the outputs, the KV
// rollback and the draw's task; then b joins the ready list. One warp.
__device__ void fin_warp(const VerifyParams& vp, const VSmem& sm, int32_t b) {
    const StatsParams& p = vp.s;
    const int lane = threadIdx.x & 31;
    const int64_t t0 = tro_at(p, b), t1 = tro_at(p, b + 1);
    const int64_t d0 = dro_at(p, b), d1 = dro_at(p, b + 1);
    const int64_t gg = d1 - d0;
    const int32_t g = (int32_t)gg;
    // The list entry releases lane 0's writes: the task and the draw's token
    // slot, the only outputs of the decision that another warp reads or
    // writes in this grid.
    auto publish = [&]() {
        __syncwarp();
        if (lane == 0) {
            const uint32_t pos = atomicAdd(vp.ready_tail, 1u);
            if (pos < (uint32_t)p.B) st_release(vp.ready + pos, (uint32_t)b + 1u);
            else atomicOr(p.err, 2u);  // more entries than sequences: offsets broke the work split
        }
        __syncwarp();
    };
    if (gg < 0 || gg > p.gmax || t1 - t0 != gg + 1 || t0 < 0 || t1 > p.rows_t || d0 < 0 || d1 > p.rows_d) {
        warp_write_error(p, b, 4, t0, g);  // SPEC_SEQ_BAD_LAYOUT
        publish();
        return;
    }
    const float T = temp_of(p, b);
    const float k = kLog2e / T;
    int32_t st = 0;
    if (!(T > 0.f) || !isfinite(T)) st = 5;  // SPEC_SEQ_BAD_TEMP
    int32_t x[2] = {0, 0};
    if (!st) {
        bool bad = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = lane + 32 * h;
            if (i < g) {
                x[h] = __ldg(p.tokens + d0 + i);
                bad |= (x[h] < 0 || x[h] >= p.V);
            }
        }
        for (int i = lane + 64; i < g; i += 32) {
            const int32_t xx = __ldg(p.tokens + d0 + i);
            bad |= (xx < 0 || xx >= p.V);
        }
        if (__any_sync(0xffffffffu, bad)) st = 1;  // SPEC_SEQ_BAD_TOKEN
    }
    const int32_t kv = p.kv_in ? __ldg(p.kv_in + b) : 0;
    if (!st && p.kv_in && kv < g) st = 2;  // SPEC_SEQ_BAD_KV
    if (st) {
        warp_write_error(p, b, st, t0, g);
        publish();
        return;
    }
    // row statistics: lane l holds positions l, l + 32, l + 64 (target) and
    // l, l + 32 (draft)
    float2 ts[3], ds[2];
    float lt[2] = {0.f, 0.f}, ld[2] = {0.f, 0.f}, ua[2] = {0.f, 0.f};
    const int tes = p.tdt == SPECV_F32 ? 4 : 2, des = p.ddt == SPECV_F32 ? 4 : 2;
#pragma unroll
    for (int h = 0; h < 3; ++h) {
        const int i = lane + 32 * h;
        ts[h] = make_float2(-INFINITY, 0.f);
        if (i <= g) {
            ts[h] = row_from_slices(vp, sm, t0 + i, false, k);
            p.row_stats[t0 + i] = ts[h];
        }
        if (h < 2) {
            ds[h] = make_float2(-INFINITY, 0.f);
            if (i < g) {
                ds[h] = row_from_slices(vp, sm, p.rows_t + d0 + i, p.probs != 0, k);
                p.row_stats[p.rows_t + d0 + i] = ds[h];
                lt[h] = ld_elem_rt((const char*)p.tgt + (t0 + i) * p.V * tes, p.tdt, x[h]);
                ld[h] = ld_elem_rt((const char*)p.dft + (d0 + i) * p.V * des, p.ddt, x[h]);
                ua[h] = p.uniforms ? __ldg(p.uniforms + 2 * (t0 + i))
                                   : draw_uniforms(p.seed, p.round, p.seq_offset + (uint32_t)b, (uint32_t)i).x;
            }
        }
    }
    // accept scan: the first position that is rejected or needs a bad row
    int32_t a = g, s2 = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int base = 32 * h;
        if (base >= g || a < g || s2) break;
        const int i = base + lane;
        bool stop = false, bad = false;
        if (i < g) {
            bad = !row_ok(ts[h], false) || !row_ok(ds[h], p.probs != 0);
            const float pxv = ex2(__fmaf_rn(lt[h], k, -__fmul_rn(ts[h].x, k))) * (1.0f / ts[h].y);
            const float qxv = p.probs ? ld[h] * (1.0f / ds[h].y)
                                      : ex2(__fmaf_rn(ld[h], k, -__fmul_rn(ds[h].x, k))) * (1.0f / ds[h].y);
            p.pq[d0 + i] = make_float2(pxv, qxv);
            stop = bad || !(__fmul_rn(ua[h], qxv) < pxv);
        }
        const uint32_t m = __ballot_sync(0xffffffffu, stop);
        if (m) {
            const int f = __ffs(m) - 1;
            if (__shfl_sync(0xffffffffu, bad, f)) s2 = 3;  // SPEC_SEQ_BAD_ROW
            else a = base + f;
        }
    }
    const float2 rsa = pick_pos(ts, a);                                   // target row at the sampled position
    const float2 rda = pick_pos(ds, a < g ? a : 0);                       // draft row there (a rejection)
    if (!s2 && a == g && !row_ok(rsa, false)) s2 = 3;
    if (s2) {
        warp_write_error(p, b, s2, t0, g);
        publish();
        return;
    }
#pragma unroll
    for (int h = 0; h < 3; ++h) {
        const int i = lane + 32 * h;
        if (i <= g && i != a) p.out_tokens[t0 + i] = (i < a) ? (h < 2 ? x[h] : __ldg(p.tokens + d0 + i)) : -1;
    }
    if (lane == 0) {
        p.out_tokens[t0 + a] = -1;  // the draw's slot, until the draw writes it
        update_ema(p, b, g, a);
        p.out_accepted[b] = a;
        if (p.kv_out || p.out_blocks) {
            const int32_t kvo = p.kv_in ? kv - (g - a) : 0;
            if (p.kv_out) p.kv_out[b] = kvo;
            if (p.out_blocks) p.out_blocks[b] = p.block_size > 0 ? (kvo + p.block_size - 1) / p.block_size : 0;
        }
        if (p.seq_status) p.seq_status[b] = 0;
        SampleTask t;
        t.mode = a < g ? kTaskResidual : kTaskBonus;
        t.probs = p.probs;
        t.trow = t0 + a;
        t.drow = a < g ? d0 + a : -1;
        t.out_slot = t0 + a;
        t.u = p.uniforms ? __ldg(p.uniforms + 2 * (t0 + a) + 1)
                         : draw_uniforms(p.seed, p.round, p.seq_offset + (uint32_t)b, (uint32_t)a).y;
        const df kk = k_pos_lo(k_of_temperature(T));
        t.k_hi = kk.hi;
        t.k_lo = kk.lo;
        t.mt = rsa.x;
        t.md = a < g ? rda.x : 0.f;
        t.it_apx = inv_norm_apx(rsa, k);
        t.id_apx = a < g ? (p.probs ? 1.0f / rda.y : inv_norm_apx(rda, k)) : 0.f;
        t.z_hi = t.z_lo = 0.f;
        t.tau_t = t.tau_d = -INFINITY;  // this path never truncates
        t.pad = 0;
        p.tasks[b] = t;
    }
    publish();
}

// ------------------------------------------------------------- streaming
// Row r of this CTA once every streaming warp has left it: merge the slice's
// warp partials into one and count the slice for the row's sequence; the
// count's last arrival takes the sequence's decision. Whole warp (the CTA's
// closer warp, so that no streaming warp stops for it).
// Lane 0 alone carries the hand-offs: it has acquired the other warps'
// partials (the row counter's atomic), merges them, stores the slice
// partial and counts it with an acquire-release add.
__device__ void close_slice(const VerifyParams& vp, const VSmem& sm, int64_t r, bool probs_row, float k) {
    const StatsParams& p = vp.s;
    const int lane = threadIdx.x & 31;
    const bool is_t = r < p.rows_t;
    const int32_t b = seq_of_row(p, !is_t, is_t ? r : r - p.rows_t);
    uint32_t old = 0;
    if (lane == 0) {
        const int64_t slot = (int64_t)blockIdx.x - row_geom(p, sm, r).c_first;
        const float2* src = p.partials + (r * p.S + slot) * p.pw;
        float2 w[kVStreamWarps];
#pragma unroll
        for (int i = 0; i < kVStreamWarps; ++i) w[i] = src[i];
#pragma unroll
        for (int h = kVStreamWarps / 2; h > 0; h >>= 1)
#pragma unroll
            for (int i = 0; i < h; ++i) w[i] = v_merge(w[i], w[i + h], probs_row, k);
        vp.spart[r * p.S + slot] = w[0];
        if (b >= 0) old = add_acq_rel_gpu(p.counters + b, 1u);
    }
    if (b < 0) return;
    old = __shfl_sync(0xffffffffu, old, 0);
    const uint32_t want = expected_slices(p, sm, b);
    if (old + 1 != want) return;
    if (lane == 0) p.counters[b] = 0;  // every slice of b is in: ready for the next call
    __syncwarp();
    fin_warp(vp, sm, b);
}

// Reduce this warp's lane states of row r; lane 0 stores the warp partial.
__device__ void v_lane_flush(const StatsParams& p, LaneAcc& a, int mode, float k, int64_t idx, bool poison) {
    const int lane = threadIdx.x & 31;
    float2 out;
    if (mode == kLogits) {
        float2 v = make_float2(a.m, a.s.x + a.s.y);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float2 w = make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o));
            v = ms_merge(v, w, k);
        }
        out = v;
    } else {
        float v = a.s.x + a.s.y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        out = make_float2(0.f, v);
    }
    if (lane == 0) {
        if (poison) out = make_float2(NAN, NAN);
        p.partials[idx] = out;
    }
    lane_reset(a);
}

// Returns false if a copy wait gave up (the warp's ring may still be written).
__device__ bool stream_warp(const VerifyParams& vp, VSmem& sm, char* ring, int warp) {
    const StatsParams& p = vp.s;
    const int lane = threadIdx.x & 31;
    const int nseg = sm.nseg, nunits = sm.nunits;
    const int64_t T = p.rows_t * p.V;
    char* myring = ring + (size_t)warp * kVRing;
    uint64_t* full = sm.full[warp];
    uint32_t issued = 0, copies = 0;
    int tseg = 0;  // lane 0: segment of the last unit taken
    auto take = [&](bool copy) -> bool {
        const int u = atomicAdd(&sm.next_unit, 1);
        if (u >= nunits) return false;
        while (tseg + 1 < nseg && u >= sm.seg[tseg + 1].u0) ++tseg;
        const int st = issued % kTmaStages;
        sm.unit_of[warp][st] = u;
        if (copy) {
            const VSeg& g = sm.seg[tseg];
            const int64_t ue = kTmaStageBytes / g.esz;
            const int64_t f = g.f0 + (int64_t)(u - g.u0) * ue, s1 = min(g.f1, f + ue);
            const char* src = f < T ? (const char*)p.tgt + f * g.esz : (const char*)p.dft + (f - T) * g.esz;
            mbar_arrive_expect_tx(&full[st], (uint32_t)((s1 - f) * g.esz));
            bulk_g2s(myring + (size_t)st * kTmaStageBytes, src, (uint32_t)((s1 - f) * g.esz), &full[st]);
            copies = issued + 1;
        }
        ++issued;
        return true;
    };
    if (lane == 0)
        for (int i = 0; i < kTmaStages; ++i)
            if (!take(true)) break;
    issued = __shfl_sync(0xffffffffu, issued, 0);
    __syncwarp();

    LaneAcc a;
    lane_reset(a);
    bool dead = false;
    uint32_t done = 0;
    // row bookkeeping: the segment the warp is in, its current row and the
    // parameters of that row
    int cs = 0;
    int64_t r = nseg > 0 ? sm.seg[0].r0 : 0, row_end = (r + 1) * p.V;
    bool touched = false;
    int mode = kLogits, dt = SPECV_BF16;
    float k = 1.f;
    int64_t param_row = -1;
    auto set_row = [&]() {
        if (param_row == r) return;
        param_row = r;
        const bool is_t = r < p.rows_t;
        dt = is_t ? p.tdt : p.ddt;
        mode = (!is_t && p.probs) ? kProbs : kLogits;
        k = 1.f;
        const int32_t b = seq_of_row(p, !is_t, is_t ? r : r - p.rows_t);
        if (b >= 0) k = kLog2e / temp_of(p, b);
    };
    auto leave_row = [&]() {  // this warp's partial of row r, then r counts as left
        set_row();
        const int64_t idx = (r * p.S + ((int64_t)blockIdx.x - row_geom(p, sm, r).c_first)) * p.pw + warp;
        if (touched) v_lane_flush(p, a, mode, k, idx, dead);
        else if (lane == 0) p.partials[idx] = v_ident(p, r);
        if (lane == 0)  // releases this warp's partial to the CTA's closer warp
            add_acq_rel_cta_smem(&sm.rowcnt[sm.seg[cs].lbase + (r - sm.seg[cs].r0)], 1u);
        touched = false;
        ++r;
        row_end += p.V;
    };
    auto seg_last_row = [&](int s) { return (sm.seg[s].f1 - 1) / p.V; };
    // leave every row before segment s, element f
    auto advance = [&](int s, int64_t f) {
        while (cs < s) {
            while (r <= seg_last_row(cs)) leave_row();
            ++cs;
            r = sm.seg[cs].r0;
            row_end = (r + 1) * p.V;
        }
        while (f >= row_end) leave_row();
    };
    int useg = 0;  // segment of the unit being consumed
    for (uint32_t kk = 0; kk < issued; ++kk) {
        const int st = kk % kTmaStages;
        if (!dead) {
            const bool ok = mbar_wait_bounded(&full[st], (kk / kTmaStages) & 1, kWaitLimit);
            dead = __any_sync(0xffffffffu, !ok);
            if (dead && lane == 0) atomicExch(&sm.failed, 1);
            if (!dead) done = kk + 1;
        }
        const int u = sm.unit_of[warp][st];
        while (useg + 1 < nseg && u >= sm.seg[useg + 1].u0) ++useg;
        const VSeg& g = sm.seg[useg];
        const int64_t ue = kTmaStageBytes / g.esz;
        const int64_t f = g.f0 + (int64_t)(u - g.u0) * ue, s1 = min(g.f1, f + ue);
        advance(useg, f);
        set_row();
        const uint32_t base = smem_addr(myring + (size_t)st * kTmaStageBytes);
        for (int64_t g0 = f; g0 < s1;) {
            const int64_t se = min(s1, row_end);
            touched = true;
            if (!dead) {
                const int esz = dt == SPECV_F32 ? 4 : 2;
                const uint32_t sa = base + (uint32_t)((g0 - f) * esz);
                const int nvec = (int)((se - g0) * esz / 16);
                const int64_t col0 = g0 - (row_end - p.V);
                if (mode == kLogits) {
                    if (dt == SPECV_F32) warp_segment<SPECV_F32, kLogits>(a, sa, nvec, col0, k, lane);
                    else warp_segment<SPECV_BF16, kLogits>(a, sa, nvec, col0, k, lane);
                } else {
                    if (dt == SPECV_F32) warp_segment<SPECV_F32, kProbs>(a, sa, nvec, col0, k, lane);
                    else warp_segment<SPECV_BF16, kProbs>(a, sa, nvec, col0, k, lane);
                }
            }
            if (se == row_end) {
                leave_row();
                if (se < s1) set_row();
            }
            g0 = se;
        }
        __syncwarp();
        if (lane == 0) {
            if (!dead) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            take(!dead);
        }
        issued = __shfl_sync(0xffffffffu, issued, 0);
        __syncwarp();
    }
    // the rest of the CTA's rows
    if (nseg > 0) {
        advance(nseg - 1, sm.seg[nseg - 1].f0);
        while (r <= seg_last_row(nseg - 1)) leave_row();
    }
    bool drained = true;
    if (lane == 0) {
        for (uint32_t q = done; q < copies; ++q)
            drained &= mbar_wait_bounded(&full[q % kTmaStages], (q / kTmaStages) & 1, kWaitLimit);
    }
    return __shfl_sync(0xffffffffu, (int)(drained && !dead), 0) != 0;
}

// ------------------------------------------------------------------ tail
// A task another CTA wrote during this grid, read from L2.
__device__ __forceinline__ SampleTask load_task(const SampleTask* src) {
    static_assert(sizeof(SampleTask) % 16 == 0, "task in 16-byte words");
    SampleTask t;
    const float4* s = reinterpret_cast<const float4*>(src);
    float4* d = reinterpret_cast<float4*>(&t);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(SampleTask) / 16); ++i) d[i] = __ldcg(s + i);
    return t;
}

__device__ __forceinline__ TileScratch scratch_of(VScratch& x, const Exp2Table& tab) {
    return TileScratch{x.q, &x.nu, x.uw, &tab};
}

// One tile item: the double-float sums of tile `tile` of sequence b's task
// rows (the sampler kernel's phase 1, one warp). Lane 0 writes the record;
// returns the tile's open columns (their list is written by any lane).
template <int TDT, int DDT>
__device__ int32_t tile_warp(const VerifyParams& vp, VScratch& x, const Exp2Table& tab, int32_t b, int32_t tile,
                             const SampleTask& t) {
    const SampleParams& p = vp.t;
    const int lane = threadIdx.x & 31;
    const bool resid = t.mode == kTaskResidual;
    const float ratio = resid ? t.id_apx / t.it_apx : 0.f;
    const float r_hi = ratio * (1.f + kMargin), r_lo = ratio * (1.f - kMargin);
    if (lane == 0) x.nu = 0;
    __syncwarp();
    const int64_t item = (int64_t)b * p.ntile + tile;
    const RowPair<TDT, DDT> rp = tile_rows<TDT, DDT>(p, t, tile);
    TileAcc acc;
    tile_sums_packed<TDT, DDT>(rp, resid, r_hi, r_lo, scratch_of(x, tab), p.open + item * kOpenCap, 0, kGroups, acc);
    const df tot = warp_sum4_df(acc.st, acc.sd, resid ? acc.a : acc.st, acc.b);
    const df tsd = shfl_df(tot, 8), ta = shfl_df(tot, 16), tb = shfl_df(tot, 24);
    __syncwarp();
    const int32_t nu = x.nu;
    if (lane == 0) {
        float4* rec = reinterpret_cast<float4*>(p.recs + item);
        rec[0] = make_float4(ta.hi, ta.lo, tb.hi, tb.lo);
        rec[1] = make_float4(tot.hi, tot.lo, tsd.hi, tsd.lo);
        rec[2] = make_float4(x.uw[0], x.uw[1], x.uw[2], x.uw[3]);
        rec[3] = make_float4(__int_as_float(nu), 0.f, 0.f, 0.f);
    }
    return nu;
}

// Exclusive warp scan of double-float values in lane order.
__device__ __forceinline__ df warp_excl_scan_df(df x) {
    const df incl = warp_scan_df(x);
    df e = shfl_up_df(incl, 1);
    if ((threadIdx.x & 31) == 0) e = df{0.f, 0.f};
    return e;
}

// The sampling weight of a column from its values, with the light-weight
// mean-error correction the tile sums apply to their light sums (clw), so
// that every level of the draw adds the same quantities.
template <int TDT, int DDT>
__device__ __forceinline__ df draw_weight(const RowPair<TDT, DDT>& rp, float lt, float ld, int mode, df It, df Id,
                                          float clw, const Exp2Table& tab) {
    df w = rp.wt(lt, tab);
    if (mode == kTaskResidual) w = resid_weight(w, rp.wd(ld, tab), It, Id);
    return is_heavy(w) ? w : light_sum_df(w.hi, clw);
}

// The draw of sequence b from its tile records (the draw kernel's steps, one
// warp): the exact normalisers S_t, S_d; each tile's sum of the sampling
// weights (A / S_t - B / S_d plus its open columns, or the tile summed again
// when more than kOpenCap columns stayed open); Z; the tile holding u * Z by
// an exclusive prefix over the tiles. In that tile, lane l holds columns
// g 256 + 8 l .. + 7 of group g (one 16-byte load per row per group, all in
// flight at once): the group, then the lane, then the column whose running
// sum first exceeds u * Z.
template <int TDT, int DDT>
__device__ __noinline__ void draw_warp(const VerifyParams& vp, VScratch& x, const Exp2Table& tab, int32_t b,
                                       const SampleTask& t) {
    const SampleParams& p = vp.t;
    const int lane = threadIdx.x & 31;
    const TileRec* recs = p.recs + (int64_t)b * p.ntile;
    const int nt = p.ntile;
    const int K = (nt + 31) / 32;
    const int t0 = lane * K, t1 = min(nt, t0 + K);
    float* w_hi = x.w_hi;
    float* w_lo = x.w_lo;
    df st{0.f, 0.f}, sd{0.f, 0.f};
#pragma unroll 4
    for (int ti = t0; ti < t1; ++ti) {
        const float4 ss = __ldcg(reinterpret_cast<const float4*>(recs + ti) + 1);
        st = df_add(st, df{ss.x, ss.y});
        sd = df_add(sd, df{ss.z, ss.w});
    }
    const df St = warp_sum_df(st);
    const df Sd = warp_sum_df(sd);
    int mode = t.mode;
    const bool resid = mode == kTaskResidual;
    const df It = resid ? df_recip(St) : df{1.f, 0.f}, Id = resid ? df_recip(Sd) : df{1.f, 0.f};
    const float cl = (resid && t.probs) ? 0.f : kEx2LightBias;
    const TileScratch ws = scratch_of(x, tab);
    df z{0.f, 0.f};
    for (int kq = 0; kq < K; ++kq) {
        const int ti = t0 + kq;
        bool dirty = false;
        if (ti < t1) {
            const float4* r = reinterpret_cast<const float4*>(recs + ti);
            df v;
            if (!resid) {
                const float4 ss = __ldcg(r + 1);
                v = df{ss.x, ss.y};
            } else {
                const int32_t nu = __ldcg(reinterpret_cast<const int32_t*>(r + 3));
                const float4 ab = __ldcg(r);
                v = resid_of_sums(df{ab.x, ab.y}, df{ab.z, ab.w}, It, Id);
                if (nu == 1) {
                    const float4 uu = __ldcg(r + 2);
                    v = df_add(v, resid_of_sums(df{uu.x, uu.y}, df{uu.z, uu.w}, It, Id));
                }
                dirty = nu > 1;
            }
            if (!dirty) {
                w_hi[ti] = v.hi;
                w_lo[ti] = v.lo;
                z = df_add(z, v);
            }
        }
        // tiles with more than one open column, summed again by the whole warp
        uint32_t dm = __ballot_sync(0xffffffffu, dirty);
        while (dm) {
            const int src = __ffs(dm) - 1;
            dm &= dm - 1;
            const int di = src * K + kq;
            const RowPair<TDT, DDT> rp = tile_rows<TDT, DDT>(p, t, di);
            const int32_t nu = __ldcg(&recs[di].nu);
            df xv;
            if (nu <= kOpenCap) {
                const uint16_t* lst = p.open + ((int64_t)b * nt + di) * kOpenCap;
                const df c = lane < nu ? col_weight(rp, (int64_t)__ldcg(lst + lane), kTaskResidual, It, Id, tab)
                                       : df{0.f, 0.f};
                const float4 ab = __ldcg(reinterpret_cast<const float4*>(recs + di));
                xv = df_add(resid_of_sums(df{ab.x, ab.y}, df{ab.z, ab.w}, It, Id), warp_sum_df(c));
            } else {
                xv = warp_sum_df(lane_tile_sum(rp, 0, mode, It, Id, cl, ws));
            }
            if (lane == src) {
                w_hi[di] = xv.hi;
                w_lo[di] = xv.lo;
                z = df_add(z, xv);
            }
        }
    }
    __syncwarp();
    df Z = warp_sum_df(z);
    if (resid && residual_empty(Z)) {  // p_i == q_i to rounding: draw from p_i instead
        mode = kTaskBonus;
        for (int ti = t0; ti < t1; ++ti) {
            const float4 ss = __ldcg(reinterpret_cast<const float4*>(recs + ti) + 1);
            w_hi[ti] = ss.x;
            w_lo[ti] = ss.y;
        }
        Z = St;
    }
    __syncwarp();
    if (lane == 0) {
        p.tasks[b].z_hi = Z.hi;
        p.tasks[b].z_lo = Z.lo;
    }
    // the tile holding the crossing u * Z (u has 24 significant bits)
    const df thr = df_add(two_prod(t.u, Z.hi), df{__fmul_rn(t.u, Z.lo), 0.f});
    df mine{0.f, 0.f};
    for (int ti = t0; ti < t1; ++ti) mine = df_add(mine, df{w_hi[ti], w_lo[ti]});
    df run = warp_excl_scan_df(mine);
    int sel_here = -1, last_here = -1;
    df start_here{0.f, 0.f};
    for (int ti = t0; ti < t1; ++ti) {
        const df v{w_hi[ti], w_lo[ti]};
        const df end = df_add(run, v);
        if (df_pos(v)) last_here = ti;
        if (sel_here < 0 && df_gt(end, thr) && !df_gt(run, thr)) {
            sel_here = ti;
            start_here = run;
        }
        run = end;
    }
    const uint32_t sm_sel = __ballot_sync(0xffffffffu, sel_here >= 0);
    int sel;
    df start;
    bool last_mass = false;
    if (sm_sel) {
        const int src = __ffs(sm_sel) - 1;
        sel = __shfl_sync(0xffffffffu, sel_here, src);
        start = shfl_df(start_here, src);
    } else {  // rounding left no crossing: the last tile with mass
        int lm = last_here;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lm = max(lm, __shfl_xor_sync(0xffffffffu, lm, o));
        sel = lm;
        last_mass = true;
    }
    if (sel < 0) return;
    // rescan of tile sel: the group sums, each lane's 8 columns per group
    // (kept as stored: four words per bf16 row, eight per f32 row)
    const float clw = (mode == kTaskResidual && t.probs) ? 0.f : kEx2LightBias;
    const bool rs = mode == kTaskResidual;
    const RowPair<TDT, DDT> rp = tile_rows<TDT, DDT>(p, t, sel);
    constexpr int NB = (TDT == SPECV_F32 || DDT == SPECV_F32) ? 1 : 2;  // groups loaded together
    df lsum[kGroups];
    int lp = -1;  // the last column of this lane with mass
#pragma unroll
    for (int g = 0; g < kGroups; g += NB) {
        Raw8<TDT> rt[NB];
        Raw8<DDT> rd[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            rt[i] = raw_load8<TDT>(rp.t, (g + i) * 256 + lane * 8);
            if (rs) rd[i] = raw_load8<DDT>(rp.d, (g + i) * 256 + lane * 8);
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            df acc{0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const df w = draw_weight(rp, raw_get(rt[i], e), rs ? raw_get(rd[i], e) : 0.f, mode, It, Id, clw, tab);
                acc_add(acc, w);
                if (df_pos(w)) lp = (g + i) * 256 + lane * 8 + e;
            }
            lsum[g + i] = df_norm(acc);
        }
    }
    int col = -1;
    if (!last_mass) {
        df gstart = start;
#pragma unroll
        for (int gi = 0; gi < kGroups; ++gi) {
            const df lstart = df_add(gstart, warp_excl_scan_df(lsum[gi]));
            const uint32_t cm = __ballot_sync(0xffffffffu, df_gt(df_add(lstart, lsum[gi]), thr));
            if (cm) {
                // the first lane of this group whose 8 columns hold the crossing
                // (read again: one 16-byte word per row, the same for every lane)
                const int L = __ffs(cm) - 1;
                const Raw8<TDT> xt = raw_load8<TDT>(rp.t, gi * 256 + L * 8);
                Raw8<DDT> xd;
                if (rs) xd = raw_load8<DDT>(rp.d, gi * 256 + L * 8);
                df run8 = shfl_df(lstart, L);
                int hit = -1, lp8 = -1;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const df w = draw_weight(rp, raw_get(xt, e), rs ? raw_get(xd, e) : 0.f, mode, It, Id, clw, tab);
                    run8 = df_add(run8, w);
                    if (df_pos(w)) lp8 = e;
                    if (hit < 0 && df_gt(run8, thr)) hit = e;
                }
                // rounding can leave no column over the threshold: the lane's last column with mass
                const int e = hit >= 0 ? hit : lp8;
                if (e >= 0) col = gi * 256 + L * 8 + e;
                break;
            }
            gstart = df_add(gstart, warp_sum_df(lsum[gi]));
        }
    }
    if (col < 0) {  // no group holds the crossing: the last column of the tile with mass
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
        col = lp;
    }
    if (lane == 0 && col >= 0) p.out_tokens[t.out_slot] = (int32_t)((int64_t)sel * kTile + col);
}

// The closers: tail warps 0 .. nclosers - 1 of each CTA close the CTA's
// rows (closer c takes every nclosers-th row, in order), each as soon as all
// streaming warps have left it (shared-memory counters), so the merges, the
// slice counts and the decisions they complete run beside the stream. Every
// wait is bounded.
__device__ void closer_warp(const VerifyParams& vp, VSmem& sm, int which, int nclosers) {
    const StatsParams& p = vp.s;
    const int lane = threadIdx.x & 31;
    for (int s = 0; s < sm.nseg; ++s) {
        const VSeg& g = sm.seg[s];
        const int64_t r1 = (g.f1 - 1) / p.V;
        for (int64_t r = g.r0; r <= r1; ++r) {
            if ((g.lbase + (r - g.r0)) % nclosers != which) continue;  // the other closer's row
            uint32_t* cnt = &sm.rowcnt[g.lbase + (r - g.r0)];
            int ok = 1;
            if (lane == 0) {
                uint32_t v;
                asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(cnt)) : "memory");
                if (v < (uint32_t)kVStreamWarps) {
                    const uint64_t t0 = global_ns();
                    unsigned ns = 32;
                    for (uint32_t it = 0; it < kPollCap; ++it) {
                        __nanosleep(ns);
                        if (ns < 512) ns <<= 1;
                        asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(cnt)) : "memory");
                        if (v >= (uint32_t)kVStreamWarps || global_ns() - t0 > vp.wait_ns) break;
                    }
                    ok = v >= (uint32_t)kVStreamWarps;
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) {  // gave up: the rest of this CTA's rows stay open
                if (lane == 0) atomicOr(p.err, 1u);
                return;
            }
            const bool is_t = r < p.rows_t;
            const int32_t b = seq_of_row(p, !is_t, is_t ? r : r - p.rows_t);
            const bool probs_row = !is_t && p.probs;
            const float k = (b >= 0 && !probs_row) ? kLog2e / temp_of(p, b) : 1.f;
            close_slice(vp, sm, r, probs_row, k);
        }
    }
}

// Tile items in ready-list order until none is left; the warp that finishes
// a sequence's last tile draws its token.
template <int TDT, int DDT>
__device__ void tail_loop(const VerifyParams& vp, VScratch& x, const Exp2Table& tab) {
    const SampleParams& p = vp.t;
    const int lane = threadIdx.x & 31;
    const int64_t items = (int64_t)vp.s.B * p.ntile;
    for (;;) {
        uint32_t kq = 0;
        if (lane == 0) kq = atomicAdd(vp.claim, 1u);
        kq = __shfl_sync(0xffffffffu, kq, 0);
        if ((int64_t)kq >= items) break;
        const int64_t pos = kq / p.ntile;
        const int32_t tile = (int32_t)(kq - pos * p.ntile);
        const uint32_t e = warp_wait_nonzero(vp.ready + pos, vp.wait_ns);
        if (!e) {  // gave up: the sequence behind this entry is not known
            if (lane == 0) atomicOr(p.err, 1u);
            break;
        }
        const int32_t b = (int32_t)(e - 1);
        const SampleTask t = load_task(p.tasks_in + b);
        const int32_t nu = t.mode != kTaskNone ? tile_warp<TDT, DDT>(vp, x, tab, b, tile, t) : 0;
        if (nu > 0) __threadfence();  // open-column lists (any lane) before the count
        __syncwarp();
        uint32_t old = 0;
        if (lane == 0) old = add_acq_rel_gpu(vp.tiles_done + b, 1u);  // releases the record, acquires the others
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old + 1 == (uint32_t)p.ntile) {  // the sequence's last tile: draw its token
            __syncwarp();
            if (lane == 0) {
                vp.tiles_done[b] = 0;
                vp.ready[pos] = 0;
            }
            if (t.mode != kTaskNone) draw_warp<TDT, DDT>(vp, x, tab, b, t);
        }
    }
}

template <int TDT, int DDT>
__global__ void __launch_bounds__(kVThreads, 1) verify_kernel(VerifyParams vp) {
    __shared__ VSmem sm;
    extern __shared__ __align__(128) char ring[];
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kVerifyMaxLocalRows; i += blockDim.x) sm.rowcnt[i] = 0;
    for (int i = threadIdx.x; i < 64; i += blockDim.x) {
        sm.tab.hi[i] = vp.t.tab.hi[i];
        sm.tab.lo[i] = vp.t.tab.lo[i];
    }
    if (threadIdx.x == 0) {
        for (int w = 0; w < kVStreamWarps; ++w)
            for (int st = 0; st < kTmaStages; ++st) mbar_init(&sm.full[w][st], 1);
        sm.next_unit = 0;
        sm.failed = 0;
        plan_waves(vp, sm);
        fence_barrier_init();
    }
    __syncthreads();
    if (warp < kVStreamWarps) {
        // sequences that own no row (offsets out of range) get their outputs
        // here: no slice will ever arrive for them
        if (vp.s.tro && warp == 0)
            for (int64_t b = blockIdx.x; b < vp.s.B; b += gridDim.x)
                if (expected_slices(vp.s, sm, (int32_t)b) == 0) fin_warp(vp, sm, (int32_t)b);
        const bool clean = stream_warp(vp, sm, ring, warp);
        // no units left: the warp's ring becomes its scratch for tile items and draws
        if (clean) tail_loop<TDT, DDT>(vp, *reinterpret_cast<VScratch*>(ring + (size_t)warp * kVRing), sm.tab);
    } else {
        if (warp - kVStreamWarps < kVClosers) closer_warp(vp, sm, warp - kVStreamWarps, kVClosers);
        tail_loop<TDT, DDT>(vp, sm.ts[warp - kVStreamWarps], sm.tab);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (sm.failed) atomicOr(vp.s.err, 1u);
        __threadfence();
        if (atomicAdd(vp.exit_count, 1u) == gridDim.x - 1) {  // every CTA is done: reset for the next call
            *vp.ready_tail = 0;
            *vp.claim = 0;
            *vp.exit_count = 0;
            __threadfence();
        }
    }
}

template <int TDT, int DDT>
cudaError_t launch_typed(const VerifyParams& p, cudaStream_t s) {
    static bool attr_done = false;
    const int smem = kVStreamWarps * kVRing;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(verify_kernel<TDT, DDT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.s.grid);
    cfg.blockDim = dim3(kVThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeCooperative;
    attr.val.cooperative = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, verify_kernel<TDT, DDT>, p);
}

// Test hook: one warp waits on *flag through the same bounded wait the
// verify kernel's hand-offs use and records what it saw (out[0]: the flag's
// value, 0 if the wait gave up; out[1]: 1 if it gave up).
__global__ void wait_probe_kernel(const uint32_t* flag, uint64_t limit_ns, uint32_t* out) {
    const uint32_t v = warp_wait_nonzero(flag, limit_ns);
    if (threadIdx.x == 0) {
        out[0] = v;
        out[1] = v ? 0u : 1u;
    }
}

}  // namespace

cudaError_t launch_wait_probe(const uint32_t* flag, uint64_t limit_ns, uint32_t* out, cudaStream_t s) {
    wait_probe_kernel<<<1, 32, 0, s>>>(flag, limit_ns, out);
    return cudaGetLastError();
}

int verify_resident_ctas(int device) {
    int sms = 0, per = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    const int smem = kVStreamWarps * kVRing;
    if (cudaFuncSetAttribute(verify_kernel<SPECV_BF16, SPECV_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
        return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, verify_kernel<SPECV_BF16, SPECV_BF16>, kVThreads, smem) !=
        cudaSuccess)
        return 0;
    return sms * per;
}

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t s) {
    if (p.s.tdt == SPECV_BF16 && p.s.ddt == SPECV_BF16) return launch_typed<SPECV_BF16, SPECV_BF16>(p, s);
    if (p.s.tdt == SPECV_BF16) return launch_typed<SPECV_BF16, SPECV_F32>(p, s);
    if (p.s.ddt == SPECV_BF16) return launch_typed<SPECV_F32, SPECV_BF16>(p, s);
    return launch_typed<SPECV_F32, SPECV_F32>(p, s);
}

}  // namespace specv
