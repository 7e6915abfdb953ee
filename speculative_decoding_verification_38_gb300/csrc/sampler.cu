// sampler.cu -- the one draw each sequence makes after its accept scan.
//
// At the first rejection i the token comes from norm(max(0, p_i - q_i)); if
// every draft was accepted it comes from p_{gamma+1} ("Speculative decoding"
// (mhtirogla.ai), How it works, steps 3-4; "Speculative decoding"
// (inference.tusharamrit.in), the residual p'(z) and its normaliser). The draw
// is an inverse-CDF pick in index order: the first j whose running sum of the
// weights exceeds u * Z, Z = the sum of all weights (the page's sampler in its
// Code section, which tolerates unnormalised weights). If Z == 0 at a
// rejection (p == q to rounding) the same rule runs on p_i; if rounding leaves
// no index, the last one with positive weight is taken.
//
// Only the selected row pair is re-read, once. The work is split into tile
// items (one sequence x one tile of kTile columns), one warp each:
//   phase 1 (every item): the weights w_t = 2^((l - l_max) k) of both rows over
//     the tile, summed over every column (the exact normalisers S_t, S_d are
//     the sums over all tiles) and over the columns that are certainly in the
//     residual's support. Support membership p > q is decided with the
//     streaming pass's approximate normalisers and a relative margin of 1e-4;
//     since the residual is linear in 1/S_t and 1/S_d on a fixed support, the
//     tile's residual sum is then exactly  A / S_t - B / S_d  plus the columns
//     the margin left open (kept apart, at most one per tile; a tile with more
//     is summed again once the normalisers are known).
//   phase 2 (a second kernel, one CTA per sequence): S_t, S_d, the tile sums
//     and Z, the tile holding u * Z by a prefix over the tile sums, and one
//     exact rescan of that tile for the column.
// Weights and their sums are double-float (precise.cuh), so the pick matches
// a float64 evaluation except within ~1e-10 of a CDF edge.
#include <math.h>

#include "precise.cuh"

namespace specv {

namespace {

constexpr int kWarps = kSampThreads / 32;
constexpr int kQCap = 128;      // entries per warp queue (power of two)
constexpr float kMargin = 1e-4f;  // relative margin of the approximate support test
constexpr int64_t kWideItems = 608;  // at most this many tile items: one CTA per item (4 CTAs x 152 SMs)

struct SampSmem {
    Exp2Table tab;
    int32_t q[kWarps][kQCap];  // per-warp queue of columns awaiting double-float evaluation
    int32_t nu[kWarps];        // open columns found by each warp in its current tile
    float uw[kWarps][4];       // the first one's weights (wt hi, lo, wd hi, lo)
    float part[kWarps][4][2];  // wide tiles: each warp's four sums, combined in warp order
};

// One row's chunk: column j (0-based within the chunk) at g + j * esz. With
// top-k truncation, columns whose value is below tau read as -inf (weight 0).
struct Src {
    const char* g;
    int64_t n;  // columns in the chunk
    float tau;  // the row's top-k threshold (-inf: no truncation)
    bool al;    // g is 16-byte aligned
};

__device__ __forceinline__ float keep_top(float v, float tau) { return v >= tau ? v : -INFINITY; }

template <int DT>
__device__ __forceinline__ float src_elem(const Src& r, int64_t j) {
    return keep_top(ld_elem<DT>(r.g, j), r.tau);
}

// Columns j..j+7 of a chunk as floats; columns past the chunk read as -inf
// (weight 0). j is a multiple of 8. Loads keep the lines in L1: columns queued
// for double-float evaluation are read again moments later.
template <int DT>
__device__ __forceinline__ void src_load8(const Src& r, int64_t j, float (&v)[8]) {
    if (j + 8 <= r.n && r.al) {
        if constexpr (DT == SPECV_BF16) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(r.g + j * 2));
            v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
            v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
        } else {
            const uint4 q0 = __ldg(reinterpret_cast<const uint4*>(r.g + j * 4));
            const uint4 q1 = __ldg(reinterpret_cast<const uint4*>(r.g + j * 4 + 16));
            v[0] = __uint_as_float(q0.x); v[1] = __uint_as_float(q0.y);
            v[2] = __uint_as_float(q0.z); v[3] = __uint_as_float(q0.w);
            v[4] = __uint_as_float(q1.x); v[5] = __uint_as_float(q1.y);
            v[6] = __uint_as_float(q1.z); v[7] = __uint_as_float(q1.w);
        }
        if (r.tau > -INFINITY) {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = keep_top(v[e], r.tau);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = (j + e < r.n) ? src_elem<DT>(r, j + e) : -INFINITY;
    }
}

template <int TDT, int DDT>
struct RowPair {
    Src t, d;
    bool probs;
    float mt, md;  // raw row maxima
    df k;

    __device__ __forceinline__ df wt(float l, const Exp2Table& tab) const {
        return logit_weight<TDT == SPECV_F32>(l, mt, k, tab);
    }
    __device__ __forceinline__ df wd(float l, const Exp2Table& tab) const {
        if (probs) return df{(l > -INFINITY) ? l : 0.f, 0.f};  // probabilities are their own weights
        return logit_weight<DDT == SPECV_F32>(l, md, k, tab);
    }
};

// A weight is "heavy" when it carries a low part (double-float path) or is
// large enough that one rounding would matter; light ones are summed in fp32
// over a short run before joining a double-float sum.
__device__ __forceinline__ bool is_heavy(df w) { return w.lo != 0.f || w.hi > 1.220703125e-4f; }

// Tiles are kTile = kGroups x 256 columns; in group g, lane l owns the 8
// consecutive columns g*256 + l*8 .. +7, so each warp-wide 16-byte load covers
// 512 contiguous bytes (no shared-memory bank conflicts).
constexpr int kGroups = kTile / 256;

// Pass B item: the double-float sampling weight of chunk column j.
template <int TDT, int DDT>
__device__ __forceinline__ df tile_item(const RowPair<TDT, DDT>& rp, int64_t j, int mode, df It, df Id,
                                        const Exp2Table& tab) {
    const df wt = rp.wt(src_elem<TDT>(rp.t, j), tab);
    if (mode != kTaskResidual) return wt;
    return resid_weight_df(wt, rp.wd(src_elem<DDT>(rp.d, j), tab), It, Id);
}

// This lane's share of a tile (its kGroups runs of 8 columns): light columns
// summed in fp32, columns with a heavy weight queued and evaluated densely.
template <int TDT, int DDT>
__device__ __forceinline__ df lane_tile_sum(const RowPair<TDT, DDT>& rp, int64_t tile_j, int mode, df It, df Id,
                                            float cl, SampSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* q = sm.q[warp];
    uint32_t head = 0, tail = 0;
    float light = 0.f;
    df acc{0.f, 0.f};
    const bool resid = mode == kTaskResidual;
#pragma unroll 1
    for (int g = 0; g < kGroups; ++g) {
        const int64_t j = tile_j + g * 256 + lane * 8;
        float lt[8], ld[8];
        src_load8<TDT>(rp.t, j, lt);
        if (resid) src_load8<DDT>(rp.d, j, ld);
        uint32_t m = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            bool ht, hd = false;
            const float wt = light_weight<TDT == SPECV_F32>(lt[e], rp.mt, rp.k, ht);
            if (!resid) {
                if (ht) m |= 1u << e; else light = __fadd_rn(light, wt);
                continue;
            }
            float qv;
            if (rp.probs) {
                const float v = ld[e] > -INFINITY ? ld[e] : 0.f;
                hd = v > 1.220703125e-4f;
                qv = __fmaf_rn(v, Id.hi, __fmul_rn(v, Id.lo));
            } else {
                const float wd = light_weight<DDT == SPECV_F32>(ld[e], rp.md, rp.k, hd);
                qv = __fmaf_rn(wd, Id.hi, __fmul_rn(wd, Id.lo));
            }
            if (ht || hd) {
                m |= 1u << e;
            } else {
                const float r = __fsub_rn(__fmaf_rn(wt, It.hi, __fmul_rn(wt, It.lo)), qv);
                light = __fadd_rn(light, r > 0.f ? r : 0.f);
            }
        }
        const auto code = [&](int b) { return (int32_t)(j + b); };
        if (!wq_push(q, head, tail, m, code)) {
            while (m) {
                const int b = __ffs(m) - 1;
                m &= m - 1;
                acc_add(acc, tile_item(rp, j + b, mode, It, Id, sm.tab));
            }
        }
        while (tail - head >= 32) {
            acc_add(acc, tile_item(rp, q[(head + lane) & (kQCap - 1)], mode, It, Id, sm.tab));
            head += 32;
            __syncwarp();
        }
    }
    if (lane < (int)(tail - head)) acc_add(acc, tile_item(rp, q[(head + lane) & (kQCap - 1)], mode, It, Id, sm.tab));
    __syncwarp();
    return df_add(df_norm(acc), light_sum_df(light, cl));
}

// Inclusive warp scan of double-float values (Hillis-Steele).
__device__ __forceinline__ df warp_scan_df(df x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        df y = shfl_up_df(x, o);
        if (lane >= o) x = df_add(y, x);
    }
    return x;
}

__device__ __forceinline__ df warp_sum_df(df x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = df_add(x, shfl_xor_df(x, o));
    return x;
}

// ---------------------------------------------------------------- queues
// Heavy weights are rare (about 1% of a row) but each takes the double-float
// path. Evaluating them in place would make the whole warp wait for every
// heavy lane; instead each warp queues them in shared memory and evaluates
// them 32 at a time.

// Warp-wide exclusive prefix of per-lane counts; returns the lane's offset and
// sets `total`.
__device__ __forceinline__ uint32_t warp_offsets(uint32_t n, uint32_t& total) {
    const int lane = threadIdx.x & 31;
    uint32_t incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    total = __shfl_sync(0xffffffffu, incl, 31);
    return incl - n;
}

// Append this lane's items (bit b of m -> code(b)) to the warp's ring
// buffer. Returns false (and appends nothing) if they do not fit.
template <class Code>
__device__ __forceinline__ bool wq_push(int32_t* q, uint32_t head, uint32_t& tail, uint32_t m, Code code) {
    uint32_t total;
    uint32_t off = warp_offsets(__popc(m), total);
    if (tail + total - head > (uint32_t)kQCap) return false;  // warp-uniform
    off += tail;
    while (m) {
        const int b = __ffs(m) - 1;
        m &= m - 1;
        q[(off++) & (kQCap - 1)] = code(b);
    }
    tail += total;
    __syncwarp();
    return true;
}

// The row pair of task t restricted to tile `tile` (columns read from global
// memory; 16-byte loads where the tile start is aligned).
template <int TDT, int DDT>
__device__ __forceinline__ RowPair<TDT, DDT> tile_rows(const SampleParams& p, const SampleTask& t, int32_t tile) {
    constexpr int te = TDT == SPECV_F32 ? 4 : 2, de = DDT == SPECV_F32 ? 4 : 2;
    const int64_t c0 = (int64_t)tile * kTile;
    const int64_t n = min((int64_t)kTile, p.V - c0);
    const bool resid = t.mode == kTaskResidual;
    RowPair<TDT, DDT> rp;
    rp.t.g = (const char*)p.tgt + (t.trow * p.V + c0) * te;
    rp.d.g = resid ? (const char*)p.dft + (t.drow * p.V + c0) * de : rp.t.g;
    rp.t.n = rp.d.n = n;
    rp.t.al = ((uintptr_t)rp.t.g & 15u) == 0;
    rp.d.al = ((uintptr_t)rp.d.g & 15u) == 0;
    rp.t.tau = t.tau_t;
    rp.d.tau = resid ? t.tau_d : t.tau_t;
    rp.probs = t.probs != 0;
    rp.mt = t.mt;
    rp.md = t.md;
    rp.k = df{t.k_hi, t.k_lo};
    return rp;
}

// The double-float weights (target, and draft for a residual) of one queued
// column, out of line with the heavy path inline inside it: the queue's three
// evaluation sites share this one copy and pay one call per column. The same
// arithmetic as RowPair::wt / wd.
template <int TDT, int DDT>
__device__ __noinline__ float4 col_weights(const char* tg, const char* dg, float tau_t, float tau_d, float mt, float md,
                                           df k, bool probs, bool resid, int64_t j, const Exp2Table& tab) {
    const df wt = logit_weight<TDT == SPECV_F32, true>(keep_top(ld_elem<TDT>(tg, j), tau_t), mt, k, tab);
    df wd{0.f, 0.f};
    if (resid) {
        const float l = keep_top(ld_elem<DDT>(dg, j), tau_d);
        wd = probs ? df{(l > -INFINITY) ? l : 0.f, 0.f} : logit_weight<DDT == SPECV_F32, true>(l, md, k, tab);
    }
    return make_float4(wt.hi, wt.lo, wd.hi, wd.lo);
}

// Phase 1 for one tile: this lane's sums (double-float) over its columns.
struct TileAcc {
    df st, sd, a, b;
};

// Every group of the tile, or (WIDE) group gw alone; sw: the shared-memory
// slot counting the tile's open columns (the warp's own, or one for the CTA).
template <int TDT, int DDT, bool WIDE>
__device__ void tile_sums(const RowPair<TDT, DDT>& rp, bool resid, float r_hi, float r_lo, SampSmem& sm,
                          uint16_t* open_list, int sw, int gw, TileAcc& out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* q = sm.q[warp];
    uint32_t head = 0, tail = 0;
    float st_l = 0.f, sd_l = 0.f, a_l = 0.f, b_l = 0.f;
    df st_h{0.f, 0.f}, sd_h{0.f, 0.f}, a_h{0.f, 0.f}, b_h{0.f, 0.f};
    constexpr int32_t kOpen = 1 << 30;  // queued light column whose weights are already in st / sd
    // one queued column: double-float weights, then the support decision
    auto eval = [&](int32_t code) {
        const int64_t j = code & (kOpen - 1);
        const float4 w4 = col_weights<TDT, DDT>(rp.t.g, rp.d.g, rp.t.tau, rp.d.tau, rp.mt, rp.md, rp.k, rp.probs, resid,
                                                j, sm.tab);
        const df wt{w4.x, w4.y};
        if (!resid) {
            acc_add(st_h, wt);
            return;
        }
        const df wd{w4.z, w4.w};
        if (!(code & kOpen)) {
            acc_add(st_h, wt);
            acc_add(sd_h, wd);
        }
        if (wt.hi == 0.f && wd.hi == 0.f) return;
        if (wt.hi > wd.hi * r_hi) {
            acc_add(a_h, wt);
            acc_add(b_h, wd);
        } else if (!(wt.hi < wd.hi * r_lo)) {  // still open: kept apart for phase 2
            const int slot = atomicAdd(&sm.nu[sw], 1);
            if (slot < kOpenCap) open_list[slot] = (uint16_t)j;  // the draw evaluates listed columns alone
            if (slot == 0) {
                sm.uw[sw][0] = wt.hi;
                sm.uw[sw][1] = wt.lo;
                sm.uw[sw][2] = wd.hi;
                sm.uw[sw][3] = wd.lo;
            }
        }
    };
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
        if (WIDE && g != gw) continue;  // uniform per warp
        const int64_t j = g * 256 + lane * 8;
        float lt[8], ld[8];
        src_load8<TDT>(rp.t, j, lt);
        if (resid) src_load8<DDT>(rp.d, j, ld);
        uint32_t m = 0, open = 0;
        // branch-free per column: selects for the sums, predicated bits for
        // the heavy and open masks (the same sums as the branching form)
        if (!resid) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                bool ht;
                const float wt = light_weight<TDT == SPECV_F32>(lt[e], rp.mt, rp.k, ht);
                st_l = __fadd_rn(st_l, ht ? 0.f : wt);
                m |= ht ? (1u << e) : 0u;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                bool ht, hd = false;
                const float wt = light_weight<TDT == SPECV_F32>(lt[e], rp.mt, rp.k, ht);
                float wd;
                if (rp.probs) {
                    wd = ld[e] > -INFINITY ? ld[e] : 0.f;
                    hd = wd > 1.220703125e-4f;
                } else {
                    wd = light_weight<DDT == SPECV_F32>(ld[e], rp.md, rp.k, hd);
                }
                const bool heavy = ht || hd;
                const bool in = !heavy && wt > wd * r_hi;  // certainly p > q
                const bool opn = !heavy && !in && !(wt < wd * r_lo) && (wt != 0.f || wd != 0.f);
                st_l = __fadd_rn(st_l, heavy ? 0.f : wt);
                sd_l = __fadd_rn(sd_l, heavy ? 0.f : wd);
                a_l = __fadd_rn(a_l, in ? wt : 0.f);
                b_l = __fadd_rn(b_l, in ? wd : 0.f);
                m |= (heavy || opn) ? (1u << e) : 0u;
                open |= opn ? (1u << e) : 0u;
            }
        }
        const auto code = [&](int bit) { return (int32_t)((j + bit) | ((open >> bit) & 1u ? kOpen : 0)); };
        if (!wq_push(q, head, tail, m, code)) {  // queue full: evaluate in place
            while (m) {
                const int bit = __ffs(m) - 1;
                m &= m - 1;
                eval(code(bit));
            }
        }
        while (tail - head >= 32) {
            eval(q[(head + lane) & (kQCap - 1)]);
            head += 32;
            __syncwarp();
        }
    }
    if (lane < (int)(tail - head)) eval(q[(head + lane) & (kQCap - 1)]);
    __syncwarp();
    const float cd = rp.probs ? 0.f : kEx2LightBias;
    out.st = df_add(df_norm(st_h), light_sum_df(st_l, kEx2LightBias));
    out.sd = df_add(df_norm(sd_h), light_sum_df(sd_l, cd));
    out.a = df_add(df_norm(a_h), light_sum_df(a_l, kEx2LightBias));
    out.b = df_add(df_norm(b_h), light_sum_df(b_l, cd));
}

// Double-float sums of four per-lane values over the warp, halving the
// exchanged data at each step: afterwards lanes 8q .. 8q + 7 hold the total
// of value q.
__device__ __forceinline__ df warp_sum4_df(df v0, df v1, df v2, df v3) {
    const int lane = threadIdx.x & 31;
    // step 16: keep values 0,1 (lanes < 16) or 2,3; add the partner's copy
    const bool up = lane & 16;
    df s0 = up ? v2 : v0, s1 = up ? v3 : v1;
    const df g0 = up ? v0 : v2, g1 = up ? v1 : v3;  // what the partner keeps
    s0 = df_add(s0, shfl_xor_df(g0, 16));
    s1 = df_add(s1, shfl_xor_df(g1, 16));
    // step 8: keep one of the two
    const bool up8 = lane & 8;
    df s = up8 ? s1 : s0;
    const df g = up8 ? s0 : s1;
    s = df_add(s, shfl_xor_df(g, 8));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) s = df_add(s, shfl_xor_df(s, o));
    return s;
}

// WIDE: one CTA per tile item, warp w summing group w (for problems with few
// items, so that one tile's double-float columns are spread over kGroups
// warps); otherwise one warp per item.
template <int TDT, int DDT, bool WIDE>
__global__ void __launch_bounds__(kSampThreads, 4) sampler_kernel(SampleParams p) {
    __shared__ SampSmem sm;
    for (int i = threadIdx.x; i < 64; i += blockDim.x) {
        sm.tab.hi[i] = p.tab.hi[i];
        sm.tab.lo[i] = p.tab.lo[i];
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sw = WIDE ? 0 : warp;  // the open-column counter of this tile
    if (WIDE && threadIdx.x == 0) sm.nu[0] = 0;
    __syncthreads();
    pdl_launch_dependents();
    pdl_wait_primary();  // tasks are written by the finalize step
    const int64_t item = WIDE ? (int64_t)blockIdx.x : (int64_t)blockIdx.x * kWarps + warp;
    if (item >= (int64_t)p.B * p.ntile) return;  // block-uniform when WIDE
    const int32_t b = (int32_t)(item / p.ntile), tile = (int32_t)(item - (int64_t)b * p.ntile);
    const SampleTask t = p.tasks_in[b];
    if (t.mode == kTaskNone) return;
    const bool resid = t.mode == kTaskResidual;
    // approximate support test p > q(1 + m) / p < q(1 - m), i.e. w_t > w_d * r
    const float ratio = resid ? t.id_apx / t.it_apx : 0.f;
    const float r_hi = ratio * (1.f + kMargin), r_lo = ratio * (1.f - kMargin);
    if (!WIDE) {
        if (lane == 0) sm.nu[warp] = 0;
        __syncwarp();
    }
    const RowPair<TDT, DDT> rp = tile_rows<TDT, DDT>(p, t, tile);
    TileAcc acc;
    if (WIDE && warp >= kGroups) acc = TileAcc{};
    else tile_sums<TDT, DDT, WIDE>(rp, resid, r_hi, r_lo, sm, p.open + item * kOpenCap, sw, warp, acc);
    df tot = warp_sum4_df(acc.st, acc.sd, resid ? acc.a : acc.st, acc.b);
    if (WIDE) {  // the groups' sums in warp order
        if (warp < kGroups && (lane & 7) == 0) {
            sm.part[warp][lane >> 3][0] = tot.hi;
            sm.part[warp][lane >> 3][1] = tot.lo;
        }
        __syncthreads();
        if (warp != 0) return;
        tot = df{0.f, 0.f};
        if ((lane & 7) == 0)
            for (int w = 0; w < kGroups; ++w) tot = df_add(tot, df{sm.part[w][lane >> 3][0], sm.part[w][lane >> 3][1]});
    }
    TileRec& r = p.recs[item];
    if ((lane & 7) == 0) {
        float* dst = lane == 0 ? r.st : (lane == 8 ? r.sd : (lane == 16 ? r.a : r.b));
        dst[0] = tot.hi;
        dst[1] = tot.lo;
    }
    if (lane == 1) {
        r.nu = sm.nu[sw];
        r.uwt[0] = sm.uw[sw][0];
        r.uwt[1] = sm.uw[sw][1];
        r.uwd[0] = sm.uw[sw][2];
        r.uwd[1] = sm.uw[sw][3];
    }
}

// ------------------------------------------------------------- phase 2
// One CTA per sequence, after every tile record is in (programmatic launch).
// Thread i owns tiles i*K .. i*K + K - 1 (K = ceil(ntile / 256) <= 8); the
// tile sums of the sampling weights live in shared memory. All arithmetic is
// double-float (the GPU's float64 rate is far below its fp32 rate).
constexpr int kMaxTiles = (int)(kMaxVocab / kTile);

struct DrawSmem {
    Exp2Table tab;
    int32_t q[kWarps][kQCap];  // lane_tile_sum's queues (tiles summed again)
    float w_hi[kMaxTiles], w_lo[kMaxTiles];  // tile sums
    float red_hi[kWarps], red_lo[kWarps];
    int32_t dirty[kMaxTiles];
    int32_t ndirty, sel, col, last;
    float start_hi, start_lo;
};

__device__ __forceinline__ df block_sum_df(df x, DrawSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    x = warp_sum_df(x);
    __syncthreads();  // red[] is free
    if (lane == 0) {
        sm.red_hi[warp] = x.hi;
        sm.red_lo[warp] = x.lo;
    }
    __syncthreads();
    df t{0.f, 0.f};
    for (int i = 0; i < kWarps; ++i) t = df_add(t, df{sm.red_hi[i], sm.red_lo[i]});
    return t;
}

// Exclusive block-wide prefix of one value per thread (thread order).
__device__ __forceinline__ df block_excl_scan_df(df x, DrawSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const df incl = warp_scan_df(x);
    __syncthreads();
    if (lane == 31) {
        sm.red_hi[warp] = incl.hi;
        sm.red_lo[warp] = incl.lo;
    }
    __syncthreads();
    df before{0.f, 0.f};
    for (int i = 0; i < warp; ++i) before = df_add(before, df{sm.red_hi[i], sm.red_lo[i]});
    df excl = shfl_up_df(incl, 1);
    if (lane == 0) excl = df{0.f, 0.f};
    return df_add(before, excl);
}

__device__ __forceinline__ df ldcg_df(const float* v) {
    const float2 x = __ldcg(reinterpret_cast<const float2*>(v));
    return df{x.x, x.y};
}

// Sampling weight of column j (0-based in the tile) as double-float.
template <int TDT, int DDT>
__device__ __forceinline__ df col_weight(const RowPair<TDT, DDT>& rp, int64_t j, int mode, df It, df Id,
                                         const Exp2Table& tab) {
    const df wt = rp.wt(src_elem<TDT>(rp.t, j), tab);
    if (mode != kTaskResidual) return wt;
    return resid_weight(wt, rp.wd(src_elem<DDT>(rp.d, j), tab), It, Id);
}

// max(0, a * It - b * Id) for one tile record's pair of sums
__device__ __forceinline__ df resid_of_sums(df a, df b, df It, df Id) {
    const df v = df_sub(df_mul(It, a), df_mul(Id, b));
    return df_pos(v) ? v : df{0.f, 0.f};
}

template <int TDT, int DDT>
__global__ void __launch_bounds__(kSampThreads) draw_kernel(SampleParams p) {
    __shared__ DrawSmem sm;
    for (int i = threadIdx.x; i < 64; i += blockDim.x) {
        sm.tab.hi[i] = p.tab.hi[i];
        sm.tab.lo[i] = p.tab.lo[i];
    }
    if (threadIdx.x == 0) sm.ndirty = 0;
    pdl_wait_primary();
    const int32_t b = blockIdx.x;
    const SampleTask t = p.tasks_in[b];
    if (t.mode == kTaskNone) return;  // block-uniform
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TileRec* recs = p.recs + (int64_t)b * p.ntile;
    const int nt = p.ntile;
    const int K = (nt + kSampThreads - 1) / kSampThreads;
    const int t0 = threadIdx.x * K, t1 = min(nt, t0 + K);
    // the exact normalisers
    df st{0.f, 0.f}, sd{0.f, 0.f};
#pragma unroll 1
    for (int ti = t0; ti < t1; ++ti) {
        const float4 ss = __ldcg(reinterpret_cast<const float4*>(recs + ti) + 1);
        st = df_add(st, df{ss.x, ss.y});
        sd = df_add(sd, df{ss.z, ss.w});
    }
    const df St = block_sum_df(st, sm);
    const df Sd = block_sum_df(sd, sm);
    int mode = t.mode;
    const bool resid = mode == kTaskResidual;
    const df It = resid ? df_recip(St) : df{1.f, 0.f}, Id = resid ? df_recip(Sd) : df{1.f, 0.f};
    float cl = (resid && t.probs) ? 0.f : kEx2LightBias;
    // tile sums of the sampling weights
    df z{0.f, 0.f};
#pragma unroll 1
    for (int ti = t0; ti < t1; ++ti) {
        const float4* r = reinterpret_cast<const float4*>(recs + ti);
        df v;
        if (!resid) {
            const float4 ss = __ldcg(r + 1);
            v = df{ss.x, ss.y};
        } else {
            const int32_t nu = __ldcg(reinterpret_cast<const int32_t*>(r + 3));
            if (nu > 1) {  // more than one open column: summed again below
                sm.dirty[atomicAdd(&sm.ndirty, 1)] = ti;
                continue;
            }
            const float4 ab = __ldcg(r);
            v = resid_of_sums(df{ab.x, ab.y}, df{ab.z, ab.w}, It, Id);
            if (nu == 1) {
                const float4 uu = __ldcg(r + 2);
                v = df_add(v, resid_of_sums(df{uu.x, uu.y}, df{uu.z, uu.w}, It, Id));
            }
        }
        sm.w_hi[ti] = v.hi;
        sm.w_lo[ti] = v.lo;
        z = df_add(z, v);
    }
    __syncthreads();
    const int nd = sm.ndirty;
#pragma unroll 1
    for (int i = warp; i < nd; i += kWarps) {  // one warp per tile, exactly
        const int ti = sm.dirty[i];
        const RowPair<TDT, DDT> rp = tile_rows<TDT, DDT>(p, t, ti);
        const int32_t nu = __ldcg(&recs[ti].nu);
        df x;
        if (nu <= kOpenCap) {  // the tile's open columns are listed: the certain part plus each of them
            const uint16_t* lst = p.open + ((int64_t)b * nt + ti) * kOpenCap;
            const df c = lane < nu ? col_weight(rp, (int64_t)__ldcg(lst + lane), kTaskResidual, It, Id, sm.tab)
                                   : df{0.f, 0.f};
            const float4 ab = __ldcg(reinterpret_cast<const float4*>(recs + ti));
            x = df_add(resid_of_sums(df{ab.x, ab.y}, df{ab.z, ab.w}, It, Id), warp_sum_df(c));
        } else {
            x = warp_sum_df(lane_tile_sum(rp, 0, mode, It, Id, cl, *reinterpret_cast<SampSmem*>(&sm)));
        }
        if (lane == 0) {
            sm.w_hi[ti] = x.hi;
            sm.w_lo[ti] = x.lo;
            z = df_add(z, x);
        }
    }
    df Z = block_sum_df(z, sm);
    if (resid && residual_empty(Z)) {  // p_i == q_i to rounding: draw from p_i instead
        mode = kTaskBonus;
        cl = kEx2LightBias;
        for (int ti = t0; ti < t1; ++ti) {
            const float4 ss = __ldcg(reinterpret_cast<const float4*>(recs + ti) + 1);
            sm.w_hi[ti] = ss.x;
            sm.w_lo[ti] = ss.y;
        }
        Z = St;
    }
    if (threadIdx.x == 0) {
        p.tasks[b].z_hi = Z.hi;
        p.tasks[b].z_lo = Z.lo;
        sm.sel = -1;
        sm.last = -1;
        sm.col = -1;
    }
    __syncthreads();
    // the tile holding the crossing u * Z (u has 24 significant bits)
    const df thr = df_add(two_prod(t.u, Z.hi), df{__fmul_rn(t.u, Z.lo), 0.f});
    df mine{0.f, 0.f};
    for (int ti = t0; ti < t1; ++ti) mine = df_add(mine, df{sm.w_hi[ti], sm.w_lo[ti]});
    df run = block_excl_scan_df(mine, sm);
    int last_here = -1;
    for (int ti = t0; ti < t1; ++ti) {
        const df v{sm.w_hi[ti], sm.w_lo[ti]};
        const df end = df_add(run, v);
        if (df_pos(v)) last_here = ti;
        if (df_gt(end, thr) && !df_gt(run, thr)) {
            sm.sel = ti;  // the only thread with a crossing
            sm.start_hi = run.hi;
            sm.start_lo = run.lo;
        }
        run = end;
    }
    atomicMax(&sm.last, last_here);
    __syncthreads();
    int sel = sm.sel;
    const bool last_mass = sel < 0;
    if (last_mass) sel = sm.last;  // rounding left no crossing: the last tile with mass
    if (sel < 0) return;
    // rescan the selected tile: warp w covers columns w*128 .. +127, 4 per lane
    const RowPair<TDT, DDT> rp = tile_rows<TDT, DDT>(p, t, sel);
    const df basef = last_mass ? df{NAN, 0.f} : df{sm.start_hi, sm.start_lo};  // NaN: no comparison succeeds
    const int64_t j0 = (int64_t)warp * 128 + lane * 4;
    df w4[4], pre[4];
    float light = 0.f;
    df heavy{0.f, 0.f};
    int lp = -1;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        w4[e] = j0 + e < rp.t.n ? col_weight(rp, j0 + e, mode, It, Id, sm.tab) : df{0.f, 0.f};
        if (is_heavy(w4[e]))
            acc_add(heavy, w4[e]);
        else
            light = __fadd_rn(light, w4[e].hi);
        pre[e] = df_add(df_norm(heavy), light_sum_df(light, cl));
        if (df_pos(w4[e])) lp = e;
    }
    // block prefix of the per-lane sums, in column order (warp-major)
    const df start = df_add(basef, block_excl_scan_df(pre[3], sm));
    int hit = -1;
#pragma unroll
    for (int e = 3; e >= 0; --e)
        if (df_gt(df_add(start, pre[e]), thr)) hit = e;
    // the first column (in order) whose running sum exceeds thr
    if (hit >= 0) atomicMin((unsigned*)&sm.col, (unsigned)(j0 + hit));
    if (lp >= 0) atomicMax(&sm.last, (int)(0x40000000 | (j0 + lp)));
    __syncthreads();
    if (threadIdx.x == 0) {
        const int64_t jt = (sm.col >= 0) ? sm.col : ((sm.last & 0x40000000) ? (sm.last & 0x3fffffff) : -1);
        if (jt >= 0) p.out_tokens[t.out_slot] = (int32_t)((int64_t)sel * kTile + jt);
    }
}

template <int TDT, int DDT>
cudaError_t launch_typed(const SampleParams& p, cudaStream_t s, bool pdl) {
    const int64_t items = (int64_t)p.B * p.ntile;
    const bool wide = items <= kWideItems;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(wide ? items : (items + kWarps - 1) / kWarps));
    cfg.blockDim = dim3(kSampThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = wide ? cudaLaunchKernelEx(&cfg, sampler_kernel<TDT, DDT, true>, p)
                         : cudaLaunchKernelEx(&cfg, sampler_kernel<TDT, DDT, false>, p);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)p.B);
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, draw_kernel<TDT, DDT>, p);
}

}  // namespace

void exp2_pairs(Exp2Pairs& t) {
    for (int i = 0; i < 64; ++i) {
        const double v = exp2((double)i / 64.0);
        t.hi[i] = (float)v;
        t.lo[i] = (float)(v - (double)t.hi[i]);
    }
}

cudaError_t launch_sampler(const SampleParams& p, cudaStream_t s, bool pdl) {
    if (p.tdt == SPECV_BF16 && p.ddt == SPECV_BF16) return launch_typed<SPECV_BF16, SPECV_BF16>(p, s, pdl);
    if (p.tdt == SPECV_BF16) return launch_typed<SPECV_BF16, SPECV_F32>(p, s, pdl);
    if (p.ddt == SPECV_BF16) return launch_typed<SPECV_F32, SPECV_BF16>(p, s, pdl);
    return launch_typed<SPECV_F32, SPECV_F32>(p, s, pdl);
}

}  // namespace specv
