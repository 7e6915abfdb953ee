// tile.cuh -- device pieces of the residual / bonus draw shared by the
// sampler kernels (sampler.cu) and the fused verify kernel (verify.cu): the
// row-pair view of one 1024-column tile, the double-float column weights,
// the per-warp queues of heavy columns and the tile sums of the first phase
// ("Speculative decoding" (mhtirogla.ai), How it works, steps 3-4;
// "Speculative decoding" (inference.tusharamrit.in), the residual p'(z) and
// its normaliser). Included by one translation unit each; everything here has
// internal linkage.
#pragma once

#include "precise.cuh"

namespace specv {

namespace {

constexpr int kWarps = kSampThreads / 32;
constexpr int kQCap = 128;      // entries per warp queue (power of two)
constexpr float kMargin = 1e-4f;  // relative margin of the approximate support test
constexpr int64_t kWideItems = 608;  // at most this many tile items: one CTA per item (4 CTAs x 152 SMs)

// The shared memory one warp uses while it sums a tile: its queue of heavy
// columns (kQCap entries), the counter of the tile's open columns and the
// first open column's weights (4 floats), and the 2^(i/64) table.
struct TileScratch {
    int32_t* q;
    int32_t* nu;
    float* uw;
    const Exp2Table* tab;
};

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
// ws: this warp's queue and the table.
template <int TDT, int DDT>
__device__ __forceinline__ df lane_tile_sum(const RowPair<TDT, DDT>& rp, int64_t tile_j, int mode, df It, df Id,
                                            float cl, const TileScratch& ws) {
    const int lane = threadIdx.x & 31;
    int32_t* q = ws.q;
    const Exp2Table& tab = *ws.tab;
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
                acc_add(acc, tile_item(rp, j + b, mode, It, Id, tab));
            }
        }
        while (tail - head >= 32) {
            acc_add(acc, tile_item(rp, q[(head + lane) & (kQCap - 1)], mode, It, Id, tab));
            head += 32;
            __syncwarp();
        }
    }
    if (lane < (int)(tail - head)) acc_add(acc, tile_item(rp, q[(head + lane) & (kQCap - 1)], mode, It, Id, tab));
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

// Every group of the tile, or (WIDE) group gw alone; ws: this warp's queue,
// the counter of the tile's open columns (the warp's own, or one for the
// CTA) with the first open column's weights, and the table.
template <int TDT, int DDT, bool WIDE>
__device__ void tile_sums(const RowPair<TDT, DDT>& rp, bool resid, float r_hi, float r_lo, const TileScratch& ws,
                          uint16_t* open_list, int gw, TileAcc& out) {
    const int lane = threadIdx.x & 31;
    int32_t* q = ws.q;
    uint32_t head = 0, tail = 0;
    float st_l = 0.f, sd_l = 0.f, a_l = 0.f, b_l = 0.f;
    df st_h{0.f, 0.f}, sd_h{0.f, 0.f}, a_h{0.f, 0.f}, b_h{0.f, 0.f};
    constexpr int32_t kOpen = 1 << 30;  // queued light column whose weights are already in st / sd
    // one queued column: double-float weights, then the support decision
    auto eval = [&](int32_t code) {
        const int64_t j = code & (kOpen - 1);
        const float4 w4 = col_weights<TDT, DDT>(rp.t.g, rp.d.g, rp.t.tau, rp.d.tau, rp.mt, rp.md, rp.k, rp.probs, resid,
                                                j, *ws.tab);
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
            const int slot = atomicAdd(ws.nu, 1);
            if (slot < kOpenCap) open_list[slot] = (uint16_t)j;  // the draw evaluates listed columns alone
            if (slot == 0) {
                ws.uw[0] = wt.hi;
                ws.uw[1] = wt.lo;
                ws.uw[2] = wd.hi;
                ws.uw[3] = wd.lo;
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
// Eight consecutive columns of a row as stored: one 16-byte word for bf16,
// two for f32.
template <int DT>
struct Raw8 {
    uint4 w[DT == SPECV_F32 ? 2 : 1];
};

// Columns j .. j + 7 of a tile's row (j % 8 == 0) as stored; columns past the
// tile's end read as -inf. 16-byte loads where the run lies inside an aligned
// row, else element loads.
template <int DT>
__device__ __forceinline__ Raw8<DT> raw_load8(const Src& r, int64_t j) {
    Raw8<DT> x;
    if (j + 8 <= r.n && r.al) {
        if constexpr (DT == SPECV_BF16) {
            x.w[0] = __ldg(reinterpret_cast<const uint4*>(r.g + j * 2));
        } else {
            x.w[0] = __ldg(reinterpret_cast<const uint4*>(r.g + j * 4));
            x.w[1] = __ldg(reinterpret_cast<const uint4*>(r.g + j * 4 + 16));
        }
    } else {
        uint32_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float f = j + e < r.n ? ld_elem<DT>(r.g, j + e) : -INFINITY;
            v[e] = DT == SPECV_BF16 ? (__float_as_uint(f) >> 16) : __float_as_uint(f);
        }
        if constexpr (DT == SPECV_BF16) {
            x.w[0] = make_uint4(v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16), v[6] | (v[7] << 16));
        } else {
            x.w[0] = make_uint4(v[0], v[1], v[2], v[3]);
            x.w[1] = make_uint4(v[4], v[5], v[6], v[7]);
        }
    }
    return x;
}

template <int DT>
__device__ __forceinline__ float raw_get(const Raw8<DT>& x, int e) {
    if constexpr (DT == SPECV_BF16) {
        const uint4& q = x.w[0];
        const uint32_t w = e < 2 ? q.x : (e < 4 ? q.y : (e < 6 ? q.z : q.w));
        return (e & 1) ? bf16_hi(w) : bf16_lo(w);
    } else {
        const uint4& q = x.w[e >> 2];
        const int c = e & 3;
        return __uint_as_float(c == 0 ? q.x : (c == 1 ? q.y : (c == 2 ? q.z : q.w)));
    }
}

template <int DT>
__device__ __forceinline__ Raw8<DT> raw_shfl(const Raw8<DT>& x, int src) {
    Raw8<DT> y;
#pragma unroll
    for (int i = 0; i < (DT == SPECV_F32 ? 2 : 1); ++i) {
        y.w[i].x = __shfl_sync(0xffffffffu, x.w[i].x, src);
        y.w[i].y = __shfl_sync(0xffffffffu, x.w[i].y, src);
        y.w[i].z = __shfl_sync(0xffffffffu, x.w[i].z, src);
        y.w[i].w = __shfl_sync(0xffffffffu, x.w[i].w, src);
    }
    return y;
}

// The exponent (l - m) k of two logits, rounded as logit_weight rounds it
// (so light weights match the draw's column weights bit for bit): for fp32
// logits l - m is carried exactly as a pair (Knuth's TwoSum; a -inf logit
// gets a zero low part), then dh k_hi + (dl k_hi + dh k_lo).
template <bool FP32IN>
__device__ __forceinline__ float2 packed_exponent(float2 l, float2 m, float2 kh, float2 kl) {
    const float2 dh = sub2(l, m);
    float2 t = mul2(dh, kl);
    if constexpr (FP32IN) {
        const float2 bb = sub2(dh, l);
        float2 dl = add2(sub2(l, sub2(dh, bb)), sub2(make_float2(-m.x, -m.y), bb));
        dl = make_float2(dh.x > -INFINITY ? dl.x : 0.f, dh.y > -INFINITY ? dl.y : 0.f);
        t = fma2(dl, kh, t);
    }
    return fma2(dh, kh, t);
}

// Tile sums with packed two-column arithmetic (the same sums as tile_sums,
// non-wide). Lane l's columns are g 256 + 8 l .. + 7 of groups g = g0 ..
// g1 - 1, all loaded at once as stored. Light weights: the exponent
// (l - m) k_hi + (l - m) k_lo (k_lo > 0, so -inf logits weigh 0) two columns
// per instruction, then the SFU's 2^x; a column is heavy when either
// exponent is above kHeavyExp (a draft probability above 2^-13), and open
// when the approximate support test cannot decide it (w_d r_lo < w_t <=
// w_d r_hi). Light columns join float sums through 0/1 factors (no
// branches); heavy and open columns are marked in a per-lane bit mask and
// evaluated in double-float once per tile, 32 at a time.
template <int TDT, int DDT>
__device__ void tile_sums_packed(const RowPair<TDT, DDT>& rp, bool resid, float r_hi, float r_lo,
                                 const TileScratch& ws, uint16_t* open_list, int g0, int g1, TileAcc& out) {
    const int lane = threadIdx.x & 31;
    // groups loaded together: two for bf16 rows, one when a row is f32
    constexpr int NB = (TDT == SPECV_F32 || DDT == SPECV_F32) ? 1 : 2;
    Raw8<TDT> rt[NB];
    Raw8<DDT> rd[NB];
    const bool trunc_t = rp.t.tau > -INFINITY, trunc_d = resid && rp.d.tau > -INFINITY;
    const float2 kh = make_float2(rp.k.hi, rp.k.hi), kl = make_float2(rp.k.lo, rp.k.lo);
    const float2 mt = make_float2(rp.mt, rp.mt), md = make_float2(rp.md, rp.md);
    const float2 rh = make_float2(r_hi, r_hi), rl = make_float2(r_lo, r_lo);
    float2 st2 = make_float2(0.f, 0.f), sd2 = st2, a2 = st2, b2 = st2;
    uint32_t flag = 0, opn = 0;  // bit 8 g + e: heavy or open / open
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
        if (g < g0 || g >= g1) continue;
        if ((g - g0) % NB == 0) {
#pragma unroll
            for (int i = 0; i < NB; ++i) {
                if (g + i >= g1) break;
                rt[i] = raw_load8<TDT>(rp.t, (g + i) * 256 + lane * 8);
                if (resid) rd[i] = raw_load8<DDT>(rp.d, (g + i) * 256 + lane * 8);
            }
        }
        const int gi = (g - g0) % NB;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            float2 lt = make_float2(raw_get(rt[gi], e), raw_get(rt[gi], e + 1));
            if (trunc_t) lt = make_float2(keep_top(lt.x, rp.t.tau), keep_top(lt.y, rp.t.tau));
            const float2 xt = packed_exponent<TDT == SPECV_F32>(lt, mt, kh, kl);
            const float2 wt = make_float2(ex2(xt.x), ex2(xt.y));
            const bool ht0 = xt.x > kHeavyExp, ht1 = xt.y > kHeavyExp;
            if (!resid) {
                const float2 f = make_float2(ht0 ? 0.f : 1.f, ht1 ? 0.f : 1.f);
                st2 = fma2(wt, f, st2);
                flag |= (ht0 ? 1u << (8 * g + e) : 0u) | (ht1 ? 2u << (8 * g + e) : 0u);
                continue;
            }
            float2 ld = make_float2(raw_get(rd[gi], e), raw_get(rd[gi], e + 1));
            if (trunc_d) ld = make_float2(keep_top(ld.x, rp.d.tau), keep_top(ld.y, rp.d.tau));
            float2 wd;
            bool hd0, hd1;
            if (rp.probs) {
                wd = make_float2(ld.x > -INFINITY ? ld.x : 0.f, ld.y > -INFINITY ? ld.y : 0.f);
                hd0 = wd.x > 1.220703125e-4f;
                hd1 = wd.y > 1.220703125e-4f;
            } else {
                const float2 xd = packed_exponent<DDT == SPECV_F32>(ld, md, kh, kl);
                wd = make_float2(ex2(xd.x), ex2(xd.y));
                hd0 = xd.x > kHeavyExp;
                hd1 = xd.y > kHeavyExp;
            }
            const bool h0 = ht0 || hd0, h1 = ht1 || hd1;
            const float2 qh = mul2(wd, rh), ql = mul2(wd, rl);
            const bool in0 = !h0 && wt.x > qh.x, in1 = !h1 && wt.y > qh.y;    // certainly p > q
            const bool op0 = !h0 && !in0 && !(wt.x <= ql.x);                   // the test cannot decide
            const bool op1 = !h1 && !in1 && !(wt.y <= ql.y);
            const float2 f = make_float2(h0 ? 0.f : 1.f, h1 ? 0.f : 1.f);
            const float2 fi = make_float2(in0 ? 1.f : 0.f, in1 ? 1.f : 0.f);
            st2 = fma2(wt, f, st2);
            sd2 = fma2(wd, f, sd2);
            a2 = fma2(wt, fi, a2);
            b2 = fma2(wd, fi, b2);
            flag |= ((h0 || op0) ? 1u << (8 * g + e) : 0u) | ((h1 || op1) ? 2u << (8 * g + e) : 0u);
            opn |= (op0 ? 1u << (8 * g + e) : 0u) | (op1 ? 2u << (8 * g + e) : 0u);
        }
    }
    // the flagged columns of the warp, 32 at a time: lane L takes flagged
    // column base + L in lane-major, bit-minor order
    df st_h{0.f, 0.f}, sd_h{0.f, 0.f}, a_h{0.f, 0.f}, b_h{0.f, 0.f};
    const uint32_t cnt = __popc(flag);
    uint32_t total;
    const uint32_t off = warp_offsets(cnt, total);
    for (uint32_t base = 0; base < total; base += 32) {
        const uint32_t idx = base + lane;
        // the lane s holding flagged column idx: the last lane whose offset is <= idx
        int s = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {
            const uint32_t o = __shfl_sync(0xffffffffu, off, s + step);
            if (o <= idx) s += step;
        }
        const uint32_t fs = __shfl_sync(0xffffffffu, flag, s), os = __shfl_sync(0xffffffffu, opn, s);
        const uint32_t os_off = __shfl_sync(0xffffffffu, off, s);
        if (idx >= total) continue;
        const int bit = __fns(fs, 0, (int)(idx - os_off) + 1);
        const int64_t j = (bit >> 3) * 256 + s * 8 + (bit & 7);
        const bool is_open = (os >> bit) & 1u;
        const float4 w4 = col_weights<TDT, DDT>(rp.t.g, rp.d.g, rp.t.tau, rp.d.tau, rp.mt, rp.md, rp.k, rp.probs,
                                                resid, j, *ws.tab);
        const df wt{w4.x, w4.y};
        if (!resid) {
            acc_add(st_h, wt);
            continue;
        }
        const df wd{w4.z, w4.w};
        if (!is_open) {  // an open column's weights are in the light sums already
            acc_add(st_h, wt);
            acc_add(sd_h, wd);
        }
        if (wt.hi == 0.f && wd.hi == 0.f) continue;
        if (wt.hi > wd.hi * r_hi) {
            acc_add(a_h, wt);
            acc_add(b_h, wd);
        } else if (!(wt.hi < wd.hi * r_lo)) {  // still open: kept apart for the draw
            const int slot = atomicAdd(ws.nu, 1);
            if (slot < kOpenCap) open_list[slot] = (uint16_t)j;
            if (slot == 0) {
                ws.uw[0] = wt.hi;
                ws.uw[1] = wt.lo;
                ws.uw[2] = wd.hi;
                ws.uw[3] = wd.lo;
            }
        }
    }
    __syncwarp();
    const float cd = rp.probs ? 0.f : kEx2LightBias;
    out.st = df_add(df_norm(st_h), light_sum_df(__fadd_rn(st2.x, st2.y), kEx2LightBias));
    out.sd = df_add(df_norm(sd_h), light_sum_df(__fadd_rn(sd2.x, sd2.y), cd));
    out.a = df_add(df_norm(a_h), light_sum_df(__fadd_rn(a2.x, a2.y), kEx2LightBias));
    out.b = df_add(df_norm(b_h), light_sum_df(__fadd_rn(b2.x, b2.y), cd));
}

}  // namespace

}  // namespace specv
