// tree.cu -- verification of a token tree: several candidates per node.
//
// Tree speculation verifies several candidate continuations in one target
// pass ("Speculative decoding" (mhtirogla.ai), Levers and Implementation
// notes; "Speculative decoding" (inference.tusharamrit.in), tree attention).
// The pages leave the multi-candidate rule open; the reading implemented
// here takes the pages' residual at every candidate in turn. At node u
// (target distribution p_u, draft distribution q_u from which its children
// were drawn), r starts at p_u; candidate j with token x passes if
// u_acc(u, j) * q_u(x) < r(x) and the walk moves to it, else r becomes
// max(0, r - q_u) / Z (unchanged if Z = 0) and the next candidate is tried.
// If none passes, the token is drawn from r by inverse CDF in index order;
// a node without children draws the bonus from p_u. Greedy follows the
// first child equal to the target's argmax. Uniforms: u_acc(u, j) = word 0
// of Philox at counter (u + 65536 j, seq_offset + b, round), u_smp(u) = word 1
// at (u, ...), so a chain-shaped tree draws exactly what the chain verify
// draws.
//
// A cluster of two CTAs per sequence walks its tree, each CTA taking half of
// the columns; their partial sums meet through distributed shared memory.
// At a visited node:
//   - pass 1 reads the target row (and, with candidates, the draft row) for
//     the maxima and the NaN checks (a probability row: its sum), and, with
//     candidates, float softmax sums for the first candidate's test, which
//     runs in float as the chain's accept test does;
//   - if that candidate fails (and at a leaf), pass 2 takes the double-float
//     normalisers and keeps the target's sums over 256-column segments in
//     shared memory;
//   - a rejected candidate costs one residual pass, which takes the next
//     normaliser and keeps the residual's segment sums;
//   - the final draw scans the kept segment sums of the distribution it
//     draws from and rescans the one segment that holds u * total (one
//     warp, 8 columns per lane), so it reads no row again.
// The residual at a column is re-evaluated from p, q and the normalisers met
// so far (r_1 = p, r_{i+1} = max(0, r_i - q) / Z_{i+1}). As in the chain's
// sampler, weights below 2^-13 of the row maximum ("light") are single
// floats whose sums carry the SFU's mean bias correction; the others, and
// all sums, are double-float. Segment s covers columns 256 s .. 256 s + 255:
// warp w reads segments w, w + 16, ..., lane l the 8 columns 256 s + 8 l ...,
// with one or two 16-byte loads when the rows start on 16-byte boundaries.
#include <float.h>
#include <math.h>

#include "internal.h"
#include "precise.cuh"

namespace specv {

namespace {

constexpr int kTrThreads = 512;
constexpr int kTrWarps = kTrThreads / 32;
constexpr int kTrMaxCand = 64;  // candidates per node whose residual normalisers are kept
constexpr int kSeg = 256;       // columns per segment
constexpr float kLightMax = 1.220703125e-4f;  // 2^-13: a probability above it is heavy
constexpr int kCS = 2;          // CTAs per tree (one cluster), each taking half of the segments

struct TreeSmem {
    Exp2Table tab;
    float fred[kTrWarps];
    int32_t ired[kTrWarps];
    df dred[kTrWarps];
    df z[kTrMaxCand + 1];           // 1 / Z of each residual level (index i: r_i -> r_{i+1})
    float zf[kTrMaxCand + 1];       // its high part, for light columns
    int32_t zlive[kTrMaxCand + 1];  // 1: that level changed r (Z > 0)
    int32_t kids[kTrMaxCand];       // the current node's children, in index order
    int32_t nkids;                  // how many it has (may exceed kTrMaxCand)
    int32_t sel, col, last;         // the draw's segment, its column, the last segment of positive weight
    df start;                       // running sum before the selected segment
    float xin[2][8];                // values the peer CTA stored here (two slots, used in turn)
};

// ------------------------------------------------------------ reductions
__device__ float block_max_f(float v, TreeSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) sm.fred[warp] = v;
    __syncthreads();
    float t = -INFINITY;
#pragma unroll
    for (int w = 0; w < kTrWarps; ++w) t = fmaxf(t, sm.fred[w]);
    return t;
}

__device__ int32_t block_min_i(int32_t v, TreeSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) sm.ired[warp] = v;
    __syncthreads();
    int32_t t = INT32_MAX;
#pragma unroll
    for (int w = 0; w < kTrWarps; ++w) t = min(t, sm.ired[w]);
    return t;
}

// Double-float sum over a warp in a fixed order (every lane gets it).
__device__ __forceinline__ df warp_sum_dfx(df v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = df_add(v, shfl_xor_df(v, o));
    return v;
}

// Double-float sum over the CTA in a fixed order (the same bits whatever the timing).
__device__ df block_sum_dfx(df v, TreeSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = warp_sum_dfx(v);
    __syncthreads();
    if (lane == 0) sm.dred[warp] = v;
    __syncthreads();
    df t{0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kTrWarps; ++w) t = df_add(t, sm.dred[w]);
    return t;
}

// Inclusive prefix over a warp's lanes (double-float, Hillis-Steele).
__device__ __forceinline__ df warp_incl_scan_dfx(df x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const df y = shfl_up_df(x, o);
        if (lane >= o) x = df_add(y, x);
    }
    return x;
}

// Prefix sums over the CTA's threads in thread order (double-float): incl
// is the sum up to and including this thread, excl the previous thread's
// incl (the same bits), total the last thread's incl. The intervals
// [excl, incl) of the threads tile [0, total) without gaps or overlaps.
__device__ void block_scan_dfx(df v, TreeSmem& sm, df& excl, df& incl, df& total) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const df x = warp_incl_scan_dfx(v);
    __syncthreads();
    if (lane == 31) sm.dred[warp] = x;
    __syncthreads();
    df before{0.f, 0.f};
    for (int w = 0; w < warp; ++w) before = df_add(before, sm.dred[w]);
    incl = df_add(before, x);
    const df up = shfl_up_df(incl, 1);
    excl = lane == 0 ? before : up;
    total = df{0.f, 0.f};
    for (int w = 0; w < kTrWarps; ++w) total = df_add(total, sm.dred[w]);
}

// ------------------------------------------------------------ the pair of CTAs
// This CTA's share of a tree: segments [s_lo, s_hi), its rank in the
// cluster and the exchange slot to use next.
struct Part {
    int64_t s_lo, s_hi;
    uint32_t rank;
    int ph;
};

struct X8 {
    float v[8];
};

// Every thread of both CTAs calls this with its CTA's values (block-uniform):
// thread 0 stores them into the peer's slot, one cluster barrier, and each
// thread reads the peer's values from its own slot. The slots alternate, so
// a slot is written again only after a barrier its reader has passed.
__device__ X8 xchg(TreeSmem& sm, Part& pt, const X8& mine) {
    if (threadIdx.x == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) st_cluster_f32(&sm.xin[pt.ph][i], pt.rank ^ 1u, mine.v[i]);
    }
    cluster_sync_all();
    X8 o;
#pragma unroll
    for (int i = 0; i < 8; ++i) o.v[i] = sm.xin[pt.ph][i];
    pt.ph ^= 1;
    return o;
}

// Sum of the two CTAs' partial sums in rank order: the same bits in both.
__device__ __forceinline__ df pair_sum(const Part& pt, df mine, df peer) {
    return pt.rank == 0 ? df_add(mine, peer) : df_add(peer, mine);
}

// ------------------------------------------------------------ the node's rows
template <int TDT, int DDT>
struct Rows {
    const char* t;  // target row
    const char* d;  // draft row (nodes with candidates)
    bool probs;     // the draft row holds probabilities
    bool vec;       // the rows read start on 16-byte boundaries
    float mt, md;   // raw maxima
    df k;           // log2(e) / T
    df It, Id;      // 1 / the rows' normalisers
};

// Columns j .. j+7 (j % 8 == 0) as floats, fill past V: one or two 16-byte
// loads when the row allows them, else element loads.
template <int DT>
__device__ __forceinline__ void load_unit(const char* row, bool vec, int64_t j, int64_t V, float fill,
                                          float (&x)[8]) {
    if (vec && j + 8 <= V) {
        if constexpr (DT == SPECV_F32) {
            const float4* q = reinterpret_cast<const float4*>(row) + (j >> 2);
            const float4 a = __ldg(q), c = __ldg(q + 1);
            x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = c.x, x[5] = c.y, x[6] = c.z, x[7] = c.w;
        } else {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(row) + (j >> 3));
            x[0] = bf16_lo(w.x), x[1] = bf16_hi(w.x), x[2] = bf16_lo(w.y), x[3] = bf16_hi(w.y);
            x[4] = bf16_lo(w.z), x[5] = bf16_hi(w.z), x[6] = bf16_lo(w.w), x[7] = bf16_hi(w.w);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = j + e < V ? ld_elem<DT>(row, j + e) : fill;
    }
}

// Target weight 2^((l - mt) k) of one column: a light one as a float
// (returns false), a heavy one in double-float (returns true).
template <int TDT, int DDT>
__device__ __forceinline__ bool tgt_col(const Rows<TDT, DDT>& n, float l, const TreeSmem& sm, float& lw, df& hw) {
    bool h;
    lw = light_weight<TDT == SPECV_F32>(l, n.mt, n.k, h);
    if (h) hw = heavy_logit_weight<TDT == SPECV_F32, true>(l, n.mt, n.k, sm.tab);
    return h;
}

// Draft weight of one column, the same way (a probability is its own weight).
template <int TDT, int DDT>
__device__ __forceinline__ bool dft_col(const Rows<TDT, DDT>& n, float l, const TreeSmem& sm, float& lw, df& hw) {
    if (n.probs) {
        lw = l;
        hw = df{l, 0.f};
        return l > kLightMax;
    }
    bool h;
    lw = light_weight<DDT == SPECV_F32>(l, n.md, n.k, h);
    if (h) hw = heavy_logit_weight<DDT == SPECV_F32, true>(l, n.md, n.k, sm.tab);
    return h;
}

// max(0, r_L - q) at one column, L >= 1. Both weights light: in float
// (returns false, value in lw); else in double-float (returns true).
template <int TDT, int DDT>
__device__ __forceinline__ bool resid_col(const Rows<TDT, DDT>& n, float xt, float xd, int L, const TreeSmem& sm,
                                          float& lw, df& hw) {
    float wt, wd;
    df Wt, Wd;
    const bool ht = tgt_col(n, xt, sm, wt, Wt);
    const bool hd = dft_col(n, xd, sm, wd, Wd);
    if (!ht && !hd) {
        const float p = __fmaf_rn(wt, n.It.hi, __fmul_rn(wt, n.It.lo));
        const float q = __fmaf_rn(wd, n.Id.hi, __fmul_rn(wd, n.Id.lo));
        float r = p;
        for (int i = 1; i < L; ++i) {
            if (!sm.zlive[i]) continue;
            const float dl = __fsub_rn(r, q);
            r = dl > 0.f ? __fmul_rn(dl, sm.zf[i]) : 0.f;
        }
        const float dl = __fsub_rn(r, q);
        lw = dl > 0.f ? dl : 0.f;
        return false;
    }
    if (!ht) Wt = df{wt, 0.f};
    if (!hd) Wd = df{wd, 0.f};
    const df q = df_mul(Wd, n.Id);
    df r = df_mul(Wt, n.It);
    for (int i = 1; i < L; ++i) {
        if (!sm.zlive[i]) continue;
        const df dl = df_sub(r, q);
        r = df_pos(dl) ? df_mul(dl, sm.z[i]) : df{0.f, 0.f};
    }
    const df dl = df_sub(r, q);
    hw = df_pos(dl) ? dl : df{0.f, 0.f};
    return true;
}

// r_L(x) and q(x) in double-float: the accept test at one column.
template <int TDT, int DDT>
__device__ df r_at(const Rows<TDT, DDT>& n, float xt, float xd, int L, const TreeSmem& sm, df& q) {
    const df Wt = logit_weight<TDT == SPECV_F32>(xt, n.mt, n.k, sm.tab);
    const df Wd = n.probs ? df{xd, 0.f} : logit_weight<DDT == SPECV_F32>(xd, n.md, n.k, sm.tab);
    q = df_mul(Wd, n.Id);
    df r = df_mul(Wt, n.It);
    for (int i = 1; i < L; ++i) {
        if (!sm.zlive[i]) continue;
        const df dl = df_sub(r, q);
        r = df_pos(dl) ? df_mul(dl, sm.z[i]) : df{0.f, 0.f};
    }
    return r;
}

// Weight of one column of the distribution a draw reads: kind 0, the target
// weight; kind L >= 1, max(0, r_L - q).
template <int TDT, int DDT>
__device__ __forceinline__ bool draw_col(const Rows<TDT, DDT>& n, int kind, float xt, float xd, const TreeSmem& sm,
                                         float& lw, df& hw) {
    return kind == 0 ? tgt_col(n, xt, sm, lw, hw) : resid_col(n, xt, xd, kind, sm, lw, hw);
}

// ------------------------------------------------------------ passes
// A lane's 8 columns as stored (bf16: four words; f32: eight), so that the
// segments in flight cost half the registers in bf16.
template <int DT>
struct Raw {
    uint32_t w[DT == SPECV_F32 ? 8 : 4];
};

template <int DT>
__device__ __forceinline__ Raw<DT> fetch_unit(const char* row, bool vec, int64_t j, int64_t V, float fill) {
    Raw<DT> r;
    if (vec && j + 8 <= V) {
        if constexpr (DT == SPECV_F32) {
            const uint4* q = reinterpret_cast<const uint4*>(row) + (j >> 2);
            const uint4 a = __ldg(q), c = __ldg(q + 1);
            r.w[0] = a.x, r.w[1] = a.y, r.w[2] = a.z, r.w[3] = a.w, r.w[4] = c.x, r.w[5] = c.y, r.w[6] = c.z,
            r.w[7] = c.w;
        } else {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(row) + (j >> 3));
            r.w[0] = a.x, r.w[1] = a.y, r.w[2] = a.z, r.w[3] = a.w;
        }
    } else {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = j + e < V ? ld_elem<DT>(row, j + e) : fill;
        if constexpr (DT == SPECV_F32) {
#pragma unroll
            for (int e = 0; e < 8; ++e) r.w[e] = __float_as_uint(x[e]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)  // the values are bf16: their high halves hold them exactly
                r.w[e] = (__float_as_uint(x[2 * e]) >> 16) | (__float_as_uint(x[2 * e + 1]) & 0xFFFF0000u);
        }
    }
    return r;
}

template <int DT>
__device__ __forceinline__ void decode_unit(const Raw<DT>& r, float (&x)[8]) {
    if constexpr (DT == SPECV_F32) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(r.w[e]);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[2 * e] = bf16_lo(r.w[e]);
            x[2 * e + 1] = bf16_hi(r.w[e]);
        }
    }
}

// f(i, j, t, d) for every segment of this CTA's share that this warp owns
// (segments s_lo + warp, s_lo + warp + 16, ...; i = s - s_lo is
// warp-uniform), j = the lane's first column, t and d its 8
// target and draft values (d only if D; columns past V read as -inf, or 0
// in a probability row). The next two segments' loads are in flight while f
// runs. Per lane, columns increase.
template <bool D, int TDT, int DDT, class F>
__device__ __forceinline__ void seg_pass(const Rows<TDT, DDT>& n, int64_t V, const Part& pt, F&& f) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int64_t s = pt.s_lo + warp;
    if (s >= pt.s_hi) return;
    const float fd = n.probs ? 0.f : -INFINITY;
    Raw<TDT> ta, tb;  // the next two segments, in flight
    Raw<DDT> da, db;
    ta = fetch_unit<TDT>(n.t, n.vec, s * kSeg + lane * 8, V, -INFINITY);
    if (D) da = fetch_unit<DDT>(n.d, n.vec, s * kSeg + lane * 8, V, fd);
    if (s + kTrWarps < pt.s_hi) {
        tb = fetch_unit<TDT>(n.t, n.vec, (s + kTrWarps) * kSeg + lane * 8, V, -INFINITY);
        if (D) db = fetch_unit<DDT>(n.d, n.vec, (s + kTrWarps) * kSeg + lane * 8, V, fd);
    }
#pragma unroll 1
    for (; s < pt.s_hi; s += kTrWarps) {
        float t[8], d[8];
        decode_unit<TDT>(ta, t);
        ta = tb;
        if (D) {
            decode_unit<DDT>(da, d);
            da = db;
        }
        const int64_t s2 = s + 2 * kTrWarps;
        if (s2 < pt.s_hi) {
            tb = fetch_unit<TDT>(n.t, n.vec, s2 * kSeg + lane * 8, V, -INFINITY);
            if (D) db = fetch_unit<DDT>(n.d, n.vec, s2 * kSeg + lane * 8, V, fd);
        }
        f(s - pt.s_lo, s * kSeg + lane * 8, t, d);
    }
}

// A lane's 8 column weights summed: light(e, l) gives a light weight in l
// (returning false) or flags a heavy column (true); heavy columns are then
// evaluated one by one, in column order, by heavy(j) in double-float, so the
// double-float code exists once per pass and runs only for them. Light
// weights are summed in float and joined with the correction cl.
template <class L, class H>
__device__ __forceinline__ df unit_sum(int64_t j, L&& light, H&& heavy, float cl) {
    float lt = 0.f;
    uint32_t hm = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float l;
        if (light(e, l)) hm |= 1u << e;
        else lt = __fadd_rn(lt, l);
    }
    df ht{0.f, 0.f};
#pragma unroll 1
    while (hm) {
        const int e = __ffs(hm) - 1;
        hm &= hm - 1;
        acc_add(ht, heavy(j + e));
    }
    return df_add(df_norm(ht), light_sum_df(lt, cl));
}

// Light parts of the column weights (true: the column is heavy).
template <int TDT, int DDT>
__device__ __forceinline__ bool tgt_light(const Rows<TDT, DDT>& n, float l, float& w) {
    bool h;
    w = light_weight<TDT == SPECV_F32>(l, n.mt, n.k, h);
    return h;
}
template <int TDT, int DDT>
__device__ __forceinline__ bool dft_light(const Rows<TDT, DDT>& n, float l, float& w) {
    if (n.probs) {
        w = l;
        return l > kLightMax;
    }
    bool h;
    w = light_weight<DDT == SPECV_F32>(l, n.md, n.k, h);
    return h;
}
template <int TDT, int DDT>
__device__ __forceinline__ bool resid_light(const Rows<TDT, DDT>& n, float xt, float xd, int L, const TreeSmem& sm,
                                            float& w) {
    float wt, wd;
    if (tgt_light(n, xt, wt) | dft_light(n, xd, wd)) return true;
    const float p = __fmaf_rn(wt, n.It.hi, __fmul_rn(wt, n.It.lo));
    const float q = __fmaf_rn(wd, n.Id.hi, __fmul_rn(wd, n.Id.lo));
    float r = p;
    for (int i = 1; i < L; ++i) {
        if (!sm.zlive[i]) continue;
        const float dl = __fsub_rn(r, q);
        r = dl > 0.f ? __fmul_rn(dl, sm.zf[i]) : 0.f;
    }
    const float dl = __fsub_rn(r, q);
    w = dl > 0.f ? dl : 0.f;
    return false;
}

// The sum of this CTA's kept segment sums in a fixed order (every thread gets it).
__device__ df seg_total(const float2* buf, const Part& pt, TreeSmem& sm) {
    df s{0.f, 0.f};
    for (int64_t i = threadIdx.x; i < pt.s_hi - pt.s_lo; i += kTrThreads) s = df_add(s, df{buf[i].x, buf[i].y});
    return block_sum_dfx(s, sm);
}

// Rescan of segment sel (global index) with warp 0: lane l takes columns
// 8 l .. 8 l + 7 with running sums formed as the pass formed the segment's
// sum; returns the first column whose running sum from start exceeds thr,
// else (rounding, or a NaN start) the segment's last column of positive
// weight, else -1. Every thread gets the result.
template <int TDT, int DDT>
__device__ int32_t rescan(const Rows<TDT, DDT>& n, int64_t V, int kind, int64_t sel, df start, df thr,
                          TreeSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        const bool D = kind > 0;
        const int64_t j = sel * kSeg + lane * 8;
        float t[8], d[8];
        load_unit<TDT>(n.t, n.vec, j, V, -INFINITY, t);
        if (D) load_unit<DDT>(n.d, n.vec, j, V, n.probs ? 0.f : -INFINITY, d);
        const float cl = (kind > 0 && n.probs) ? 0.f : kEx2LightBias;
        df pre[8];
        float lt = 0.f;
        df ht{0.f, 0.f};
        int lp = -1;
#pragma unroll 1
        for (int e = 0; e < 8; ++e) {
            float l;
            df h;
            const bool heavy = draw_col(n, kind, t[e], D ? d[e] : 0.f, sm, l, h);
            if (heavy) acc_add(ht, h);
            else lt = __fadd_rn(lt, l);
            if (heavy ? df_pos(h) : l > 0.f) lp = e;
            pre[e] = df_add(df_norm(ht), light_sum_df(lt, cl));
        }
        const df incl_l = warp_incl_scan_dfx(pre[7]);
        const df up = shfl_up_df(incl_l, 1);
        const df base = df_add(start, lane == 0 ? df{0.f, 0.f} : up);
        int hit = -1;
#pragma unroll
        for (int e = 7; e >= 0; --e)
            if (df_gt(df_add(base, pre[e]), thr)) hit = e;
        const uint32_t hm = __ballot_sync(0xffffffffu, hit >= 0);
        const uint32_t pm = __ballot_sync(0xffffffffu, lp >= 0);
        if (hm) {
            if (lane == __ffs(hm) - 1) sm.col = (int32_t)(j + hit);
        } else if (pm) {
            if (lane == 31 - __clz(pm)) sm.col = (int32_t)(j + lp);
        } else if (lane == 0) {
            sm.col = -1;
        }
    }
    __syncthreads();
    const int32_t c = sm.col;
    __syncthreads();  // sm.col is written again only after every thread has read it
    return c;
}

// Inverse CDF in index order over the distribution whose segment sums are
// buf (this CTA's share; kind as draw_col): the first column whose running
// sum exceeds u * total; if rounding leaves none, the last column of
// positive weight; -1 if no column has weight. Rank 0's prefix sums start at
// 0, rank 1's at rank 0's total, so the two CTAs' intervals tile [0, total).
// Thread t scans this CTA's segments [t K, t K + K); the thread whose
// interval holds u * total finds the segment, which warp 0 rescans. All
// threads of both CTAs get the same column.
template <int TDT, int DDT>
__device__ int32_t draw_from(const Rows<TDT, DDT>& n, int64_t V, int kind, const float2* buf, float us, Part& pt,
                             TreeSmem& sm) {
    const int64_t ns = pt.s_hi - pt.s_lo;
    const int64_t K = (ns + kTrThreads - 1) / kTrThreads;
    const int64_t s0 = min(ns, (int64_t)threadIdx.x * K), s1 = min(ns, s0 + K);
    if (threadIdx.x == 0) {
        sm.sel = -1;
        sm.last = -1;
    }
    df mine{0.f, 0.f};
    int32_t lastseg = -1;
    for (int64_t i = s0; i < s1; ++i) {
        const df v{buf[i].x, buf[i].y};
        if (df_pos(v)) lastseg = (int32_t)(pt.s_lo + i);
        mine = df_add(mine, v);
    }
    df excl, incl, tl;
    block_scan_dfx(mine, sm, excl, incl, tl);  // its barriers order the resets above
    if (lastseg >= 0) atomicMax(&sm.last, lastseg);
    __syncthreads();
    X8 x{};
    x.v[0] = tl.hi, x.v[1] = tl.lo, x.v[2] = __int_as_float(sm.last);
    const X8 y = xchg(sm, pt, x);
    const df tp{y.v[0], y.v[1]};
    const int32_t last_all = max(sm.last, __float_as_int(y.v[2]));
    const df t0 = pt.rank == 0 ? tl : tp;
    const df total = pair_sum(pt, tl, tp);
    const df thr = df_mul_f(total, us);
    if (pt.rank != 0) {
        excl = df_add(t0, excl);
        incl = df_add(t0, incl);
    }
    if (!df_gt(excl, thr) && df_gt(incl, thr)) {  // at most one thread of the two CTAs
        df run = excl;
        int64_t found = -1;
        for (int64_t i = s0; i < s1; ++i) {
            const df end = df_add(run, df{buf[i].x, buf[i].y});
            if (df_gt(end, thr)) {
                found = i;
                break;
            }
            run = end;
        }
        sm.sel = (int32_t)(found >= 0 ? pt.s_lo + found : lastseg);
        sm.start = found >= 0 ? run : df{NAN, 0.f};  // NaN: no comparison succeeds, the last column wins
    }
    __syncthreads();
    const int32_t sel = sm.sel;
    const df start = sm.start;
    int32_t c = INT32_MAX;
    if (sel >= 0) {  // block-uniform
        c = rescan(n, V, kind, sel, start, thr, sm);
        if (c < 0) c = INT32_MAX;
    }
    x.v[0] = __int_as_float(c);
    const int32_t cp = __float_as_int(xchg(sm, pt, x).v[0]);
    c = min(c, cp);
    if (c != INT32_MAX) return c;
    // rounding left no crossing in either CTA: the last column of positive weight
    if (last_all < 0) return -1;
    int32_t lc = -1;
    if (last_all >= pt.s_lo && last_all < pt.s_hi) lc = rescan(n, V, kind, last_all, df{NAN, 0.f}, thr, sm);
    x.v[0] = __int_as_float(lc);
    const int32_t lp = __float_as_int(xchg(sm, pt, x).v[0]);
    return max(lc, lp);
}

// First index of the largest target value (NaN read as -inf; a row of -inf
// or NaN gives 0).
template <int TDT, int DDT>
__device__ int32_t row_argmax(const Rows<TDT, DDT>& n, int64_t V, Part& pt, TreeSmem& sm) {
    float best = -INFINITY;
    int32_t bi = INT32_MAX;
    seg_pass<false>(n, V, pt, [&](int64_t, int64_t j, const float (&t)[8], const float (&)[8]) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (t[e] > best) {  // NaN never passes; per lane j increases: the first of equals stays
                best = t[e];
                bi = (int32_t)(j + e);
            }
    });
    const float m = block_max_f(best, sm);
    const int32_t i = block_min_i(best == m ? bi : INT32_MAX, sm);
    X8 x{};
    x.v[0] = m, x.v[1] = __int_as_float(i);
    const X8 y = xchg(sm, pt, x);
    const float M = fmaxf(m, y.v[0]);
    const int32_t k = min(m == M ? i : INT32_MAX, y.v[0] == M ? __float_as_int(y.v[1]) : INT32_MAX);
    return k == INT32_MAX ? 0 : k;
}

__device__ void write_error(const TreeParams& p, int32_t b, int32_t st, int64_t o, int64_t n) {
    if (st != 4)  // SPEC_SEQ_BAD_LAYOUT: the sequence's slots are unknown
        for (int64_t k = threadIdx.x; k < n; k += kTrThreads) {
            p.out_tokens[o + k] = -1;
            if (p.out_path) p.out_path[o + k] = -1;
        }
    if (threadIdx.x == 0) {
        p.out_accepted[b] = 0;
        if (p.seq_status) p.seq_status[b] = st;
    }
}

// A cluster of kCS CTAs per tree; both CTAs run the same walk on the same
// exchanged values, so they take the same branches and pass the same
// cluster barriers; rank 0 writes the outputs. Dynamic shared memory: two
// buffers of this CTA's segment sums, (hi, lo) per segment.
template <int TDT, int DDT>
__global__ void __cluster_dims__(kCS, 1, 1) __launch_bounds__(kTrThreads) tree_kernel(const TreeParams p) {
    __shared__ TreeSmem sm;
    extern __shared__ float2 segbuf[];
    const uint32_t rank = cluster_ctarank();
    const int32_t b = (int32_t)(blockIdx.x / kCS);
    const bool writer = rank == 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t V = p.V, segs = (V + kSeg - 1) / kSeg, half = (segs + kCS - 1) / kCS;
    Part pt{min(segs, (int64_t)rank * half), min(segs, (int64_t)rank * half + half), rank, 0};
    // statuses that need no row, in the documented order (both CTAs alike)
    const int64_t o = __ldg(p.node_off + b), N = __ldg(p.node_off + b + 1) - o;
    if (N < 1 || o < 0 || o + N > p.nodes) {
        if (writer) write_error(p, b, 4, o, N);  // SPEC_SEQ_BAD_LAYOUT
        return;
    }
    bool bad = threadIdx.x == 0 && __ldg(p.parent + o) != -1;
    for (int64_t v = 1 + threadIdx.x; v < N; v += kTrThreads) {
        const int32_t q = __ldg(p.parent + o + v);
        bad |= q < 0 || q >= v;
    }
    if (__syncthreads_or(bad)) {
        if (writer) write_error(p, b, 4, o, N);
        return;
    }
    const float T = p.temps ? __ldg(p.temps + b) : p.temperature;
    if (!p.greedy && (!(T > 0.f) || !isfinite(T))) {
        if (writer) write_error(p, b, 5, o, N);  // SPEC_SEQ_BAD_TEMP
        return;
    }
    bad = false;
    for (int64_t v = 1 + threadIdx.x; v < N; v += kTrThreads) {
        const int32_t x = __ldg(p.tokens + o + v);
        bad |= x < 0 || x >= V;
    }
    if (__syncthreads_or(bad)) {
        if (writer) write_error(p, b, 1, o, N);  // SPEC_SEQ_BAD_TOKEN
        return;
    }
    for (int i = threadIdx.x; i < 64; i += kTrThreads) {
        sm.tab.hi[i] = p.tab.hi[i];
        sm.tab.lo[i] = p.tab.lo[i];
    }
    __syncthreads();
    cluster_sync_all();  // both CTAs are running before either stores into the other

    constexpr int64_t tes = TDT == SPECV_F32 ? 4 : 2, des = DDT == SPECV_F32 ? 4 : 2;
    Rows<TDT, DDT> n;
    n.probs = p.probs != 0;
    n.k = p.greedy ? df{0.f, 0.f} : k_of_temperature(T);
    n.d = nullptr;
    n.md = 0.f;
    int64_t u = 0;
    int32_t acc = 0, emit = -1;
    const uint32_t seq = p.seq_offset + (uint32_t)b;
    for (;;) {
        n.t = (const char*)p.tgt + (o + u) * V * tes;
        if (p.greedy) {
            n.vec = ((uintptr_t)n.t & 15) == 0;
            const int32_t g = row_argmax(n, V, pt, sm);
            int32_t c = INT32_MAX;
            for (int64_t v = u + 1 + threadIdx.x; v < N; v += kTrThreads)
                if (__ldg(p.parent + o + v) == u && __ldg(p.tokens + o + v) == g) {
                    c = (int32_t)v;  // increasing v per thread: the first match is its smallest
                    break;
                }
            c = block_min_i(c, sm);
            if (c == INT32_MAX) {
                emit = g;
                break;
            }
            if (writer && threadIdx.x == 0) {
                p.out_tokens[o + acc] = g;
                if (p.out_path) p.out_path[o + acc] = c;
            }
            ++acc;
            u = c;
            continue;
        }
        // the node's candidates, in index order (warp 0), once every thread
        // is done with the previous node's list
        __syncthreads();
        if (warp == 0) {
            int32_t cnt = 0;
            for (int64_t base = u + 1; base < N; base += 32) {
                const int64_t v = base + lane;
                const bool is = v < N && __ldg(p.parent + o + v) == u;
                const uint32_t m = __ballot_sync(0xffffffffu, is);
                const int32_t pos = cnt + __popc(m & ((1u << lane) - 1u));
                if (is && pos < kTrMaxCand) sm.kids[pos] = (int32_t)v;
                cnt += __popc(m);
            }
            if (lane == 0) sm.nkids = cnt;
        }
        __syncthreads();
        const int32_t m = sm.nkids;
        if (m > kTrMaxCand) {
            if (writer) write_error(p, b, kSeqUnsupported, o, N);
            return;
        }
        const bool D = m > 0;  // the draft row is read at nodes with candidates
        n.d = D ? (const char*)p.dft + (o + u) * V * des : nullptr;
        n.vec = ((uintptr_t)n.t & 15) == 0 && (!D || ((uintptr_t)n.d & 15) == 0);
        // pass 1: maxima and NaN checks; with candidates also float softmax
        // sums of both rows (online, per lane; a probability row: its
        // double-float sum) for the float test of the first candidate
        const float kf = n.k.hi;
        float mt = -INFINITY, md = -INFINITY;
        float om_t = -FLT_MAX, os_t = 0.f, om_d = -FLT_MAX, os_d = 0.f;  // online maxima and sums
        bool hnt = false, hnd = false;
        df sd{0.f, 0.f};
        auto fold = [&](float x, float& om, float& os) {
            if (x > om) {
                os = __fmaf_rn(os, ex2(__fmul_rn(__fsub_rn(om, x), kf)), 1.f);
                om = x;
            } else {
                os = __fadd_rn(os, ex2(__fmul_rn(__fsub_rn(x, om), kf)));
            }
        };
        if (D) {
            seg_pass<true>(n, V, pt, [&](int64_t, int64_t, const float (&t)[8], const float (&d)[8]) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    mt = fmaxf(mt, t[e]);
                    hnt |= t[e] != t[e];
                    hnd |= d[e] != d[e];
                    fold(t[e], om_t, os_t);
                    if (n.probs) {
                        acc_add(sd, d[e]);
                    } else {
                        md = fmaxf(md, d[e]);
                        fold(d[e], om_d, os_d);
                    }
                }
            });
        } else {
            seg_pass<false>(n, V, pt, [&](int64_t, int64_t, const float (&t)[8], const float (&)[8]) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    mt = fmaxf(mt, t[e]);
                    hnt |= t[e] != t[e];
                }
            });
        }
        hnt = __syncthreads_or(hnt);
        hnd = __syncthreads_or(hnd);
        mt = block_max_f(mt, sm);
        md = block_max_f(md, sm);
        sd = block_sum_dfx(df_norm(sd), sm);
        // the lanes' float sums relative to this CTA's maxima (NaN-free: an
        // empty lane has os = 0; a bad row's sums are never used)
        auto rel = [&](float os, float om, float M) {
            return (os > 0.f && M > -INFINITY) ? __fmul_rn(os, ex2(__fmul_rn(__fsub_rn(om, M), kf))) : 0.f;
        };
        const float fs_t = D ? block_sum_dfx(df{rel(os_t, om_t, mt), 0.f}, sm).hi : 0.f;
        const float fs_d = (D && !n.probs) ? block_sum_dfx(df{rel(os_d, om_d, md), 0.f}, sm).hi : 0.f;
        float St_f, Sd_f;
        {
            X8 x{};
            x.v[0] = mt, x.v[1] = md, x.v[2] = sd.hi, x.v[3] = sd.lo, x.v[4] = (float)(hnt ? 1 : 0) + (hnd ? 2 : 0);
            x.v[5] = fs_t, x.v[6] = fs_d;
            const X8 y = xchg(sm, pt, x);
            n.mt = fmaxf(mt, y.v[0]);
            n.md = fmaxf(md, y.v[1]);
            sd = pair_sum(pt, sd, df{y.v[2], y.v[3]});
            const int fl = (int)x.v[4] | (int)y.v[4];
            hnt = fl & 1;
            hnd = fl & 2;
            // rank order: rank 0's part first
            const float a_t = pt.rank == 0 ? fs_t : y.v[5], b_t = pt.rank == 0 ? y.v[5] : fs_t;
            const float ma_t = pt.rank == 0 ? mt : y.v[0], mb_t = pt.rank == 0 ? y.v[0] : mt;
            const float a_d = pt.rank == 0 ? fs_d : y.v[6], b_d = pt.rank == 0 ? y.v[6] : fs_d;
            const float ma_d = pt.rank == 0 ? md : y.v[1], mb_d = pt.rank == 0 ? y.v[1] : md;
            St_f = __fadd_rn(rel(a_t, ma_t, n.mt), rel(b_t, mb_t, n.mt));
            Sd_f = __fadd_rn(rel(a_d, ma_d, n.md), rel(b_d, mb_d, n.md));
        }
        bad = hnt || !isfinite(n.mt);
        if (D) bad |= n.probs ? (hnd || !(sd.hi > 0.f) || !isfinite(sd.hi)) : (hnd || !isfinite(n.md));
        if (bad) {
            if (writer) write_error(p, b, 3, o, N);  // SPEC_SEQ_BAD_ROW
            return;
        }
        const float us = draw_uniforms(p.seed, p.round, seq, (uint32_t)u).y;
        int32_t next = -1;
        if (D) {  // the first candidate's test, in float (every thread of both CTAs: the same bits)
            const int32_t c = sm.kids[0];
            const int32_t x = __ldg(p.tokens + o + c);
            const float ua = draw_uniforms(p.seed, p.round, seq, (uint32_t)u).x;
            const float px = __fdiv_rn(ex2(__fmul_rn(__fsub_rn(ld_elem<TDT>(n.t, x), n.mt), kf)), St_f);
            const float qv = ld_elem<DDT>(n.d, x);
            const float qx = n.probs ? __fdiv_rn(qv, sd.hi) : __fdiv_rn(ex2(__fmul_rn(__fsub_rn(qv, n.md), kf)), Sd_f);
            if (__fmul_rn(ua, qx) < px) next = c;
        }
        if (next >= 0) {
            if (writer && threadIdx.x == 0) {
                p.out_tokens[o + acc] = __ldg(p.tokens + o + next);
                if (p.out_path) p.out_path[o + acc] = next;
            }
            ++acc;
            u = next;
            continue;
        }
        // pass 2: the double-float normalisers, and the target's segment sums into buffer 0
        float2* cur = segbuf;         // segment sums of the distribution a draw would read
        float2* spare = segbuf + half;
        int kind = 0;                 // what cur holds (draw_col)
        const bool DL = D && !n.probs;
        df sdl{0.f, 0.f};
        auto tgt_heavy = [&](int64_t c) {
            return heavy_logit_weight<TDT == SPECV_F32, true>(ld_elem<TDT>(n.t, c), n.mt, n.k, sm.tab);
        };
        auto tgt_seg = [&](int64_t i, int64_t j, const float (&t)[8]) {
            const df v = warp_sum_dfx(
                unit_sum(j, [&](int e, float& l) { return tgt_light(n, t[e], l); }, tgt_heavy, kEx2LightBias));
            if (lane == 0) cur[i] = make_float2(v.hi, v.lo);
        };
        if (DL) {  // the draft row is read only when its logits need a normaliser
            auto dft_heavy = [&](int64_t c) {
                return heavy_logit_weight<DDT == SPECV_F32, true>(ld_elem<DDT>(n.d, c), n.md, n.k, sm.tab);
            };
            seg_pass<true>(n, V, pt, [&](int64_t i, int64_t j, const float (&t)[8], const float (&d)[8]) {
                tgt_seg(i, j, t);
                sdl = df_add(sdl, unit_sum(j, [&](int e, float& l) { return dft_light(n, d[e], l); }, dft_heavy,
                                           kEx2LightBias));
            });
        } else {
            seg_pass<false>(n, V, pt,
                            [&](int64_t i, int64_t j, const float (&t)[8], const float (&)[8]) { tgt_seg(i, j, t); });
        }
        __syncthreads();
        df st = seg_total(cur, pt, sm);
        if (DL) sd = block_sum_dfx(sdl, sm);
        {
            X8 x{};
            x.v[0] = st.hi, x.v[1] = st.lo, x.v[2] = sd.hi, x.v[3] = sd.lo;
            const X8 y = xchg(sm, pt, x);
            st = pair_sum(pt, st, df{y.v[0], y.v[1]});
            if (DL) sd = pair_sum(pt, sd, df{y.v[2], y.v[3]});
        }
        n.It = df_recip(st);
        if (!D) {  // a leaf: the bonus token from p
            emit = draw_from(n, V, 0, cur, us, pt, sm);
            break;
        }
        n.Id = df_recip(sd);
        const float cl = n.probs ? 0.f : kEx2LightBias;
        // candidate 0 failed above; from here each rejection costs a residual pass
        int level = 1;
        for (int32_t j = 0; j < m; ++j) {
            const int32_t c = sm.kids[j];
            if (j > 0) {
                const int32_t x = __ldg(p.tokens + o + c);
                const float ua = draw_uniforms(p.seed, p.round, seq, (uint32_t)(u + (int64_t)j * 65536)).x;
                df qx;  // every thread of both CTAs: the same bits, no broadcast
                const df rx = r_at(n, ld_elem<TDT>(n.t, x), ld_elem<DDT>(n.d, x), level, sm, qx);
                if (df_gt(rx, df_mul_f(qx, ua))) {
                    next = c;
                    break;
                }
            }
            // the next residual: its normaliser and segment sums
            auto res_heavy = [&](int64_t cc) {
                float l;
                df h;
                resid_col(n, ld_elem<TDT>(n.t, cc), ld_elem<DDT>(n.d, cc), level, sm, l, h);
                return h;
            };
            seg_pass<true>(n, V, pt, [&](int64_t i, int64_t jj, const float (&t)[8], const float (&d)[8]) {
                const df v = warp_sum_dfx(unit_sum(
                    jj, [&](int e, float& l) { return resid_light(n, t[e], d[e], level, sm, l); }, res_heavy, cl));
                if (lane == 0) spare[i] = make_float2(v.hi, v.lo);
            });
            __syncthreads();
            df z = seg_total(spare, pt, sm);
            {
                X8 xx{};
                xx.v[0] = z.hi, xx.v[1] = z.lo;
                const X8 y = xchg(sm, pt, xx);
                z = pair_sum(pt, z, df{y.v[0], y.v[1]});
            }
            const bool live = !residual_empty(z);
            if (threadIdx.x == 0) {
                sm.zlive[level] = live;
                sm.z[level] = df_recip(z);
                sm.zf[level] = sm.z[level].hi;
            }
            if (live) {  // r changed: the draw would read these sums
                float2* t2 = cur;
                cur = spare;
                spare = t2;
                kind = level;
            }
            __syncthreads();
            ++level;
        }
        if (next >= 0) {
            if (writer && threadIdx.x == 0) {
                p.out_tokens[o + acc] = __ldg(p.tokens + o + next);
                if (p.out_path) p.out_path[o + acc] = next;
            }
            ++acc;
            u = next;
            continue;
        }
        emit = draw_from(n, V, kind, cur, us, pt, sm);
        break;
    }
    // the emitted token, then -1 over the sequence's remaining slots
    if (writer) {
        for (int64_t k = acc + threadIdx.x; k < N; k += kTrThreads) {
            p.out_tokens[o + k] = k == acc ? emit : -1;
            if (p.out_path) p.out_path[o + k] = -1;
        }
        if (threadIdx.x == 0) {
            p.out_accepted[b] = acc;
            if (p.seq_status) p.seq_status[b] = 0;
        }
    }
}

template <int TDT, int DDT>
cudaError_t launch_tree_t(const TreeParams& p, cudaStream_t s) {
    const int64_t segs = (p.V + kSeg - 1) / kSeg;
    const size_t dyn = sizeof(float2) * 2 * (size_t)((segs + kCS - 1) / kCS);
    if (dyn > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(tree_kernel<TDT, DDT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        if (e != cudaSuccess) return e;
    }
    tree_kernel<TDT, DDT><<<(unsigned)p.B * kCS, kTrThreads, dyn, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tree(const TreeParams& p, cudaStream_t s) {
    if (p.B == 0) return cudaSuccess;
    const int ddt = p.greedy ? p.tdt : p.ddt;  // greedy reads no draft row
    if (p.tdt == SPECV_F32)
        return ddt == SPECV_F32 ? launch_tree_t<SPECV_F32, SPECV_F32>(p, s) : launch_tree_t<SPECV_F32, SPECV_BF16>(p, s);
    return ddt == SPECV_F32 ? launch_tree_t<SPECV_BF16, SPECV_F32>(p, s) : launch_tree_t<SPECV_BF16, SPECV_BF16>(p, s);
}

}  // namespace specv
