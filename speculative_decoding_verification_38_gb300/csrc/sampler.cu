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
// Only the selected row pair is re-read. Each sequence gets one thread-block
// cluster of nsplit CTAs, CTA c owning a contiguous column chunk:
//   pass A (residual only): the exact normalisers S_p = sum_j 2^((l_j - l_max) k)
//     of both rows, reduced over the cluster through distributed shared memory;
//   pass B: the weights r_j (= max(0, p_j - q_j), or p_j's weight for a bonus)
//     tile by tile (a tile = 32 lanes x 8 consecutive columns), each tile's sum
//     kept in shared memory; chunk sums are exchanged across the cluster so
//     every CTA knows Z and where its chunk starts in the CDF;
//   the CTA whose interval holds u * Z finds the tile with one warp-wide
//   prefix over its tile sums and rescans that tile to find the column.
// Weights, sums and prefixes are double-float (precise.cuh), so the pick
// matches a float64 evaluation except within ~1e-10 of a CDF edge.
#include <math.h>

#include "precise.cuh"

namespace specv {

namespace {

constexpr int kWarps = kSampThreads / 32;

struct SampSmem {
    Exp2Table tab;
    df tile_sum[kMaxTilesPerCta];
    df norm_t[kMaxCluster], norm_d[kMaxCluster];
    df zc[kMaxCluster], zc2[kMaxCluster];
    df red_t[kWarps], red_d[kWarps];
    int32_t sel_tile;
    df sel_base;
};

// Eight consecutive columns c..c+7 of a row as floats; columns at or past
// `lim` read as -inf (weight 0).
template <int DT>
__device__ __forceinline__ void load8(const char* row, int64_t c, int64_t lim, bool aligned, float (&v)[8]) {
    if (aligned && c + 8 <= lim) {
        if constexpr (DT == SPECV_BF16) {
            uint4 q = ld_stream_v4(row + c * 2);
            v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
            v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
        } else {
            uint4 q0 = ld_stream_v4(row + c * 4), q1 = ld_stream_v4(row + c * 4 + 16);
            v[0] = __uint_as_float(q0.x); v[1] = __uint_as_float(q0.y);
            v[2] = __uint_as_float(q0.z); v[3] = __uint_as_float(q0.w);
            v[4] = __uint_as_float(q1.x); v[5] = __uint_as_float(q1.y);
            v[6] = __uint_as_float(q1.z); v[7] = __uint_as_float(q1.w);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = (c + e < lim) ? ld_elem<DT>(row, c + e) : -INFINITY;
    }
}

template <int TDT, int DDT>
struct RowPair {
    const char* trow;
    const char* drow;
    bool tal, dal, probs;
    int64_t lim;
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

// Weights of the 8 columns c..c+7 of this lane: residual, or p's weight only.
template <int TDT, int DDT>
__device__ __forceinline__ void lane_weights(const RowPair<TDT, DDT>& rp, int64_t c, int mode, df It, df Id,
                                             const Exp2Table& tab, df (&w)[8]) {
    float lt[8];
    load8<TDT>(rp.trow, c, rp.lim, rp.tal, lt);
    if (mode == kTaskResidual) {
        float ld[8];
        load8<DDT>(rp.drow, c, rp.lim, rp.dal, ld);
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = resid_weight(rp.wt(lt[e], tab), rp.wd(ld[e], tab), It, Id);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = rp.wt(lt[e], tab);
    }
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

// Total of a lane's 8 weights.
__device__ __forceinline__ df lane_total(const df (&w)[8]) {
    df acc{0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 8; ++e) acc_add(acc, w[e]);
    return df_norm(acc);
}

// Pass A: exact normalisers of both rows over this CTA's chunk (block sums,
// valid in warp 0).
template <int TDT, int DDT>
__device__ void chunk_norms(const RowPair<TDT, DDT>& rp, int64_t cs, int64_t ce, SampSmem& sm, df& St, df& Sd) {
    df at{0.f, 0.f}, ad{0.f, 0.f};
    for (int64_t c = cs + (int64_t)threadIdx.x * 8; c < ce; c += (int64_t)blockDim.x * 8) {
        float lt[8], ld[8];
        load8<TDT>(rp.trow, c, rp.lim, rp.tal, lt);
        load8<DDT>(rp.drow, c, rp.lim, rp.dal, ld);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            acc_add(at, rp.wt(lt[e], sm.tab));
            acc_add(ad, rp.wd(ld[e], sm.tab));
        }
    }
    at = warp_sum_df(df_norm(at));
    ad = warp_sum_df(df_norm(ad));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        sm.red_t[warp] = at;
        sm.red_d[warp] = ad;
    }
    __syncthreads();
    if (warp == 0) {
        at = lane < kWarps ? sm.red_t[lane] : df{0.f, 0.f};
        ad = lane < kWarps ? sm.red_d[lane] : df{0.f, 0.f};
        at = warp_sum_df(at);
        ad = warp_sum_df(ad);
    }
    St = at;
    Sd = ad;
}

// Pass B: tile sums in index order into smem; returns the chunk total (warp 0).
template <int TDT, int DDT>
__device__ df chunk_tiles(const RowPair<TDT, DDT>& rp, int64_t cs, int ntiles, int mode, df It, df Id,
                          SampSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int ti = warp; ti < ntiles; ti += kWarps) {
        df w[8];
        lane_weights(rp, cs + (int64_t)ti * kTile + lane * 8, mode, It, Id, sm.tab, w);
        const df incl = warp_scan_df(lane_total(w));
        if (lane == 31) sm.tile_sum[ti] = incl;
    }
    __syncthreads();
    df z{0.f, 0.f};
    if (warp == 0) {
        for (int ti = lane; ti < ntiles; ti += 32) z = df_add(z, sm.tile_sum[ti]);
        z = warp_sum_df(z);
    }
    return z;
}

// Publish thread 0's value into slot c of every CTA in the cluster.
__device__ __forceinline__ void cluster_publish(df* slots, uint32_t c, int ns, df v) {
    if (threadIdx.x == 0)
        for (int r = 0; r < ns; ++r) {
            st_cluster_f32(&slots[c].hi, r, v.hi);
            st_cluster_f32(&slots[c].lo, r, v.lo);
        }
    cluster_sync_all();
}

template <int TDT, int DDT>
__global__ void __launch_bounds__(kSampThreads) sampler_kernel(SampleParams p) {
    __shared__ SampSmem sm;
    pdl_wait_primary();  // tasks are written by the streaming pass

    const int32_t b = blockIdx.x / p.nsplit;
    const uint32_t c = cluster_ctarank();
    const SampleTask t = p.tasks_in[b];
    if (t.mode == kTaskNone) return;  // uniform across the cluster: nobody reaches a barrier
    exp2_table_init(sm.tab);

    const int64_t cs = (int64_t)c * p.vchunk;
    const int64_t ce = min(p.V, cs + p.vchunk);
    const int ntiles = ce > cs ? (int)((ce - cs + kTile - 1) / kTile) : 0;
    constexpr int te = TDT == SPECV_F32 ? 4 : 2, de = DDT == SPECV_F32 ? 4 : 2;
    RowPair<TDT, DDT> rp;
    rp.trow = (const char*)p.tgt + t.trow * p.V * te;
    rp.drow = t.drow >= 0 ? (const char*)p.dft + t.drow * p.V * de : rp.trow;
    rp.tal = ((uintptr_t)rp.trow & 15u) == 0;
    rp.dal = ((uintptr_t)rp.drow & 15u) == 0;
    rp.lim = ce;
    rp.probs = t.probs != 0;
    rp.mt = t.mt;
    rp.md = t.md;
    rp.k = df{t.k_hi, t.k_lo};
    __syncthreads();  // exp2 table ready

    int mode = t.mode;
    df It{1.f, 0.f}, Id{1.f, 0.f};
    if (mode == kTaskResidual) {
        df St, Sd;
        chunk_norms(rp, cs, ce, sm, St, Sd);
        cluster_publish(sm.norm_t, c, p.nsplit, St);
        cluster_publish(sm.norm_d, c, p.nsplit, Sd);
        df Tt{0.f, 0.f}, Td{0.f, 0.f};
        for (int r = 0; r < p.nsplit; ++r) {
            Tt = df_add(Tt, sm.norm_t[r]);
            Td = df_add(Td, sm.norm_d[r]);
        }
        It = df_recip(Tt);
        Id = df_recip(Td);
        if (c == 0 && threadIdx.x == 0) {
            p.tasks[b].st_hi = Tt.hi;
            p.tasks[b].st_lo = Tt.lo;
            p.tasks[b].sd_hi = Td.hi;
            p.tasks[b].sd_lo = Td.lo;
        }
    }

    df zc = chunk_tiles(rp, cs, ntiles, mode, It, Id, sm);
    cluster_publish(sm.zc, c, p.nsplit, zc);
    const df* zs = sm.zc;
    df Z{0.f, 0.f}, lo{0.f, 0.f};
    for (int r = 0; r < p.nsplit; ++r) {
        if (r == (int)c) lo = Z;
        Z = df_add(Z, zs[r]);
    }
    if (mode == kTaskResidual && !df_pos(Z)) {
        // p_i == q_i to rounding: draw from p_i instead
        mode = kTaskBonus;
        __syncthreads();
        zc = chunk_tiles(rp, cs, ntiles, mode, It, Id, sm);
        cluster_publish(sm.zc2, c, p.nsplit, zc);
        zs = sm.zc2;
        Z = df{0.f, 0.f};
        for (int r = 0; r < p.nsplit; ++r) {
            if (r == (int)c) lo = Z;
            Z = df_add(Z, zs[r]);
        }
    }
    if (c == 0 && threadIdx.x == 0) {
        p.tasks[b].z_hi = Z.hi;
        p.tasks[b].z_lo = Z.lo;
    }
    // threshold u * Z; u has 24 significant bits
    const df thr = df_add(two_prod(t.u, Z.hi), df{__fmul_rn(t.u, Z.lo), 0.f});
    const df hi_edge = df_add(lo, zs[c]);
    bool owner = !df_gt(lo, thr) && df_gt(hi_edge, thr) && df_pos(zs[c]);
    bool fallback = false;
    if (!df_gt(Z, thr)) {
        int last = -1;
        for (int r = 0; r < p.nsplit; ++r)
            if (df_pos(zs[r])) last = r;
        owner = (last == (int)c);
        fallback = true;
    }
    if (!owner) return;

    // locate the tile holding the crossing: one warp, 32 tiles per step
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int sel = -1;
        df base = lo;
        if (!fallback) {
            df run = lo;
            for (int t0 = 0; t0 < ntiles && sel < 0; t0 += 32) {
                const int ti = t0 + lane;
                const df v = ti < ntiles ? sm.tile_sum[ti] : df{0.f, 0.f};
                const df end = df_add(run, warp_scan_df(v));
                const unsigned hit = __ballot_sync(0xffffffffu, ti < ntiles && df_gt(end, thr));
                if (hit) {
                    const int src = __ffs(hit) - 1;
                    sel = t0 + src;
                    base = shfl_df(df_sub(end, v), src);  // run + exclusive prefix
                } else {
                    run = shfl_df(end, 31);
                }
            }
        }
        int mark = 0;
        if (sel < 0) {  // rounding left no crossing here: the last tile with mass
            for (int hi_t = ntiles - 1; hi_t >= 0 && sel < 0; hi_t -= 32) {
                const int ti = hi_t - lane;
                const unsigned pos = __ballot_sync(0xffffffffu, ti >= 0 && df_pos(sm.tile_sum[ti >= 0 ? ti : 0]));
                if (pos) sel = hi_t - (__ffs(pos) - 1);
            }
            mark = 1;
        }
        if (lane == 0) {
            sm.sel_tile = sel;
            sm.sel_base = mark ? df{NAN, 0.f} : base;  // NaN: no comparison succeeds
        }
    }
    __syncthreads();
    if (threadIdx.x >= 32 || sm.sel_tile < 0) return;

    // one warp rescans the selected tile in index order
    const int lane = threadIdx.x;
    const int64_t col0 = cs + (int64_t)sm.sel_tile * kTile + lane * 8;
    df w[8];
    lane_weights(rp, col0, mode, It, Id, sm.tab, w);
    df cum[8];
    df acc{0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        acc_add(acc, w[e]);
        cum[e] = df_norm(acc);
    }
    const df incl = warp_scan_df(cum[7]);
    df excl = shfl_up_df(incl, 1);
    if (lane == 0) excl = df{0.f, 0.f};
    const df base = sm.sel_base;
    int hit = -1, lastpos = -1;
#pragma unroll
    for (int e = 7; e >= 0; --e) {
        if (df_gt(df_add(base, df_add(excl, cum[e])), thr)) hit = e;
        if (lastpos < 0 && df_pos(w[e])) lastpos = e;
    }
    const unsigned hm = __ballot_sync(0xffffffffu, hit >= 0);
    int64_t tok = -1;
    if (hm) {
        const int src = __ffs(hm) - 1;
        const int e = __shfl_sync(0xffffffffu, hit, src);
        tok = cs + (int64_t)sm.sel_tile * kTile + src * 8 + e;
    } else {
        const unsigned pm = __ballot_sync(0xffffffffu, lastpos >= 0);
        if (pm) {
            const int src = 31 - __clz(pm);
            const int e = __shfl_sync(0xffffffffu, lastpos, src);
            tok = cs + (int64_t)sm.sel_tile * kTile + src * 8 + e;
        }
    }
    if (lane == 0 && tok >= 0) p.out_tokens[t.out_slot] = (int32_t)tok;
}

template <int TDT, int DDT>
cudaError_t launch_typed(const SampleParams& p, int32_t B, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * p.nsplit));
    cfg.blockDim = dim3(kSampThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = (unsigned)p.nsplit;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
    if (pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, sampler_kernel<TDT, DDT>, p);
}

}  // namespace

int sampler_nsplit(int device, int64_t B, int64_t V) {
    int sms = 152;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    int64_t n = (4 * (int64_t)sms + B - 1) / B;
    const int64_t by_v = V / 4096;  // keep chunks of at least 4096 columns
    if (n > by_v) n = by_v;
    const int64_t need = (V + (int64_t)kMaxTilesPerCta * kTile - 1) / ((int64_t)kMaxTilesPerCta * kTile);
    if (n < need) n = need;
    if (n < 1) n = 1;
    if (n > kMaxCluster) n = kMaxCluster;
    return (int)n;
}

cudaError_t launch_sampler(const SampleParams& p, int32_t B, cudaStream_t s, bool pdl) {
    cudaError_t e;
    if (p.tdt == SPECV_BF16 && p.ddt == SPECV_BF16)
        e = launch_typed<SPECV_BF16, SPECV_BF16>(p, B, s, pdl);
    else if (p.tdt == SPECV_BF16)
        e = launch_typed<SPECV_BF16, SPECV_F32>(p, B, s, pdl);
    else if (p.ddt == SPECV_BF16)
        e = launch_typed<SPECV_F32, SPECV_BF16>(p, B, s, pdl);
    else
        e = launch_typed<SPECV_F32, SPECV_F32>(p, B, s, pdl);
    return e;
}

}  // namespace specv
