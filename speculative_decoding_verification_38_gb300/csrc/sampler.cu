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

#include "tile.cuh"

namespace specv {

namespace {

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
    else tile_sums_packed<TDT, DDT>(rp, resid, r_hi, r_lo, TileScratch{sm.q[warp], &sm.nu[sw], sm.uw[sw], &sm.tab},
                                    p.open + item * kOpenCap, WIDE ? warp : 0, WIDE ? warp + 1 : kGroups, acc);
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
    float red_hi[kWarps], red_lo[kWarps], red2_hi[kWarps], red2_lo[kWarps];
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

// Two block sums at once (one pair of barriers).
__device__ __forceinline__ void block_sum_df2(df& x, df& y, DrawSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    x = warp_sum_df(x);
    y = warp_sum_df(y);
    __syncthreads();  // red[] is free
    if (lane == 0) {
        sm.red_hi[warp] = x.hi;
        sm.red_lo[warp] = x.lo;
        sm.red2_hi[warp] = y.hi;
        sm.red2_lo[warp] = y.lo;
    }
    __syncthreads();
    x = y = df{0.f, 0.f};
    for (int i = 0; i < kWarps; ++i) {
        x = df_add(x, df{sm.red_hi[i], sm.red_lo[i]});
        y = df_add(y, df{sm.red2_hi[i], sm.red2_lo[i]});
    }
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
    // the exact normalisers; a thread with one tile (V up to 256 tiles) keeps
    // its whole record for the tile sums below
    df st{0.f, 0.f}, sd{0.f, 0.f};
    const bool one = K == 1;
    float4 r_ab = make_float4(0.f, 0.f, 0.f, 0.f), r_ss = r_ab, r_uu = r_ab;
    int32_t r_nu = 0;
    if (one) {
        if (t0 < t1) {
            const float4* r = reinterpret_cast<const float4*>(recs + t0);
            r_ab = __ldcg(r);
            r_ss = __ldcg(r + 1);
            r_uu = __ldcg(r + 2);
            r_nu = __ldcg(reinterpret_cast<const int32_t*>(r + 3));
            st = df{r_ss.x, r_ss.y};
            sd = df{r_ss.z, r_ss.w};
        }
    } else {
#pragma unroll 1
        for (int ti = t0; ti < t1; ++ti) {
            const float4 ss = __ldcg(reinterpret_cast<const float4*>(recs + ti) + 1);
            st = df_add(st, df{ss.x, ss.y});
            sd = df_add(sd, df{ss.z, ss.w});
        }
    }
    block_sum_df2(st, sd, sm);
    const df St = st, Sd = sd;
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
            const float4 ss = one ? r_ss : __ldcg(r + 1);
            v = df{ss.x, ss.y};
        } else {
            const int32_t nu = one ? r_nu : __ldcg(reinterpret_cast<const int32_t*>(r + 3));
            if (nu > 1) {  // more than one open column: summed again below
                sm.dirty[atomicAdd(&sm.ndirty, 1)] = ti;
                continue;
            }
            const float4 ab = one ? r_ab : __ldcg(r);
            v = resid_of_sums(df{ab.x, ab.y}, df{ab.z, ab.w}, It, Id);
            if (nu == 1) {
                const float4 uu = one ? r_uu : __ldcg(r + 2);
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
            x = warp_sum_df(lane_tile_sum(rp, 0, mode, It, Id, cl, TileScratch{sm.q[warp], nullptr, nullptr, &sm.tab}));
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
