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
// no index the last one with positive weight is taken.
//
// Only the selected row pair is re-read. Each sequence gets one thread-block
// cluster of nsplit CTAs; CTA c owns a contiguous column chunk, computes the
// weights tile by tile (a tile = 32 lanes x 8 consecutive columns), keeps each
// tile's sum in shared memory, and publishes its chunk sum to every CTA of the
// cluster through distributed shared memory. Every CTA then forms the same
// prefix over chunk sums; the CTA whose interval holds u * Z walks its tile
// sums and rescans one tile (L2-resident by then) to find the column.
#include <math.h>

#include "common.cuh"

namespace specv {

namespace {

constexpr int kWarps = kSampThreads / 32;

struct SampSmem {
    float tile_sum[kMaxTilesPerCta];
    float zc[kMaxCluster];
    float zc2[kMaxCluster];
    float red[kWarps];
    int32_t sel_tile;
    float sel_base;
    int32_t token;
};

// Eight consecutive columns c..c+7 of a row as floats; columns at or past
// `lim` read as -inf (their weight is masked to zero by the caller).
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

// Weight of one column. Explicit round-to-nearest intrinsics keep the value
// bit-identical between the summing pass and the rescan.
__device__ __forceinline__ float weight_p(float lt, const SampleTask& t) {
    return __fmul_rn(ex2(__fmaf_rn(lt, t.kt, -t.mt)), t.inv_st);
}
__device__ __forceinline__ float weight_resid(float lt, float ld, const SampleTask& t) {
    const float pt = weight_p(lt, t);
    const float qd = t.probs ? __fmul_rn(ld, t.inv_sd) : __fmul_rn(ex2(__fmaf_rn(ld, t.kd, -t.md)), t.inv_sd);
    return fmaxf(__fsub_rn(pt, qd), 0.f);
}

template <int TDT, int DDT>
struct RowPair {
    const char* trow;
    const char* drow;
    bool tal, dal;
    int64_t lim;  // one past the last column of this CTA's chunk
    // weights of the 8 columns c..c+7 owned by this lane of a tile
    __device__ __forceinline__ void weights(int64_t c, bool resid, const SampleTask& t, float (&w)[8]) const {
        float lt[8];
        load8<TDT>(trow, c, lim, tal, lt);
        if (resid) {
            float ld[8];
            load8<DDT>(drow, c, lim, dal, ld);
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = (c + e < lim) ? weight_resid(lt[e], ld[e], t) : 0.f;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = (c + e < lim) ? weight_p(lt[e], t) : 0.f;
        }
    }
};

// Inclusive warp scan of the lane sums (Hillis-Steele); also returns the
// lane's exclusive prefix as the inclusive value of the lane below.
__device__ __forceinline__ void warp_scan(float x, float& incl, float& excl) {
    const int lane = threadIdx.x & 31;
    incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl = __fadd_rn(incl, y);
    }
    excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
}

// Sum of a tile as the rescan will see it at its last column: the exclusive
// prefix of lane 31 plus lane 31's own sequential sum.
__device__ __forceinline__ float tile_total(const float (&w)[8]) {
    float ls = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ls = __fadd_rn(ls, w[e]);
    float incl, excl;
    warp_scan(ls, incl, excl);
    const float t = __fadd_rn(excl, ls);
    return __shfl_sync(0xffffffffu, t, 31);
}

// Pass over this CTA's tiles: tile sums into smem; returns their in-order sum.
template <int TDT, int DDT>
__device__ float chunk_pass(const RowPair<TDT, DDT>& rp, int64_t cs, int ntiles, bool resid, const SampleTask& t,
                            SampSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int ti = warp; ti < ntiles; ti += 2 * kWarps) {
        const int tj = ti + kWarps;
        float w0[8], w1[8];
        rp.weights(cs + (int64_t)ti * kTile + lane * 8, resid, t, w0);
        if (tj < ntiles) rp.weights(cs + (int64_t)tj * kTile + lane * 8, resid, t, w1);
        const float s0 = tile_total(w0);
        if (lane == 0) sm.tile_sum[ti] = s0;
        if (tj < ntiles) {
            const float s1 = tile_total(w1);
            if (lane == 0) sm.tile_sum[tj] = s1;
        }
    }
    __syncthreads();
    float z = 0.f;
    if (threadIdx.x == 0)
        for (int ti = 0; ti < ntiles; ++ti) z = __fadd_rn(z, sm.tile_sum[ti]);
    return z;  // thread 0
}

template <int TDT, int DDT>
__global__ void __launch_bounds__(kSampThreads) sampler_kernel(SampleParams p) {
    __shared__ SampSmem sm;
    pdl_wait_primary();  // tasks are written by the streaming pass

    const int32_t b = blockIdx.x / p.nsplit;
    const uint32_t c = cluster_ctarank();
    const SampleTask t = p.tasks_in[b];
    if (t.mode == kTaskNone) return;  // uniform across the cluster: nobody reaches a barrier

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
    bool resid = t.mode == kTaskResidual;

    // chunk sums -> every CTA of the cluster
    float zc = chunk_pass(rp, cs, ntiles, resid, t, sm);
    if (threadIdx.x == 0)
        for (int r = 0; r < p.nsplit; ++r) st_cluster_f32(&sm.zc[c], r, zc);
    cluster_sync_all();
    float pre = 0.f, Z = 0.f, lo = 0.f;
    for (int r = 0; r < p.nsplit; ++r) {
        if (r == (int)c) lo = pre;
        pre = __fadd_rn(pre, sm.zc[r]);
    }
    Z = pre;
    const float* zs = sm.zc;
    if (resid && !(Z > 0.f)) {
        // p_i == q_i to rounding: draw from p_i instead
        resid = false;
        __syncthreads();
        zc = chunk_pass(rp, cs, ntiles, resid, t, sm);
        if (threadIdx.x == 0)
            for (int r = 0; r < p.nsplit; ++r) st_cluster_f32(&sm.zc2[c], r, zc);
        cluster_sync_all();
        pre = 0.f;
        for (int r = 0; r < p.nsplit; ++r) {
            if (r == (int)c) lo = pre;
            pre = __fadd_rn(pre, sm.zc2[r]);
        }
        Z = pre;
        zs = sm.zc2;
    }
    const float thr = __fmul_rn(t.u, Z);
    const float hi = __fadd_rn(lo, zs[c]);
    bool owner = (lo <= thr) && (thr < hi);
    bool fallback = false;
    if (!(thr < Z)) {
        // rounding put u * Z at or past the total: last chunk with positive mass
        int last = -1;
        for (int r = 0; r < p.nsplit; ++r)
            if (zs[r] > 0.f) last = r;
        owner = (last == (int)c);
        fallback = true;
    }
    if (c == 0 && threadIdx.x == 0) p.tasks[b].z = Z;
    if (!owner) return;

    // locate the tile holding the crossing
    if (threadIdx.x == 0) {
        int sel = -1;
        float run = lo, base = lo;
        if (!fallback) {
            for (int ti = 0; ti < ntiles; ++ti) {
                const float nxt = __fadd_rn(run, sm.tile_sum[ti]);
                if (nxt > thr) {
                    sel = ti;
                    base = run;
                    break;
                }
                run = nxt;
            }
        }
        if (sel < 0) {  // no crossing by this CTA's own running sum: last tile with mass
            for (int ti = ntiles - 1; ti >= 0; --ti)
                if (sm.tile_sum[ti] > 0.f) {
                    sel = ti;
                    break;
                }
            base = NAN;  // no comparison succeeds: the last-positive rule applies inside the tile
        }
        sm.sel_tile = sel;
        sm.sel_base = base;
    }
    __syncthreads();
    if (threadIdx.x >= 32 || sm.sel_tile < 0) return;

    // one warp rescans the selected tile in index order
    const int lane = threadIdx.x;
    const int64_t col0 = cs + (int64_t)sm.sel_tile * kTile + lane * 8;
    float w[8];
    rp.weights(col0, resid, t, w);
    float cum[8], ls = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        ls = __fadd_rn(ls, w[e]);
        cum[e] = ls;
    }
    float incl, excl;
    warp_scan(ls, incl, excl);
    const float base = sm.sel_base;
    int hit = -1, lastpos = -1;
#pragma unroll
    for (int e = 7; e >= 0; --e) {
        if (__fadd_rn(base, __fadd_rn(excl, cum[e])) > thr) hit = e;
        if (lastpos < 0 && w[e] > 0.f) lastpos = e;
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
