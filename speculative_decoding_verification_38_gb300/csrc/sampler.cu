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
// cluster of nsplit CTAs, CTA c owning a contiguous column chunk, which it
// stages into shared memory with one TMA bulk copy per row (rows whose chunk
// is not 16-byte aligned are read from global memory instead). Then:
//   pass A (residual only): the exact normalisers S = sum_j 2^((l_j - l_max) k)
//     of both rows, reduced over the cluster through distributed shared memory;
//   pass B: the weights r_j (= max(0, p_j - q_j), or p_j's weight for a bonus)
//     tile by tile (a tile = 32 lanes x 32 consecutive columns), each tile's
//     sum kept in shared memory; chunk sums are exchanged across the cluster so
//     every CTA knows Z and where its chunk starts in the CDF;
//   the CTA whose interval holds u * Z finds the tile with one warp-wide
//   prefix over its tile sums and rescans that tile to find the column.
// Weights, sums and prefixes are double-float (precise.cuh), so the pick
// matches a float64 evaluation except within ~1e-10 of a CDF edge.
#include <math.h>

#include <mutex>

#include "precise.cuh"

namespace specv {

namespace {

constexpr int kWarps = kSampThreads / 32;
constexpr int kQCap = 128;  // entries per warp queue (power of two)

struct SampSmem {
    Exp2Table tab;
    df tile_sum[kMaxTilesPerCta];
    df norm_t[kMaxCluster], norm_d[kMaxCluster];
    df zc[kMaxCluster], zc2[kMaxCluster];
    df red_t[kWarps], red_d[kWarps];
    float okflag[kMaxCluster];
    int32_t q[kWarps][kQCap];  // per-warp queue of heavy items awaiting dense evaluation
    uint64_t bar;
    int32_t sel_tile;
    df sel_base;
};

// One row's chunk: column j (0-based within the chunk) lives in shared memory
// at s + j * esz when staged, else in global memory at g + j * esz.
struct Src {
    const char* g;
    uint32_t s;
    int64_t n;  // columns in the chunk
    bool staged, al;
};

template <int DT>
__device__ __forceinline__ float src_elem(const Src& r, int64_t j) {
    if (r.staged) {
        if constexpr (DT == SPECV_BF16) {
            unsigned short h;
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(r.s + (uint32_t)(j * 2)));
            return __uint_as_float(((uint32_t)h) << 16);
        } else {
            float f;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(f) : "r"(r.s + (uint32_t)(j * 4)));
            return f;
        }
    }
    return ld_elem<DT>(r.g, j);
}

__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// Columns j..j+7 of a chunk as floats; columns past the chunk read as -inf
// (weight 0). j is a multiple of 8.
template <int DT>
__device__ __forceinline__ void src_load8(const Src& r, int64_t j, float (&v)[8]) {
    if (j + 8 <= r.n && (r.staged || r.al)) {
        if constexpr (DT == SPECV_BF16) {
            const uint4 q = r.staged ? lds_v4(r.s + (uint32_t)(j * 2)) : ld_stream_v4(r.g + j * 2);
            v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
            v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
        } else {
            uint4 q0, q1;
            if (r.staged) {
                q0 = lds_v4(r.s + (uint32_t)(j * 4));
                q1 = lds_v4(r.s + (uint32_t)(j * 4 + 16));
            } else {
                q0 = ld_stream_v4(r.g + j * 4);
                q1 = ld_stream_v4(r.g + j * 4 + 16);
            }
            v[0] = __uint_as_float(q0.x); v[1] = __uint_as_float(q0.y);
            v[2] = __uint_as_float(q0.z); v[3] = __uint_as_float(q0.w);
            v[4] = __uint_as_float(q1.x); v[5] = __uint_as_float(q1.y);
            v[6] = __uint_as_float(q1.z); v[7] = __uint_as_float(q1.w);
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

// Weights of the 8 chunk columns j..j+7: residual, or p's weight only.
template <int TDT, int DDT>
__device__ __forceinline__ void weights8(const RowPair<TDT, DDT>& rp, int64_t j, int mode, df It, df Id,
                                         const Exp2Table& tab, df (&w)[8]) {
    float lt[8];
    src_load8<TDT>(rp.t, j, lt);
    if (mode == kTaskResidual) {
        float ld[8];
        src_load8<DDT>(rp.d, j, ld);
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = resid_weight(rp.wt(lt[e], tab), rp.wd(ld[e], tab), It, Id);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = rp.wt(lt[e], tab);
    }
}

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

// Pass A item: bit 30 = draft row, low bits = chunk column.
template <int TDT, int DDT>
__device__ __forceinline__ void norm_item(const RowPair<TDT, DDT>& rp, int32_t it, const Exp2Table& tab, df& at,
                                          df& ad) {
    const int64_t j = it & 0x3fffffff;
    if (it & (1 << 30)) {
        const float l = src_elem<DDT>(rp.d, j);
        acc_add(ad, rp.probs ? df{l, 0.f} : heavy_logit_weight<DDT == SPECV_F32>(l, rp.md, rp.k, tab));
    } else {
        acc_add(at, heavy_logit_weight<TDT == SPECV_F32>(src_elem<TDT>(rp.t, j), rp.mt, rp.k, tab));
    }
}

// Pass A: exact normalisers of both rows over this CTA's chunk (block sums,
// valid in warp 0). Each warp covers 256 contiguous columns per step.
template <int TDT, int DDT>
__device__ void chunk_norms(const RowPair<TDT, DDT>& rp, int64_t n, SampSmem& sm, df& St, df& Sd) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* q = sm.q[warp];
    uint32_t head = 0, tail = 0;
    df at{0.f, 0.f}, ad{0.f, 0.f};
    for (int64_t base = (int64_t)warp * 256; base < n; base += (int64_t)kWarps * 256) {
        const int64_t j = base + lane * 8;
        float lt[8], ld[8];
        src_load8<TDT>(rp.t, j, lt);
        src_load8<DDT>(rp.d, j, ld);
        float gt = 0.f, gd = 0.f;
        uint32_t m = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            bool h;
            const float w = light_weight<TDT == SPECV_F32>(lt[e], rp.mt, rp.k, h);
            if (h) m |= 1u << e; else gt = __fadd_rn(gt, w);
            if (rp.probs) {
                const float v = ld[e] > -INFINITY ? ld[e] : 0.f;
                if (v > 1.220703125e-4f) m |= 1u << (8 + e); else gd = __fadd_rn(gd, v);
            } else {
                const float wd = light_weight<DDT == SPECV_F32>(ld[e], rp.md, rp.k, h);
                if (h) m |= 1u << (8 + e); else gd = __fadd_rn(gd, wd);
            }
        }
        acc_add(at, light_sum_df(gt, kEx2LightBias));
        acc_add(ad, light_sum_df(gd, rp.probs ? 0.f : kEx2LightBias));
        const auto code = [&](int b) { return (int32_t)((j + (b & 7)) | (b >= 8 ? (1 << 30) : 0)); };
        if (!wq_push(q, head, tail, m, code)) {  // queue full: evaluate in place
            while (m) {
                const int b = __ffs(m) - 1;
                m &= m - 1;
                norm_item(rp, code(b), sm.tab, at, ad);
            }
        }
        while (tail - head >= 32) {
            norm_item(rp, q[(head + lane) & (kQCap - 1)], sm.tab, at, ad);
            head += 32;
            __syncwarp();
        }
    }
    if (lane < (int)(tail - head)) norm_item(rp, q[(head + lane) & (kQCap - 1)], sm.tab, at, ad);
    at = warp_sum_df(df_norm(at));
    ad = warp_sum_df(df_norm(ad));
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
__device__ df chunk_tiles(const RowPair<TDT, DDT>& rp, int ntiles, int mode, df It, df Id, float cl,
                          SampSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int ti = warp; ti < ntiles; ti += kWarps) {
        const df tot = warp_sum_df(lane_tile_sum(rp, (int64_t)ti * kTile, mode, It, Id, cl, sm));
        if (lane == 0) sm.tile_sum[ti] = tot;
    }
    __syncthreads();
    df z{0.f, 0.f};
    if (warp == 0) {
        for (int ti = lane; ti < ntiles; ti += 32) z = df_add(z, sm.tile_sum[ti]);
        z = warp_sum_df(z);
    }
    return z;
}

// One warp walks the selected tile in index order from CDF position `base`
// and returns the first chunk column whose running sum exceeds thr (or, if
// rounding leaves none, the last column with weight; -1 if the tile has none).
template <int TDT, int DDT>
__device__ int64_t rescan_tile(const RowPair<TDT, DDT>& rp, int64_t tile_j, int mode, df It, df Id, float cl,
                               df base, df thr, const Exp2Table& tab) {
    const int lane = threadIdx.x & 31;
    df run = base;
    int64_t last = -1;
#pragma unroll 1
    for (int g = 0; g < kGroups; ++g) {
        df w[8];
        const int64_t j0 = tile_j + g * 256 + lane * 8;
        weights8(rp, j0, mode, It, Id, tab, w);
        // this lane's prefix at each of its 8 columns, then the warp-wide prefix
        df pre[8];
        float light = 0.f;
        df heavy{0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (is_heavy(w[e]))
                acc_add(heavy, w[e]);
            else
                light = __fadd_rn(light, w[e].hi);
            pre[e] = df_add(df_norm(heavy), light_sum_df(light, cl));
        }
        const df incl = warp_scan_df(pre[7]);
        df excl = shfl_up_df(incl, 1);
        if (lane == 0) excl = df{0.f, 0.f};
        const df start = df_add(run, excl);
        int hit = -1, lp = -1;
#pragma unroll
        for (int e = 7; e >= 0; --e) {
            if (df_gt(df_add(start, pre[e]), thr)) hit = e;
            if (lp < 0 && df_pos(w[e])) lp = e;
        }
        const unsigned hm = __ballot_sync(0xffffffffu, hit >= 0);
        if (hm) {
            const int src = __ffs(hm) - 1;
            return tile_j + g * 256 + src * 8 + __shfl_sync(0xffffffffu, hit, src);
        }
        const unsigned pm = __ballot_sync(0xffffffffu, lp >= 0);
        if (pm) {
            const int src = 31 - __clz(pm);
            last = tile_j + g * 256 + src * 8 + __shfl_sync(0xffffffffu, lp, src);
        }
        run = df_add(run, shfl_df(incl, 31));
    }
    return last;
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

// Stage one row chunk (n columns of esz bytes at g) into shared memory at s:
// a bulk copy of the 16-byte aligned body (thread 0), plain loads for the
// short tail.
__device__ __forceinline__ void stage_row(const char* g, char* s, int64_t n, int esz, uint64_t* bar) {
    const uint32_t bytes = (uint32_t)(n * esz);
    const uint32_t body = bytes & ~15u;
    if (threadIdx.x == 0 && body) bulk_g2s(s, g, body, bar);
    for (uint32_t b = body + threadIdx.x; b < bytes; b += blockDim.x) s[b] = __ldg(g + b);
}

template <int TDT, int DDT>
__global__ void __launch_bounds__(kSampThreads) sampler_kernel(SampleParams p) {
    __shared__ SampSmem sm;
    extern __shared__ __align__(128) char dyn[];
    pdl_wait_primary();  // tasks are written by the streaming pass

    const int32_t b = blockIdx.x / p.nsplit;
    const uint32_t c = cluster_ctarank();
    const SampleTask t = p.tasks_in[b];
    if (t.mode == kTaskNone) return;  // uniform across the cluster: nobody reaches a barrier
    exp2_table_init(sm.tab);

    const int64_t cs = (int64_t)c * p.vchunk;
    const int64_t ce = min(p.V, cs + p.vchunk);
    const int64_t n = ce > cs ? ce - cs : 0;
    const int ntiles = (int)((n + kTile - 1) / kTile);
    constexpr int te = TDT == SPECV_F32 ? 4 : 2, de = DDT == SPECV_F32 ? 4 : 2;
    const bool resid0 = t.mode == kTaskResidual;
    RowPair<TDT, DDT> rp;
    rp.t.g = (const char*)p.tgt + (t.trow * p.V + cs) * te;
    rp.d.g = resid0 ? (const char*)p.dft + (t.drow * p.V + cs) * de : rp.t.g;
    rp.t.n = rp.d.n = n;
    rp.t.al = ((uintptr_t)rp.t.g & 15u) == 0;
    rp.d.al = ((uintptr_t)rp.d.g & 15u) == 0;
    rp.t.staged = p.stage_bytes > 0 && rp.t.al && n * te <= (int64_t)p.stage_bytes;
    rp.d.staged = resid0 && p.stage_bytes > 0 && rp.d.al && n * de <= (int64_t)p.stage_bytes;
    rp.t.s = smem_addr(dyn);
    rp.d.s = smem_addr(dyn + p.stage_bytes);
    rp.probs = t.probs != 0;
    rp.mt = t.mt;
    rp.md = t.md;
    rp.k = df{t.k_hi, t.k_lo};

    // stage the chunk of both rows into shared memory
    bool ok = true;
    if (rp.t.staged || rp.d.staged) {
        if (threadIdx.x == 0) {
            mbar_init(&sm.bar, 1);
            fence_barrier_init();
        }
        __syncthreads();
        const uint32_t tb = rp.t.staged ? (uint32_t)(n * te) & ~15u : 0u;
        const uint32_t db = rp.d.staged ? (uint32_t)(n * de) & ~15u : 0u;
        if (threadIdx.x == 0) mbar_arrive_expect_tx(&sm.bar, tb + db);
        if (rp.t.staged) stage_row(rp.t.g, dyn, n, te, &sm.bar);
        if (rp.d.staged) stage_row(rp.d.g, dyn + p.stage_bytes, n, de, &sm.bar);
        if (!mbar_wait_bounded(&sm.bar, 0, kWaitLimit)) {
            ok = false;
            mbar_wait_bounded(&sm.bar, 0, kWaitLimit);  // let copies in flight land before leaving
        }
    }
    ok = __syncthreads_and(ok);  // also publishes the plain-load tails
    if (threadIdx.x == 0)
        for (int r = 0; r < p.nsplit; ++r) st_cluster_f32(&sm.okflag[c], r, ok ? 1.f : 0.f);
    cluster_sync_all();
    bool all_ok = true;
    for (int r = 0; r < p.nsplit; ++r) all_ok = all_ok && sm.okflag[r] > 0.f;
    if (!all_ok) {  // the whole cluster gives up together
        if (c == 0 && threadIdx.x == 0) {
            atomicOr(p.err, 1u);
            if (p.seq_status) p.seq_status[b] = kSeqTimeout;
        }
        return;
    }

    int mode = t.mode;
    df It{1.f, 0.f}, Id{1.f, 0.f};
    if (mode == kTaskResidual) {
        df St, Sd;
        chunk_norms(rp, n, sm, St, Sd);
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

    // light-sum correction of the sampling weights: both rows' light weights
    // carry the same SFU bias unless the draft is given as probabilities
    float cl = (mode == kTaskResidual && rp.probs) ? 0.f : kEx2LightBias;
    df zc = chunk_tiles(rp, ntiles, mode, It, Id, cl, sm);
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
        cl = kEx2LightBias;
        __syncthreads();
        zc = chunk_tiles(rp, ntiles, mode, It, Id, cl, sm);
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
    const int64_t jt = rescan_tile(rp, (int64_t)sm.sel_tile * kTile, mode, It, Id, cl, sm.sel_base, thr, sm.tab);
    const int64_t tok = jt >= 0 ? cs + jt : -1;
    if (lane == 0 && tok >= 0) p.out_tokens[t.out_slot] = (int32_t)tok;
}

template <int TDT, int DDT>
cudaError_t launch_typed(const SampleParams& p, int32_t B, cudaStream_t s, bool pdl) {
    static bool attr_done = false;  // per instantiation
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(sampler_kernel<TDT, DDT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSampStageMax);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * p.nsplit));
    cfg.blockDim = dim3(kSampThreads);
    cfg.dynamicSmemBytes = 2 * (size_t)p.stage_bytes;
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

namespace {

template <int TDT, int DDT>
int active_clusters(int nsplit, uint32_t stage_bytes) {
    static bool attr_done = false;  // per instantiation
    if (!attr_done) {
        if (cudaFuncSetAttribute(sampler_kernel<TDT, DDT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSampStageMax) != cudaSuccess)
            return 0;
        attr_done = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nsplit);
    cfg.blockDim = dim3(kSampThreads);
    cfg.dynamicSmemBytes = 2 * (size_t)stage_bytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)nsplit;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)sampler_kernel<TDT, DDT>, &cfg) != cudaSuccess) return 0;
    return n;
}

int active_clusters_rt(int tdt, int ddt, int nsplit, uint32_t stage_bytes) {
    if (tdt == SPECV_BF16 && ddt == SPECV_BF16) return active_clusters<SPECV_BF16, SPECV_BF16>(nsplit, stage_bytes);
    if (tdt == SPECV_BF16) return active_clusters<SPECV_BF16, SPECV_F32>(nsplit, stage_bytes);
    if (ddt == SPECV_BF16) return active_clusters<SPECV_F32, SPECV_BF16>(nsplit, stage_bytes);
    return active_clusters<SPECV_F32, SPECV_F32>(nsplit, stage_bytes);
}

struct PlanKey {
    int device, tdt, ddt;
    int64_t B, V;
};
std::mutex g_plan_mu;
PlanKey g_plan_key[8];
SampPlan g_plan_val[8];
int g_plan_n = 0, g_plan_next = 0;

}  // namespace

// CTAs per sequence (cluster size) and shared-memory staging. Each candidate
// split n keeps chunks of at least 4096 columns and at most kMaxTilesPerCta
// tiles; its cost is the number of waves the B clusters need (from the
// occupancy calculator, which knows how clusters pack into GPCs) times the
// columns each CTA handles. Staging the row pair in shared memory is used
// when it fits and does not cost a wave; the cheapest candidate wins, larger
// splits first on ties. Plans are cached per (device, B, V, dtypes).
SampPlan sampler_plan(int device, int64_t B, int64_t V, int tdt, int ddt) {
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        for (int i = 0; i < g_plan_n; ++i) {
            const PlanKey& k = g_plan_key[i];
            if (k.device == device && k.B == B && k.V == V && k.tdt == tdt && k.ddt == ddt) return g_plan_val[i];
        }
    }
    const int64_t et = tdt == SPECV_F32 ? 4 : 2, ed = ddt == SPECV_F32 ? 4 : 2;
    const int64_t need = (V + (int64_t)kMaxTilesPerCta * kTile - 1) / ((int64_t)kMaxTilesPerCta * kTile);
    int64_t hi = V / 4096;
    if (hi > kMaxCluster) hi = kMaxCluster;
    if (hi < need) hi = need;
    if (hi < 1) hi = 1;
    SampPlan best{};
    double best_cost = -1.0;
    for (int64_t n = hi; n >= (need < 1 ? 1 : need); --n) {
        const int64_t per = (V + n - 1) / n;
        const int64_t vchunk = (per + kTile - 1) / kTile * kTile;
        const int64_t row_bytes = (vchunk * (et > ed ? et : ed) + 15) / 16 * 16;
        for (int staged = 1; staged >= 0; --staged) {
            if (staged && 2 * row_bytes > (int64_t)kSampStageMax) continue;
            const uint32_t sb = staged ? (uint32_t)row_bytes : 0u;
            const int act = active_clusters_rt(tdt, ddt, (int)n, sb);
            if (act < 1) continue;
            const int64_t waves = (B + act - 1) / act;
            const double cost = (double)waves * (double)vchunk;
            if (best_cost < 0.0 || cost < best_cost) {
                best_cost = cost;
                best.nsplit = (int)n;
                best.vchunk = vchunk;
                best.stage_bytes = sb;
            }
        }
    }
    if (best_cost < 0.0) {  // no occupancy answer: one CTA per sequence, direct reads
        best.nsplit = (int)(need < 1 ? 1 : need);
        const int64_t per = (V + best.nsplit - 1) / best.nsplit;
        best.vchunk = (per + kTile - 1) / kTile * kTile;
        best.stage_bytes = 0;
    }
    std::lock_guard<std::mutex> lk(g_plan_mu);
    const int slot = g_plan_n < 8 ? g_plan_n++ : (g_plan_next++ & 7);
    g_plan_key[slot] = PlanKey{device, tdt, ddt, B, V};
    g_plan_val[slot] = best;
    return best;
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
