// stats.cu -- the streaming pass of the verify step and its finalize tail.
//
// One persistent grid streams every vocabulary row the decision needs exactly
// once: the target rows p_1..p_{gamma+1} and (sampling) the draft rows
// q_1..q_gamma ("Speculative decoding" (mhtirogla.ai), How it works, steps
// 1-2). The rows are flattened into one element range and cut into equal
// contiguous slices, one per CTA, so every CTA moves the same number of bytes
// whatever the ragged row structure. For each (row, slice) piece a CTA
// produces a partial statistic:
//   sampling, logits rows:  online (m, s), m = max l*k, s = sum 2^(l*k - m),
//                           k = log2(e)/T (the softmax of l/T in base 2);
//   sampling, probs rows:   s = sum q (the row is later divided by it);
//   greedy:                 first-index argmax (value, index), NaN as -inf.
// After its pieces of a sequence are stored, a CTA bumps that sequence's
// arrival counter; the CTA that completes the count merges the sequence's
// partials and runs the decision: the left-to-right accept scan u*q(x) < p(x)
// to the first rejection (same page, step 3; its Code section's division-free
// test), or the greedy match count ("Speculative Decoding" (tokentrails.org),
// One round), plus the KV-length rollback (mhtirogla.ai, step 5). Cross-CTA
// hand-off uses only the counter (no CTA ever waits on another), and the last
// arriver resets the counter for the next call.
#include <math.h>

#include "precise.cuh"

namespace specv {

namespace {

constexpr int kWarps = kStatsThreads / 32;
constexpr int kMaxGamma = 64;
constexpr int kUnroll = 4;

enum Mode { kLogits = 0, kProbs = 1, kArgmax = 2 };

struct Smem {
    float2 red[kWarps];
    int32_t redi[kWarps];
    // finalize
    float2 rs[2 * kMaxGamma + 1];  // merged row stats of the sequence
    float px[kMaxGamma], qx[kMaxGamma];
    float ua[kMaxGamma + 1], us[kMaxGamma + 1];
    int32_t xt[kMaxGamma];
    int32_t pick[kMaxGamma + 1];
    int32_t status, accepted, flag_tok, is_last;
};

__device__ __forceinline__ int64_t tro_at(const StatsParams& p, int64_t b) {
    return p.tro ? p.tro[b] : b * (int64_t)(p.gmax + 1);
}
__device__ __forceinline__ int64_t dro_at(const StatsParams& p, int64_t b) {
    return p.dro ? p.dro[b] : b * (int64_t)p.gmax;
}

// Sequence owning local row lr of the target (draft = false) or draft tensor,
// or -1 if no sequence owns it (offsets that do not start at 0 / end early).
__device__ int32_t seq_of_row(const StatsParams& p, bool draft, int64_t lr) {
    const int64_t* off = draft ? p.dro : p.tro;
    if (!off) {
        int64_t per = draft ? p.gmax : p.gmax + 1;
        int64_t b = lr / per;
        return b < p.B ? (int32_t)b : -1;
    }
    // largest b in [0, B) with off[b] <= lr
    int32_t lo = 0, hi = p.B - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) >> 1;
        if (off[mid] <= lr)
            lo = mid;
        else
            hi = mid - 1;
    }
    if (lr < off[lo] || lr >= off[lo + 1]) return -1;
    return lo;
}

__device__ __forceinline__ uint32_t nseg_of(int64_t r, int64_t V, int64_t chunk) {
    return (uint32_t)(((r + 1) * V - 1) / chunk - (r * V) / chunk + 1);
}

// Number of (row, slice) pieces the streaming pass produces for sequence b.
__device__ uint32_t expected_arrivals(const StatsParams& p, int32_t b) {
    int64_t t0 = max((int64_t)0, tro_at(p, b)), t1 = min(p.rows_t, tro_at(p, b + 1));
    uint32_t n = 0;
    for (int64_t r = t0; r < t1; ++r) n += nseg_of(r, p.V, p.chunk);
    if (!p.greedy) {
        int64_t d0 = max((int64_t)0, dro_at(p, b)), d1 = min(p.rows_d, dro_at(p, b + 1));
        for (int64_t r = d0; r < d1; ++r) n += nseg_of(p.rows_t + r, p.V, p.chunk);
    }
    return n;
}

__device__ __forceinline__ float temp_of(const StatsParams& p, int32_t b) {
    return p.temps ? __ldg(p.temps + b) : p.temperature;
}

// ------------------------------------------------------------ block reductions
__device__ float2 block_ms(float2 v, float k, Smem& sm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float2 w = make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o));
        v = ms_merge(v, w, k);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sm.red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < kWarps ? sm.red[lane] : make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float2 w = make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o));
            v = ms_merge(v, w, k);
        }
    }
    __syncthreads();
    return v;  // valid in thread 0
}

__device__ float block_sum(float v, Smem& sm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sm.red[warp].x = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < kWarps ? sm.red[lane].x : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    }
    __syncthreads();
    return v;
}

__device__ __forceinline__ void am_merge_shfl(float& v, int32_t& i, int o) {
    float w = __shfl_xor_sync(0xffffffffu, v, o);
    int32_t j = __shfl_xor_sync(0xffffffffu, i, o);
    if (am_better(w, j, v, i)) {
        v = w;
        i = j;
    }
}

__device__ void block_argmax(float& v, int32_t& i, Smem& sm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am_merge_shfl(v, i, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        sm.red[warp].x = v;
        sm.redi[warp] = i;
    }
    __syncthreads();
    if (warp == 0) {
        v = lane < kWarps ? sm.red[lane].x : -INFINITY;
        i = lane < kWarps ? sm.redi[lane] : INT32_MAX;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am_merge_shfl(v, i, o);
    }
    __syncthreads();
}

// ------------------------------------------------------------ per-thread updates
template <int DT>
struct VecTraits;
template <>
struct VecTraits<SPECV_BF16> {
    static constexpr int kEsz = 2, kVec = 8;
    __device__ static __forceinline__ void unpack(const uint4& q, float* v) {
        v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
        v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
    }
    static constexpr uint32_t kNegInfWord = 0xFF80FF80u;
};
template <>
struct VecTraits<SPECV_F32> {
    static constexpr int kEsz = 4, kVec = 4;
    __device__ static __forceinline__ void unpack(const uint4& q, float* v) {
        v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
        v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
    }
    static constexpr uint32_t kNegInfWord = 0xFF800000u;
};

// Running state of one thread over its share of a row slice.
struct ThreadAcc {
    float m;    // logits: largest raw logit seen; argmax: best value
    float s;    // logits/probs: running sum
    float neg;  // logits: -(m * k), or 0 while nothing finite was seen
    int32_t idx;  // argmax: index of best
};

template <int MODE>
__device__ __forceinline__ void acc_scalar(ThreadAcc& a, float v, float k, int32_t col) {
    if constexpr (MODE == kLogits) {
        if (v > a.m) {
            float nneg = -(v * k);
            if (a.s != 0.f) a.s *= ex2(nneg - a.neg);
            a.m = v;
            a.neg = nneg;
        }
        a.s += ex2(__fmaf_rn(v, k, a.neg));
    } else if constexpr (MODE == kProbs) {
        a.s += v;
    } else {
        if (v > a.m) {
            a.m = v;
            a.idx = col;
        }
    }
}

// n values v[0..n) in increasing column order; col_of(j) gives the column of v[j].
template <int MODE, int NV>
__device__ __forceinline__ void acc_block(ThreadAcc& a, const float (&v)[NV], float k, const int32_t (&cols)[NV]) {
    float bm = v[0];
#pragma unroll
    for (int j = 1; j < NV; ++j) bm = fmaxf(bm, v[j]);
    if constexpr (MODE == kLogits) {
        if (bm > a.m) {
            float nneg = -(bm * k);
            if (a.s != 0.f) a.s *= ex2(nneg - a.neg);
            a.m = bm;
            a.neg = nneg;
        }
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < NV; j += 2) {
            s0 += ex2(__fmaf_rn(v[j], k, a.neg));
            s1 += ex2(__fmaf_rn(v[j + 1], k, a.neg));
        }
        a.s += s0 + s1;
    } else if constexpr (MODE == kProbs) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < NV; j += 2) {
            s0 += v[j];
            s1 += v[j + 1];
        }
        a.s += s0 + s1;
    } else {
        if (bm > a.m) {
            int32_t c = cols[NV - 1];
#pragma unroll
            for (int j = NV - 1; j >= 0; --j)
                if (v[j] == bm) c = cols[j];
            a.m = bm;
            a.idx = c;
        }
    }
}

// Stream columns [c0, c1) of one row; returns the CTA's partial in thread 0.
template <int DT, int MODE>
__device__ float2 seg_pass(const char* row, int64_t c0, int64_t c1, float k, Smem& sm) {
    using VT = VecTraits<DT>;
    constexpr int ESZ = VT::kEsz, VEC = VT::kVec;
    ThreadAcc a;
    a.m = -INFINITY;
    a.s = 0.f;
    a.neg = 0.f;
    a.idx = INT32_MAX;
    const int tid = threadIdx.x;
    const uintptr_t addr0 = (uintptr_t)(row + c0 * ESZ);
    int64_t head = (int64_t)(((16u - (uint32_t)(addr0 & 15u)) & 15u) / ESZ);
    if (head > c1 - c0) head = c1 - c0;
    if (tid < head) {
        int64_t c = c0 + tid;
        acc_scalar<MODE>(a, ld_elem<DT>(row, c), k, (int32_t)c);
    }
    const int64_t v0 = c0 + head;
    const int64_t nvec = (c1 - v0) / VEC;
    const uint4* vp = reinterpret_cast<const uint4*>(row + v0 * ESZ);
    constexpr int64_t kStep = (int64_t)kUnroll * kStatsThreads;
    int64_t i = tid;
    // full iterations: kUnroll vectors per thread, all in range
    for (; i + (kUnroll - 1) * kStatsThreads < nvec; i += kStep) {
        uint4 q[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) q[u] = ld_stream_v4(vp + i + u * kStatsThreads);
        float v[kUnroll * VEC];
        int32_t cols[kUnroll * VEC];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            VT::unpack(q[u], v + u * VEC);
#pragma unroll
            for (int e = 0; e < VEC; ++e) cols[u * VEC + e] = (int32_t)(v0 + (i + u * kStatsThreads) * VEC + e);
        }
        acc_block<MODE>(a, v, k, cols);
    }
    // last partial iteration
    if (i < nvec) {
        uint4 q[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            int64_t j = i + u * kStatsThreads;
            if (j < nvec) {
                q[u] = ld_stream_v4(vp + j);
            } else {
                uint32_t f = (MODE == kProbs) ? 0u : VT::kNegInfWord;
                q[u] = make_uint4(f, f, f, f);
            }
        }
        float v[kUnroll * VEC];
        int32_t cols[kUnroll * VEC];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            VT::unpack(q[u], v + u * VEC);
#pragma unroll
            for (int e = 0; e < VEC; ++e) cols[u * VEC + e] = (int32_t)(v0 + (i + u * kStatsThreads) * VEC + e);
        }
        acc_block<MODE>(a, v, k, cols);
    }
    // tail scalars
    const int64_t t0 = v0 + nvec * VEC;
    if (tid < c1 - t0) {
        int64_t c = t0 + tid;
        acc_scalar<MODE>(a, ld_elem<DT>(row, c), k, (int32_t)c);
    }
    // reduce across the CTA
    if constexpr (MODE == kLogits) {
        return block_ms(make_float2(a.m, a.s), k, sm);  // (raw max, sum relative to it)
    } else if constexpr (MODE == kProbs) {
        return make_float2(0.f, block_sum(a.s, sm));
    } else {
        float v = a.m;
        int32_t ix = a.idx;
        block_argmax(v, ix, sm);
        if (ix == INT32_MAX) ix = (int32_t)c0;  // every element -inf or NaN: first one
        return make_float2(v, __int_as_float(ix));
    }
}

__device__ float2 run_segment(const StatsParams& p, bool is_t, int64_t lr, int64_t c0, int64_t c1, float k,
                              Smem& sm) {
    const int dt = is_t ? p.tdt : p.ddt;
    const int esz = dt == SPECV_F32 ? 4 : 2;
    const char* row = (const char*)(is_t ? p.tgt : p.dft) + lr * p.V * esz;
    if (p.greedy) {
        return dt == SPECV_F32 ? seg_pass<SPECV_F32, kArgmax>(row, c0, c1, k, sm)
                               : seg_pass<SPECV_BF16, kArgmax>(row, c0, c1, k, sm);
    }
    if (!is_t && p.probs) {
        return dt == SPECV_F32 ? seg_pass<SPECV_F32, kProbs>(row, c0, c1, k, sm)
                               : seg_pass<SPECV_BF16, kProbs>(row, c0, c1, k, sm);
    }
    return dt == SPECV_F32 ? seg_pass<SPECV_F32, kLogits>(row, c0, c1, k, sm)
                           : seg_pass<SPECV_BF16, kLogits>(row, c0, c1, k, sm);
}

// -------------------------------------------------------------- finalize
__device__ __forceinline__ bool row_ok(float2 st, bool probs_row) {
    if (probs_row) return isfinite(st.y) && st.y > 0.f;
    return isfinite(st.x) && isfinite(st.y) && st.y > 0.f;
}

// Checks that do not depend on the logits, in the documented order.
__device__ int32_t precheck(const StatsParams& p, int32_t b, Smem& sm, int64_t& t0, int64_t& d0, int32_t& g) {
    if (threadIdx.x == 0) {
        sm.status = 0;
        sm.flag_tok = 0;
    }
    __syncthreads();
    t0 = tro_at(p, b);
    d0 = dro_at(p, b);
    const int64_t t1 = tro_at(p, b + 1), d1 = dro_at(p, b + 1);
    const int64_t gg = d1 - d0;
    g = (int32_t)gg;
    int32_t st = 0;
    if (gg < 0 || gg > p.gmax || t1 - t0 != gg + 1 || t0 < 0 || t1 > p.rows_t || d0 < 0 || d1 > p.rows_d)
        st = 4;  // SPEC_SEQ_BAD_LAYOUT
    if (!st && !p.greedy) {
        float T = temp_of(p, b);
        if (!(T > 0.f) || !isfinite(T)) st = 5;  // SPEC_SEQ_BAD_TEMP
    }
    if (!st) {
        for (int i = threadIdx.x; i < g; i += blockDim.x) {
            int32_t x = __ldg(p.tokens + d0 + i);
            if (x < 0 || x >= p.V) atomicOr(&sm.flag_tok, 1);
        }
        __syncthreads();
        if (sm.flag_tok) st = 1;  // SPEC_SEQ_BAD_TOKEN
    }
    if (!st && p.kv_in && __ldg(p.kv_in + b) < g) st = 2;  // SPEC_SEQ_BAD_KV
    return st;
}

__device__ void write_error(const StatsParams& p, int32_t b, int32_t st, int64_t t0, int32_t g) {
    if (st != 4) {
        for (int i = threadIdx.x; i <= g; i += blockDim.x) p.out_tokens[t0 + i] = -1;
    }
    if (threadIdx.x == 0) {
        p.out_accepted[b] = 0;
        int32_t kv = p.kv_in ? p.kv_in[b] : 0;
        if (p.kv_out) p.kv_out[b] = kv;
        if (p.out_blocks) p.out_blocks[b] = p.block_size > 0 ? (kv + p.block_size - 1) / p.block_size : 0;
        if (p.seq_status) p.seq_status[b] = st;
        if (!p.greedy) p.tasks[b].mode = kTaskNone;
    }
}

__device__ void write_ok(const StatsParams& p, int32_t b, int32_t g, int32_t a) {
    p.out_accepted[b] = a;
    if (p.kv_out || p.out_blocks) {
        int32_t kv = p.kv_in ? p.kv_in[b] - (g - a) : 0;
        if (p.kv_out) p.kv_out[b] = kv;
        if (p.out_blocks) p.out_blocks[b] = p.block_size > 0 ? (kv + p.block_size - 1) / p.block_size : 0;
    }
    if (p.seq_status) p.seq_status[b] = 0;
}

// Merge the partials of row r (flat index) with one warp; result in lane 0.
__device__ float2 merge_row_ms(const StatsParams& p, int64_t r, bool probs_row, float k) {
    const int lane = threadIdx.x & 31;
    const uint32_t ns = nseg_of(r, p.V, p.chunk);
    float2 acc = make_float2(probs_row ? 0.f : -INFINITY, 0.f);
    for (uint32_t j = lane; j < ns; j += 32) {
        float2 v = ld_cg_f2(p.partials + r * p.S + j);
        acc = probs_row ? make_float2(0.f, acc.y + v.y) : ms_merge(acc, v, k);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float2 w = make_float2(__shfl_xor_sync(0xffffffffu, acc.x, o), __shfl_xor_sync(0xffffffffu, acc.y, o));
        acc = probs_row ? make_float2(0.f, acc.y + w.y) : ms_merge(acc, w, k);
    }
    return acc;
}

__device__ void merge_row_am(const StatsParams& p, int64_t r, float& v, int32_t& ix) {
    const int lane = threadIdx.x & 31;
    const uint32_t ns = nseg_of(r, p.V, p.chunk);
    v = -INFINITY;
    ix = INT32_MAX;
    for (uint32_t j = lane; j < ns; j += 32) {
        float2 w = ld_cg_f2(p.partials + r * p.S + j);
        int32_t wi = __float_as_int(w.y);
        if (am_better(w.x, wi, v, ix)) {
            v = w.x;
            ix = wi;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am_merge_shfl(v, ix, o);
}

__device__ void finalize_sample(const StatsParams& p, int32_t b, Smem& sm) {
    int64_t t0, d0;
    int32_t g;
    int32_t st = precheck(p, b, sm, t0, d0, g);
    if (st) {
        write_error(p, b, st, t0, g);
        return;
    }
    const float k = kLog2e / temp_of(p, b);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrows = 2 * g + 1;  // rows 0..g target, g+1..2g draft
    for (int j = warp; j < nrows; j += kWarps) {
        const bool is_t = j <= g;
        const int64_t r = is_t ? (t0 + j) : (p.rows_t + d0 + (j - g - 1));
        const bool probs_row = !is_t && p.probs;
        float2 v = merge_row_ms(p, r, probs_row, k);
        if (lane == 0) {
            sm.rs[j] = v;
            p.row_stats[r] = v;
        }
    }
    __syncthreads();
    // p_i(x_i), q_i(x_i) and the uniforms of every position
    for (int i = threadIdx.x; i <= g; i += blockDim.x) {
        if (i < g) {
            const int32_t x = __ldg(p.tokens + d0 + i);
            const float2 ts = sm.rs[i], ds = sm.rs[g + 1 + i];
            const float lt = ld_elem_rt((const char*)p.tgt + (t0 + i) * p.V * (p.tdt == SPECV_F32 ? 4 : 2), p.tdt, x);
            const float ld = ld_elem_rt((const char*)p.dft + (d0 + i) * p.V * (p.ddt == SPECV_F32 ? 4 : 2), p.ddt, x);
            const float pxv = ex2(__fmaf_rn(lt, k, -__fmul_rn(ts.x, k))) * (1.0f / ts.y);
            const float qxv =
                p.probs ? ld * (1.0f / ds.y) : ex2(__fmaf_rn(ld, k, -__fmul_rn(ds.x, k))) * (1.0f / ds.y);
            sm.px[i] = pxv;
            sm.qx[i] = qxv;
            sm.xt[i] = x;
            p.pq[d0 + i] = make_float2(pxv, qxv);
        }
        float2 u;
        if (p.uniforms) {
            u = __ldg(reinterpret_cast<const float2*>(p.uniforms) + t0 + i);
        } else {
            u = draw_uniforms(p.seed, p.round, p.seq_offset + (uint32_t)b, (uint32_t)i);
        }
        sm.ua[i] = u.x;
        sm.us[i] = u.y;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t a = g, s2 = 0;
        for (int i = 0; i < g; ++i) {
            if (!row_ok(sm.rs[i], false) || !row_ok(sm.rs[g + 1 + i], p.probs != 0)) {
                s2 = 3;  // SPEC_SEQ_BAD_ROW
                break;
            }
            if (!(__fmul_rn(sm.ua[i], sm.qx[i]) < sm.px[i])) {  // reject x_i
                a = i;
                break;
            }
        }
        if (!s2 && a == g && !row_ok(sm.rs[g], false)) s2 = 3;
        sm.status = s2;
        sm.accepted = a;
        if (!s2) {
            write_ok(p, b, g, a);
            SampleTask t;
            t.mode = a < g ? kTaskResidual : kTaskBonus;
            t.probs = p.probs;
            t.trow = t0 + a;
            t.drow = a < g ? d0 + a : -1;
            t.out_slot = t0 + a;
            t.u = sm.us[a];
            const df kk = k_of_temperature(temp_of(p, b));
            t.k_hi = kk.hi;
            t.k_lo = kk.lo;
            t.mt = sm.rs[a].x;
            t.md = a < g ? sm.rs[g + 1 + a].x : 0.f;
            t.z_hi = t.z_lo = t.st_hi = t.st_lo = t.sd_hi = t.sd_lo = 0.f;
            t.pad = 0;
            p.tasks[b] = t;
        }
    }
    __syncthreads();
    if (sm.status) {
        write_error(p, b, sm.status, t0, g);
        return;
    }
    const int32_t a = sm.accepted;
    for (int i = threadIdx.x; i <= g; i += blockDim.x) p.out_tokens[t0 + i] = (i < a) ? sm.xt[i] : -1;
}

__device__ void finalize_greedy(const StatsParams& p, int32_t b, Smem& sm) {
    int64_t t0, d0;
    int32_t g;
    int32_t st = precheck(p, b, sm, t0, d0, g);
    if (st) {
        write_error(p, b, st, t0, g);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j <= g; j += kWarps) {
        float v;
        int32_t ix;
        merge_row_am(p, t0 + j, v, ix);
        if (lane == 0) {
            sm.pick[j] = ix;
            p.row_stats[t0 + j] = make_float2(v, __int_as_float(ix));
        }
    }
    for (int i = threadIdx.x; i < g; i += blockDim.x) sm.xt[i] = __ldg(p.tokens + d0 + i);
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t a = 0;
        while (a < g && sm.xt[a] == sm.pick[a]) ++a;
        sm.accepted = a;
        write_ok(p, b, g, a);
    }
    __syncthreads();
    const int32_t a = sm.accepted;
    for (int i = threadIdx.x; i <= g; i += blockDim.x)
        p.out_tokens[t0 + i] = (i < a) ? sm.xt[i] : (i == a ? sm.pick[a] : -1);
}

__device__ __forceinline__ void finalize(const StatsParams& p, int32_t b, Smem& sm) {
    if (p.greedy)
        finalize_greedy(p, b, sm);
    else
        finalize_sample(p, b, sm);
}

// Count `cnt` pieces of sequence b as done; the CTA that completes the count
// finalizes b. Block-uniform arguments.
__device__ void arrive(const StatsParams& p, int32_t b, uint32_t cnt, Smem& sm) {
    if (b < 0 || cnt == 0) return;
    if (threadIdx.x == 0) {
        __threadfence();  // this CTA's partials before its arrival
        const uint32_t expected = expected_arrivals(p, b);
        const uint32_t old = atomicAdd(p.counters + b, cnt);
        sm.is_last = (old + cnt == expected);
        if (sm.is_last) {
            p.counters[b] = 0;  // every piece of b has arrived: ready for the next call
            __threadfence();
        }
    }
    __syncthreads();
    if (sm.is_last) finalize(p, b, sm);
    __syncthreads();
}

__global__ void __launch_bounds__(kStatsThreads, 2) stats_kernel(StatsParams p) {
    __shared__ Smem sm;
    // The residual sampler (next launch) may be scheduled now; it waits for
    // this grid's completion before reading anything this grid writes.
    pdl_launch_dependents();

    // Sequences that own no row at all (only possible with broken offsets)
    // still get their outputs written.
    if (p.tro) {
        for (int32_t b = blockIdx.x; b < p.B; b += gridDim.x) {
            if (expected_arrivals(p, b) == 0) {
                finalize(p, b, sm);
                __syncthreads();
            }
        }
    }

    int64_t e = (int64_t)blockIdx.x * p.chunk;
    const int64_t end = min(p.N, e + p.chunk);
    int32_t pend_b = -1;
    uint32_t pend_n = 0;
    bool pend_draft = false;
    while (e < end) {
        const int64_t r = e / p.V;
        const int64_t c0 = e - r * p.V;
        const int64_t seg_end = min(end, (r + 1) * p.V);
        const int64_t c1 = seg_end - r * p.V;
        const bool is_t = r < p.rows_t;
        const int64_t lr = is_t ? r : r - p.rows_t;
        const int32_t b = seq_of_row(p, !is_t, lr);
        float k = 1.f;
        if (!p.greedy && b >= 0) k = kLog2e / temp_of(p, b);
        const float2 part = run_segment(p, is_t, lr, c0, c1, k, sm);
        if (threadIdx.x == 0) p.partials[r * p.S + (blockIdx.x - (r * p.V) / p.chunk)] = part;
        if (b != pend_b || (!is_t) != pend_draft) {
            arrive(p, pend_b, pend_n, sm);
            pend_b = b;
            pend_n = 0;
            pend_draft = !is_t;
        }
        if (b >= 0) ++pend_n;
        e = seg_end;
    }
    arrive(p, pend_b, pend_n, sm);
}

}  // namespace

Layout make_layout(int64_t B, int64_t V, int64_t rows_t, int64_t rows_d, int greedy, int64_t grid_cap) {
    Layout L;
    L.rows_total = rows_t + (greedy ? 0 : rows_d);
    L.N = L.rows_total * V;
    int64_t cap = grid_cap < 1 ? 1 : grid_cap;
    int64_t chunk = (L.N + cap - 1) / cap;
    chunk = (chunk + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
    if (chunk < kMinChunk) chunk = kMinChunk;
    L.chunk = chunk;
    L.grid = (int32_t)((L.N + chunk - 1) / chunk);
    L.S = (int32_t)((V - 1) / chunk + 2);
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    size_t off = al(kHeaderBytes);
    L.off_partials = off;
    off = al(off + (size_t)L.rows_total * L.S * sizeof(float2));
    L.off_rowstats = off;
    off = al(off + (size_t)L.rows_total * sizeof(float2));
    L.off_pq = off;
    off = al(off + (greedy ? 0 : (size_t)rows_d * sizeof(float2)));
    L.off_tasks = off;
    off = al(off + (greedy ? 0 : (size_t)B * sizeof(SampleTask)));
    L.total = off;
    return L;
}

int stats_resident_ctas(int device, int greedy) {
    (void)greedy;
    int sms = 0, per = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, stats_kernel, kStatsThreads, 0) != cudaSuccess)
        return 0;
    if (per < 1) per = 1;
    return sms * per;
}

cudaError_t launch_stats(const StatsParams& p, cudaStream_t s) {
    stats_kernel<<<p.grid, kStatsThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace specv
