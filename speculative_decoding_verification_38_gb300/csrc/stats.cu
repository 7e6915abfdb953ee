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

#include "stream.cuh"

namespace specv {

namespace {

constexpr int kWarps = kStatsThreads / 32;
constexpr int kUnroll = 4;


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




// Elements (rows x V) the streaming pass folds for sequence b: every CTA
// adds the elements of b it has folded to b's counter, and the one that
// brings the counter to this total finalizes b.
__device__ uint32_t expected_elements(const StatsParams& p, int32_t b) {
    const int64_t t0 = max((int64_t)0, tro_at(p, b)), t1 = min(p.rows_t, tro_at(p, b + 1));
    int64_t rows = max((int64_t)0, t1 - t0);
    if (!p.greedy) {
        const int64_t d0 = max((int64_t)0, dro_at(p, b)), d1 = min(p.rows_d, dro_at(p, b + 1));
        rows += max((int64_t)0, d1 - d0);
    }
    return (uint32_t)(rows * p.V);
}
static_assert((2 * 64 + 1) * kMaxVocab < (int64_t)1 << 32, "per-sequence element count fits 32 bits");


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

// NV values v[] in increasing column order; for argmax, value j sits at
// column cb[j / VEC] + j % VEC (computed only when a new maximum appears).
template <int MODE, int NV, int VEC>
__device__ __forceinline__ void acc_block(ThreadAcc& a, const float (&v)[NV], float k, const int32_t (&cb)[NV / VEC]) {
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
            int32_t c = INT32_MAX;
#pragma unroll
            for (int j = NV - 1; j >= 0; --j)
                if (v[j] == bm) c = cb[j / VEC] + (j % VEC);
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
        int32_t cb[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            VT::unpack(q[u], v + u * VEC);
            cb[u] = (int32_t)(v0 + (i + u * kStatsThreads) * VEC);
        }
        acc_block<MODE, kUnroll * VEC, VEC>(a, v, k, cb);
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
        int32_t cb[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            VT::unpack(q[u], v + u * VEC);
            cb[u] = (int32_t)(v0 + (i + u * kStatsThreads) * VEC);
        }
        acc_block<MODE, kUnroll * VEC, VEC>(a, v, k, cb);
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



// Merge the partials of row r (flat index) with one warp; result in lane 0.
__device__ float2 merge_row_ms(const StatsParams& p, int64_t r, bool probs_row, float k) {
    const int lane = threadIdx.x & 31;
    const uint32_t ns = nseg_of(r, p.V, p.chunk);
    float2 acc = make_float2(probs_row ? 0.f : -INFINITY, 0.f);
    for (uint32_t j = lane; j < ns * (uint32_t)p.pw; j += 32) {
        float2 v = ld_cg_f2(p.partials + r * p.S * p.pw + j);
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
    for (uint32_t j = lane; j < ns * (uint32_t)p.pw; j += 32) {
        float2 w = ld_cg_f2(p.partials + r * p.S * p.pw + j);
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
    const int nwarps = blockDim.x >> 5;
    for (int j = warp; j < nrows; j += nwarps) {
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
            const df kk = k_pos_lo(k_of_temperature(temp_of(p, b)));
            t.k_hi = kk.hi;
            t.k_lo = kk.lo;
            t.mt = sm.rs[a].x;
            t.md = a < g ? sm.rs[g + 1 + a].x : 0.f;
            t.it_apx = inv_norm_apx(sm.rs[a], k);
            t.id_apx = a < g ? (p.probs ? 1.0f / sm.rs[g + 1 + a].y : inv_norm_apx(sm.rs[g + 1 + a], k)) : 0.f;
            t.z_hi = t.z_lo = 0.f;
            t.tau_t = t.tau_d = -INFINITY;  // this path never truncates
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
    const int nwarps = blockDim.x >> 5;
    for (int j = warp; j <= g; j += nwarps) {
        float v;
        int32_t ix;
        merge_row_am(p, t0 + j, v, ix);
        if (ix == INT32_MAX) ix = 0;  // every logit -inf or NaN: the first index
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

// Count `cnt` elements of sequence b as folded; the CTA that completes the
// count finalizes b. Block-uniform arguments.
__device__ void arrive(const StatsParams& p, int32_t b, uint32_t cnt, Smem& sm) {
    if (b < 0 || cnt == 0) return;
    if (threadIdx.x == 0) {
        __threadfence();  // this CTA's partials before its arrival
        const uint32_t expected = expected_elements(p, b);
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
            if (expected_elements(p, b) == 0) {
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
        if (threadIdx.x == 0) p.partials[(r * p.S + (blockIdx.x - (r * p.V) / p.chunk)) * p.pw] = part;
        if (b != pend_b || (!is_t) != pend_draft) {
            arrive(p, pend_b, pend_n, sm);
            pend_b = b;
            pend_n = 0;
            pend_draft = !is_t;
        }
        if (b >= 0) pend_n += (uint32_t)(seg_end - e);
        e = seg_end;
    }
    arrive(p, pend_b, pend_n, sm);
}

// ------------------------------------------------------------ TMA variant
// One CTA per SM; its element range is cut into one contiguous piece per warp.
// Every warp streams its own piece through a private ring of shared-memory
// stages filled by 1-D bulk copies (cp.async.bulk, completion counted on a
// per-stage mbarrier that lane 0 arms), folds each stage into per-lane
// states with packed f32x2 arithmetic and, whenever a row ends, reduces its
// lanes and stores one partial per (row, CTA slice, warp). Warps never wait
// on one another while streaming. Every mbarrier wait is bounded; a warp that
// gives up poisons its partials (NaN), so the affected sequences report
// SPEC_SEQ_BAD_ROW, and sets the workspace error word.
constexpr int kWarpRing = kTmaStages * (int)kTmaStageBytes;  // bytes of one warp's ring






// ------------------------------------------------- finalize helpers (TMA variant)
// Partials of row r: nseg_of(r) CTA slices of pw warp partials each, stored
// contiguously from (r * S) * pw; a warp that folded nothing of the row
// stored the identity.
__device__ __forceinline__ int32_t pieces_of_row(const StatsParams& p, int64_t r) {
    return (int32_t)nseg_of(r, p.V, p.chunk) * p.pw;
}


__device__ __forceinline__ float2 ident_partial(const StatsParams& p, int64_t r) {
    if (p.greedy) return make_float2(-INFINITY, __int_as_float(INT32_MAX));
    if (r >= p.rows_t && p.probs) return make_float2(0.f, 0.f);
    return make_float2(-INFINITY, 0.f);
}

__device__ __forceinline__ int64_t partial_index(const StatsParams& p, int64_t r, int warp) {
    const int64_t slot = (int64_t)blockIdx.x - (r * p.V) / p.chunk;
    return (r * p.S + slot) * p.pw + warp;
}

// Reduce the lane states of row r over the warp; lane 0 stores the partial
// (NaN if the warp gave up on a copy).
__device__ void lane_flush(const StatsParams& p, LaneAcc& a, int mode, float k, int64_t r, int warp, bool poison) {
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
    } else if (mode == kProbs) {
        float v = a.s.x + a.s.y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        out = make_float2(0.f, v);
    } else {
        float v = a.m;
        int32_t ix = a.idx;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am_merge_shfl(v, ix, o);
        out = make_float2(v, __int_as_float(ix));
    }
    if (lane == 0) {
        if (poison) out = make_float2(NAN, NAN);
        p.partials[partial_index(p, r, warp)] = out;
    }
    lane_reset(a);
}

struct WarpRing {
    uint64_t full[kTmaConsumerWarps][kTmaStages];
    int64_t unit_of[kTmaConsumerWarps][kTmaStages];  // unit held by each stage of each warp's ring
    int next_unit;                                     // next unit of this CTA's range to hand out
    int failed;
};

__global__ void __launch_bounds__(kTmaThreads, 1) stats_tma_kernel(StatsParams p) {
    __shared__ WarpRing wr;
    extern __shared__ __align__(128) char ring[];
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int w = 0; w < kTmaConsumerWarps; ++w)
            for (int st = 0; st < kTmaStages; ++st) mbar_init(&wr.full[w][st], 1);
        wr.next_unit = 0;
        wr.failed = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const int64_t e0 = (int64_t)blockIdx.x * p.chunk;
    const int64_t e1 = min(p.N, e0 + p.chunk);
    // The range is handed out in units of one stage: units of the target part
    // [e0, m) first, then of the draft part [m, e1); m = the first draft element.
    const int64_t T = p.rows_t * p.V;
    const int tesz = p.tdt == SPECV_F32 ? 4 : 2, desz = p.ddt == SPECV_F32 ? 4 : 2;
    const int64_t m = max(e0, min(e1, T));
    const int64_t ut = kTmaStageBytes / tesz, ud = kTmaStageBytes / desz;  // elements per unit
    const int64_t nut = (m - e0 + ut - 1) / ut, nud = (e1 - m + ud - 1) / ud;
    const int64_t nunits = nut + nud;
    auto unit_start = [&](int64_t u) { return u < nut ? e0 + u * ut : m + (u - nut) * ud; };
    auto unit_end = [&](int64_t u) { return u < nut ? min(m, e0 + (u + 1) * ut) : min(e1, m + (u - nut + 1) * ud); };

    char* myring = ring + (size_t)warp * kWarpRing;
    uint64_t* full = wr.full[warp];
    // lane 0 takes the next unit and, unless the warp gave up, starts its copy
    uint32_t issued = 0, copies = 0;  // stages handed to this warp / of those, stages with a copy
    auto take = [&](bool copy) -> bool {
        const int64_t u = atomicAdd(&wr.next_unit, 1);
        if (u >= nunits) return false;
        const int st = issued % kTmaStages;
        wr.unit_of[warp][st] = u;
        if (copy) {
            const int64_t f = unit_start(u), s1 = unit_end(u);
            const bool tgt = f < T;
            const int esz = tgt ? tesz : desz;
            const char* src = tgt ? (const char*)p.tgt + f * esz : (const char*)p.dft + (f - T) * esz;
            mbar_arrive_expect_tx(&full[st], (uint32_t)((s1 - f) * esz));
            bulk_g2s(myring + (size_t)st * kTmaStageBytes, src, (uint32_t)((s1 - f) * esz), &full[st]);
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
    uint32_t done = 0;  // stages whose copy completed
    // row bookkeeping: the current row r of the CTA range, whether this warp
    // has folded any of it, and its parameters
    const int64_t R0 = e0 < e1 ? e0 / p.V : 0, R1 = e0 < e1 ? (e1 - 1) / p.V : -1;
    int64_t r = R0, row_end = (R0 + 1) * p.V;
    bool touched = false;
    int mode = kLogits, dt = SPECV_BF16;
    float k = 1.f;
    int64_t param_row = -1;  // row the parameters above belong to
    auto set_row = [&]() {
        if (param_row == r) return;
        param_row = r;
        const bool is_t = r < p.rows_t;
        dt = is_t ? p.tdt : p.ddt;
        mode = p.greedy ? kArgmax : ((!is_t && p.probs) ? kProbs : kLogits);
        k = 1.f;
        if (!p.greedy) {
            const int32_t b = seq_of_row(p, !is_t, is_t ? r : r - p.rows_t);
            if (b >= 0) k = kLog2e / temp_of(p, b);
        }
    };
    auto leave_row = [&]() {  // store this warp's partial of row r, then move to r + 1
        if (touched) lane_flush(p, a, mode, k, r, warp, dead);
        else if (lane == 0) p.partials[partial_index(p, r, warp)] = ident_partial(p, r);
        touched = false;
        ++r;
        row_end += p.V;
    };
    if (R0 <= R1) set_row();

    for (uint32_t kk = 0; kk < issued; ++kk) {
        const int st = kk % kTmaStages;
        if (!dead) {
            const bool ok = mbar_wait_bounded(&full[st], (kk / kTmaStages) & 1, kWaitLimit);
            dead = __any_sync(0xffffffffu, !ok);
            if (dead && lane == 0) atomicExch(&wr.failed, 1);
            if (!dead) done = kk + 1;
        }
        const int64_t u = wr.unit_of[warp][st];
        const int64_t f = unit_start(u), s1 = unit_end(u);
        while (f >= row_end) leave_row();
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
                } else if (mode == kProbs) {
                    if (dt == SPECV_F32) warp_segment<SPECV_F32, kProbs>(a, sa, nvec, col0, k, lane);
                    else warp_segment<SPECV_BF16, kProbs>(a, sa, nvec, col0, k, lane);
                } else {
                    if (dt == SPECV_F32) warp_segment<SPECV_F32, kArgmax>(a, sa, nvec, col0, k, lane);
                    else warp_segment<SPECV_BF16, kArgmax>(a, sa, nvec, col0, k, lane);
                }
            }
            if (se == row_end) {  // the row ends inside this unit
                leave_row();
                if (se < s1) set_row();
            }
            g0 = se;
        }
        // refill the slot just consumed (the reads above are done once the warp converges)
        __syncwarp();
        if (lane == 0) {
            if (!dead) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            take(!dead);
        }
        issued = __shfl_sync(0xffffffffu, issued, 0);
        __syncwarp();  // lane 0's record of the unit is seen by the warp even without a wait
    }
    while (r <= R1) leave_row();  // the rest of the CTA range's rows
    // never leave while a copy into this warp's ring may be in flight
    if (lane == 0) {
        for (uint32_t q = done; q < copies; ++q)
            mbar_wait_bounded(&full[q % kTmaStages], (q / kTmaStages) & 1, kWaitLimit);
    }
    __syncthreads();
    if (threadIdx.x == 0 && wr.failed) atomicOr(p.err, 1u);

}

// Finalize of the TMA variant: one CTA per sequence, after the streaming grid
// has completed (programmatic launch; the wait returns once every partial of
// that grid is visible). The same decisions as finalize_sample /
// finalize_greedy, arranged for few dependent memory round trips: warp 0
// issues every check's load at once, the CTA's warps merge one row each
// (lane q loads partial q of the row, a coalesced read), and warp 0 takes the
// accept decisions by ballot.
constexpr int kFinThreads = 256;
constexpr int kFinWarps = kFinThreads / 32;

struct FinSmem {
    float2 rs[2 * kMaxGamma + 1];
    int64_t t0, d0;
    int32_t g, status;
};



__global__ void __launch_bounds__(kFinThreads) finalize_kernel(StatsParams p) {
    __shared__ FinSmem fs;
    pdl_launch_dependents();
    pdl_wait_primary();
    const int32_t b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Layout first (every thread: the offsets are a broadcast load); with a
    // valid layout warps 1.. merge rows at once while warp 0 runs the other
    // status checks and, for positions lane and lane + 32, fetches the draft
    // token, the two logits at it and u_acc.
    const int64_t t0 = tro_at(p, b), t1 = tro_at(p, b + 1);
    const int64_t d0 = dro_at(p, b), d1 = dro_at(p, b + 1);
    const int64_t gg = d1 - d0;
    const int32_t g = (int32_t)gg;
    if (gg < 0 || gg > p.gmax || t1 - t0 != gg + 1 || t0 < 0 || t1 > p.rows_t || d0 < 0 || d1 > p.rows_d) {
        if (warp == 0) warp_write_error(p, b, 4, t0, g);  // SPEC_SEQ_BAD_LAYOUT
        return;
    }
    const float T = p.greedy ? 1.f : temp_of(p, b);
    const float k = p.greedy ? 1.f : kLog2e / T;
    const int nrows = p.greedy ? g + 1 : 2 * g + 1;  // rows 0..g target, g+1..2g draft
    int32_t x[2] = {0, 0};
    float lt[2] = {0.f, 0.f}, ld[2] = {0.f, 0.f}, ua[2] = {0.f, 0.f};
    int32_t kv = 0;
    if (warp == 0) {
        kv = p.kv_in ? __ldg(p.kv_in + b) : 0;
        int32_t st = 0;
        if (!p.greedy && (!(T > 0.f) || !isfinite(T))) st = 5;  // SPEC_SEQ_BAD_TEMP
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
            for (int i = lane + 64; i < g; i += 32) {  // gamma_max <= 64: at most one more
                const int32_t xx = __ldg(p.tokens + d0 + i);
                bad |= (xx < 0 || xx >= p.V);
            }
            if (__any_sync(0xffffffffu, bad)) st = 1;  // SPEC_SEQ_BAD_TOKEN
        }
        if (!st && p.kv_in && kv < g) st = 2;  // SPEC_SEQ_BAD_KV
        if (lane == 0) fs.status = st;
        if (!st && !p.greedy) {
            const int tes = p.tdt == SPECV_F32 ? 4 : 2, des = p.ddt == SPECV_F32 ? 4 : 2;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h;
                if (i < g) {
                    lt[h] = ld_elem_rt((const char*)p.tgt + (t0 + i) * p.V * tes, p.tdt, x[h]);
                    ld[h] = ld_elem_rt((const char*)p.dft + (d0 + i) * p.V * des, p.ddt, x[h]);
                    ua[h] = p.uniforms ? __ldg(p.uniforms + 2 * (t0 + i))
                                       : draw_uniforms(p.seed, p.round, p.seq_offset + (uint32_t)b, (uint32_t)i).x;
                }
            }
        }
    } else {
        for (int j = warp - 1; j < nrows; j += kFinWarps - 1) {
            const bool is_t = j <= g;
            const int64_t r = is_t ? (t0 + j) : (p.rows_t + d0 + (j - g - 1));
            float2 v;
            if (p.direct) {  // the top-k pass wrote the row's statistics whole
                if (lane == 0) fs.rs[j] = __ldcg(p.row_stats + r);
                continue;
            }
            const float2* src = p.partials + r * p.S * p.pw;
            const int32_t n = pieces_of_row(p, r);
            if (p.greedy) {
                int32_t ix;
                warp_merge_am(src, n, v.x, ix);
                if (ix == INT32_MAX) ix = 0;  // every logit -inf or NaN: the first index
                v.y = __int_as_float(ix);
            } else {
                v = warp_merge_ms(src, n, !is_t && p.probs, k);
            }
            if (lane == 0) fs.rs[j] = v;
        }
    }
    __syncthreads();
    if (fs.status) {
        if (warp == 0) warp_write_error(p, b, fs.status, t0, g);
        return;
    }
    if (!p.direct)
        for (int j = threadIdx.x; j < nrows; j += kFinThreads)
            p.row_stats[j <= g ? t0 + j : p.rows_t + d0 + (j - g - 1)] = fs.rs[j];
    if (warp != 0) return;
    if (p.greedy) {
        int32_t a = g;
        for (int base = 0; base < g; base += 32) {
            const int i = base + lane;
            const int32_t xi = base == 0 ? x[0] : (base == 32 ? x[1] : (i < g ? __ldg(p.tokens + d0 + i) : 0));
            const bool miss = i < g && xi != __float_as_int(fs.rs[i].y);
            const uint32_t m = __ballot_sync(0xffffffffu, miss);
            if (m) {
                a = base + __ffs(m) - 1;
                break;
            }
        }
        for (int i = lane; i <= g; i += 32)
            p.out_tokens[t0 + i] = (i < a) ? __ldg(p.tokens + d0 + i) : (i == a ? __float_as_int(fs.rs[a].y) : -1);
        if (lane == 0) write_ok(p, b, g, a);
        return;
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
            const float2 ts = fs.rs[i], ds = fs.rs[g + 1 + i];
            bad = !row_ok(ts, false) || !row_ok(ds, p.probs != 0);
            float pxv = ex2(__fmaf_rn(lt[h], k, -__fmul_rn(ts.x, k))) * (1.0f / ts.y);
            float qxv =
                p.probs ? ld[h] * (1.0f / ds.y) : ex2(__fmaf_rn(ld[h], k, -__fmul_rn(ds.x, k))) * (1.0f / ds.y);
            if (p.tau) {  // a token outside a row's top-k has probability 0 there
                if (!(lt[h] >= __ldcg(p.tau + t0 + i))) pxv = 0.f;
                if (!(ld[h] >= __ldcg(p.tau + p.rows_t + d0 + i))) qxv = 0.f;
            }
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
    if (!s2 && a == g && !row_ok(fs.rs[g], false)) s2 = 3;
    if (s2) {
        warp_write_error(p, b, s2, t0, g);
        return;
    }
#pragma unroll
    for (int h = 0; h < 3; ++h) {
        const int i = lane + 32 * h;
        if (i <= g) p.out_tokens[t0 + i] = (i < a) ? (h < 2 ? x[h] : __ldg(p.tokens + d0 + i)) : -1;
    }
    if (lane == 0) {
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
        const df kk = k_pos_lo(k_of_temperature(temp_of(p, b)));
        t.k_hi = kk.hi;
        t.k_lo = kk.lo;
        t.mt = fs.rs[a].x;
        t.md = a < g ? fs.rs[g + 1 + a].x : 0.f;
        t.it_apx = inv_norm_apx(fs.rs[a], k);
        t.id_apx = a < g ? (p.probs ? 1.0f / fs.rs[g + 1 + a].y : inv_norm_apx(fs.rs[g + 1 + a], k)) : 0.f;
        t.z_hi = t.z_lo = 0.f;
        t.tau_t = p.tau ? __ldcg(p.tau + t0 + a) : -INFINITY;
        t.tau_d = (p.tau && a < g) ? __ldcg(p.tau + p.rows_t + d0 + a) : -INFINITY;
        t.pad = 0;
        p.tasks[b] = t;
    }
}

}  // namespace

Layout make_layout(int64_t B, int64_t V, int64_t rows_t, int64_t rows_d, int greedy, int64_t grid_cap, int pw,
                   bool topp) {
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
    off = al(off + (size_t)L.rows_total * L.S * pw * sizeof(float2));
    L.off_rowstats = off;
    off = al(off + (size_t)L.rows_total * sizeof(float2));
    L.off_pq = off;
    off = al(off + (greedy ? 0 : (size_t)rows_d * sizeof(float2)));
    L.off_tasks = off;
    off = al(off + (greedy ? 0 : (size_t)B * sizeof(SampleTask)));
    L.off_recs = off;
    off = al(off + (greedy ? 0 : (size_t)B * ((V + kTile - 1) / kTile) * sizeof(TileRec)));
    L.off_open = off;
    off = al(off + (greedy ? 0 : (size_t)B * ((V + kTile - 1) / kTile) * kOpenCap * sizeof(uint16_t)));
    L.off_tau = off;
    off = al(off + (greedy ? 0 : (size_t)L.rows_total * sizeof(float)));
    const bool keep = topp && !greedy;
    L.off_keep = off;
    off = al(off + (keep ? (size_t)L.rows_total * kKeepCap * sizeof(uint32_t) : 0));
    L.off_keepn = off;
    off = al(off + (keep ? (size_t)L.rows_total * sizeof(int32_t) : 0));
    L.off_spart = off;
    off = al(off + (greedy ? 0 : (size_t)L.rows_total * L.S * sizeof(float2)));
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

cudaError_t launch_finalize(const StatsParams& p, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.B);
    cfg.blockDim = dim3(kFinThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, finalize_kernel, p);
}

cudaError_t launch_stats(const StatsParams& p, cudaStream_t s) {
    if (p.tma) {
        static bool attr_done = false;
        if (!attr_done) {
            cudaError_t e = cudaFuncSetAttribute(stats_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kTmaConsumerWarps * kWarpRing);
            if (e != cudaSuccess) return e;
            attr_done = true;
        }
        stats_tma_kernel<<<p.grid, kTmaThreads, kTmaConsumerWarps * kWarpRing, s>>>(p);
    } else {
        stats_kernel<<<p.grid, kStatsThreads, 0, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace specv
