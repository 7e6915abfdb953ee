// stream.cuh -- device pieces of the streaming pass and of the per-sequence
// decision shared by stats.cu (the streaming and finalize kernels) and
// verify.cu (the fused verify kernel): row and sequence bookkeeping, the
// per-lane online softmax / argmax fold of staged row data, the merge of
// partial statistics, and the outputs of a finished sequence ("Speculative
// decoding" (mhtirogla.ai), How it works, steps 2-5). Included by one
// translation unit each; everything here has internal linkage.
#pragma once

#include <math.h>

#include "precise.cuh"

namespace specv {

namespace {

constexpr int kMaxGamma = 64;

enum Mode { kLogits = 0, kProbs = 1, kArgmax = 2 };

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

__device__ __forceinline__ float temp_of(const StatsParams& p, int32_t b) {
    return p.temps ? __ldg(p.temps + b) : p.temperature;
}

__device__ __forceinline__ void am_merge_shfl(float& v, int32_t& i, int o) {
    float w = __shfl_xor_sync(0xffffffffu, v, o);
    int32_t j = __shfl_xor_sync(0xffffffffu, i, o);
    if (am_better(w, j, v, i)) {
        v = w;
        i = j;
    }
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

// -------------------------------------------------------------- finalize
__device__ __forceinline__ bool row_ok(float2 st, bool probs_row) {
    if (probs_row) return isfinite(st.y) && st.y > 0.f;
    return isfinite(st.x) && isfinite(st.y) && st.y > 0.f;
}

// The running acceptance of sequence b after a round with a of its g drafts
// accepted: the round performed t = a + 1 accept tests if a draft was
// rejected, else g; ema += lambda * (a / t - ema), each step rounded to
// float32 in that order. Rounds with g = 0 leave it.
__device__ __forceinline__ void update_ema(const StatsParams& p, int32_t b, int32_t g, int32_t a) {
    if (!p.ema || g <= 0) return;
    const int32_t t = a < g ? a + 1 : g;
    const float x = __fdiv_rn((float)a, (float)t);
    const float e = p.ema[b];
    p.ema[b] = __fadd_rn(e, __fmul_rn(p.ema_lambda, __fsub_rn(x, e)));
}

__device__ void write_ok(const StatsParams& p, int32_t b, int32_t g, int32_t a) {
    update_ema(p, b, g, a);
    p.out_accepted[b] = a;
    if (p.kv_out || p.out_blocks) {
        int32_t kv = p.kv_in ? p.kv_in[b] - (g - a) : 0;
        if (p.kv_out) p.kv_out[b] = kv;
        if (p.out_blocks) p.out_blocks[b] = p.block_size > 0 ? (kv + p.block_size - 1) / p.block_size : 0;
    }
    if (p.seq_status) p.seq_status[b] = 0;
}

// 1 / (the sampler's normaliser of a logits row), from the streaming pass's
// (raw max m, s = sum 2^(l k - fl(m k))): the sampler's weights 2^((l - m) k)
// are s's terms times 2^(fl(m k) - m k). Good to ~1e-6, which is all the
// sampler's support test asks of it.
__device__ __forceinline__ float inv_norm_apx(float2 rsv, float k) {
    const float mk = __fmul_rn(rsv.x, k);
    const float e = __fmaf_rn(rsv.x, k, -mk);  // m k - fl(m k), exact
    return 1.0f / (rsv.y * ex2(-e));
}

__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// Per-lane state of the warp-streaming pass: raw max m, neg = -fl(m*k) (0
// while nothing finite was seen), a two-lane running sum, argmax index.
struct LaneAcc {
    float m, neg;
    float2 s;
    int32_t idx;
};

__device__ __forceinline__ void lane_reset(LaneAcc& a) {
    a.m = -INFINITY;
    a.neg = 0.f;
    a.s = make_float2(0.f, 0.f);
    a.idx = INT32_MAX;
}

// Fold NV values (NV a multiple of 8, increasing columns; value j at column
// cb[j / VEC] + j % VEC) into a lane state. Maxima and sums run in four
// independent chains so that consecutive instructions do not wait on one another.
template <int MODE, int NV, int VEC>
__device__ __forceinline__ void lane_block(LaneAcc& a, const float (&v)[NV], float k, const int32_t (&cb)[NV / VEC]) {
    static_assert(NV % 8 == 0, "block of 8");
    if constexpr (MODE == kProbs) {
        float2 c[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) c[q] = make_float2(v[2 * q], v[2 * q + 1]);
#pragma unroll
        for (int j = 8; j < NV; j += 2) c[(j / 2) % 4] = add2(c[(j / 2) % 4], make_float2(v[j], v[j + 1]));
        a.s = add2(a.s, add2(add2(c[0], c[1]), add2(c[2], c[3])));
    } else {
        float mx[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) mx[q] = fmaxf(v[2 * q], v[2 * q + 1]);
#pragma unroll
        for (int j = 8; j < NV; j += 2) mx[(j / 2) % 4] = max3(mx[(j / 2) % 4], v[j], v[j + 1]);
        const float bm = max3(max3(a.m, mx[0], mx[1]), mx[2], mx[3]);
        if constexpr (MODE == kLogits) {
            if (bm > a.m) {
                const float nneg = -(bm * k);
                const float f = ex2(nneg - a.neg);
                if (a.s.x != 0.f) a.s.x *= f;
                if (a.s.y != 0.f) a.s.y *= f;
                a.m = bm;
                a.neg = nneg;
            }
            const float2 kk = make_float2(k, k), nn = make_float2(a.neg, a.neg);
            float2 c[4];
#pragma unroll
            for (int j = 0; j < NV; j += 2) {
                const float2 t = fma2(make_float2(v[j], v[j + 1]), kk, nn);
                const float2 e = make_float2(ex2(t.x), ex2(t.y));
                if (j < 8) c[j / 2] = e;
                else c[(j / 2) % 4] = add2(c[(j / 2) % 4], e);
            }
            a.s = add2(a.s, add2(add2(c[0], c[1]), add2(c[2], c[3])));
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
}

// Fold the nvec 16-byte vectors of one row segment held in shared memory at
// sa (first column col0) into the lane states of one warp.
template <int DT, int MODE>
__device__ __forceinline__ void warp_segment(LaneAcc& a, uint32_t sa, int nvec, int64_t col0, float k, int lane) {
    using VT = VecTraits<DT>;
    constexpr int VEC = VT::kVec;
    constexpr int U = 4;
    int i = lane;
    for (; i + 32 * (U - 1) < nvec; i += 32 * U) {
        uint4 q[U];
#pragma unroll
        for (int u = 0; u < U; ++u) q[u] = lds_v4(sa + (uint32_t)(i + 32 * u) * 16u);
        float v[U * VEC];
        int32_t cb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            VT::unpack(q[u], v + u * VEC);
            cb[u] = (int32_t)(col0 + (int64_t)(i + 32 * u) * VEC);
        }
        lane_block<MODE, U * VEC, VEC>(a, v, k, cb);
    }
    for (; i < nvec; i += 32) {  // leftover vectors, one at a time (f32 pads with -inf / 0)
        const uint4 q = lds_v4(sa + (uint32_t)i * 16u);
        float v[8];
        VT::unpack(q, v);
        if constexpr (VEC == 4) {
#pragma unroll
            for (int j = 4; j < 8; ++j) v[j] = MODE == kProbs ? 0.f : -INFINITY;
        }
        const int32_t cb[8 / VEC] = {(int32_t)(col0 + (int64_t)i * VEC)};
        lane_block<MODE, 8, VEC>(a, v, k, cb);
    }
}

__device__ void warp_write_error(const StatsParams& p, int32_t b, int32_t st, int64_t t0, int32_t g) {
    const int lane = threadIdx.x & 31;
    if (st != 4)
        for (int i = lane; i <= g; i += 32) p.out_tokens[t0 + i] = -1;
    if (lane == 0) {
        p.out_accepted[b] = 0;
        const int32_t kv = p.kv_in ? p.kv_in[b] : 0;
        if (p.kv_out) p.kv_out[b] = kv;
        if (p.out_blocks) p.out_blocks[b] = p.block_size > 0 ? (kv + p.block_size - 1) / p.block_size : 0;
        if (p.seq_status) p.seq_status[b] = st;
        if (!p.greedy) p.tasks[b].mode = kTaskNone;
    }
}

// Merge the n partials at src over the warp (all lanes get the result).
__device__ float2 warp_merge_ms(const float2* src, int32_t n, bool probs_row, float k) {
    const int lane = threadIdx.x & 31;
    float2 acc = make_float2(probs_row ? 0.f : -INFINITY, 0.f);
    for (int32_t q = lane; q < n; q += 32) {
        const float2 v = ld_cg_f2(src + q);
        acc = probs_row ? make_float2(0.f, acc.y + v.y) : ms_merge(acc, v, k);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float2 w = make_float2(__shfl_xor_sync(0xffffffffu, acc.x, o), __shfl_xor_sync(0xffffffffu, acc.y, o));
        acc = probs_row ? make_float2(0.f, acc.y + w.y) : ms_merge(acc, w, k);
    }
    return acc;
}

__device__ void warp_merge_am(const float2* src, int32_t n, float& v, int32_t& ix) {
    const int lane = threadIdx.x & 31;
    v = -INFINITY;
    ix = INT32_MAX;
    for (int32_t q = lane; q < n; q += 32) {
        const float2 w = ld_cg_f2(src + q);
        const int32_t wi = __float_as_int(w.y);
        if (am_better(w.x, wi, v, ix)) {
            v = w.x;
            ix = wi;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am_merge_shfl(v, ix, o);
}

}  // namespace

}  // namespace specv
