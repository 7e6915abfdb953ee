// misc.cu -- the standalone KV-length rollback and the test hooks.
#include <math.h>

#include "precise.cuh"

namespace specv {

namespace {

// kv' = kv - (gamma_b - accepted_b): drop the cache entries of the rejected
// drafts ("Speculative decoding" (mhtirogla.ai), How it works step 5; paged KV
// makes it a length truncate, Implementation notes).
__global__ void kv_rollback_kernel(const int32_t* kv_in, int32_t* kv_out, const int32_t* accepted,
                                   const int32_t* gammas, int32_t gmax, int32_t B, int32_t block_size,
                                   int32_t* out_blocks, int32_t* seq_status) {
    const int32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int32_t g = gammas ? gammas[b] : gmax;
    const int32_t a = accepted[b];
    const int32_t kv = kv_in[b];
    int32_t st = 0;
    if (g < 0 || a < 0 || a > g)
        st = 4;  // SPEC_SEQ_BAD_LAYOUT
    else if (kv < g)
        st = 2;  // SPEC_SEQ_BAD_KV
    const int32_t kv2 = st ? kv : kv - (g - a);
    kv_out[b] = kv2;
    if (out_blocks) out_blocks[b] = block_size > 0 ? (kv2 + block_size - 1) / block_size : 0;
    if (seq_status) seq_status[b] = st;
}

// Adaptive gamma for the next round: per request, the smallest g in
// [0, gmax] with the largest E(a, g) / (1 + g c) ("Speculative decoding"
// (inference.tusharamrit.in), actual speedup), a the running acceptance
// clamped to [0, 1], E(a, g) = 1 + a + ... + a^g summed term by term.
// Float32, every operation an explicit correctly rounded one in a fixed
// order (no contraction), so any IEEE machine gets the same gammas. Then
// speculation is off for the whole batch if its verify positions sum
// (g_b + 1) exceed max_positions (> 0) ("Speculative decoding"
// (mhtirogla.ai), Implementation notes).
constexpr int kAdaptThreads = 1024;  // one CTA: batches up to this size
constexpr int kAdaptBlock = 256;     // larger batches: one request per thread

__device__ int32_t best_gamma(float ema, int32_t gmax, float c) {
    float a = ema;
    if (!(a >= 0.f)) a = 0.f;
    if (a > 1.f) a = 1.f;
    float pw = 1.f, E = 1.f, best_sp = 0.f;
    int32_t best = 0;
#pragma unroll 4
    for (int32_t g = 0; g <= gmax; ++g) {  // the divisions of successive g overlap
        if (g > 0) {
            pw = __fmul_rn(pw, a);
            E = __fadd_rn(E, pw);
        }
        const float sp = __fdiv_rn(E, __fadd_rn(1.f, __fmul_rn((float)g, c)));
        if (g == 0 || sp > best_sp) {
            best_sp = sp;
            best = g;
        }
    }
    return best;
}

__device__ long long block_sum_ll(long long v, long long* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    long long t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
    return t;
}

// The whole batch in one CTA (B <= kAdaptThreads): choice, sum and switch.
__global__ void __launch_bounds__(kAdaptThreads) adapt_gamma_small(const float* ema, int32_t B, int32_t gmax, float c,
                                                                    int64_t max_positions, int32_t* gammas,
                                                                    int64_t* total) {
    __shared__ long long red[kAdaptThreads / 32];
    const int b = threadIdx.x;
    const int32_t g = b < B ? best_gamma(ema[b], gmax, c) : 0;
    const long long t = block_sum_ll(b < B ? g + 1 : 0, red);
    if (b < B) gammas[b] = (max_positions > 0 && t > max_positions) ? 0 : g;
    if (b == 0 && total) *total = t;
}

// Larger batches: each request's choice, and the positions summed into
// *total (zeroed before; integer atomics, so the sum does not depend on order).
__global__ void __launch_bounds__(kAdaptBlock) adapt_gamma_choose(const float* ema, int32_t B, int32_t gmax, float c,
                                                                   int32_t* gammas, unsigned long long* total) {
    __shared__ long long red[kAdaptBlock / 32];
    const int32_t b = blockIdx.x * kAdaptBlock + threadIdx.x;
    const int32_t g = b < B ? best_gamma(ema[b], gmax, c) : 0;
    if (b < B) gammas[b] = g;
    if (!total) return;
    const long long t = block_sum_ll(b < B ? g + 1 : 0, red);
    if (threadIdx.x == 0) atomicAdd(total, (unsigned long long)t);
}

// The switch for larger batches, after the sum is complete.
__global__ void __launch_bounds__(kAdaptBlock) adapt_gamma_switch(int32_t B, int64_t max_positions, int32_t* gammas,
                                                                   const int64_t* total) {
    const int32_t b = blockIdx.x * kAdaptBlock + threadIdx.x;
    if (b < B && *total > max_positions) gammas[b] = 0;
}

__global__ void debug_philox_kernel(uint64_t seed, uint64_t round, uint32_t seq_offset, int32_t B, int32_t npos,
                                    float* out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * npos) return;
    const int32_t b = (int32_t)(i / npos), pos = (int32_t)(i % npos);
    const float2 u = draw_uniforms(seed, round, seq_offset + (uint32_t)b, (uint32_t)pos);
    out[2 * i] = u.x;
    out[2 * i + 1] = u.y;
}

__global__ void debug_light_exp2_kernel(const float* x, float* y, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const df w = light_sum_df(light_exp2(x[i]), kEx2LightBias);
        y[2 * i] = w.hi;
        y[2 * i + 1] = w.lo;
    }
}

__global__ void debug_rowstats_kernel(const float2* rs, int64_t rows, int greedy, float* a, float* bb,
                                      int32_t* idx) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const float2 v = rs[r];
    if (a) a[r] = v.x;
    if (greedy) {
        if (idx) idx[r] = __float_as_int(v.y);
    } else if (bb) {
        bb[r] = v.y;
    }
}

constexpr int kDbgThreads = 1024;

__device__ df dbg_block_sum_df(df v, df* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = df_add(v, shfl_xor_df(v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    df t{0.f, 0.f};
    for (int w = 0; w < kDbgThreads / 32; ++w) t = df_add(t, red[w]);  // same order in every thread
    __syncthreads();
    return t;
}

__device__ __forceinline__ df dbg_weight(const char* row, int dt, int64_t j, float lmax, df k, bool probs,
                                         float tau, const Exp2Table& tab) {
    const float l = ld_elem_rt(row, dt, j);
    if (!(l >= tau)) return df{0.f, 0.f};  // below the row's top-k threshold (or NaN)
    if (probs) return df{(l > -INFINITY) ? l : 0.f, 0.f};
    return dt == SPECV_F32 ? logit_weight<true>(l, lmax, k, tab) : logit_weight<false>(l, lmax, k, tab);
}

// p_pos, q_pos and the normalised sampling weights of one position with the
// sampler's own weight, normaliser and residual arithmetic.
__global__ void __launch_bounds__(kDbgThreads) debug_probs_kernel(StatsParams p, int32_t seq, int32_t pos,
                                                                  float* out_p, float* out_q, float* out_w,
                                                                  float* out_sc) {
    __shared__ df red[kDbgThreads / 32];
    __shared__ Exp2Table tab;
    exp2_table_init(tab);
    const int64_t t0 = p.tro ? p.tro[seq] : (int64_t)seq * (p.gmax + 1);
    const int64_t d0 = p.dro ? p.dro[seq] : (int64_t)seq * p.gmax;
    const int64_t d1 = p.dro ? p.dro[seq + 1] : (int64_t)(seq + 1) * p.gmax;
    const int32_t g = (int32_t)(d1 - d0);
    if (pos > g || t0 < 0 || t0 + pos >= p.rows_t || d0 < 0 || (pos < g && d0 + pos >= p.rows_d)) {
        if (out_sc && threadIdx.x == 0)
            for (int i = 0; i < 4; ++i) out_sc[i] = NAN;
        return;
    }
    __syncthreads();
    const float T = p.temps ? p.temps[seq] : p.temperature;
    const df k = k_of_temperature(T);
    const bool draftpos = pos < g;
    const float mt = p.row_stats[t0 + pos].x;
    const float md = draftpos ? p.row_stats[p.rows_t + d0 + pos].x : 0.f;
    const int te = p.tdt == SPECV_F32 ? 4 : 2, de = p.ddt == SPECV_F32 ? 4 : 2;
    const char* trow = (const char*)p.tgt + (t0 + pos) * p.V * te;
    const char* drow = draftpos ? (const char*)p.dft + (d0 + pos) * p.V * de : trow;
    const bool probs = p.probs != 0;
    const float tt = p.tau ? p.tau[t0 + pos] : -INFINITY;
    const float td = (p.tau && draftpos) ? p.tau[p.rows_t + d0 + pos] : -INFINITY;
    df at{0.f, 0.f}, ad{0.f, 0.f};
    for (int64_t j = threadIdx.x; j < p.V; j += blockDim.x) {
        acc_add(at, dbg_weight(trow, p.tdt, j, mt, k, false, tt, tab));
        if (draftpos) acc_add(ad, dbg_weight(drow, p.ddt, j, md, k, probs, td, tab));
    }
    const df St = dbg_block_sum_df(df_norm(at), red);
    const df Sd = draftpos ? dbg_block_sum_df(df_norm(ad), red) : df{1.f, 0.f};
    const df It = df_recip(St), Id = df_recip(Sd);
    df az{0.f, 0.f};
    for (int64_t j = threadIdx.x; j < p.V; j += blockDim.x) {
        const df wt = dbg_weight(trow, p.tdt, j, mt, k, false, tt, tab);
        const df pv = df_mul(wt, It);
        df qv{0.f, 0.f};
        if (draftpos) {
            const df wd = dbg_weight(drow, p.ddt, j, md, k, probs, td, tab);
            qv = df_mul(wd, Id);
            acc_add(az, resid_weight(wt, wd, It, Id));
        }
        if (out_p) out_p[j] = pv.hi;
        if (out_q) out_q[j] = qv.hi;
    }
    const df Z = draftpos ? dbg_block_sum_df(df_norm(az), red) : df{1.f, 0.f};
    const bool use_r = draftpos && !residual_empty(Z);
    const df Iz = use_r ? df_recip(Z) : df{1.f, 0.f};
    if (out_w) {
        for (int64_t j = threadIdx.x; j < p.V; j += blockDim.x) {
            const df wt = dbg_weight(trow, p.tdt, j, mt, k, false, tt, tab);
            df w = df_mul(wt, It);
            if (use_r) w = df_mul(resid_weight(wt, dbg_weight(drow, p.ddt, j, md, k, probs, td, tab), It, Id), Iz);
            out_w[j] = w.hi;
        }
    }
    if (out_sc && threadIdx.x == 0) {
        const float2 pq = draftpos ? p.pq[d0 + pos] : make_float2(0.f, 0.f);
        out_sc[0] = pq.x;
        out_sc[1] = pq.y;
        out_sc[2] = draftpos ? Z.hi : -1.f;
        out_sc[3] = 0.f;
    }
}

}  // namespace

cudaError_t launch_kv_rollback(const int32_t* kv_in, int32_t* kv_out, const int32_t* accepted,
                               const int32_t* gammas, int32_t gmax, int32_t B, int32_t block_size,
                               int32_t* out_blocks, int32_t* seq_status, cudaStream_t s) {
    const int th = 256;
    kv_rollback_kernel<<<(B + th - 1) / th, th, 0, s>>>(kv_in, kv_out, accepted, gammas, gmax, B, block_size,
                                                        out_blocks, seq_status);
    return cudaGetLastError();
}

cudaError_t launch_debug_philox(uint64_t seed, uint64_t round, uint32_t seq_offset, int32_t B, int32_t npos,
                                float* out, cudaStream_t s) {
    const int64_t n = (int64_t)B * npos;
    const int th = 256;
    debug_philox_kernel<<<(unsigned)((n + th - 1) / th), th, 0, s>>>(seed, round, seq_offset, B, npos, out);
    return cudaGetLastError();
}

cudaError_t launch_debug_light_exp2(const float* x, float* y, int64_t n, cudaStream_t s) {
    const int th = 256;
    debug_light_exp2_kernel<<<(unsigned)((n + th - 1) / th), th, 0, s>>>(x, y, n);
    return cudaGetLastError();
}

cudaError_t launch_debug_rowstats(const float2* row_stats, int64_t rows, int greedy, float* out_a, float* out_b,
                                  int32_t* out_idx, cudaStream_t s) {
    const int th = 256;
    debug_rowstats_kernel<<<(unsigned)((rows + th - 1) / th), th, 0, s>>>(row_stats, rows, greedy, out_a, out_b,
                                                                          out_idx);
    return cudaGetLastError();
}

cudaError_t launch_adapt_gamma(const float* ema, int32_t B, int32_t gmax, float c, int64_t max_positions,
                               int32_t* gammas, int64_t* total, cudaStream_t s) {
    if (B <= kAdaptThreads) {
        adapt_gamma_small<<<1, kAdaptThreads, 0, s>>>(ema, B, gmax, c, max_positions, gammas, total);
        return cudaGetLastError();
    }
    const unsigned grid = (unsigned)((B + kAdaptBlock - 1) / kAdaptBlock);
    if (total && cudaMemsetAsync(total, 0, sizeof(int64_t), s) != cudaSuccess) return cudaErrorUnknown;
    adapt_gamma_choose<<<grid, kAdaptBlock, 0, s>>>(ema, B, gmax, c, gammas, (unsigned long long*)total);
    if (max_positions > 0) adapt_gamma_switch<<<grid, kAdaptBlock, 0, s>>>(B, max_positions, gammas, total);
    return cudaGetLastError();
}

cudaError_t launch_debug_probs(const StatsParams& p, int32_t seq, int32_t pos, float* out_p, float* out_q,
                               float* out_w, float* out_scalars, cudaStream_t s) {
    debug_probs_kernel<<<1, kDbgThreads, 0, s>>>(p, seq, pos, out_p, out_q, out_w, out_scalars);
    return cudaGetLastError();
}

}  // namespace specv
