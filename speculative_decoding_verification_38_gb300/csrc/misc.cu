// misc.cu -- the standalone KV-length rollback and the test hooks.
#include <math.h>

#include "common.cuh"

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

__global__ void debug_philox_kernel(uint64_t seed, uint64_t round, uint32_t seq_offset, int32_t B, int32_t npos,
                                    float* out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * npos) return;
    const int32_t b = (int32_t)(i / npos), pos = (int32_t)(i % npos);
    const float2 u = draw_uniforms(seed, round, seq_offset + (uint32_t)b, (uint32_t)pos);
    out[2 * i] = u.x;
    out[2 * i + 1] = u.y;
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

__device__ float dbg_block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    if (threadIdx.x == 0)
        for (int w = 0; w < kDbgThreads / 32; ++w) t += red[w];
    __syncthreads();
    if (threadIdx.x == 0) red[0] = t;
    __syncthreads();
    t = red[0];
    __syncthreads();
    return t;
}

// p_pos, q_pos and the normalised sampling weights of one position, from the
// row statistics the last sampling call stored (same formulas as the sampler).
__global__ void __launch_bounds__(kDbgThreads) debug_probs_kernel(StatsParams p, int32_t seq, int32_t pos,
                                                                  float* out_p, float* out_q, float* out_w,
                                                                  float* out_sc) {
    __shared__ float red[kDbgThreads / 32];
    const int64_t t0 = p.tro ? p.tro[seq] : (int64_t)seq * (p.gmax + 1);
    const int64_t d0 = p.dro ? p.dro[seq] : (int64_t)seq * p.gmax;
    const int64_t d1 = p.dro ? p.dro[seq + 1] : (int64_t)(seq + 1) * p.gmax;
    const int32_t g = (int32_t)(d1 - d0);
    if (pos > g || t0 < 0 || t0 + pos >= p.rows_t || d0 < 0 || (pos < g && d0 + pos >= p.rows_d)) {
        if (out_sc && threadIdx.x == 0)
            for (int i = 0; i < 4; ++i) out_sc[i] = NAN;
        return;
    }
    const float T = p.temps ? p.temps[seq] : p.temperature;
    const float k = kLog2e / T;
    const bool draftpos = pos < g;
    const float2 ts = p.row_stats[t0 + pos];
    const float2 ds = draftpos ? p.row_stats[p.rows_t + d0 + pos] : make_float2(0.f, 1.f);
    const int te = p.tdt == SPECV_F32 ? 4 : 2, de = p.ddt == SPECV_F32 ? 4 : 2;
    const char* trow = (const char*)p.tgt + (t0 + pos) * p.V * te;
    const char* drow = draftpos ? (const char*)p.dft + (d0 + pos) * p.V * de : trow;
    const float inv_st = 1.0f / ts.y, inv_sd = 1.0f / ds.y;
    float zpart = 0.f;
    for (int64_t j = threadIdx.x; j < p.V; j += blockDim.x) {
        const float pv = __fmul_rn(ex2(__fmaf_rn(ld_elem_rt(trow, p.tdt, j), k, -ts.x)), inv_st);
        float qv = 0.f;
        if (draftpos) {
            const float l = ld_elem_rt(drow, p.ddt, j);
            qv = p.probs ? __fmul_rn(l, inv_sd) : __fmul_rn(ex2(__fmaf_rn(l, k, -ds.x)), inv_sd);
        }
        if (out_p) out_p[j] = pv;
        if (out_q) out_q[j] = qv;
        zpart += draftpos ? fmaxf(pv - qv, 0.f) : pv;
    }
    const float Z = dbg_block_sum(zpart, red);
    const bool use_r = draftpos && Z > 0.f;
    float wsum = use_r ? Z : 1.f;
    if (!use_r && draftpos) {
        float s2 = 0.f;
        for (int64_t j = threadIdx.x; j < p.V; j += blockDim.x)
            s2 += __fmul_rn(ex2(__fmaf_rn(ld_elem_rt(trow, p.tdt, j), k, -ts.x)), inv_st);
        wsum = dbg_block_sum(s2, red);
    }
    if (out_w) {
        for (int64_t j = threadIdx.x; j < p.V; j += blockDim.x) {
            const float pv = __fmul_rn(ex2(__fmaf_rn(ld_elem_rt(trow, p.tdt, j), k, -ts.x)), inv_st);
            float w = pv;
            if (use_r) {
                const float l = ld_elem_rt(drow, p.ddt, j);
                const float qv = p.probs ? __fmul_rn(l, inv_sd) : __fmul_rn(ex2(__fmaf_rn(l, k, -ds.x)), inv_sd);
                w = fmaxf(pv - qv, 0.f);
            }
            out_w[j] = w / wsum;
        }
    }
    if (out_sc && threadIdx.x == 0) {
        const float2 pq = draftpos ? p.pq[d0 + pos] : make_float2(0.f, 0.f);
        const SampleTask tk = p.tasks[seq];
        const bool sampled_here = tk.mode != kTaskNone && tk.out_slot == t0 + pos;
        out_sc[0] = pq.x;
        out_sc[1] = pq.y;
        out_sc[2] = (sampled_here && draftpos) ? tk.z : (draftpos ? Z : -1.f);
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

cudaError_t launch_debug_rowstats(const float2* row_stats, int64_t rows, int greedy, float* out_a, float* out_b,
                                  int32_t* out_idx, cudaStream_t s) {
    const int th = 256;
    debug_rowstats_kernel<<<(unsigned)((rows + th - 1) / th), th, 0, s>>>(row_stats, rows, greedy, out_a, out_b,
                                                                          out_idx);
    return cudaGetLastError();
}

cudaError_t launch_debug_probs(const StatsParams& p, int32_t seq, int32_t pos, float* out_p, float* out_q,
                               float* out_w, float* out_scalars, cudaStream_t s) {
    debug_probs_kernel<<<1, kDbgThreads, 0, s>>>(p, seq, pos, out_p, out_q, out_w, out_scalars);
    return cudaGetLastError();
}

}  // namespace specv
