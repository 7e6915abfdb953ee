// ngram.cu -- the n-gram (prompt lookup) drafter.
//
// Draft tokens at no model cost: search the sequence's own context for its
// last n tokens and propose what followed their latest earlier occurrence
// ("Speculative decoding" (mhtirogla.ai), Implementation notes: copy the
// continuation of the last matching n-gram; "Speculative decoding"
// (inference.tusharamrit.in), n-gram / prompt lookup). The search covers
// the whole context, n falls back from n_max to n_min, and the draft is at
// most gamma tokens, clipped at the end of the context.
//
// One CTA per sequence and one backward pass for every n at once. For a
// continuation position p (the token after a candidate occurrence), l(p) is
// the length, capped at n_max, of the common suffix of ctx[0 .. p) and of
// the whole context ctx[0 .. L); an n-gram match with start j = p - n exists
// iff l(p) >= n. Scanning p from L - 1 down, the first p at which l exceeds
// the best length so far is the latest position with that length, so the
// pair kept at the end is (the largest n with a match, its latest start):
// the fallback from n_max to n_min in one pass, which stops as soon as a
// match of n_max is found. Each thread tests kNgPer positions per chunk; a
// warp reduction and one barrier per chunk (per-warp results
// double-buffered) give the chunk's best.
#include "common.cuh"
#include "internal.h"

namespace specv {

namespace {

constexpr int kNgThreads = 1024;
constexpr int kNgWarps = kNgThreads / 32;
constexpr int kNgPer = 8;                       // positions per thread and chunk
constexpr int kNgChunk = kNgThreads * kNgPer;   // positions per chunk
constexpr uint32_t kIdxBits = 13;               // chunk index field (kNgChunk <= 8192)
static_assert(kNgChunk <= (1 << kIdxBits), "chunk index field");

// Encodes (length, position index within the chunk) so that the maximum is
// the longest match and, among equal lengths, the latest position.
__device__ __forceinline__ uint32_t ng_key(int32_t len, int32_t idx) {
    return ((uint32_t)len << kIdxBits) | (uint32_t)((1 << kIdxBits) - 1 - idx);
}

__global__ void __launch_bounds__(kNgThreads) ngram_kernel(const int32_t* ctx, const int64_t* off, int32_t nmax,
                                                           int32_t nmin, int32_t gamma, int32_t* draft,
                                                           int32_t* n_draft, int64_t* match_pos, int32_t* match_n) {
    __shared__ int32_t suf[kNgMaxN];              // suf[k - 1] = ctx[L - k]
    __shared__ uint32_t wbest[2][kNgWarps];
    const int32_t b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t o = __ldg(off + b), L = __ldg(off + b + 1) - o;
    const int32_t* c = ctx + o;
    const int32_t kmax = (int32_t)min((int64_t)nmax, L);  // the suffix cannot be longer than the context
    if (threadIdx.x < kmax) suf[threadIdx.x] = __ldg(c + L - 1 - threadIdx.x);
    __syncthreads();
    int32_t best_len = 0;
    int64_t best_p = -1;
    int par = 0;
    for (int64_t hi = L - 1; hi >= 1 && best_len < nmax; hi -= kNgChunk) {  // the same decisions in every thread
        uint32_t key = 0;
#pragma unroll
        for (int u = 0; u < kNgPer; ++u) {
            const int32_t idx = u * kNgThreads + threadIdx.x;
            const int64_t p = hi - idx;
            if (p < 1) continue;
            const int32_t lim = (int32_t)min((int64_t)kmax, p);
            int32_t len = 0;
            while (len < lim && __ldg(c + p - 1 - len) == suf[len]) ++len;
            if (len > 0) key = max(key, ng_key(len, idx));
        }
        key = __reduce_max_sync(0xffffffffu, key);
        if (lane == 0) wbest[par][warp] = key;
        __syncthreads();
        uint32_t k = 0;
#pragma unroll
        for (int w = 0; w < kNgWarps; ++w) k = max(k, wbest[par][w]);
        par ^= 1;
        const int32_t len = (int32_t)(k >> kIdxBits);
        if (len > best_len) {  // later chunks (earlier positions) replace only with a longer match
            best_len = len;
            best_p = hi - ((1 << kIdxBits) - 1 - (int32_t)(k & ((1u << kIdxBits) - 1)));
        }
    }
    const bool found = best_len >= nmin;
    const int32_t n = found ? best_len : 0;
    const int64_t j = found ? best_p - n : -1;
    const int64_t from = found ? best_p : 0;  // first drafted position
    for (int32_t i = threadIdx.x; i < gamma; i += kNgThreads) {
        const bool has = found && from + i < L;
        draft[(int64_t)b * gamma + i] = has ? __ldg(c + from + i) : -1;
    }
    if (threadIdx.x == 0) {
        n_draft[b] = found ? (int32_t)min((int64_t)gamma, L - from) : 0;
        if (match_pos) match_pos[b] = j;
        if (match_n) match_n[b] = n;
    }
}

}  // namespace

cudaError_t launch_ngram(const int32_t* ctx, const int64_t* off, int32_t B, int32_t nmax, int32_t nmin, int32_t gamma,
                         int32_t* draft, int32_t* n_draft, int64_t* match_pos, int32_t* match_n, cudaStream_t s) {
    ngram_kernel<<<(unsigned)B, kNgThreads, 0, s>>>(ctx, off, nmax, nmin, gamma, draft, n_draft, match_pos, match_n);
    return cudaGetLastError();
}

}  // namespace specv
