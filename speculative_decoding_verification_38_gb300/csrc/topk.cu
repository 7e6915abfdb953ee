// topk.cu -- top-k truncation for the sampling verify.
//
// Both models' rows go through the same processing ("Speculative decoding"
// (mhtirogla.ai), Implementation notes), so a sequence that samples from its
// top k truncates its target rows and its draft rows alike: a row keeps every
// column whose value is at least tau, the row's k-th largest value (NaN ranks
// as -inf; ties at tau all stay), and its distribution is renormalised over
// the kept columns. For every row this pass writes tau and the statistics the
// rest of the step reads: logits rows (m, s), m the raw maximum and
// s = sum over kept columns of 2^(l k - fl(m k)), k = log2(e) / T;
// probabilities rows (0, sum of the kept values).
//
// One CTA per row (four resident per SM) and one read of the row from HBM.
// Each warp filters its share of the row against a threshold that only
// rises and keeps, in a shared-memory buffer, every value at least that
// large. The threshold starts, after the first batch of loads, at the k-th
// largest of the maxima of every 16-byte vector the CTA loaded (k distinct
// vectors each hold a value at least that large, so it cannot pass tau),
// found by a CTA bisection on order-preserving keys. When a warp's buffer
// fills, the warp raises its threshold to the k-th largest of its entries,
// drops what lies below and shares the new bound with the other warps. Every
// threshold is a proven lower bound of tau, so the buffers together hold
// every kept column; the CTA then bisects for tau over the buffers and sums
// the kept entries' weights in a fixed order (the result does not depend on
// timing). Rows where that cannot work (k past half a buffer, more equal
// values than a buffer holds, k off) select over the row itself in L2, one
// read per radix digit, and sum it in one more read.
//
// With top-p as well, a top-p row's kept values go to the workspace and a
// second kernel (nucleus_kernel) takes the nucleus inside them, one warp per
// row, with the loads done: the streaming pass keeps no serial tail. A row
// with top-p but no top-k passes through this pass whole (its maximum and
// sum) and a third kernel (alone_kernel) takes the nucleus of the whole row,
// one CTA per row.
#include <math.h>

#include <algorithm>

#include "precise.cuh"

namespace specv {

namespace {

constexpr int kTkThreads = 256;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkUnroll = 8;        // 16-byte loads in flight per lane
constexpr int kBufBytes = 4096;     // candidate buffer per warp
constexpr unsigned kFull = 0xffffffffu;

struct TkSmem {
    uint32_t buf[kTkWarps][kBufBytes / 4];  // candidate value bits (u16 for bf16, u32 for f32)
    uint32_t hist[256];                     // the CTA's radix histogram
    uint32_t thr_key;                       // largest threshold key any warp has proven (a lower bound of tau's)
    int32_t cnt[kTkWarps];
    int32_t ovf[kTkWarps];
    float mx[kTkWarps];
    int32_t nan[kTkWarps];
    float red[kTkWarps];
    uint32_t sel_bin, sel_above;
    uint32_t bis[2][3][kTkWarps];  // block bisection: per-warp counts, double-buffered
    int32_t kc[kTkWarps];          // per-warp counts of kept values (top-p rows)
};
constexpr size_t kTkSmemBytes = sizeof(TkSmem);

// --------------------------------------------------------- order-preserving keys
// Storage bits of one value with -0 folded into +0, so that equal values have
// equal bits. bf16: the 16-bit pattern; f32: the 32-bit pattern.
template <int DT>
struct KeyTraits;
template <>
struct KeyTraits<SPECV_BF16> {
    using Bits = uint16_t;
    static constexpr int kDigits = 2;  // 16-bit keys
    static constexpr int kEsz = 2;
    __device__ static uint32_t canon(uint32_t h) { return h == 0x8000u ? 0u : h; }
    __device__ static float value(uint32_t h) { return __uint_as_float(h << 16); }
    // unsigned key whose order is the order of the values (NaN excluded)
    __device__ static uint32_t key(uint32_t h) { return h ^ ((h & 0x8000u) ? 0xFFFFu : 0x8000u); }
    __device__ static uint32_t bits_of_key(uint32_t k) { return k ^ ((k & 0x8000u) ? 0x8000u : 0xFFFFu); }
};
template <>
struct KeyTraits<SPECV_F32> {
    using Bits = uint32_t;
    static constexpr int kDigits = 4;  // 32-bit keys
    static constexpr int kEsz = 4;
    __device__ static uint32_t canon(uint32_t h) { return h == 0x80000000u ? 0u : h; }
    __device__ static float value(uint32_t h) { return __uint_as_float(h); }
    __device__ static uint32_t key(uint32_t h) { return h ^ ((h & 0x80000000u) ? 0xFFFFFFFFu : 0x80000000u); }
    __device__ static uint32_t bits_of_key(uint32_t k) {
        return k ^ ((k & 0x80000000u) ? 0x80000000u : 0xFFFFFFFFu);
    }
};

// Key of a loaded value for the selects over the row: NaN ranks lowest
// (as -inf would), -0 as +0.
template <int DT>
__device__ __forceinline__ uint32_t key_of_value(float v) {
    using KT = KeyTraits<DT>;
    if (v != v) return 0u;
    const uint32_t b = DT == SPECV_BF16 ? (__float_as_uint(v) >> 16) : __float_as_uint(v);
    return KT::key(KT::canon(b));
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Find, in a 256-bin histogram, the digit b holding the `remaining`-th
// largest key: sum_{b' > b} h[b'] < remaining <= sum_{b' >= b} h[b']. One
// warp; lane L reads bins 8L..8L+7. Needs 1 <= remaining <= sum h. Returns b
// and (in `above`) the count in the bins above it, in every lane.
__device__ __forceinline__ uint32_t warp_find_bin(const uint32_t* h, uint32_t remaining, uint32_t& above) {
    const int lane = threadIdx.x & 31;
    uint32_t c[8], t = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        c[j] = h[lane * 8 + j];
        t += c[j];
    }
    uint32_t s = t;  // inclusive suffix sum over lanes lane..31
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(kFull, s, o);
        if (lane + o < 32) s += v;
    }
    const uint32_t hi = s - t;  // keys in the bins of higher lanes
    const bool mine = hi < remaining && remaining <= s;
    uint32_t bin = 0, ab = 0;
    if (mine) {
        uint32_t acc = hi;
#pragma unroll
        for (int j = 7; j >= 0; --j) {
            if (acc + c[j] >= remaining) {
                bin = lane * 8 + j;
                ab = acc;
                break;
            }
            acc += c[j];
        }
    }
    const uint32_t owner = __ballot_sync(kFull, mine);
    const int src = owner ? __ffs(owner) - 1 : 0;
    above = __shfl_sync(kFull, ab, src);
    return __shfl_sync(kFull, bin, src);
}

// The kk-th largest key among a warp's buffer entries (1 <= kk <= cnt): the
// largest K with #{key >= K} >= kk, found bit by bit from the top.
template <int DT>
__device__ uint32_t warp_kth_buf(const typename KeyTraits<DT>::Bits* wb, int cnt, uint32_t kk) {
    using KT = KeyTraits<DT>;
    const int lane = threadIdx.x & 31;
    uint32_t prefix = 0;
#pragma unroll 1
    for (int b = 8 * KT::kDigits - 1; b >= 0; --b) {
        const uint32_t cand = prefix | (1u << b);
        uint32_t c = 0;
        for (int e = lane; e < cnt; e += 32) c += KT::key(wb[e]) >= cand ? 1u : 0u;
        if (__reduce_add_sync(kFull, c) >= kk) prefix = cand;
    }
    return prefix;
}

// Keep the entries whose key is at least kmin, in order (in place).
template <int DT>
__device__ int warp_compact(typename KeyTraits<DT>::Bits* wb, int cnt, uint32_t kmin) {
    using KT = KeyTraits<DT>;
    const int lane = threadIdx.x & 31;
    int out = 0;
    for (int base = 0; base < cnt; base += 32) {
        const int e = base + lane;
        const uint32_t bits = e < cnt ? (uint32_t)wb[e] : 0u;
        const bool keep = e < cnt && KT::key(bits) >= kmin;
        const uint32_t bal = __ballot_sync(kFull, keep);
        __syncwarp();  // every lane has read its entry before any write
        if (keep) wb[out + __popc(bal & lanemask_lt())] = (typename KT::Bits)bits;
        out += __popc(bal);
        __syncwarp();
    }
    return out;
}

// ------------------------------------------------------- the filtering pass
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ float max_nan_f32(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// Largest of the values in one 16-byte vector; NaN if any is NaN.
template <int DT>
__device__ __forceinline__ float vec_max(const uint4& q) {
    if constexpr (DT == SPECV_BF16) {
        const uint32_t m2 = max_nan_bf16x2(max_nan_bf16x2(q.x, q.y), max_nan_bf16x2(q.z, q.w));
        return max_nan_f32(bf16_lo(m2), bf16_hi(m2));
    } else {
        return max_nan_f32(max_nan_f32(__uint_as_float(q.x), __uint_as_float(q.y)),
                           max_nan_f32(__uint_as_float(q.z), __uint_as_float(q.w)));
    }
}

// Append this lane's values of one vector that are >= thr (when `need`) to
// the warp's buffer: lanes in order, each lane's values in column order.
template <int DT>
__device__ __noinline__ void warp_append(typename KeyTraits<DT>::Bits* wb, int& cnt, const uint4& q, bool need,
                                            float thr) {
    using KT = KeyTraits<DT>;
    constexpr int EPV = 16 / KT::kEsz;
    const int lane = threadIdx.x & 31;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint32_t bits[EPV];
    bool c[EPV];
    int n = 0;
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
        bits[e] = DT == SPECV_BF16 ? ((e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu)) : w[e];
        c[e] = need && KT::value(bits[e]) >= thr;
        n += c[e] ? 1 : 0;
    }
    int incl = n;  // inclusive scan of the counts over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
    }
    int pos = cnt + incl - n;
#pragma unroll
    for (int e = 0; e < EPV; ++e)
        if (c[e]) wb[pos++] = (typename KT::Bits)KT::canon(bits[e]);
    cnt += __shfl_sync(kFull, incl, 31);
}

// Threshold state of one warp: a key every value it must keep reaches, and
// the value of that key (-inf while no key is known).
struct WarpThr {
    uint32_t key;
    float val;
};

template <int DT>
__device__ __forceinline__ void raise_thr(WarpThr& t, uint32_t k) {
    using KT = KeyTraits<DT>;
    if (k > t.key) {
        t.key = k;
        t.val = KT::value(KT::bits_of_key(k));
    }
}

// Make room in a full buffer: drop the entries below the warp's threshold
// (another warp may have raised it); if that is not enough, raise the
// threshold to the kk-th largest entry and drop again. Returns false when
// the survivors (ties) still leave fewer than `room` free entries.
template <int DT>
__device__ __noinline__ bool warp_make_room(typename KeyTraits<DT>::Bits* wb, int& cnt, uint32_t kk, WarpThr& thr,
                               uint32_t* shared_key, int room) {
    constexpr int C = kBufBytes / KeyTraits<DT>::kEsz;
    cnt = warp_compact<DT>(wb, cnt, thr.key);
    if (cnt <= C - room) return true;
    const uint32_t K = warp_kth_buf<DT>(wb, cnt, kk);  // cnt > C - room >= kk
    raise_thr<DT>(thr, K);
    if ((threadIdx.x & 31) == 0) atomicMax(shared_key, K);
    cnt = warp_compact<DT>(wb, cnt, thr.key);
    return cnt <= C - room;
}

// The kk-th largest key over the keys every thread counts (the largest K
// with #{key >= K} >= kk; 0 if there are fewer than kk), two bits per
// round: count(c1, c2, c3, n1, n2, n3) gives this thread's numbers of keys
// at least c1 < c2 < c3. One barrier per round (the per-warp totals are
// double-buffered). Every thread of the CTA calls it and gets the result.
template <int BITS, class Count>
__device__ uint32_t block_kth(uint32_t kk, TkSmem& sm, const Count& count) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t prefix = 0;
#pragma unroll 1
    for (int b = BITS - 2; b >= 0; b -= 2) {
        const uint32_t c1 = prefix | (1u << b), c2 = prefix | (2u << b), c3 = prefix | (3u << b);
        uint32_t n1 = 0, n2 = 0, n3 = 0;
        count(c1, c2, c3, n1, n2, n3);
        n1 = __reduce_add_sync(kFull, n1);
        n2 = __reduce_add_sync(kFull, n2);
        n3 = __reduce_add_sync(kFull, n3);
        const int par = (b >> 1) & 1;
        if (lane == 0) {
            sm.bis[par][0][warp] = n1;
            sm.bis[par][1][warp] = n2;
            sm.bis[par][2][warp] = n3;
        }
        __syncthreads();
        uint32_t t1 = 0, t2 = 0, t3 = 0;
#pragma unroll
        for (int w = 0; w < kTkWarps; ++w) {
            t1 += sm.bis[par][0][w];
            t2 += sm.bis[par][1][w];
            t3 += sm.bis[par][2][w];
        }
        prefix = t3 >= kk ? c3 : (t2 >= kk ? c2 : (t1 >= kk ? c1 : prefix));
    }
    return prefix;
}

// One warp's share of the row: vectors it + u * kTkThreads + warp * 32 + lane
// (u < kTkUnroll) of every iteration, plus, for warp 0, the columns before
// the first 16-byte boundary and after the last full vector. With `filt`,
// the warp keeps in its buffer (in the order met) every value of its share
// at least as large as its threshold. The threshold starts at the kk-th
// largest of the maxima of every vector the CTA's first iteration loaded
// (kk vectors each hold a value at least that large, so it cannot pass tau)
// and rises with every select any warp makes (shared through sm.thr_key).
// The warp's maximum, NaN flag, entry count and overflow flag go to shared
// memory.
template <int DT>
__device__ void filter_pass(const char* row, int64_t V, uint32_t kk, bool filt, TkSmem& sm) {
    using KT = KeyTraits<DT>;
    using Bits = typename KT::Bits;
    constexpr int ESZ = KT::kEsz, EPV = 16 / ESZ, C = kBufBytes / ESZ, STEP = 32 * EPV;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Bits* wb = reinterpret_cast<Bits*>(sm.buf[warp]);
    volatile uint32_t* shared_key = &sm.thr_key;
    int64_t head = (int64_t)(((16u - (uint32_t)((uintptr_t)row & 15u)) & 15u) / ESZ);
    if (head > V) head = V;
    const int64_t nvec = (V - head) / EPV;
    const int64_t tail0 = head + nvec * EPV;
    const uint4* vrow = reinterpret_cast<const uint4*>(row + head * ESZ);
    WarpThr thr{0u, -INFINITY};
    float lmax = -INFINITY;
    int cnt = 0;
    bool nan = false, ovf = false;

    if (filt && nvec > 0) {  // the first threshold (the whole CTA; its loads come back from L2 in the loop)
        float mx[kTkUnroll];
#pragma unroll
        for (int u = 0; u < kTkUnroll; ++u) {
            const int64_t vi = warp * 32 + lane + (int64_t)u * kTkThreads;
            mx[u] = vi < nvec ? vec_max<DT>(ld_stream_v4(vrow + vi)) : -INFINITY;
        }
        const uint32_t K0 = block_kth<8 * KT::kDigits>(
            kk, sm, [&](uint32_t c1, uint32_t c2, uint32_t c3, uint32_t& n1, uint32_t& n2, uint32_t& n3) {
#pragma unroll
                for (int u = 0; u < kTkUnroll; ++u) {
                    const uint32_t key = key_of_value<DT>(mx[u]);
                    n1 += key >= c1 ? 1u : 0u;
                    n2 += key >= c2 ? 1u : 0u;
                    n3 += key >= c3 ? 1u : 0u;
                }
            });
        raise_thr<DT>(thr, K0);
        if (threadIdx.x == 0 && K0) atomicMax(&sm.thr_key, K0);
    }

    for (int64_t it = 0; it < nvec; it += (int64_t)kTkUnroll * kTkThreads) {
        const int64_t v0 = it + warp * 32 + lane;
        uint4 q[kTkUnroll];
#pragma unroll
        for (int u = 0; u < kTkUnroll; ++u) {
            const int64_t vi = v0 + (int64_t)u * kTkThreads;
            q[u] = vi < nvec ? ld_stream_v4(vrow + vi) : make_uint4(0u, 0u, 0u, 0u);
        }
        float mx[kTkUnroll];
#pragma unroll
        for (int u = 0; u < kTkUnroll; ++u) {
            const bool valid = v0 + (int64_t)u * kTkThreads < nvec;
            const float m = vec_max<DT>(q[u]);
            nan |= valid && m != m;
            mx[u] = valid ? m : -INFINITY;
            lmax = fmaxf(lmax, mx[u]);
        }
        if (!filt) continue;
        raise_thr<DT>(thr, *shared_key);
#pragma unroll
        for (int u = 0; u < kTkUnroll; ++u) {
            const bool valid = v0 + (int64_t)u * kTkThreads < nvec;
            bool need = valid && mx[u] >= thr.val;
            if (!__any_sync(kFull, need)) continue;
            if (cnt > C - STEP) {
                raise_thr<DT>(thr, *shared_key);
                if (!warp_make_room<DT>(wb, cnt, kk, thr, &sm.thr_key, STEP)) {
                    filt = false;
                    ovf = true;
                    break;
                }
                need = valid && mx[u] >= thr.val;
            }
            warp_append<DT>(wb, cnt, q[u], need, thr.val);
        }
    }
    if (warp == 0) {  // the ragged ends: at most EPV - 1 columns each
        int64_t col = -1;
        if (lane < head)
            col = lane;
        else if (lane >= 16 && (int64_t)(lane - 16) < V - tail0)
            col = tail0 + (lane - 16);
        const float v = col >= 0 ? ld_elem<DT>(row, col) : -INFINITY;
        nan |= v != v;
        lmax = fmaxf(lmax, v);
        if (filt) {
            bool need = col >= 0 && v >= thr.val;
            if (__any_sync(kFull, need)) {
                bool ok = true;
                if (cnt > C - 32) {
                    ok = warp_make_room<DT>(wb, cnt, kk, thr, &sm.thr_key, 32);
                    need = col >= 0 && v >= thr.val;
                }
                if (ok) {
                    const uint32_t bits = DT == SPECV_BF16 ? (__float_as_uint(v) >> 16) : __float_as_uint(v);
                    const uint32_t bal = __ballot_sync(kFull, need);
                    if (need) wb[cnt + __popc(bal & lanemask_lt())] = (Bits)KT::canon(bits);
                    cnt += __popc(bal);
                } else {
                    ovf = true;
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(kFull, lmax, o));
    nan = __any_sync(kFull, nan);
    if (lane == 0) {
        sm.cnt[warp] = cnt;
        sm.ovf[warp] = ovf;
        sm.mx[warp] = lmax;
        sm.nan[warp] = nan;
    }
}

// ------------------------------------------------------------ CTA level
// The kk-th largest key over every key `each` visits (each thread visits its
// own share; 1 <= kk <= their number), by MSD radix select with the CTA's
// histogram hist[0].
template <int DT, class Each>
__device__ uint32_t block_select(uint32_t kk, TkSmem& sm, const Each& each) {
    using KT = KeyTraits<DT>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t* h = sm.hist;
    uint32_t prefix = 0, remaining = kk;
#pragma unroll 1
    for (int d = KT::kDigits - 1; d >= 0; --d) {
        const int sh = 8 * d;
        __syncthreads();  // the last users of h and sel_* are done
        for (int i = threadIdx.x; i < 256; i += kTkThreads) h[i] = 0;
        __syncthreads();
        each([&](uint32_t key) {
            if (d == KT::kDigits - 1 || (key >> (sh + 8)) == (prefix >> (sh + 8)))
                atomicAdd(&h[(key >> sh) & 255u], 1u);
        });
        __syncthreads();
        if (warp == 0) {
            uint32_t above;
            const uint32_t bin = warp_find_bin(h, remaining, above);
            if (lane == 0) {
                sm.sel_bin = bin;
                sm.sel_above = above;
            }
        }
        __syncthreads();
        prefix |= sm.sel_bin << sh;
        remaining -= sm.sel_above;
    }
    return prefix;
}

// Sum over the CTA, the same association whatever the timing.
__device__ float block_sum_fixed(float v, TkSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    if (lane == 0) sm.red[warp] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kTkWarps; ++w) t += sm.red[w];
    return t;
}

// Weight of a kept value: 2^(l k - fl(m k)) for logits, the value itself for
// probabilities.
__device__ __forceinline__ float kept_weight(float v, bool probs_row, float k2, float nmk) {
    return probs_row ? v : ex2(__fmaf_rn(v, k2, nmk));
}

template <int DT>
__device__ void row_topk(const StatsParams& p, int64_t r, const char* row, int64_t kk, bool off, bool probs_row,
                         float k2, float tp, TkSmem& sm) {
    using KT = KeyTraits<DT>;
    using Bits = typename KT::Bits;
    constexpr int C = kBufBytes / KT::kEsz;
    const int64_t V = p.V;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool filt = !off && kk <= C / 2;
    const bool topp = !off && tp > 0.f && tp < 1.f && p.keep;  // the nucleus kernel takes this row next
    if (threadIdx.x == 0) sm.thr_key = 0u;
    __syncthreads();
    filter_pass<DT>(row, V, (uint32_t)kk, filt, sm);
    __syncthreads();
    float m = -INFINITY;
    bool nan = false, ovf = false;
#pragma unroll
    for (int w = 0; w < kTkWarps; ++w) {
        m = fmaxf(m, sm.mx[w]);
        nan |= sm.nan[w] != 0;
        ovf |= sm.ovf[w] != 0;
    }
    const float nmk = -__fmul_rn(m, k2);
    float tau = -INFINITY, acc = 0.f;
    if (!off && filt && !ovf) {
        // tau over the union of the buffers, then the kept entries' weights
        const Bits* wb = reinterpret_cast<const Bits*>(sm.buf[warp]);
        const int cnt = sm.cnt[warp];
        const uint32_t K = block_kth<8 * KT::kDigits>(
            (uint32_t)kk, sm, [&](uint32_t c1, uint32_t c2, uint32_t c3, uint32_t& n1, uint32_t& n2, uint32_t& n3) {
                for (int e = lane; e < cnt; e += 32) {
                    const uint32_t key = KT::key(wb[e]);
                    n1 += key >= c1 ? 1u : 0u;
                    n2 += key >= c2 ? 1u : 0u;
                    n3 += key >= c3 ? 1u : 0u;
                }
            });
        tau = KT::value(KT::bits_of_key(K));
        for (int e = lane; e < cnt; e += 32) {
            const float v = KT::value(wb[e]);
            if (v >= tau) acc += kept_weight(v, probs_row, k2, nmk);
        }
        if (topp) {  // the kept values' keys for the nucleus kernel, warp by warp, in buffer order
            int c = 0;
            for (int e = lane; e < cnt; e += 32) c += KT::value(wb[e]) >= tau ? 1 : 0;
            c = (int)__reduce_add_sync(kFull, (uint32_t)c);
            if (lane == 0) sm.kc[warp] = c;
            __syncthreads();
            int off_w = 0, tot = 0;
#pragma unroll
            for (int w = 0; w < kTkWarps; ++w) {
                off_w += w < warp ? sm.kc[w] : 0;
                tot += sm.kc[w];
            }
            if (tot <= kKeepCap) {
                uint32_t* dst = p.keep + r * kKeepCap + off_w;
                int base = 0;
                for (int e0 = 0; e0 < cnt; e0 += 32) {
                    const int e = e0 + lane;
                    const bool keep = e < cnt && KT::value(wb[e]) >= tau;
                    const uint32_t bal = __ballot_sync(kFull, keep);
                    if (keep) dst[base + __popc(bal & lanemask_lt())] = KT::key(wb[e]);
                    base += __popc(bal);
                }
            }
            if (threadIdx.x == 0) p.keep_n[r] = tot <= kKeepCap ? tot : -1;
        }
    } else {
        // over the row itself (in L2 after the pass)
        if (!off) {
            const uint32_t K = block_select<DT>((uint32_t)kk, sm, [&](auto&& f) {
                for (int64_t j = threadIdx.x; j < V; j += kTkThreads) f(key_of_value<DT>(ld_elem<DT>(row, j)));
            });
            tau = KT::value(KT::bits_of_key(K));
        }
        for (int64_t j = threadIdx.x; j < V; j += kTkThreads) {
            const float v = ld_elem<DT>(row, j);
            if (v >= tau) acc += kept_weight(v, probs_row, k2, nmk);
        }
        if (topp && threadIdx.x == 0) p.keep_n[r] = -1;  // the nucleus kernel reads the row
    }
    float s = block_sum_fixed(acc, sm);
    if (threadIdx.x == 0) {
        if (nan) s = NAN;  // a NaN anywhere makes the row invalid
        p.row_stats[r] = make_float2(probs_row ? 0.f : m, s);
        p.tau[r] = tau;
    }
}

// Sequence owning local row lr of the target (draft = false) or draft
// tensor, or -1 if none does.
__device__ int32_t row_seq(const StatsParams& p, bool draft, int64_t lr) {
    const int64_t* off = draft ? p.dro : p.tro;
    if (!off) {
        const int64_t per = draft ? p.gmax : p.gmax + 1;
        const int64_t b = per > 0 ? lr / per : p.B;
        return b < p.B ? (int32_t)b : -1;
    }
    int32_t lo = 0, hi = p.B - 1;  // largest b with off[b] <= lr
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (__ldg(off + mid) <= lr)
            lo = mid;
        else
            hi = mid - 1;
    }
    if (lr < __ldg(off + lo) || lr >= __ldg(off + lo + 1)) return -1;
    return lo;
}

// Whether row r is a bf16 logits row of a sequence that samples from its
// top-p nucleus with top-k off: whole_nucleus_kernel takes such a row whole
// (its maximum, nucleus and sum over the nucleus), and the top-k pass and
// alone_kernel leave it. Only with p.keep (some top-p on).
__device__ bool whole_bf16_row(const StatsParams& p, int64_t r) {
    if (!p.keep) return false;
    const bool is_t = r < p.rows_t;
    if ((is_t ? p.tdt : p.ddt) != SPECV_BF16 || (!is_t && p.probs != 0)) return false;
    const int32_t b = row_seq(p, !is_t, is_t ? r : r - p.rows_t);
    if (b < 0) return false;
    const int64_t kk = p.top_ks ? (int64_t)__ldg(p.top_ks + b) : (int64_t)p.top_k;
    const float tp = p.top_ps ? __ldg(p.top_ps + b) : p.top_p;
    return !(kk >= 1 && kk < p.V) && tp > 0.f && tp < 1.f;
}

__global__ void __launch_bounds__(kTkThreads, 4) topk_kernel(StatsParams p) {
    extern __shared__ __align__(16) unsigned char tk_raw[];
    TkSmem& sm = *reinterpret_cast<TkSmem*>(tk_raw);
    pdl_launch_dependents();
    const int64_t r = blockIdx.x;
    if (whole_bf16_row(p, r)) return;
    const bool is_t = r < p.rows_t;
    const int64_t lr = is_t ? r : r - p.rows_t;
    const int32_t b = row_seq(p, !is_t, lr);
    const int dt = is_t ? p.tdt : p.ddt;
    const bool probs_row = !is_t && p.probs != 0;
    const int64_t kk = b < 0 ? 0 : (p.top_ks ? (int64_t)__ldg(p.top_ks + b) : (int64_t)p.top_k);
    const bool off = kk <= 0 || kk >= p.V;
    float T = b < 0 ? 1.f : (p.temps ? __ldg(p.temps + b) : p.temperature);
    if (!(T > 0.f) || !isfinite(T)) T = 1.f;  // the finalize reports the sequence's bad temperature
    const float k2 = kLog2e / T;
    const float tp = b < 0 ? 0.f : (p.top_ps ? __ldg(p.top_ps + b) : p.top_p);
    const int64_t esz = dt == SPECV_F32 ? 4 : 2;
    const char* row = (const char*)(is_t ? p.tgt : p.dft) + lr * p.V * esz;
    if (dt == SPECV_F32)
        row_topk<SPECV_F32>(p, r, row, kk, off, probs_row, k2, tp, sm);
    else
        row_topk<SPECV_BF16>(p, r, row, kk, off, probs_row, k2, tp, sm);
}

// ------------------------------------------------- top-p without top-k
// One CTA of 1024 threads per SM: about 152 rows are in flight at a time
// (39 MB of bf16 rows at V = 128256), so the passes after the first read
// their row from L2.
constexpr int kAlThreads = 1024, kAlWarps = kAlThreads / 32;
constexpr int kAlBinBits = 14, kAlBins = 1 << kAlBinBits;  // one narrowing pass's float histogram
constexpr int kAlBinsPerThread = kAlBins / kAlThreads;
constexpr size_t kAlSmemBytes = kAlBins * sizeof(float);   // dynamic: the histogram

// Shared memory of alone_kernel (besides the histogram).
struct AloneSmem {
    Exp2Table tab;
    df dsum[2][5][kAlWarps];  // block sums: each warp's, double-buffered
    float fsum[2][5][kAlWarps];
    df dfin[2][5];            // block sums: the CTA's
    float ffin[2][5];
    float wtot[kAlWarps];     // histogram choice: each warp's bins
    int bin;                  // histogram choice: the bin
    float bin_above;          // histogram choice: the float mass above the bin
    uint32_t tail_key;        // 1 + the largest key left out of the histogram (0: none)
};

// f(v) for each value of one 16-byte vector, in column order.
template <int DT, typename F>
__device__ __forceinline__ void vec_each(const uint4& q, F&& f) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if constexpr (DT == SPECV_BF16) {
            f(bf16_lo(w[e]));
            f(bf16_hi(w[e]));
        } else {
            f(__uint_as_float(w[e]));
        }
    }
}

// N double-float and N float sums over the CTA, the same in every thread:
// each warp reduces its lanes, warp 0 reduces the warps' sums and every
// thread reads the result. par alternates between calls, so that a call's
// writes never meet the previous call's reads.
template <int N>
__device__ void block_sum(df (&d)[N], float (&f)[N], int par, AloneSmem& sm) {
    static_assert(kAlWarps == 32, "warp 0 reduces one warp sum per lane");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < N; ++i) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            d[i] = df_add(d[i], shfl_xor_df(d[i], o));
            f[i] += __shfl_xor_sync(kFull, f[i], o);
        }
    }
    if (lane == 0)
#pragma unroll
        for (int i = 0; i < N; ++i) {
            sm.dsum[par][i][warp] = d[i];
            sm.fsum[par][i][warp] = f[i];
        }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            df x = sm.dsum[par][i][lane];
            float y = sm.fsum[par][i][lane];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                x = df_add(x, shfl_xor_df(x, o));
                y += __shfl_xor_sync(kFull, y, o);
            }
            if (lane == 0) {
                sm.dfin[par][i] = x;
                sm.ffin[par][i] = y;
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < N; ++i) {
        d[i] = sm.dfin[par][i];
        f[i] = sm.ffin[par][i];
    }
}

// One narrowing choice over the float histogram, for the whole CTA: the
// highest bin j with above + (the bins from j up) >= target, else bin 0.
// above becomes the float mass above bin j. With first, target is first set
// to top_p of above + every bin + below (mass left out of the histogram,
// under its bins). Each thread sums its own bins and the warps combine from
// the top, in a fixed order. The choice is a guess that the double-float
// pass checks.
__device__ int hist_pick(const float* hist, float& above, float& target, bool first, float tp, float below,
                         AloneSmem& sm) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    float loc[kAlBinsPerThread];
    const float4* h4 = reinterpret_cast<const float4*>(hist) + t * (kAlBinsPerThread / 4);
    float cs = 0.f;
#pragma unroll
    for (int i = 0; i < kAlBinsPerThread / 4; ++i) {
        const float4 q = h4[i];
        loc[4 * i] = q.x;
        loc[4 * i + 1] = q.y;
        loc[4 * i + 2] = q.z;
        loc[4 * i + 3] = q.w;
    }
#pragma unroll
    for (int i = 0; i < kAlBinsPerThread; ++i) cs += loc[i];
    float x = cs;  // this lane's bins and every higher lane's
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_down_sync(kFull, x, o);
        if (lane + o < 32) x += y;
    }
    float ex = __shfl_down_sync(kFull, x, 1);  // the higher lanes' alone
    if (lane == 31) ex = 0.f;
    if (lane == 0) sm.wtot[warp] = x;
    if (t == 0) sm.bin = 0;
    __syncthreads();
    float up = above, all = above;  // above + the higher warps' bins; above + every bin
    for (int w = kAlWarps - 1; w >= 0; --w) {
        const float v = sm.wtot[w];
        if (w > warp) up += v;
        all += v;
    }
    if (first) target = tp * (all + below);
    const float base = up + ex;  // above + every bin above this thread's
    float run = base;
    int cand = -1;
#pragma unroll
    for (int i = kAlBinsPerThread - 1; i >= 0; --i) {
        run += loc[i];
        if (cand < 0 && !(target > run)) cand = t * kAlBinsPerThread + i;
    }
    if (cand >= 0) atomicMax(&sm.bin, cand);
    __syncthreads();
    const int j = sm.bin;
    if (t == j / kAlBinsPerThread) {  // the bin's thread: the mass above the bin, summed as in the search
        float a = base;
#pragma unroll
        for (int i = kAlBinsPerThread - 1; i >= 0; --i)
            if (i > j % kAlBinsPerThread) a += loc[i];
        sm.bin_above = a;
    }
    __syncthreads();
    above = sm.bin_above;
    return j;
}

// The nucleus of a whole row (top-p without top-k): the largest key K whose
// values at or above it carry at least top_p of the row's double-float mass
// (the nucleus kernel's weights and decision).
//  1. Float narrowing: each pass spreads the float mass of the keys in
//     [P, P + 2^R) over kAlBins bins of 2^(R-14) keys and keeps the bin where
//     the float mass from the top reaches top_p of the row's, until R <= 4
//     (one pass for bf16 keys, two for f32). The first pass also sums the
//     row's double-float mass for the target, and bins only the values that
//     weigh at least 2^-16 of the row's largest (few in a peaked row), the
//     rest being summed apart: if the bin found may hold such a value, that
//     pass runs again over every value.
//  2. Double-float two-bit bisection over the kept range. Its first round
//     also weighs the keys above the range and checks that the target falls
//     inside it: mass(>= P) >= target > mass(>= P + 2^R). If the float guess
//     was wrong, the bisection runs again over the whole key range.
// Each round's range [prefix, hi) holds the keys still undecided; the mass of
// the keys at or above hi is carried. Float sums of the sampler's weights go
// along, for the row's sum over the nucleus.
template <int DT>
__device__ void row_nucleus_whole(const StatsParams& p, int64_t r, const char* row, float T, float tp, bool probs_row,
                                  AloneSmem& sm, float* hist, const float2 rs) {
    using KT = KeyTraits<DT>;
    constexpr int ESZ = KT::kEsz, EPV = 16 / ESZ, W = 8 * KT::kDigits;
    if (!(rs.y == rs.y)) return;  // an invalid row stays invalid
    const float m = rs.x;
    const int64_t V = p.V;
    const df kd = k_of_temperature(T);
    const float k2 = kLog2e / T, nmk = -__fmul_rn(m, k2);
    auto weight = [&](float v) -> df {
        return probs_row ? df{v, 0.f} : logit_weight<DT == SPECV_F32>(v, m, kd, sm.tab);
    };
    // 16-byte vectors from the row's first 16-byte boundary; the columns
    // before it (head) and after the last full vector (from tail0) one by one
    int64_t head = (int64_t)(((16u - (uint32_t)((uintptr_t)row & 15u)) & 15u) / ESZ);
    if (head > V) head = V;
    const int64_t nvec = (V - head) / EPV, tail0 = head + nvec * EPV;
    const uint4* vrow = reinterpret_cast<const uint4*>(row + head * ESZ);
    auto each = [&](auto&& f) {  // f(v) for every value of the row
        for (int64_t vi = threadIdx.x; vi < nvec; vi += 2 * kAlThreads) {  // two loads in flight
            const bool two = vi + kAlThreads < nvec;
            const uint4 q0 = __ldcg(vrow + vi);
            const uint4 q1 = two ? __ldcg(vrow + vi + kAlThreads) : make_uint4(0u, 0u, 0u, 0u);
            vec_each<DT>(q0, f);
            if (two) vec_each<DT>(q1, f);
        }
        if (threadIdx.x < head) f(ld_elem<DT>(row, threadIdx.x));
        if (tail0 + threadIdx.x < V) f(ld_elem<DT>(row, tail0 + threadIdx.x));
    };

    // 1. float narrowing
    df target{0.f, 0.f};
    uint32_t P = 0;
    int R = W, par = 0;
    float above_h = 0.f, target_f = 0.f;
    const float light = probs_row ? m * 0x1p-16f : 0x1p-16f;  // the first pass bins weights from here up
    bool skip = true;
#pragma unroll 1
    while (R > 4) {
        const int s = R - kAlBinBits;
        const bool first = R == W && skip;
        const uint64_t span = 1ull << R;
        for (int i = threadIdx.x; i < kAlBins; i += kAlThreads) hist[i] = 0.f;
        if (threadIdx.x == 0) sm.tail_key = 0u;
        __syncthreads();
        df tot[1] = {{0.f, 0.f}};
        float tail[1] = {0.f};  // the float mass left out of the histogram
        uint32_t tk = 0u;       // 1 + the largest key left out
        each([&](float v) {
            const uint32_t key = key_of_value<DT>(v);
            if (first) tot[0] = df_add(tot[0], weight(v));
            const uint32_t off = key - P;  // wraps above span for key < P
            if ((uint64_t)off >= span) return;
            const float fw = kept_weight(v, probs_row, k2, nmk);
            if (!(fw > 0.f)) return;
            if (first && fw < light) {
                tail[0] += fw;
                tk = max(tk, key + 1u);
                return;
            }
            atomicAdd(hist + (off >> s), fw);
        });
        if (tk) atomicMax(&sm.tail_key, tk);
        if (first) {
            block_sum<1>(tot, tail, par, sm);
            par ^= 1;
            target = df_mul_f(tot[0], tp);
        }
        __syncthreads();  // the histogram is complete
        const uint32_t tkb = sm.tail_key;
        float ah = above_h;
        const int j = hist_pick(hist, ah, target_f, first, tp, first ? tail[0] : 0.f, sm);
        if (first && tkb && j <= (int)((tkb - 1u - P) >> s)) {  // the bin may hold values left out
            skip = false;
            continue;
        }
        skip = false;
        above_h = ah;
        P += (uint32_t)j << s;
        R = s;
    }

    // 2. double-float bisection
    df above{0.f, 0.f};
    float above_f = 0.f, nucleus_f = 0.f;
    uint32_t prefix = P;
#pragma unroll 1
    for (int attempt = 0; attempt < 2; ++attempt) {
        const int b0 = attempt ? W - 2 : R - 2;
        if (attempt) {  // the float guess was wrong: the whole key range
            prefix = 0;
            above = df{0.f, 0.f};
            above_f = 0.f;
        }
        bool ok = true;
#pragma unroll 1
        for (int b = b0; b >= 0; b -= 2) {
            const bool edge = attempt == 0 && b == b0;  // also weigh the keys at or above hi
            const uint32_t c1 = prefix | (1u << b), c2 = prefix | (2u << b), c3 = prefix | (3u << b);
            const uint64_t hi = (uint64_t)prefix + (4ull << b);
            // d[i] / f[i], i < 4: the range's values at or above c_i (c_0 = prefix);
            // d[4] / f[4]: the values at or above hi (edge round)
            df d[5] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
            float f[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
            each([&](float v) {
                const uint32_t key = key_of_value<DT>(v);
                if ((uint64_t)key >= hi) {
                    if (edge) {
                        d[4] = df_add(d[4], weight(v));
                        f[4] += kept_weight(v, probs_row, k2, nmk);
                    }
                    return;
                }
                if (key < prefix) return;
                const df w = weight(v);
                const float fw = kept_weight(v, probs_row, k2, nmk);
                d[0] = df_add(d[0], w);
                f[0] += fw;
                if (key >= c1) {
                    d[1] = df_add(d[1], w);
                    f[1] += fw;
                }
                if (key >= c2) {
                    d[2] = df_add(d[2], w);
                    f[2] += fw;
                }
                if (key >= c3) {
                    d[3] = df_add(d[3], w);
                    f[3] += fw;
                }
            });
            block_sum<5>(d, f, par, sm);
            par ^= 1;
            if (edge) {
                above = d[4];
                above_f = f[4];
                if (!df_gt(target, above) || df_gt(target, df_add(above, d[0]))) {  // the same in every thread
                    ok = false;
                    break;
                }
            }
            const df t3 = df_add(above, d[3]), t2 = df_add(above, d[2]), t1 = df_add(above, d[1]);
            if (!df_gt(target, t3)) {
                prefix = c3;
                nucleus_f = above_f + f[3];
            } else if (!df_gt(target, t2)) {
                prefix = c2;
                above = t3;
                nucleus_f = above_f + f[2];
                above_f += f[3];
            } else if (!df_gt(target, t1)) {
                prefix = c1;
                above = t2;
                nucleus_f = above_f + f[1];
                above_f += f[2];
            } else {
                above = t1;
                nucleus_f = above_f + f[0];
                above_f += f[1];
            }
        }
        if (ok) break;
    }
    if (threadIdx.x == 0) {
        p.row_stats[r] = make_float2(rs.x, nucleus_f);
        p.tau[r] = KT::value(KT::bits_of_key(prefix));
    }
}

// Rows with top-p and no top-k, after the top-k pass (which gave them their
// maximum): the nucleus of the whole row. One CTA per row; the other rows
// return at once.
__global__ void __launch_bounds__(kAlThreads, 1) alone_kernel(StatsParams p) {
    __shared__ AloneSmem sm;
    extern __shared__ float4 al_hist[];
    pdl_launch_dependents();
    pdl_wait_primary();  // the top-k pass's row statistics
    const int64_t r = blockIdx.x;
    const bool is_t = r < p.rows_t;
    const int64_t lr = is_t ? r : r - p.rows_t;
    const int32_t b = row_seq(p, !is_t, lr);
    if (b < 0) return;
    const int64_t kk = p.top_ks ? (int64_t)__ldg(p.top_ks + b) : (int64_t)p.top_k;
    const float tp = p.top_ps ? __ldg(p.top_ps + b) : p.top_p;
    if ((kk >= 1 && kk < p.V) || !(tp > 0.f && tp < 1.f)) return;  // top-k on, or no top-p
    float T = p.temps ? __ldg(p.temps + b) : p.temperature;
    if (!(T > 0.f) || !isfinite(T)) T = 1.f;  // the finalize reports the sequence's bad temperature
    const int dt = is_t ? p.tdt : p.ddt;
    const bool probs_row = !is_t && p.probs != 0;
    if (dt == SPECV_BF16 && !probs_row) return;  // whole_nucleus_kernel's row
    const char* row = (const char*)(is_t ? p.tgt : p.dft) + lr * p.V * (dt == SPECV_F32 ? 4 : 2);
    if (threadIdx.x < 64) {
        sm.tab.hi[threadIdx.x] = p.tab.hi[threadIdx.x];
        sm.tab.lo[threadIdx.x] = p.tab.lo[threadIdx.x];
    }
    __syncthreads();
    float* hist = reinterpret_cast<float*>(al_hist);
    const float2 rs = __ldcg(p.row_stats + r);
    if (dt == SPECV_F32) row_nucleus_whole<SPECV_F32>(p, r, row, T, tp, probs_row, sm, hist, rs);
    else row_nucleus_whole<SPECV_BF16>(p, r, row, T, tp, probs_row, sm, hist, rs);
}

// ---------------------------------------------------------------- top-p
// The nucleus of each top-p row inside its top-k set: the largest key K
// whose kept values at or above it carry at least top_p of the kept mass,
// the masses double-float sums of the sampler's weights (so the boundary is
// decided as the float64 reading decides it). One warp per row, after the
// top-k pass: the row's kept values come from p.keep (or from the row
// itself when they did not fit). The warp then rewrites the row's threshold
// and its sum over the kept columns.
constexpr int kNuThreads = 256;
constexpr int kNuReg = 4;  // kept values per lane whose weights stay in registers
constexpr int kNuWarps = kNuThreads / 32;

__device__ __forceinline__ df warp_sum_df(df v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = df_add(v, shfl_xor_df(v, o));
    return v;
}

template <int DT>
__device__ void row_nucleus(const StatsParams& p, int64_t r, const char* row, float T, float tp, bool probs_row,
                            const Exp2Table& tab) {
    using KT = KeyTraits<DT>;
    const int lane = threadIdx.x & 31;
    const float2 rs = __ldcg(p.row_stats + r);
    if (!(rs.y == rs.y)) return;  // an invalid row stays invalid
    const float m = rs.x, tk = __ldcg(p.tau + r);
    const df kd = k_of_temperature(T);
    const int32_t n = __ldcg(p.keep_n + r);
    const uint32_t* kept = p.keep + r * kKeepCap;
    auto weight = [&](float v) -> df {
        if (probs_row) return df{v, 0.f};
        return logit_weight<DT == SPECV_F32>(v, m, kd, tab);
    };
    auto visit = [&](auto&& f) {  // (key, value) of this lane's kept values
        if (n >= 0) {
            for (int e = lane; e < n; e += 32) {
                const uint32_t key = __ldcg(kept + e);
                f(key, KT::value(KT::bits_of_key(key)));
            }
        } else {
            for (int64_t j = lane; j < p.V; j += 32) {
                const float v = ld_elem<DT>(row, j);
                if (v >= tk) f(key_of_value<DT>(v), v);
            }
        }
    };
    // Rows keeping at most 32 * kNuReg values keep each lane's keys and
    // weights in registers: the rounds below then only compare and add, in
    // the same per-lane order as the uncached walk (the same sums).
    const bool cached = n >= 0 && n <= 32 * kNuReg;
    uint32_t ck[kNuReg];
    df cw[kNuReg];
    if (cached) {
#pragma unroll
        for (int i = 0; i < kNuReg; ++i) {
            const int e = lane + 32 * i;
            ck[i] = e < n ? __ldcg(kept + e) : 0u;  // key 0 is below every round's bounds
            cw[i] = e < n ? weight(KT::value(KT::bits_of_key(ck[i]))) : df{0.f, 0.f};
        }
    }
    df S{0.f, 0.f};
    if (cached) {
#pragma unroll
        for (int i = 0; i < kNuReg; ++i)
            if (lane + 32 * i < n) S = df_add(S, cw[i]);
    } else {
        visit([&](uint32_t, float v) { S = df_add(S, weight(v)); });
    }
    S = warp_sum_df(S);
    const df target = df_mul_f(S, tp);
    uint32_t prefix = 0;
#pragma unroll 1
    for (int b = 8 * KT::kDigits - 2; b >= 0; b -= 2) {
        const uint32_t c1 = prefix | (1u << b), c2 = prefix | (2u << b), c3 = prefix | (3u << b);
        df m1{0.f, 0.f}, m2{0.f, 0.f}, m3{0.f, 0.f};
        auto take = [&](uint32_t key, const df& w) {
            if (key < c1) return;
            m1 = df_add(m1, w);
            if (key >= c2) m2 = df_add(m2, w);
            if (key >= c3) m3 = df_add(m3, w);
        };
        if (cached) {
#pragma unroll
            for (int i = 0; i < kNuReg; ++i) take(ck[i], cw[i]);
        } else {
            visit([&](uint32_t key, float v) {
                if (key >= c1) take(key, weight(v));
            });
        }
        m1 = warp_sum_df(m1);
        m2 = warp_sum_df(m2);
        m3 = warp_sum_df(m3);
        prefix = !df_gt(target, m3) ? c3 : (!df_gt(target, m2) ? c2 : (!df_gt(target, m1) ? c1 : prefix));
    }
    const float tau = KT::value(KT::bits_of_key(prefix));
    // the row's sum over the nucleus, as the top-k pass sums its kept columns
    const float k2 = kLog2e / T, nmk = -__fmul_rn(m, k2);
    float acc = 0.f;
    visit([&](uint32_t, float v) {
        if (v >= tau) acc += kept_weight(v, probs_row, k2, nmk);
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
    if (lane == 0) {
        p.row_stats[r] = make_float2(rs.x, acc);
        p.tau[r] = tau;
    }
}

__global__ void __launch_bounds__(kNuThreads) nucleus_kernel(StatsParams p) {
    __shared__ Exp2Table tab;
    for (int i = threadIdx.x; i < 64; i += kNuThreads) {
        tab.hi[i] = p.tab.hi[i];
        tab.lo[i] = p.tab.lo[i];
    }
    __syncthreads();
    pdl_launch_dependents();
    pdl_wait_primary();
    const int64_t r = (int64_t)blockIdx.x * kNuWarps + (threadIdx.x >> 5);
    if (r >= p.rows_t + p.rows_d) return;
    const bool is_t = r < p.rows_t;
    const int64_t lr = is_t ? r : r - p.rows_t;
    const int32_t b = row_seq(p, !is_t, lr);
    if (b < 0) return;
    const int64_t kk = p.top_ks ? (int64_t)__ldg(p.top_ks + b) : (int64_t)p.top_k;
    const float tp = p.top_ps ? __ldg(p.top_ps + b) : p.top_p;
    if (!(kk >= 1 && kk < p.V) || !(tp > 0.f && tp < 1.f)) return;  // no nucleus for this row
    float T = p.temps ? __ldg(p.temps + b) : p.temperature;
    if (!(T > 0.f) || !isfinite(T)) T = 1.f;  // the finalize reports the sequence's bad temperature
    const int dt = is_t ? p.tdt : p.ddt;
    const bool probs_row = !is_t && p.probs != 0;
    const char* row = (const char*)(is_t ? p.tgt : p.dft) + lr * p.V * (dt == SPECV_F32 ? 4 : 2);
    if (dt == SPECV_F32)
        row_nucleus<SPECV_F32>(p, r, row, T, tp, probs_row, tab);
    else
        row_nucleus<SPECV_BF16>(p, r, row, T, tp, probs_row, tab);
}

// ------------------------------------------ top-p without top-k, bf16 logits
// The nucleus of a whole bf16 logits row (top-p with top-k off), one CTA per
// SM taking rows in turn. The rows reach shared memory through a ring of
// two 32 KB bulk-copy stages filled by one thread a stage ahead of the CTA,
// across the CTA's rows (the next row's first chunk arrives while the CTA
// decides the current one).
//  1. One pass over the row, chunk by chunk. Each chunk first raises the
//     running maximum (its packed bf16 maxima, over the CTA). A bf16 logit's
//     weight depends only on its 16-bit pattern, so the heavy columns
//     (weight above 2^-13 of the running maximum's) are counted per pattern
//     in shared memory (16-bit counters, two to a word), while the light
//     ones are summed as they come: the SFU's 2^x, eight at a time and then
//     in double-float, rescaled exactly whenever the maximum rises, with a
//     bound on the sum's error (the SFU's relative error, the exponent's
//     rounding, the summation's).
//  2. Over the counts: each pattern's double-float weight times its count,
//     summed from the highest pattern down (the patterns present spread over
//     the threads, then a block scan); the total is those masses plus the
//     light sum; the nucleus edge is the highest pattern whose mass at or
//     above it reaches top_p of the total, found by the thread where the
//     running mass crosses the target walking its patterns (with its warp
//     when it holds many).
//  3. The edge stands if it holds for every total within the light sum's
//     bound and its pattern was heavy against the final maximum (so every
//     column at or above it was counted). If not, or if the edge lies among
//     the light columns, the row is counted again with every column by
//     pattern and every pattern weighed in double-float (a pass with no light
//     sum). A pattern held by 65536 columns or more wraps its counter; the
//     counts then fall short of the columns counted and the row goes through
//     the narrowing search of row_nucleus_whole instead.
constexpr int kWnThreads = 1024, kWnWarps = kWnThreads / 32;
constexpr int kWnKeys = 65536;
constexpr int kWnWordsPerThread = kWnKeys / 2 / kWnThreads;     // 32 words: 64 consecutive patterns
constexpr size_t kWnHistBytes = kWnKeys * sizeof(uint16_t);     // the counters (128 KB)
constexpr int kWnStages = 2;                                    // ring stages
constexpr uint32_t kWnChunk = 32u << 10;                        // bytes per stage: two 16-byte vectors per thread
constexpr int kWnList = 4096;                                   // patterns present listed for the decision
constexpr size_t kWnSmemBytes = kWnHistBytes + kWnStages * kWnChunk + kWnList * 6;  // counters, ring, list
constexpr int kWnLoads = 4;                                     // 16-byte loads in flight per thread (recount)
constexpr float kWnHeavy = -13.0f;  // exponents above this are counted by pattern, those below summed
// Bound on the relative error of the SFU's 2^x used for the light sum (its
// measured maximum on GB300 is 1.44e-7).
constexpr float kWnEx2Err = 2.4e-7f;
constexpr float kWnU = 5.9604645e-8f;  // 2^-24
static_assert(kWnThreads == kAlThreads, "the narrowing search runs with the same CTA");
static_assert(kWnHistBytes >= kAlSmemBytes, "the narrowing search reuses the counters' memory");
static_assert(kWnWordsPerThread == 32, "each warp's counters are 8 x 32 vectors of 8 patterns");
static_assert(kWnChunk == 32u * kWnThreads, "two vectors per thread per chunk");

struct WholeSmem {
    AloneSmem al;                    // the narrowing search's (its exp2 table serves every step)
    df ws[kWnWarps], wf[kWnWarps];   // warp totals: masses, kept weights
    df as[kWnWarps], af[kWnWarps];   // the same summed over the higher warps
    df tot_s, tot_f;                 // the row's
    df above_s, above_f;             // above the crossing thread's patterns
    df lsum;                         // the light weights' sum
    uint64_t full[kWnStages];        // ring: a stage's copy has landed
    uint32_t wnz[kWnWarps];          // patterns present per warp
    uint32_t cmax[3];                // a chunk step's maximum as an ordered key, by step modulo 3
    uint32_t cnan, failed;
    uint32_t negz, count, mink, maxk, nheavy;
    int32_t tstar, verdict;
};

__device__ __forceinline__ df shfl_down_df(df v, int o) {
    return df{__shfl_down_sync(kFull, v.hi, o), __shfl_down_sync(kFull, v.lo, o)};
}

// The value of a bf16 pattern key (the inverse of KeyTraits<SPECV_BF16>::key).
__device__ __forceinline__ float bf16_of_key(uint32_t k) {
    return __uint_as_float((k ^ ((k & 0x8000u) ? 0x8000u : 0xFFFFu)) << 16);
}

// Count one bf16 pattern (or both of a 32-bit word) under its order-preserving
// key; -0 keeps a key of its own, joined to +0's when the counts are read.
__device__ __forceinline__ void count_one(uint32_t* hist, uint32_t h) {
    const uint32_t k = h ^ ((h & 0x8000u) ? 0xFFFFu : 0x8000u);
    atomicAdd(hist + (k >> 1), 1u << ((k & 1u) << 4));
}
__device__ __forceinline__ void count_pair(uint32_t* hist, uint32_t w) {
    const uint32_t sg = (w >> 15) & 0x00010001u;            // each half's sign bit
    const uint32_t k = w ^ ((sg * 0x7FFFu) | 0x80008000u);  // both keys
    const uint32_t k0 = k & 0xFFFFu, k1 = k >> 16;
    atomicAdd(hist + (k0 >> 1), 1u << ((k0 & 1u) << 4));
    atomicAdd(hist + (k1 >> 1), 1u << ((k1 & 1u) << 4));
}

// Both halves' maxima of two bf16 pairs, NaN propagating.
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Row r's address.
__device__ __forceinline__ const char* row_addr(const StatsParams& p, int64_t r) {
    const bool is_t = r < p.rows_t;
    const int dt = is_t ? p.tdt : p.ddt;
    return (const char*)(is_t ? p.tgt : p.dft) + (is_t ? r : r - p.rows_t) * p.V * (dt == SPECV_F32 ? 4 : 2);
}

// A bf16 row as 16-byte vectors from its first 16-byte boundary, with the
// columns before it (head) and after the last full vector (from tail0).
struct RowSplit {
    const uint4* vec;
    int64_t head, nvec, tail0;
};
__device__ __forceinline__ RowSplit split_row(const char* row, int64_t V) {
    RowSplit s;
    s.head = (int64_t)(((16u - (uint32_t)((uintptr_t)row & 15u)) & 15u) / 2u);
    if (s.head > V) s.head = V;
    s.nvec = (V - s.head) / 8;
    s.tail0 = s.head + s.nvec * 8;
    s.vec = reinterpret_cast<const uint4*>(row + s.head * 2);
    return s;
}

// f(q) for this thread's vectors, kWnLoads loads in flight; g(bits) for its
// head and tail columns.
template <typename F, typename G>
__device__ __forceinline__ void each_vec(const char* row, int64_t V, F&& f, G&& g) {
    const RowSplit rs = split_row(row, V);
    const int t = threadIdx.x;
    for (int64_t v0 = t; v0 < rs.nvec; v0 += kWnLoads * kWnThreads) {
        uint4 q[kWnLoads];
#pragma unroll
        for (int i = 0; i < kWnLoads; ++i)
            if (v0 + i * kWnThreads < rs.nvec) q[i] = ld_stream_v4(rs.vec + v0 + i * kWnThreads);
#pragma unroll
        for (int i = 0; i < kWnLoads; ++i)
            if (v0 + i * kWnThreads < rs.nvec) f(q[i]);
    }
    const uint16_t* row16 = reinterpret_cast<const uint16_t*>(row);
    if (t < rs.head) g((uint32_t)__ldg(row16 + t));
    if (rs.tail0 + t < V) g((uint32_t)__ldg(row16 + rs.tail0 + t));
}

// Weight of a bf16 pattern relative to the maximum, double-float down to
// 2^-120 (a single float below).
__device__ __forceinline__ df pattern_weight(float v, float m, df kd, const Exp2Table& tab) {
    const float dh = __fsub_rn(v, m);
    if (!(dh > -INFINITY)) return df{0.f, 0.f};
    const float x = __fmaf_rn(dh, kd.hi, __fmul_rn(dh, kd.lo));
    if (x > -120.f) return heavy_weight(dh, 0.f, kd, tab);
    return df{ex2(x), 0.f};
}

// The edge from the counts in hist (and, for the counts of heavy columns
// only, the light sum L with error bound E), written to row r unless it is
// not certain. expect: the columns counted. The patterns present are listed
// in ascending order (when they fit the list) and split evenly over the
// threads, so that their double-float weights are spread over the CTA (a row
// with more patterns than the list holds splits the range of patterns
// present instead, at most 64 to a thread). Returns 0 when written, 1 when
// the edge needs every column counted, 2 when a counter wrapped. Every
// thread returns the same.
static __device__ __noinline__ int decide_edge(const StatsParams& p, int64_t r, uint32_t* hist, WholeSmem& sm,
                                               float m, df kd, float k2, float tp, uint32_t expect, bool all, df L,
                                               float E) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const uint16_t* h16 = reinterpret_cast<const uint16_t*>(hist);
    uint16_t* lkey = reinterpret_cast<uint16_t*>(reinterpret_cast<char*>(hist) + kWnHistBytes + kWnStages * kWnChunk);
    uint32_t* lcnt = reinterpret_cast<uint32_t*>(lkey + kWnList);
    const float nmk = -__fmul_rn(m, k2);
    const uint32_t negz = h16[0x7FFF];  // -0's count, joined to +0's
    // this warp's counters: vectors warp*256 + i*32 + lane (i = 0..7), so that
    // a warp reads contiguous words; vector v holds the patterns 8v .. 8v+7
    const uint4* hw = reinterpret_cast<const uint4*>(hist) + warp * 256 + lane;

    // A. the columns counted, the range of patterns present, and the number
    // of patterns present in this warp's 2048 (list positions: the lower
    // warps' come first, the list ascending)
    {
        uint32_t cnt = 0u, kmin = 0xFFFFFFFFu, kmax = 0u, nz = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 q = hw[i * 32];
            if ((q.x | q.y | q.z | q.w) == 0u) continue;
            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
            const uint32_t kb = 8u * (uint32_t)(warp * 256 + i * 32 + lane);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t key = kb + 2u * j, c0 = wv[j] & 0xFFFFu, c1 = wv[j] >> 16;
                cnt += c0 + c1;
                nz += (c0 ? 1u : 0u) + (c1 ? 1u : 0u);
                if (c0) {
                    kmin = min(kmin, key);
                    kmax = key + 1u;
                }
                if (c1) {
                    kmin = min(kmin, key + 1u);
                    kmax = key + 2u;
                }
            }
        }
        if (warp == 0x7FFF / 2048 && lane == 31 && negz) --nz;                  // key 0x7FFF is no pattern of its own
        if (warp == 0x8000 / 2048 && lane == 0 && negz && h16[0x8000] == 0u) ++nz;  // +0 present through -0 alone
        cnt = __reduce_add_sync(kFull, cnt);
        kmin = __reduce_min_sync(kFull, kmin);
        kmax = __reduce_max_sync(kFull, kmax);
        nz = __reduce_add_sync(kFull, nz);
        if (lane == 0) {
            atomicAdd(&sm.count, cnt);
            atomicMin(&sm.mink, kmin);
            atomicMax(&sm.maxk, kmax);
            sm.wnz[warp] = nz;
        }
        __syncthreads();
    }
    if (sm.count != expect) return 2;
    uint32_t klo = sm.mink, khi = sm.maxk - 1u;
    if (klo == 0x7FFFu) klo = 0x8000u;  // -0 as +0
    if (khi == 0x7FFFu) khi = 0x8000u;
    uint32_t NZ = 0u, base = 0u;
#pragma unroll 8
    for (int w = 0; w < kWnWarps; ++w) {
        const uint32_t v = sm.wnz[w];
        NZ += v;
        if (w < warp) base += v;
    }
    const bool listed = NZ <= (uint32_t)kWnList;
    if (listed) {  // this warp's patterns, ascending, at its list position
        uint32_t o = base;
#pragma unroll 1
        for (int i = 0; i < 8; ++i) {
            const uint4 q = hw[i * 32];
            const bool zero = (q.x | q.y | q.z | q.w) == 0u;
            if (__all_sync(kFull, zero) && !(negz && warp == 0x8000 / 2048 && i == 0)) continue;
            const uint32_t kb = 8u * (uint32_t)(warp * 256 + i * 32 + lane);
            uint32_t c[8];
            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) c[e] = (e & 1) ? wv[e >> 1] >> 16 : wv[e >> 1] & 0xFFFFu;
            if (negz && (warp == 0x7FFF / 2048 || warp == 0x8000 / 2048)) {
                if (kb + 7u == 0x7FFFu) c[7] = 0u;  // -0 ...
                if (kb == 0x8000u) c[0] += negz;    // ... counts as +0
            }
            uint32_t n = 0u;
#pragma unroll
            for (int e = 0; e < 8; ++e) n += c[e] ? 1u : 0u;
            uint32_t x = n;  // inclusive prefix over the lanes
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t y = __shfl_up_sync(kFull, x, d);
                if (lane >= d) x += y;
            }
            uint32_t pos = o + x - n;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (c[e]) {
                    lkey[pos] = (uint16_t)(kb + e);
                    lcnt[pos] = c[e];
                    ++pos;
                }
            o += __shfl_sync(kFull, x, 31);
        }
        __syncthreads();
    }
    // thread tt's items, highest first: list entries, or the patterns of its range
    const uint32_t per = listed ? (NZ + kWnThreads - 1) / kWnThreads : (khi - klo + kWnThreads) / kWnThreads;
    auto items = [&](int tt) -> uint32_t {
        const uint32_t b0 = listed ? min((uint32_t)tt * per, NZ) : min(klo + (uint32_t)tt * per, khi + 1u);
        const uint32_t b1 = listed ? min(b0 + per, NZ) : min(b0 + per, khi + 1u);
        return b1 - b0;
    };
    auto item = [&](int tt, uint32_t j, uint32_t& key) -> uint32_t {  // count of item j, its key in key
        if (listed) {
            const uint32_t e = min(min((uint32_t)tt * per, NZ) + per, NZ) - 1u - j;
            key = lkey[e];
            return lcnt[e];
        }
        const uint32_t b1 = min(min(klo + (uint32_t)tt * per, khi + 1u) + per, khi + 1u);
        key = b1 - 1u - j;
        uint32_t c = h16[key];
        if (key == 0x7FFFu) c = 0u;
        if (key == 0x8000u) c += negz;
        return c;
    };

    // B. each thread's masses over its items, from the highest down
    df S{0.f, 0.f}, F{0.f, 0.f};
    {
        const uint32_t n = items(t);
#pragma unroll 1
        for (uint32_t j = 0; j < n; ++j) {
            uint32_t key;
            const uint32_t c = item(t, j, key);
            if (c == 0u) continue;
            const float v = bf16_of_key(key), cf = (float)c;
            S = df_add(S, df_mul_f(pattern_weight(v, m, kd, sm.al.tab), cf));
            F = df_add(F, two_prod(kept_weight(v, false, k2, nmk), cf));
        }
    }

    // C. masses above each thread's items: suffix sums over the lanes, then the warps
    df xs = S, xf = F;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const df ys = shfl_down_df(xs, o), yf = shfl_down_df(xf, o);
        if (lane + o < 32) {
            xs = df_add(xs, ys);
            xf = df_add(xf, yf);
        }
    }
    df es = shfl_down_df(xs, 1), ef = shfl_down_df(xf, 1);  // the higher lanes' alone
    if (lane == 31) es = ef = df{0.f, 0.f};
    if (lane == 0) {
        sm.ws[warp] = xs;
        sm.wf[warp] = xf;
    }
    __syncthreads();
    if (warp == 0) {
        df ys = sm.ws[lane], yf = sm.wf[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const df zs = shfl_down_df(ys, o), zf = shfl_down_df(yf, o);
            if (lane + o < 32) {
                ys = df_add(ys, zs);
                yf = df_add(yf, zf);
            }
        }
        df us = shfl_down_df(ys, 1), uf = shfl_down_df(yf, 1);
        if (lane == 31) us = uf = df{0.f, 0.f};
        sm.as[lane] = us;
        sm.af[lane] = uf;
        if (lane == 0) {
            sm.tot_s = ys;
            sm.tot_f = yf;
        }
    }
    __syncthreads();
    const df wa = sm.as[warp];
    const df tot = df_add(sm.tot_s, L);
    const df target = df_mul_f(tot, tp);

    // D. the crossing thread: the highest one whose items reach the target
    const bool cand = df_pos(S) && !df_gt(target, df_add(wa, xs));
    const uint32_t tc = __reduce_max_sync(kFull, cand ? (uint32_t)t + 1u : 0u);
    if (lane == 0 && tc) atomicMax(&sm.tstar, (int32_t)tc);
    __syncthreads();
    const int32_t ts = sm.tstar - 1;
    if (ts < 0) {
        if (!all) return 1;  // the edge lies among the light columns
        // nothing reaches the target (rounding): the whole row
        if (t == 0) {
            const df f = sm.tot_f;
            p.row_stats[r] = make_float2(m, __fadd_rn(f.hi, f.lo));
            p.tau[r] = bf16_of_key(klo);
        }
        return 0;
    }
    if (listed && per <= 4u) {
        // E. few items a thread: the crossing thread walks its own, highest first
        if (t == ts) {
            const uint32_t n = items(ts);
            const df above = df_add(wa, es);
            df run = above, prev{0.f, 0.f}, at{0.f, 0.f};
            uint32_t K = 0xFFFFFFFFu, lo = 0xFFFFFFFFu;
#pragma unroll 1
            for (uint32_t j = 0; j < n; ++j) {
                uint32_t key;
                const uint32_t c = item(ts, j, key);
                if (c == 0u) continue;
                const df pw = df_mul_f(pattern_weight(bf16_of_key(key), m, kd, sm.al.tab), (float)c);
                if (!df_pos(pw)) continue;
                const df before = run;
                run = df_add(run, pw);
                lo = key;
                if (K == 0xFFFFFFFFu && !df_gt(target, run)) {
                    K = key;
                    prev = before;
                    at = run;
                }
            }
            int verdict = 0;
            if (K == 0xFFFFFFFFu) {  // none within the thread (rounding): its lowest pattern with weight
                K = lo;
                verdict = all ? 0 : 1;
            } else if (!all) {
                // the edge holds for every total within E of the estimate:
                // the mass at or above K reaches the highest target, the mass
                // above K stays under the lowest; and K is heavy against the
                // reference the columns were classified by, so every column
                // at or above it was counted
                const df thi = df_mul_f(df_add(tot, df{E, 0.f}), tp);
                const df tlo = df_mul_f(df_add(tot, df{-E, 0.f}), tp);
                const float dk = __fsub_rn(bf16_of_key(K), m);
                const bool heavy = __fmaf_rn(dk, kd.hi, __fmul_rn(dk, kd.lo)) > kWnHeavy;
                verdict = (heavy && !df_gt(thi, at) && df_gt(tlo, prev)) ? 0 : 1;
            }
            if (verdict == 0) {
                df f = df_add(sm.af[warp], ef);
#pragma unroll 1
                for (uint32_t j = 0; j < n; ++j) {
                    uint32_t key;
                    const uint32_t c = item(ts, j, key);
                    if (c != 0u && key >= K) f = df_add(f, two_prod(kept_weight(bf16_of_key(key), false, k2, nmk), (float)c));
                }
                p.row_stats[r] = make_float2(m, __fadd_rn(f.hi, f.lo));
                p.tau[r] = bf16_of_key(K);
            }
            sm.verdict = verdict;
        }
        __syncthreads();
        return sm.verdict;
    }
    if (t == ts) {
        sm.above_s = df_add(wa, es);
        sm.above_f = df_add(sm.af[warp], ef);
    }
    __syncthreads();
    if (warp == (ts >> 5)) {
        // E. the crossing thread's items, two per lane, lane 0 the highest
        const uint32_t n = items(ts), j1 = 2u * (uint32_t)lane, j0 = j1 + 1u;
        uint32_t key1 = 0u, key0 = 0u;
        const uint32_t n1 = j1 < n ? item(ts, j1, key1) : 0u, n0 = j0 < n ? item(ts, j0, key0) : 0u;
        df p1{0.f, 0.f}, p0{0.f, 0.f}, g1{0.f, 0.f}, g0{0.f, 0.f};
        if (n1) {
            const float v = bf16_of_key(key1);
            p1 = df_mul_f(pattern_weight(v, m, kd, sm.al.tab), (float)n1);
            g1 = two_prod(kept_weight(v, false, k2, nmk), (float)n1);
        }
        if (n0) {
            const float v = bf16_of_key(key0);
            p0 = df_mul_f(pattern_weight(v, m, kd, sm.al.tab), (float)n0);
            g0 = two_prod(kept_weight(v, false, k2, nmk), (float)n0);
        }
        df x = df_add(p1, p0);  // inclusive prefix over the lanes (items downward)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const df y = shfl_up_df(x, o);
            if (lane >= o) x = df_add(y, x);
        }
        df ex = shfl_up_df(x, 1);
        if (lane == 0) ex = df{0.f, 0.f};
        const df base = df_add(sm.above_s, ex);
        const df run1 = df_add(base, p1), run0 = df_add(run1, p0);
        // 1 + the highest pattern whose mass at or above it reaches the
        // target, with the mass above that pattern and at it
        uint32_t kc = 0u;
        df prev{0.f, 0.f}, at{0.f, 0.f};
        if (df_pos(p1) && !df_gt(target, run1)) {
            kc = key1 + 1u;
            prev = base;
            at = run1;
        } else if (df_pos(p0) && !df_gt(target, run0)) {
            kc = key0 + 1u;
            prev = run1;
            at = run0;
        }
        const uint32_t kbest = __reduce_max_sync(kFull, kc);
        int verdict = 0;
        uint32_t K;
        if (kbest == 0u) {
            // none within the thread (rounding): its lowest pattern with weight
            const uint32_t lo = df_pos(p0) ? key0 : (df_pos(p1) ? key1 : 0xFFFFFFFFu);
            K = __reduce_min_sync(kFull, lo);
            verdict = all ? 0 : 1;
        } else {
            K = kbest - 1u;
            if (!all) {
                // the edge holds for every total within E of the estimate:
                // the mass at or above K reaches the highest target, the
                // mass above K stays under the lowest
                const int src = __ffs(__ballot_sync(kFull, kc == kbest)) - 1;
                const df pv = shfl_df(prev, src), av = shfl_df(at, src);
                const df thi = df_mul_f(df_add(tot, df{E, 0.f}), tp);
                const df tlo = df_mul_f(df_add(tot, df{-E, 0.f}), tp);
                // and K heavy against the final maximum: then it was heavy
                // against every running maximum, so every column at or
                // above it was counted
                const float dk = __fsub_rn(bf16_of_key(K), m);
                const bool heavy = __fmaf_rn(dk, kd.hi, __fmul_rn(dk, kd.lo)) > kWnHeavy;
                verdict = (heavy && !df_gt(thi, av) && df_gt(tlo, pv)) ? 0 : 1;
            }
        }
        if (verdict == 0) {
            df gs = (n1 && key1 >= K) ? g1 : df{0.f, 0.f};
            if (n0 && key0 >= K) gs = df_add(gs, g0);
            gs = warp_sum_df(gs);
            if (lane == 0) {
                const df f = df_add(sm.above_f, gs);
                p.row_stats[r] = make_float2(m, __fadd_rn(f.hi, f.lo));
                p.tau[r] = bf16_of_key(K);
            }
        }
        if (lane == 0) sm.verdict = verdict;
    }
    __syncthreads();
    return sm.verdict;
}

// Reset the counters and the scalars the counting steps accumulate into.
__device__ __forceinline__ void clear_counts(uint32_t* hist, WholeSmem& sm) {
    __syncthreads();  // earlier readers of the counters are done
    uint4* h4 = reinterpret_cast<uint4*>(hist);
#pragma unroll
    for (int i = 0; i < kWnWordsPerThread / 4; ++i) h4[threadIdx.x + i * kWnThreads] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        sm.count = 0u;
        sm.mink = 0xFFFFFFFFu;
        sm.maxk = 0u;
        sm.tstar = 0;
        sm.nheavy = 0u;
        sm.cnan = 0u;
        sm.lsum = df{0.f, 0.f};
    }
    __syncthreads();
}

// Float bits as an unsigned key of the same order (NaN excluded).
__device__ __forceinline__ uint32_t ord_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
constexpr uint32_t kOrdNegInf = 0x007FFFFFu;  // ord_key(-inf)
constexpr uint32_t kOrdPosInf = 0xFF800000u;  // ord_key(+inf)

// The ring's producer (thread 0): the CTA's rows in turn, each row's
// 16-byte-aligned body in chunks of kWnChunk bytes.
struct RingFeed {
    int64_t row;      // the row being issued (>= rows: none left)
    const char* src;  // the rest of its body
    uint32_t left;    // bytes of it not yet issued
    uint32_t g;       // chunks issued so far
};
__device__ __forceinline__ int64_t next_whole_row(const StatsParams& p, int64_t r, int64_t rows) {
    while (r < rows && !whole_bf16_row(p, r)) r += gridDim.x;
    return r;
}
__device__ void feed_set(RingFeed& f, const StatsParams& p, int64_t r, int64_t rows) {
    for (;;) {
        f.row = next_whole_row(p, r, rows);
        f.left = 0u;
        if (f.row >= rows) return;
        const RowSplit rs = split_row(row_addr(p, f.row), p.V);
        f.src = reinterpret_cast<const char*>(rs.vec);
        f.left = (uint32_t)(rs.nvec * 16);
        if (f.left) return;
        r = f.row + gridDim.x;  // no full vector in this row: nothing to copy
    }
}
__device__ void feed_issue(RingFeed& f, const StatsParams& p, int64_t rows, WholeSmem& sm, char* ring) {
    if (f.row >= rows) return;
    const uint32_t st = f.g % kWnStages, n = min(f.left, kWnChunk);
    mbar_arrive_expect_tx(&sm.full[st], n);
    bulk_g2s(ring + (size_t)st * kWnChunk, f.src, n, &sm.full[st]);
    ++f.g;
    f.src += n;
    f.left -= n;
    if (f.left == 0u) feed_set(f, p, f.row + gridDim.x, rows);
}

// A row whose edge the counts of its heavy columns could not settle (out of
// line: rare). Unless a counter already wrapped, every column is counted by
// pattern and every pattern weighed in double-float; a wrapped counter sends
// the row to the narrowing search.
static __device__ __noinline__ void whole_slow(const StatsParams& p, int64_t r, const char* row, float T, float tp,
                                               uint32_t* hist, WholeSmem& sm, float m, df kd, float k2,
                                               bool wrapped) {
    const int64_t V = p.V;
    int v = 2;
    if (!wrapped) {
        clear_counts(hist, sm);
        each_vec(
            row, V,
            [&](const uint4& q) {
                count_pair(hist, q.x);
                count_pair(hist, q.y);
                count_pair(hist, q.z);
                count_pair(hist, q.w);
            },
            [&](uint32_t h) { count_one(hist, h); });
        __syncthreads();
        v = decide_edge(p, r, hist, sm, m, kd, k2, tp, (uint32_t)V, true, df{0.f, 0.f}, 0.f);
    }
    if (v == 2) {
        __syncthreads();  // the counters' readers are done: the search reuses their memory
        row_nucleus_whole<SPECV_BF16>(p, r, row, T, tp, false, sm.al, reinterpret_cast<float*>(hist),
                                      make_float2(m, 0.f));
    }
}

// 1. One pass over a row through the ring: the running maximum (chunk by
// chunk, over the CTA), heavy columns counted by pattern, light ones summed
// (out of line, so that the calls after it leave its registers alone).
// Returns false if a ring wait gave up.
static __device__ __noinline__ bool stream_row(const StatsParams& p, uint32_t* hist, char* ring, WholeSmem& sm,
                                               uint32_t& g_io, uint32_t& cs_io, RingFeed& feed, int64_t rows,
                                               uint32_t body, uint32_t nch, uint32_t eh, bool has_e, df kd,
                                               float& m_out, df& l_out, uint32_t& nh_out, bool& nan_out) {
    const int t = threadIdx.x, lane = t & 31;
    uint32_t g = g_io, cs = cs_io;
    df lacc{0.f, 0.f};
    uint32_t nh = 0u;
    float mrun = -INFINITY;
    bool nan_row = false;
    // the light weights of a vector's eight columns against the running
    // maximum, summed in three levels; heavy columns counted instead
    auto vec = [&](const uint4& q, float mr) -> float {
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float dh = __fsub_rn((e & 1) ? bf16_hi(wv[e >> 1]) : bf16_lo(wv[e >> 1]), mr);
            x[e] = __fmaf_rn(dh, kd.hi, __fmul_rn(dh, kd.lo));
        }
        const float xm = fmaxf(max3(x[0], x[1], x[2]), fmaxf(max3(x[3], x[4], x[5]), fmaxf(x[6], x[7])));
        if (xm > kWnHeavy) {  // some column of the vector is heavy (rare)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (x[e] > kWnHeavy) {
                    count_one(hist, (e & 1) ? wv[e >> 1] >> 16 : wv[e >> 1] & 0xFFFFu);
                    ++nh;
                }
        }
        float w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = x[e] > kWnHeavy ? 0.f : ex2(x[e]);
        return ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
    };
    const uint4 ninf = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    const uint32_t steps = nch > 0u ? nch : 1u;
#pragma unroll 1
    for (uint32_t c = 0; c < steps; ++c) {
        const bool has = c < nch;
        const uint32_t st = g % kWnStages;
        if (t == 0) sm.cmax[(cs + 1u) % 3u] = kOrdNegInf;  // its readers (step cs - 2) are past the last barrier
        bool ok = true;
        if (has) ok = mbar_wait_bounded(&sm.full[st], (g / kWnStages) & 1u, kWaitLimit);
        const uint32_t nbytes = has ? min(kWnChunk, body - c * kWnChunk) : 0u;
        const uint4* sv = reinterpret_cast<const uint4*>(ring + (size_t)st * kWnChunk);
        const bool in0 = ok && (uint32_t)t * 16u < nbytes, in1 = ok && ((uint32_t)t + kWnThreads) * 16u < nbytes;
        const uint4 q0 = in0 ? sv[t] : ninf, q1 = in1 ? sv[t + kWnThreads] : ninf;
        uint32_t a = bmax2(bmax2(bmax2(q0.x, q0.y), bmax2(q0.z, q0.w)), bmax2(bmax2(q1.x, q1.y), bmax2(q1.z, q1.w)));
        if (c == 0u && has_e) a = bmax2(a, eh | (eh << 16));
        // the chunk's maximum over the CTA as an ordered key (a NaN, canonical
        // from the packed maxima, ranks above +inf)
        const uint32_t km = __reduce_max_sync(kFull, max(ord_key(bf16_lo(a)), ord_key(bf16_hi(a))));
        if (lane == 0) atomicMax(&sm.cmax[cs % 3u], km);
        // every thread has its vectors of this chunk: the stage is free again
        if (__syncthreads_or(!ok)) {
            g_io = g;
            cs_io = cs;
            return false;
        }
        if (t == 0 && has) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the reads above before the refill
            feed_issue(feed, p, rows, sm, ring);
        }
        const uint32_t kc = sm.cmax[cs % 3u];
        nan_row = nan_row || kc > kOrdPosInf;
        const float mnew = nan_row ? mrun : fmaxf(mrun, ord_value(kc));
        if (!nan_row && mnew < INFINITY && mnew > -INFINITY) {
            if (mnew > mrun && mrun > -INFINITY) {
                // rescale the light sum to the new maximum: 2^((mrun - mnew) k) in double-float
                const df d = two_sum(mrun, -mnew);
                const float x = __fmaf_rn(d.hi, kd.hi, __fmul_rn(d.hi, kd.lo));
                lacc = x > -120.f ? df_mul(lacc, heavy_weight_t<true>(d.hi, d.lo, kd, sm.al.tab)) : df{0.f, 0.f};
            }
            mrun = mnew;
            if (in0) acc_add(lacc, vec(q0, mrun));
            if (in1) acc_add(lacc, vec(q1, mrun));
            if (c == 0u && has_e) {
                const float dh = __fsub_rn(__uint_as_float(eh << 16), mrun);
                const float x = __fmaf_rn(dh, kd.hi, __fmul_rn(dh, kd.lo));
                if (x > kWnHeavy) {
                    count_one(hist, eh);
                    ++nh;
                } else {
                    acc_add(lacc, ex2(x));
                }
            }
        } else {
            mrun = mnew;
        }
        if (has) ++g;
        ++cs;
    }
    g_io = g;
    cs_io = cs;
    m_out = mrun;
    l_out = lacc;
    nh_out = nh;
    nan_out = nan_row;
    return true;
}

// One row (every thread). g: chunks taken from the ring so far; cs: chunk
// steps so far (a row with no full vector takes one step with no chunk).
// Returns false if a ring wait gave up (the CTA then stops).
__device__ bool whole_row_bf16(const StatsParams& p, int64_t r, uint32_t* hist, char* ring, WholeSmem& sm,
                               uint32_t& g, uint32_t& cs, RingFeed& feed, int64_t rows) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const bool is_t = r < p.rows_t;
    const int32_t b = row_seq(p, !is_t, is_t ? r : r - p.rows_t);
    float T = p.temps ? __ldg(p.temps + b) : p.temperature;
    if (!(T > 0.f) || !isfinite(T)) T = 1.f;  // the finalize reports the sequence's bad temperature
    const float tp = p.top_ps ? __ldg(p.top_ps + b) : p.top_p;
    const char* row = row_addr(p, r);
    const int64_t V = p.V;
    const RowSplit rs = split_row(row, V);
    const uint32_t body = (uint32_t)(rs.nvec * 16), nch = (body + kWnChunk - 1u) / kWnChunk;
    // the positive-low-part k: -inf logits give exponent -inf, not NaN
    const df kd = k_pos_lo(k_of_temperature(T));
    const float k2 = kLog2e / T;
    // the columns outside the body: threads 0..7 the head, 8..15 the tail
    uint32_t eh = 0xFF80u;  // -inf
    bool has_e = false;
    {
        const uint16_t* row16 = reinterpret_cast<const uint16_t*>(row);
        if (t < rs.head) {
            eh = __ldg(row16 + t);
            has_e = true;
        } else if (t >= 8 && t < 16 && rs.tail0 + (t - 8) < V) {
            eh = __ldg(row16 + rs.tail0 + (t - 8));
            has_e = true;
        }
    }
    clear_counts(hist, sm);

    // 1. one pass: the running maximum, heavy columns counted, light ones summed
    float mrun;
    df lacc;
    uint32_t nh;
    bool nan_row;
    if (!stream_row(p, hist, ring, sm, g, cs, feed, rows, body, nch, eh, has_e, kd, mrun, lacc, nh, nan_row))
        return false;
    const float m = mrun;
    if (nan_row || !(m > -INFINITY && m < INFINITY)) {  // NaN anywhere, or an infinite maximum: invalid
        if (t == 0) {
            p.row_stats[r] = make_float2(m, NAN);
            p.tau[r] = -INFINITY;
        }
        return true;
    }
    lacc = df_norm(lacc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lacc = df_add(lacc, shfl_xor_df(lacc, o));
    nh = __reduce_add_sync(kFull, nh);
    if (lane == 0) {
        sm.ws[warp] = lacc;
        atomicAdd(&sm.nheavy, nh);
    }
    __syncthreads();  // the counts and the warps' sums are complete
    if (warp == 0) {
        df y = sm.ws[lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) y = df_add(y, shfl_xor_df(y, o));
        if (lane == 0) sm.lsum = y;
    }
    __syncthreads();
    const df L = sm.lsum;
    // |light sum - exact| <= E: each weight's SFU error; the exponent's two
    // roundings (the difference v - m and the product by k, each within
    // 2^-24 |x|, times ln 2 in the weight), where the sum over the light
    // columns of w |x| = w log2(1/w) is at most L log2(n / L) for n columns
    // (concavity), and at least 13 L; the summation's three roundings within
    // each group of eight (the double-float sums and rescalings after them
    // add no more than 2^-40 of the sum). Half again for margin.
    const float lg = L.hi > 0.f ? fmaxf(-kWnHeavy, __log2f((float)V) - __log2f(L.hi) + 0.5f) : 0.f;
    const float E = 1.5f * __fmul_rn(kWnEx2Err + 3.f * kWnU + 0x1p-40f + 2.f * 0.6931472f * kWnU * lg, L.hi);

    // 2-3. the edge from the counts, else every column counted
    const int v = decide_edge(p, r, hist, sm, m, kd, k2, tp, sm.nheavy, false, L, E);
    if (v != 0) whole_slow(p, r, row, T, tp, hist, sm, m, kd, k2, v == 2);
    return true;
}

// Every row whole_bf16_row selects, one CTA per SM taking rows in turn.
// Launched after the top-k pass (or as the step's first kernel when it takes
// every row); before it exits it waits for the kernel before it, so that the
// kernels after it see both.
__global__ void __launch_bounds__(kWnThreads, 1) whole_nucleus_kernel(StatsParams p) {
    __shared__ WholeSmem sm;
    extern __shared__ __align__(128) unsigned char wn_raw[];
    uint32_t* hist = reinterpret_cast<uint32_t*>(wn_raw);
    char* ring = reinterpret_cast<char*>(wn_raw + kWnHistBytes);
    const int64_t rows = p.rows_t + p.rows_d;
    if (threadIdx.x < 64) {
        sm.al.tab.hi[threadIdx.x] = p.tab.hi[threadIdx.x];
        sm.al.tab.lo[threadIdx.x] = p.tab.lo[threadIdx.x];
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kWnStages; ++i) mbar_init(&sm.full[i], 1);
        sm.cmax[0] = sm.cmax[1] = sm.cmax[2] = kOrdNegInf;
        sm.failed = 0u;
        fence_barrier_init();
    }
    __syncthreads();
    RingFeed feed{rows, nullptr, 0u, 0u};  // thread 0's
    if (threadIdx.x == 0) {
        feed_set(feed, p, blockIdx.x, rows);
        for (int i = 0; i < kWnStages; ++i) feed_issue(feed, p, rows, sm, ring);
    }
    uint32_t g = 0u, cs = 0u;
    bool alive = true;
    for (int64_t r = next_whole_row(p, blockIdx.x, rows); r < rows; r = next_whole_row(p, r + gridDim.x, rows)) {
        if (!whole_row_bf16(p, r, hist, ring, sm, g, cs, feed, rows)) {
            alive = false;
            break;
        }
    }
    // never leave while a copy into the ring may be in flight
    if (threadIdx.x == 0) {
        for (uint32_t q = g; q < feed.g; ++q)
            mbar_wait_bounded(&sm.full[q % kWnStages], (q / kWnStages) & 1u, kWaitLimit);
        if (!alive) atomicOr(p.err, 1u);
    }
    pdl_wait_primary();
}

}  // namespace

cudaError_t launch_nucleus(const StatsParams& p, cudaStream_t s) {
    const int64_t rows = p.rows_t + p.rows_d;
    if (rows < 1) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + kNuWarps - 1) / kNuWarps));
    cfg.blockDim = dim3(kNuThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, nucleus_kernel, p);
}

cudaError_t launch_alone(const StatsParams& p, cudaStream_t s) {
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e =
            cudaFuncSetAttribute(alone_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAlSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int64_t rows = p.rows_t + p.rows_d;
    if (rows < 1) return cudaSuccess;
    if (!p.top_ks && p.top_k >= 1 && p.top_k < p.V) return cudaSuccess;  // top-k on for every sequence
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows);
    cfg.blockDim = dim3(kAlThreads);
    cfg.dynamicSmemBytes = kAlSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, alone_kernel, p);
}

cudaError_t launch_whole(const StatsParams& p, int sms, bool after_topk, cudaStream_t s) {
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e = cudaFuncSetAttribute(whole_nucleus_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)kWnSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int64_t rows = p.rows_t + p.rows_d;
    if (rows < 1 || !p.keep) return cudaSuccess;
    if (!p.top_ks && p.top_k >= 1 && p.top_k < p.V) return cudaSuccess;  // top-k on for every sequence
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>(rows, std::max(sms, 1)));
    cfg.blockDim = dim3(kWnThreads);
    cfg.dynamicSmemBytes = kWnSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = after_topk ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, whole_nucleus_kernel, p);
}

cudaError_t launch_topk(const StatsParams& p, cudaStream_t s) {
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e =
            cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTkSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int64_t rows = p.rows_t + p.rows_d;
    if (rows < 1) return cudaSuccess;
    topk_kernel<<<(unsigned)rows, kTkThreads, kTkSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace specv
