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
__device__ __forceinline__ void warp_append(typename KeyTraits<DT>::Bits* wb, int& cnt, const uint4& q, bool need,
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
__device__ bool warp_make_room(typename KeyTraits<DT>::Bits* wb, int& cnt, uint32_t kk, WarpThr& thr,
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

__global__ void __launch_bounds__(kTkThreads, 4) topk_kernel(StatsParams p) {
    extern __shared__ __align__(16) unsigned char tk_raw[];
    TkSmem& sm = *reinterpret_cast<TkSmem*>(tk_raw);
    pdl_launch_dependents();
    const int64_t r = blockIdx.x;
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
                                  AloneSmem& sm, float* hist) {
    using KT = KeyTraits<DT>;
    constexpr int ESZ = KT::kEsz, EPV = 16 / ESZ, W = 8 * KT::kDigits;
    const float2 rs = __ldcg(p.row_stats + r);
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
    const char* row = (const char*)(is_t ? p.tgt : p.dft) + lr * p.V * (dt == SPECV_F32 ? 4 : 2);
    if (threadIdx.x < 64) {
        sm.tab.hi[threadIdx.x] = p.tab.hi[threadIdx.x];
        sm.tab.lo[threadIdx.x] = p.tab.lo[threadIdx.x];
    }
    __syncthreads();
    float* hist = reinterpret_cast<float*>(al_hist);
    if (dt == SPECV_F32) row_nucleus_whole<SPECV_F32>(p, r, row, T, tp, probs_row, sm, hist);
    else row_nucleus_whole<SPECV_BF16>(p, r, row, T, tp, probs_row, sm, hist);
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
