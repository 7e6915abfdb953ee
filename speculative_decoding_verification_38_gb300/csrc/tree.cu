// tree.cu -- verification of a token tree: several candidates per node.
//
// Tree speculation verifies several candidate continuations in one target
// pass ("Speculative decoding" (mhtirogla.ai), Levers and Implementation
// notes; "Speculative decoding" (inference.tusharamrit.in), tree attention).
// The pages leave the multi-candidate rule open; the reading implemented
// here takes the pages' residual at every candidate in turn. At node u
// (target distribution p_u, draft distribution q_u from which its children
// were drawn), r starts at p_u; candidate j with token x passes if
// u_acc(u, j) * q_u(x) < r(x) and the walk moves to it, else r becomes
// max(0, r - q_u) / Z (unchanged if Z = 0) and the next candidate is tried.
// If none passes, the token is drawn from r by inverse CDF in index order;
// a node without children draws the bonus from p_u. Greedy follows the
// first child equal to the target's argmax. Uniforms: u_acc(u, j) = word 0
// of Philox at counter (u + 65536 j, seq_offset + b, round), u_smp(u) = word 1
// at (u, ...), so a chain-shaped tree draws exactly what the chain verify
// draws.
//
// One CTA per sequence walks its tree. A visited node costs full-row passes
// (the maximum and the double-float normaliser of p and of q, one pass per
// failed candidate for the next residual normaliser, and the draw), read
// from global memory; the residual at a column is re-evaluated from p, q
// and the normalisers met so far (r_1 = p, r_{i+1} = max(0, r_i - q) / Z_{i+1}).
#include <math.h>

#include "internal.h"
#include "precise.cuh"

namespace specv {

namespace {

constexpr int kTrThreads = 512;
constexpr int kTrWarps = kTrThreads / 32;
constexpr int kTrMaxCand = 64;  // candidates per node whose residual normalisers are kept

struct TreeSmem {
    Exp2Table tab;
    float fred[kTrWarps];
    int32_t ired[kTrWarps];
    df dred[kTrWarps];
    df z[kTrMaxCand + 1];   // residual normalisers Z_2 .. of the current node (index i: r_{i+1})
    int32_t zlive[kTrMaxCand + 1];  // 1: that level changed r (Z > 0)
    int32_t kids[kTrMaxCand];       // the current node's children, in index order
    int32_t nkids;                  // how many it has (may exceed kTrMaxCand)
    int32_t flag;
};

// ------------------------------------------------------------ reductions
__device__ float block_max_f(float v, TreeSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) sm.fred[warp] = v;
    __syncthreads();
    float t = -INFINITY;
#pragma unroll
    for (int w = 0; w < kTrWarps; ++w) t = fmaxf(t, sm.fred[w]);
    return t;
}

__device__ int32_t block_min_i(int32_t v, TreeSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) sm.ired[warp] = v;
    __syncthreads();
    int32_t t = INT32_MAX;
#pragma unroll
    for (int w = 0; w < kTrWarps; ++w) t = min(t, sm.ired[w]);
    return t;
}

// Double-float sum over the CTA in a fixed order (the same bits whatever the timing).
__device__ df block_sum_dfx(df v, TreeSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = df_add(v, shfl_xor_df(v, o));
    __syncthreads();
    if (lane == 0) sm.dred[warp] = v;
    __syncthreads();
    df t{0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kTrWarps; ++w) t = df_add(t, sm.dred[w]);
    return t;
}

// Prefix sums over the CTA's threads in thread order (double-float): incl
// is the sum up to and including this thread, excl the previous thread's
// incl (the same bits), total the last thread's incl. The intervals
// [excl, incl) of the threads tile [0, total) without gaps or overlaps.
__device__ void block_scan_dfx(df v, TreeSmem& sm, df& excl, df& incl, df& total) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    df x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const df y = shfl_up_df(x, o);
        if (lane >= o) x = df_add(y, x);
    }
    __syncthreads();
    if (lane == 31) sm.dred[warp] = x;
    __syncthreads();
    df before{0.f, 0.f};
    for (int w = 0; w < warp; ++w) before = df_add(before, sm.dred[w]);
    incl = df_add(before, x);
    const df up = shfl_up_df(incl, 1);
    excl = lane == 0 ? before : up;
    total = df{0.f, 0.f};
    for (int w = 0; w < kTrWarps; ++w) total = df_add(total, sm.dred[w]);
}

// ------------------------------------------------------------ row passes
// The node's two rows and what the walk has learnt about them.
struct NodeRows {
    const char* t;  // target row
    const char* d;  // draft row
    int tdt, ddt;
    bool probs;
    bool vec;       // the rows read start on 16-byte boundaries: 16-byte loads
    float mt, md;   // raw maxima
    df k;           // log2(e) / T
    df It, Id;      // 1 / the rows' normalisers
};

__device__ __forceinline__ df tgt_weight(const NodeRows& n, float l, const Exp2Table& tab) {
    return n.tdt == SPECV_F32 ? logit_weight<true>(l, n.mt, n.k, tab) : logit_weight<false>(l, n.mt, n.k, tab);
}
__device__ __forceinline__ df dft_weight(const NodeRows& n, float l, const Exp2Table& tab) {
    if (n.probs) return df{l, 0.f};  // a probability row is used as given, divided by its sum
    return n.ddt == SPECV_F32 ? logit_weight<true>(l, n.md, n.k, tab) : logit_weight<false>(l, n.md, n.k, tab);
}

__device__ __forceinline__ df p_of(const NodeRows& n, float xt, const TreeSmem& sm) {
    return df_mul(tgt_weight(n, xt, sm.tab), n.It);
}

// r_level at a column with values xt (target) and xd (draft), and q there:
// r_1 = p, r_{i+1} = max(0, r_i - q) / Z_{i+1} for the levels that changed r
// (the others left it as it was).
__device__ df r_of(const NodeRows& n, float xt, float xd, int level, const TreeSmem& sm, df& q) {
    const df p = p_of(n, xt, sm);
    q = df_mul(dft_weight(n, xd, sm.tab), n.Id);
    df t = p;
    for (int i = 1; i < level; ++i) {
        if (!sm.zlive[i]) continue;
        const df dlt = df_sub(t, q);
        t = df_pos(dlt) ? df_mul(dlt, sm.z[i]) : df{0.f, 0.f};  // sm.z holds 1 / Z
    }
    return t;
}

// Columns j .. j+7 of a row (j % 8 == 0): one or two 16-byte loads when the
// row starts on a 16-byte boundary, else eight element loads.
__device__ __forceinline__ void ld8(const char* row, int dt, bool vec, int64_t j, float (&x)[8]) {
    if (vec) {
        if (dt == SPECV_F32) {
            const float4* q = reinterpret_cast<const float4*>(row) + (j >> 2);
            const float4 a = __ldg(q), c = __ldg(q + 1);
            x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = c.x, x[5] = c.y, x[6] = c.z, x[7] = c.w;
        } else {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(row) + (j >> 3));
            x[0] = bf16_lo(w.x), x[1] = bf16_hi(w.x), x[2] = bf16_lo(w.y), x[3] = bf16_hi(w.y);
            x[4] = bf16_lo(w.z), x[5] = bf16_hi(w.z), x[6] = bf16_lo(w.w), x[7] = bf16_hi(w.w);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = ld_elem_rt(row, dt, j + e);
    }
}

constexpr int kTrU = 2;  // 8-column units in flight per thread

// f(j, xt, xd) for every column of the node's rows (xd = 0 unless D), each
// thread taking 8-column units kTrThreads apart, kTrU loaded at a time, then
// the columns past the last whole unit. Per thread, j increases.
template <bool D, class F>
__device__ __forceinline__ void node_pass(const NodeRows& n, int64_t V, F&& f) {
    const int64_t units = V >> 3;
    for (int64_t k0 = threadIdx.x; k0 < units; k0 += (int64_t)kTrThreads * kTrU) {
        float t[kTrU][8], d[kTrU][8];
#pragma unroll
        for (int u = 0; u < kTrU; ++u) {
            const int64_t k = k0 + (int64_t)u * kTrThreads;
            if (k < units) {
                ld8(n.t, n.tdt, n.vec, k << 3, t[u]);
                if (D) ld8(n.d, n.ddt, n.vec, k << 3, d[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kTrU; ++u) {
            const int64_t k = k0 + (int64_t)u * kTrThreads;
            if (k < units)
#pragma unroll
                for (int e = 0; e < 8; ++e) f((k << 3) + e, t[u][e], D ? d[u][e] : 0.f);
        }
    }
    for (int64_t j = (units << 3) + threadIdx.x; j < V; j += kTrThreads)
        f(j, ld_elem_rt(n.t, n.tdt, j), D ? ld_elem_rt(n.d, n.ddt, j) : 0.f);
}

// f(j, xt, xd) for the columns [j0, j1) of one thread's contiguous chunk
// (j0 % 8 == 0), in increasing j.
template <class F>
__device__ __forceinline__ void chunk_pass(const NodeRows& n, bool D, int64_t j0, int64_t j1, F&& f) {
    int64_t j = j0;
    for (; j + 8 * kTrU <= j1; j += 8 * kTrU) {
        float t[kTrU][8], d[kTrU][8];
#pragma unroll
        for (int u = 0; u < kTrU; ++u) {
            ld8(n.t, n.tdt, n.vec, j + 8 * u, t[u]);
            if (D) ld8(n.d, n.ddt, n.vec, j + 8 * u, d[u]);
        }
#pragma unroll
        for (int u = 0; u < kTrU; ++u)
#pragma unroll
            for (int e = 0; e < 8; ++e) f(j + 8 * u + e, t[u][e], D ? d[u][e] : 0.f);
    }
    for (; j < j1; ++j) f(j, ld_elem_rt(n.t, n.tdt, j), D ? ld_elem_rt(n.d, n.ddt, j) : 0.f);
}

// First index of the largest target value (NaN read as -inf; a row of -inf
// or NaN gives 0).
__device__ int64_t row_argmax(const NodeRows& n, int64_t V, TreeSmem& sm) {
    float best = -INFINITY;
    int32_t bi = INT32_MAX;
    node_pass<false>(n, V, [&](int64_t j, float x, float) {
        if (x > best) {  // NaN never passes; per thread j increases: the first of equals stays
            best = x;
            bi = (int32_t)j;
        }
    });
    const float m = block_max_f(best, sm);
    const int32_t i = block_min_i(best == m ? bi : INT32_MAX, sm);
    return i == INT32_MAX ? 0 : i;
}

// Inverse CDF in index order over w(j) = r_level(j) (level 0: p, the target
// row alone): the first index whose running sum exceeds u * total; if
// rounding leaves none, the last index of positive weight. Each thread owns
// a contiguous chunk of whole 8-column units; the thread whose prefix
// interval holds u * total rescans its chunk.
__device__ int64_t draw_index(const NodeRows& n, int level, float us, int64_t V, TreeSmem& sm) {
    const int64_t C = (((V + 7) >> 3) + kTrThreads - 1) / kTrThreads * 8;
    const int64_t j0 = min(V, (int64_t)threadIdx.x * C), j1 = min(V, j0 + C);
    const bool D = level > 0;
    auto w = [&](float xt, float xd) {
        df q;
        return D ? r_of(n, xt, xd, level, sm, q) : p_of(n, xt, sm);
    };
    df s{0.f, 0.f};
    int32_t last = -1;
    chunk_pass(n, D, j0, j1, [&](int64_t j, float xt, float xd) {
        const df x = w(xt, xd);
        if (df_pos(x)) last = (int32_t)j;
        acc_add(s, x);
    });
    df excl, incl, total;
    block_scan_dfx(df_norm(s), sm, excl, incl, total);
    const df t = df_mul_f(total, us);
    int32_t pick = INT32_MAX;
    if (!df_gt(excl, t) && df_gt(incl, t)) {
        df c = excl;
        chunk_pass(n, D, j0, j1, [&](int64_t j, float xt, float xd) {
            if (pick != INT32_MAX) return;
            c = df_add(c, w(xt, xd));
            if (df_gt(c, t)) pick = (int32_t)j;
        });
        if (pick == INT32_MAX) pick = last;
    }
    pick = block_min_i(pick, sm);
    if (pick != INT32_MAX && pick >= 0) return pick;
    return -block_min_i(-last, sm);  // the last index of positive weight
}

__device__ void write_error(const TreeParams& p, int32_t b, int32_t st, int64_t o, int64_t n) {
    if (st != 4)  // SPEC_SEQ_BAD_LAYOUT: the sequence's slots are unknown
        for (int64_t k = threadIdx.x; k < n; k += kTrThreads) {
            p.out_tokens[o + k] = -1;
            if (p.out_path) p.out_path[o + k] = -1;
        }
    if (threadIdx.x == 0) {
        p.out_accepted[b] = 0;
        if (p.seq_status) p.seq_status[b] = st;
    }
}

__global__ void __launch_bounds__(kTrThreads) tree_kernel(const TreeParams p) {
    __shared__ TreeSmem sm;
    const int32_t b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t V = p.V;
    // statuses that need no row, in the documented order
    const int64_t o = __ldg(p.node_off + b), N = __ldg(p.node_off + b + 1) - o;
    if (N < 1 || o < 0 || o + N > p.nodes) {
        write_error(p, b, 4, o, N);  // SPEC_SEQ_BAD_LAYOUT
        return;
    }
    bool bad = threadIdx.x == 0 && __ldg(p.parent + o) != -1;
    for (int64_t v = 1 + threadIdx.x; v < N; v += kTrThreads) {
        const int32_t q = __ldg(p.parent + o + v);
        bad |= q < 0 || q >= v;
    }
    if (__syncthreads_or(bad)) {
        write_error(p, b, 4, o, N);
        return;
    }
    const float T = p.temps ? __ldg(p.temps + b) : p.temperature;
    if (!p.greedy && (!(T > 0.f) || !isfinite(T))) {
        write_error(p, b, 5, o, N);  // SPEC_SEQ_BAD_TEMP
        return;
    }
    bad = false;
    for (int64_t v = 1 + threadIdx.x; v < N; v += kTrThreads) {
        const int32_t x = __ldg(p.tokens + o + v);
        bad |= x < 0 || x >= V;
    }
    if (__syncthreads_or(bad)) {
        write_error(p, b, 1, o, N);  // SPEC_SEQ_BAD_TOKEN
        return;
    }
    for (int i = threadIdx.x; i < 64; i += kTrThreads) {
        sm.tab.hi[i] = p.tab.hi[i];
        sm.tab.lo[i] = p.tab.lo[i];
    }
    __syncthreads();

    const int64_t tes = p.tdt == SPECV_F32 ? 4 : 2, des = p.ddt == SPECV_F32 ? 4 : 2;
    NodeRows n;
    n.tdt = p.tdt;
    n.ddt = p.ddt;
    n.probs = p.probs != 0;
    n.k = p.greedy ? df{0.f, 0.f} : k_of_temperature(T);
    n.d = nullptr;
    int64_t u = 0;
    int32_t acc = 0, emit = -1;
    const uint32_t seq = p.seq_offset + (uint32_t)b;
    for (;;) {
        n.t = (const char*)p.tgt + (o + u) * V * tes;
        if (p.greedy) {
            n.vec = ((uintptr_t)n.t & 15) == 0;
            const int32_t g = (int32_t)row_argmax(n, V, sm);
            int32_t c = INT32_MAX;
            for (int64_t v = u + 1 + threadIdx.x; v < N; v += kTrThreads)
                if (__ldg(p.parent + o + v) == u && __ldg(p.tokens + o + v) == g) {
                    c = (int32_t)v;  // increasing v per thread: the first match is its smallest
                    break;
                }
            c = block_min_i(c, sm);
            if (c == INT32_MAX) {
                emit = g;
                break;
            }
            if (threadIdx.x == 0) {
                p.out_tokens[o + acc] = g;
                if (p.out_path) p.out_path[o + acc] = c;
            }
            ++acc;
            u = c;
            continue;
        }
        // the node's candidates, in index order (warp 0), once every thread
        // is done with the previous node's list
        __syncthreads();
        if (warp == 0) {
            int32_t cnt = 0;
            for (int64_t base = u + 1; base < N; base += 32) {
                const int64_t v = base + lane;
                const bool is = v < N && __ldg(p.parent + o + v) == u;
                const uint32_t m = __ballot_sync(0xffffffffu, is);
                const int32_t pos = cnt + __popc(m & ((1u << lane) - 1u));
                if (is && pos < kTrMaxCand) sm.kids[pos] = (int32_t)v;
                cnt += __popc(m);
            }
            if (lane == 0) sm.nkids = cnt;
        }
        __syncthreads();
        const int32_t m = sm.nkids;
        if (m > kTrMaxCand) {
            write_error(p, b, kSeqUnsupported, o, N);
            return;
        }
        const bool D = m > 0;  // the draft row is read at nodes with candidates
        n.d = D ? (const char*)p.dft + (o + u) * V * des : nullptr;
        n.vec = ((uintptr_t)n.t & 15) == 0 && (!D || ((uintptr_t)n.d & 15) == 0);
        // pass 1: maxima (a probability row: its sum) and NaN checks of both rows
        float mt = -INFINITY, md = -INFINITY;
        bool hnt = false, hnd = false;
        df sd{0.f, 0.f};
        if (D) {
            node_pass<true>(n, V, [&](int64_t, float xt, float xd) {
                mt = fmaxf(mt, xt);
                hnt |= xt != xt;
                hnd |= xd != xd;
                if (n.probs) acc_add(sd, xd);
                else md = fmaxf(md, xd);
            });
        } else {
            node_pass<false>(n, V, [&](int64_t, float xt, float) {
                mt = fmaxf(mt, xt);
                hnt |= xt != xt;
            });
        }
        hnt = __syncthreads_or(hnt);
        hnd = __syncthreads_or(hnd);
        n.mt = block_max_f(mt, sm);
        bool bad = hnt || !isfinite(n.mt);
        if (D) {
            if (n.probs) {
                sd = block_sum_dfx(df_norm(sd), sm);
                bad |= hnd || !(sd.hi > 0.f) || !isfinite(sd.hi);
            } else {
                n.md = block_max_f(md, sm);
                bad |= hnd || !isfinite(n.md);
            }
        }
        if (bad) {
            write_error(p, b, 3, o, N);  // SPEC_SEQ_BAD_ROW
            return;
        }
        // pass 2: the normalisers
        df st{0.f, 0.f};
        if (D && !n.probs) {
            df s2{0.f, 0.f};
            node_pass<true>(n, V, [&](int64_t, float xt, float xd) {
                acc_add(st, tgt_weight(n, xt, sm.tab));
                acc_add(s2, dft_weight(n, xd, sm.tab));
            });
            sd = block_sum_dfx(df_norm(s2), sm);
        } else {
            node_pass<false>(n, V, [&](int64_t, float xt, float) { acc_add(st, tgt_weight(n, xt, sm.tab)); });
        }
        st = block_sum_dfx(df_norm(st), sm);
        n.It = df_recip(st);
        const float us = draw_uniforms(p.seed, p.round, seq, (uint32_t)u).y;
        if (!D) {  // a leaf: the bonus token from p
            emit = (int32_t)draw_index(n, 0, us, V, sm);
            break;
        }
        n.Id = df_recip(sd);
        int level = 1;
        int32_t next = -1;
        for (int32_t j = 0; j < m; ++j) {
            const int32_t c = sm.kids[j];
            const int32_t x = __ldg(p.tokens + o + c);
            const float ua = draw_uniforms(p.seed, p.round, seq, (uint32_t)(u + (int64_t)j * 65536)).x;
            df qx;  // every thread: the same bits, no broadcast
            const df rx = r_of(n, ld_elem_rt(n.t, p.tdt, x), ld_elem_rt(n.d, p.ddt, x), level, sm, qx);
            if (df_gt(rx, df_mul_f(qx, ua))) {
                next = c;
                break;
            }
            // the next residual's normaliser
            df z{0.f, 0.f};
            node_pass<true>(n, V, [&](int64_t, float xt, float xd) {
                df qv;
                const df dl = df_sub(r_of(n, xt, xd, level, sm, qv), qv);
                if (df_pos(dl)) acc_add(z, dl);
            });
            z = block_sum_dfx(df_norm(z), sm);
            if (threadIdx.x == 0) {
                sm.zlive[level] = !residual_empty(z);
                sm.z[level] = df_recip(z);
            }
            __syncthreads();
            ++level;
        }
        if (next >= 0) {
            if (threadIdx.x == 0) {
                p.out_tokens[o + acc] = __ldg(p.tokens + o + next);
                if (p.out_path) p.out_path[o + acc] = next;
            }
            ++acc;
            u = next;
            continue;
        }
        emit = (int32_t)draw_index(n, level, us, V, sm);
        break;
    }
    // the emitted token, then -1 over the sequence's remaining slots
    for (int64_t k = acc + threadIdx.x; k < N; k += kTrThreads) {
        p.out_tokens[o + k] = k == acc ? emit : -1;
        if (p.out_path) p.out_path[o + k] = -1;
    }
    if (threadIdx.x == 0) {
        p.out_accepted[b] = acc;
        if (p.seq_status) p.seq_status[b] = 0;
    }
}

}  // namespace

cudaError_t launch_tree(const TreeParams& p, cudaStream_t s) {
    if (p.B == 0) return cudaSuccess;
    tree_kernel<<<(unsigned)p.B, kTrThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace specv
