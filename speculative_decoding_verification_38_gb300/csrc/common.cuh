// common.cuh -- device helpers shared by the verify kernels (sm_103a).
//
// Nothing here is shared with the CPU oracle: the Philox generator below is
// this library's own restatement of the SC'11 definition (Salmon, Moraes,
// Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", Philox S-box and
// key schedule).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace specv {

constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ Philox
// Four 32-bit counter words, two key words, ten rounds. Each round multiplies
// counter words 0 and 2 by the round constants (full 64-bit products), mixes
// the high halves with words 1/3 and the key, and swaps lanes; the key advances
// by the Weyl increments between rounds.
struct Philox4 {
    uint32_t w[4];
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                  uint32_t k0, uint32_t k1) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        uint32_t lo0 = M0 * c0, hi0 = __umulhi(M0, c0);
        uint32_t lo1 = M1 * c2, hi1 = __umulhi(M1, c2);
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += W0;
        k1 += W1;
    }
    Philox4 o;
    o.w[0] = c0;
    o.w[1] = c1;
    o.w[2] = c2;
    o.w[3] = c3;
    return o;
}

// 24-bit uniform in [0, 1): the top 24 bits of a word, scaled by 2^-24 (exact in fp32).
__device__ __forceinline__ float u24(uint32_t w) { return (float)(w >> 8) * (1.0f / 16777216.0f); }

// (u_acc, u_smp) of global sequence `seq` at position `pos` of round `round`.
__device__ __forceinline__ float2 draw_uniforms(uint64_t seed, uint64_t round, uint32_t seq, uint32_t pos) {
    Philox4 r = philox4x32_10(pos, seq, (uint32_t)round, (uint32_t)(round >> 32), (uint32_t)seed,
                              (uint32_t)(seed >> 32));
    return make_float2(u24(r.w[0]), u24(r.w[1]));
}

// ------------------------------------------------------------- arithmetic
// 2^x on the SFU (ex2.approx, subnormal results flushed to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Packed two-lane fp32 arithmetic (one instruction for two IEEE
// round-to-nearest operations) and the three-input maximum.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ------------------------------------------------------------------ loads
// Streaming 16-byte load through the non-coherent path, not kept in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// One element of a row as float (exact for both storage types).
template <int DT>
__device__ __forceinline__ float ld_elem(const void* row, int64_t j) {
    if constexpr (DT == SPECV_F32) {
        return __ldg(reinterpret_cast<const float*>(row) + j);
    } else {
        uint16_t h = __ldg(reinterpret_cast<const unsigned short*>(row) + j);
        return __uint_as_float(((uint32_t)h) << 16);
    }
}

__device__ __forceinline__ float ld_elem_rt(const void* row, int dt, int64_t j) {
    return dt == SPECV_F32 ? ld_elem<SPECV_F32>(row, j) : ld_elem<SPECV_BF16>(row, j);
}

// L2-coherent loads of values other CTAs wrote during this grid.
__device__ __forceinline__ float2 ld_cg_f2(const float2* p) { return __ldcg(p); }

// ------------------------------------------------------ cluster (DSMEM)
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store a float into the same shared-memory variable of CTA `rank` of this cluster.
__device__ __forceinline__ void st_cluster_f32(float* local, uint32_t rank, float v) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(local), ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}

// ------------------------------------------ TMA bulk copies and mbarriers
// One-dimensional bulk copies global -> this CTA's shared memory (no
// multicast), completed through a transaction-counting mbarrier. Source,
// destination and size must be multiples of 16 bytes.
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for phase `parity` of the barrier, giving up after `limit` attempts
// (each attempt itself suspends for a bounded time). Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
constexpr uint32_t kWaitLimit = 1u << 24;  // ~seconds: never reached by a healthy copy

// ------------------------------------------------- programmatic launch
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------- softmax state
// Online max/sum of one row slice in the base-2 domain with 1/T folded in:
// state (m, s) with m = the largest raw logit and s = sum_j 2^(l_j*k - fl(m*k)),
// k = log2(e) / T. Merging two states rescales each sum to the larger max. A
// zero sum contributes nothing (so an all -inf slice never poisons the merge)
// while a NaN sum propagates.
__device__ __forceinline__ float2 ms_merge(float2 a, float2 b, float k) {
    const float M = fmaxf(a.x, b.x);
    const float Ms = __fmul_rn(M, k);
    const float sa = (a.y == 0.f) ? 0.f : a.y * ex2(__fmul_rn(a.x, k) - Ms);
    const float sb = (b.y == 0.f) ? 0.f : b.y * ex2(__fmul_rn(b.x, k) - Ms);
    return make_float2(M, sa + sb);
}

// Argmax state (value, first index); larger value wins, equal values keep the smaller index.
__device__ __forceinline__ bool am_better(float va, int32_t ia, float vb, int32_t ib) {
    return (va > vb) || (va == vb && ia < ib);
}

}  // namespace specv
