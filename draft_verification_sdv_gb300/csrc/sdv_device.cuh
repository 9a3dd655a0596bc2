// sdv_device.cuh -- device helpers of libsdv: streaming loads, exp2, the
// counter-based generator, mbarrier / bulk-copy / cluster primitives.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sdv {

constexpr float kLog2e = 1.4426950408889634f;   // log2(e)
constexpr float kLn2 = 0.6931471805599453f;      // ln(2)

// -------------------------------------------------------------------------
// Loads
// -------------------------------------------------------------------------

// 16-byte streaming load through the non-coherent path, not kept in L1: every
// logit byte of the row pass is read exactly once.
__device__ __forceinline__ uint4 ld_stream(const uint4* ptr) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

// One logit as fp32 (bf16 widens exactly).
__device__ __forceinline__ float load_logit(const void* base, int64_t idx, bool bf16) {
    if (bf16) {
        const unsigned short h = static_cast<const unsigned short*>(base)[idx];
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    return static_cast<const float*>(base)[idx];
}

// Low and high bf16 halves of a 32-bit word, widened to fp32.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Elementwise max of two packed bf16 pairs.
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// -------------------------------------------------------------------------
// Arithmetic
// -------------------------------------------------------------------------

// 2^x on the special-function unit (relative error about 2^-22; results
// below 2^-126 flush to zero, which is far below any term that matters for
// a row sum normalised to its maximum).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Max of the logits of N 16-byte vectors (packed pairs for bf16); NaN
// propagates so that a NaN row is caught.
template <bool BF16, int N>
__device__ __forceinline__ float vec_max_n(const uint4 (&v)[N]) {
    if constexpr (BF16) {
        uint32_t m[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
#pragma unroll
        for (int u = 1; u < N; ++u) {
            asm("max.NaN.bf16x2 %0, %0, %1;" : "+r"(m[0]) : "r"(v[u].x));
            asm("max.NaN.bf16x2 %0, %0, %1;" : "+r"(m[1]) : "r"(v[u].y));
            asm("max.NaN.bf16x2 %0, %0, %1;" : "+r"(m[2]) : "r"(v[u].z));
            asm("max.NaN.bf16x2 %0, %0, %1;" : "+r"(m[3]) : "r"(v[u].w));
        }
        asm("max.NaN.bf16x2 %0, %0, %1;" : "+r"(m[0]) : "r"(m[1]));
        asm("max.NaN.bf16x2 %0, %0, %1;" : "+r"(m[2]) : "r"(m[3]));
        asm("max.NaN.bf16x2 %0, %0, %1;" : "+r"(m[0]) : "r"(m[2]));
        float r;
        asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(bf16_lo(m[0])), "f"(bf16_hi(m[0])));
        return r;
    } else {
        float r = __uint_as_float(v[0].x);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const float e[4] = {__uint_as_float(v[u].x), __uint_as_float(v[u].y),
                                __uint_as_float(v[u].z), __uint_as_float(v[u].w)};
#pragma unroll
            for (int i = 0; i < 4; ++i) asm("max.NaN.f32 %0, %0, %1;" : "+f"(r) : "f"(e[i]));
        }
        return r;
    }
}

// Sum of 2^{(l - m) c} over the logits of one 16-byte vector (pairwise tree).
template <bool BF16>
__device__ __forceinline__ float vec_exp_sum(const uint4& v, float m, float c) {
    if constexpr (BF16) {
        const float e0 = ex2((bf16_lo(v.x) - m) * c), e1 = ex2((bf16_hi(v.x) - m) * c);
        const float e2 = ex2((bf16_lo(v.y) - m) * c), e3 = ex2((bf16_hi(v.y) - m) * c);
        const float e4 = ex2((bf16_lo(v.z) - m) * c), e5 = ex2((bf16_hi(v.z) - m) * c);
        const float e6 = ex2((bf16_lo(v.w) - m) * c), e7 = ex2((bf16_hi(v.w) - m) * c);
        return ((e0 + e1) + (e2 + e3)) + ((e4 + e5) + (e6 + e7));
    } else {
        const float e0 = ex2((__uint_as_float(v.x) - m) * c);
        const float e1 = ex2((__uint_as_float(v.y) - m) * c);
        const float e2 = ex2((__uint_as_float(v.z) - m) * c);
        const float e3 = ex2((__uint_as_float(v.w) - m) * c);
        return (e0 + e1) + (e2 + e3);
    }
}

// Merge two partial softmax statistics (max m, sum s of 2^{(l - m) c}).
// NaN sums propagate; an empty partial (s == 0) contributes nothing.
__device__ __forceinline__ void merge_stat(float& m, float& s, float m2, float s2, float c) {
    if (m2 > m) {
        const float t = m; m = m2; m2 = t;
        const float u = s; s = s2; s2 = u;
    }
    if (s2 != 0.0f) s += s2 * ex2((m2 - m) * c);
}

// -------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of the
// 4x32 multiply-xor S-box, key advanced by the Weyl increments between rounds.
// -------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 x, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t a_hi = __umulhi(0xD2511F53u, x.x);
        const uint32_t a_lo = 0xD2511F53u * x.x;
        const uint32_t b_hi = __umulhi(0xCD9E8D57u, x.z);
        const uint32_t b_lo = 0xCD9E8D57u * x.z;
        x = make_uint4(b_hi ^ x.y ^ k0, b_lo, a_hi ^ x.w ^ k1, a_lo);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return x;
}

// 24-bit uniform in [0, 1 - 2^-24], exact in fp32.
__device__ __forceinline__ float uniform24(uint32_t word) {
    return static_cast<float>(word >> 8) * 5.9604644775390625e-8f;   // 2^-24
}

// -------------------------------------------------------------------------
// Shared memory, mbarrier, bulk copy, cluster
// -------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
    // make the initialised barrier visible to the async (bulk-copy) proxy
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Bounded wait for phase `parity` of an mbarrier.  Returns false if the
// barrier did not complete within `max_polls` polls (each try_wait may itself
// suspend the thread for a short, hardware-defined time).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t max_polls) {
    const uint32_t addr = smem_u32(bar);
    for (uint32_t i = 0; i < max_polls; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// 1-D bulk copy (TMA engine) global -> this CTA's shared memory, completion
// counted in bytes on `bar`.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Hardware cluster barrier (every thread of every CTA of the cluster).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

}  // namespace sdv
