// common.cuh -- device helpers shared by the MoE kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace strata {

constexpr int kWarp = 32;

// Workspace control block (offset 0 of every workspace).
struct Ctl {
    uint32_t err;       // latched strata_status (first error wins; a timeout replaces it)
    uint32_t where[7];  // first timed-out wait: site, block, warp, slot, round, item, 1
    uint32_t pad[56];
};

__device__ __forceinline__ void latch(uint32_t* err, uint32_t code) {
    atomicCAS(err, 0u, code);
}

// latch() from the lowest lane of `bad` (a ballot of the lanes that hit the
// condition), skipped once the word holds a code: many threads that meet
// the same condition send one atomic a warp, not one each, to one address.
__device__ __forceinline__ void latch_warp(uint32_t* err, uint32_t code, uint32_t bad) {
    if (bad != 0u && int(threadIdx.x & 31) == __ffs(bad) - 1 &&
        *reinterpret_cast<const volatile uint32_t*>(err) == 0u)
        atomicCAS(err, 0u, code);
}

// Nonzero when either fp16 half of w has an all-ones exponent (inf or NaN).
__device__ __forceinline__ uint32_t f16x2_not_finite(uint32_t w) {
    return uint32_t((w & 0x7c00u) == 0x7c00u) | uint32_t((w & 0x7c000000u) == 0x7c000000u);
}
// Nonzero when either bf16 half of w is not finite.
__device__ __forceinline__ uint32_t bf16x2_not_finite(uint32_t w) {
    return uint32_t((w & 0x7f80u) == 0x7f80u) | uint32_t((w & 0x7f800000u) == 0x7f800000u);
}
// Nonzero when either bf16 half of w has no finite fp16 value: |v| >= 65536
// (the bf16 value below it, 65280, converts exactly), infinite or NaN.  A
// half at or above 0x4780 carries into its top bit when 0x3880 is added.
__device__ __forceinline__ uint32_t bf16x2_over_f16(uint32_t w) {
    return ((w & 0x7fff7fffu) + 0x38803880u) & 0x80008000u;
}
// w with each infinite half replaced by the largest finite value of its sign
// (+-65504) and each NaN by 0: tensor-core operands stay finite.
__device__ __forceinline__ uint32_t f16x2_saturate(uint32_t w) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t h = (w >> (16 * k)) & 0xffffu;
        if ((h & 0x7c00u) == 0x7c00u) {
            const uint32_t f = (h & 0x03ffu) != 0u ? 0u : ((h & 0x8000u) | 0x7bffu);
            w = (w & ~(0xffffu << (16 * k))) | (f << (16 * k));
        }
    }
    return w;
}

// A bounded wait ran out: latch STRATA_ETIMEOUT over any code latched
// before (the waits that give up early look for that code) and record where
// (the first one only).  `err` points at Ctl::err.
__device__ __forceinline__ void latch_timeout(uint32_t* err, uint32_t site, uint32_t slot,
                                              uint32_t round, uint32_t item) {
    atomicExch(err, 4u /* STRATA_ETIMEOUT */);
    uint32_t* w = err + 1;
    if (atomicCAS(&w[6], 0u, 1u) == 0u) {
        w[0] = site;
        w[1] = blockIdx.x;
        w[2] = threadIdx.x >> 5;
        w[3] = slot;
        w[4] = round;
        w[5] = item;
    }
}

// ------------------------------------------------------------------ formats
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float f16_to_f32(uint16_t h) {
    float f;
    asm("{ .reg .b16 t; mov.b16 t, %1; cvt.f32.f16 %0, t; }" : "=f"(f) : "h"(h));
    return f;
}

// fp32 -> bf16 bits, round to nearest even (NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

// ----------------------------------------------------- packed fp32 (f32x2)
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t pku(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ float2 upk(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// ------------------------------------------------------ int4 dot products
//
// A 16-byte chunk holds 32 consecutive int4 weights of one row (one scale
// group): byte b of word w holds element 8w+2b in bits 0..3 and 8w+2b+1 in
// bits 4..7, offset-binary (weight = scale * (u - 8)).
//
// Each nibble u becomes the fp32 value 1 + u/128 without any conversion
// instruction: OR-ing 0x80 into the byte and placing it under the exponent
// byte 0x3F gives the bit pattern 0x3F80_0000 | u << 16.  With
//   A = sum_j (1 + u_j/128) x_j   and   X = sum_j x_j
// the group's integer dot product is
//   sum_j (u_j - 8) x_j = 128 (A - X) - 8 X = 128 A - 136 X.
// Every step is exact except the fp32 sums, whose rounding error relative to
// the result stays near 1e-5 for |u| <= 15.
__device__ __forceinline__ uint32_t place_byte(uint32_t bytes, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(bytes), "r"(0x3F000000u), "r"(sel));
    return r;
}

// x2[16]: the chunk's 32 activations as pairs (x[2j], x[2j+1]).
// Returns A = sum_j (1 + u_j/128) x_j.
__device__ __forceinline__ float dot_chunk(const uint4& q, const uint64_t* x2) {
    uint64_t acc0 = 0ull, acc1 = 0ull;
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t lo = (words[w] & 0x0F0F0F0Fu) | 0x80808080u;
        const uint32_t hi = ((words[w] >> 4) & 0x0F0F0F0Fu) | 0x80808080u;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t sel = 0x7044u | (uint32_t(b) << 8);
            const uint64_t f = pku(place_byte(lo, sel), place_byte(hi, sel));
            if (b & 1)
                acc1 = ffma2(f, x2[4 * w + b], acc1);
            else
                acc0 = ffma2(f, x2[4 * w + b], acc0);
        }
    }
    const float2 a0 = upk(acc0), a1 = upk(acc1);
    return (a0.x + a0.y) + (a1.x + a1.y);
}

// d = a * b + c with a, b one bf16 half each of a 32-bit word (HI_A /
// HI_B: the upper half) and c, d fp32; the product of two bf16 is exact in
// fp32, so this rounds once, as fmaf on the widened values does.
template <bool HI_A, bool HI_B>
__device__ __forceinline__ float fma_bf16(uint32_t a, uint32_t b, float c) {
    float d;
    if (!HI_A && !HI_B)
        asm("{ .reg .b16 a0, a1, b0, b1; mov.b32 {a0, a1}, %1; mov.b32 {b0, b1}, %2;\n"
            "  fma.rn.f32.bf16 %0, a0, b0, %3; }" : "=f"(d) : "r"(a), "r"(b), "f"(c));
    else if (!HI_A && HI_B)
        asm("{ .reg .b16 a0, a1, b0, b1; mov.b32 {a0, a1}, %1; mov.b32 {b0, b1}, %2;\n"
            "  fma.rn.f32.bf16 %0, a0, b1, %3; }" : "=f"(d) : "r"(a), "r"(b), "f"(c));
    else if (HI_A && !HI_B)
        asm("{ .reg .b16 a0, a1, b0, b1; mov.b32 {a0, a1}, %1; mov.b32 {b0, b1}, %2;\n"
            "  fma.rn.f32.bf16 %0, a1, b0, %3; }" : "=f"(d) : "r"(a), "r"(b), "f"(c));
    else
        asm("{ .reg .b16 a0, a1, b0, b1; mov.b32 {a0, a1}, %1; mov.b32 {b0, b1}, %2;\n"
            "  fma.rn.f32.bf16 %0, a1, b1, %3; }" : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}

// dot_chunk times 128, bit for bit, against bf16 activations left packed:
// xb[k] holds elements 2k, 2k + 1.  A weight becomes the bf16 128 + u (one
// mask-and-or makes two), multiplied by x with fp32 accumulation in the
// same four chains, in the same order, as dot_chunk (elements {0,4},
// {1,5}, {2,6}, {3,7} of each word); 128 * (1 + u/128) = 128 + u exactly,
// so each partial sum is 128 times dot_chunk's.
__device__ __forceinline__ float dot_chunk_bf16(const uint4& q, const uint32_t* xb) {
    float c0 = 0.0f, c1 = 0.0f, c2 = 0.0f, c3 = 0.0f;
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t v = words[w];
        const uint32_t p04 = (v & 0x000F000Fu) | 0x43004300u;
        const uint32_t p15 = ((v >> 4) & 0x000F000Fu) | 0x43004300u;
        const uint32_t p26 = ((v >> 8) & 0x000F000Fu) | 0x43004300u;
        const uint32_t p37 = ((v >> 12) & 0x000F000Fu) | 0x43004300u;
        const uint32_t x0 = xb[4 * w], x1 = xb[4 * w + 1], x2 = xb[4 * w + 2], x3 = xb[4 * w + 3];
        c0 = fma_bf16<false, false>(p04, x0, c0);
        c0 = fma_bf16<true, false>(p04, x2, c0);
        c1 = fma_bf16<false, true>(p15, x0, c1);
        c1 = fma_bf16<true, true>(p15, x2, c1);
        c2 = fma_bf16<false, false>(p26, x1, c2);
        c2 = fma_bf16<true, false>(p26, x3, c2);
        c3 = fma_bf16<false, true>(p37, x1, c3);
        c3 = fma_bf16<true, true>(p37, x3, c3);
    }
    return (c0 + c1) + (c2 + c3);
}

// Scaled group dot product: scale * sum_j (u_j - 8) x_j.
__device__ __forceinline__ float group_dot(float A, float X, float scale) {
    return scale * fmaf(128.0f, A, -136.0f * X);
}
// The same from dot_chunk_bf16's sum (128 A): -136 X rounded, then one
// rounding of 128 A plus it, as in group_dot (the explicit roundings keep
// the compiler from fusing the two into one).
__device__ __forceinline__ float group_dot128(float A128, float X, float scale) {
    return scale * __fadd_rn(A128, __fmul_rn(-136.0f, X));
}

// ------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over aligned groups of `width` lanes (width a power of two <= 32).
__device__ __forceinline__ float group_sum(float v, int width) {
    for (int o = width >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + expf(-g)) * u;
}

// ------------------------------------------------------------ global loads
__device__ __forceinline__ uint4 ldg_stream(const void* p) {   // weights: read once
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint16_t ldg_u16(const uint16_t* p) {
    uint16_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}
__device__ __forceinline__ uint4 ldg_keep(const void* p) {     // activations: reused
    return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ float4 ldcg_f4(const float* p) {    // written by an earlier kernel
    return __ldcg(reinterpret_cast<const float4*>(p));
}

// --------------------------------------------- programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

}  // namespace strata

namespace strata {

// ------------------------------------------------- mbarrier + bulk copies
// One-dimensional bulk copies (global -> this CTA's shared memory) complete
// on an mbarrier's transaction count.  Every wait is bounded: a wait that
// runs out returns false and the caller latches STRATA_ETIMEOUT.
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// Explicit shared-memory loads by 32-bit shared address: used where a
// pointer reaches a non-inlined routine, which would otherwise read shared
// memory through generic addressing.  volatile keeps them after the waits
// that make the data ready.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds_u2(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint16_t lds_u16(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ int lds_s32(uint32_t a) {
    int v;
    asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// dst, src 16-byte aligned; bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace strata
