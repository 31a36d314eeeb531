// e4m3_rule.cuh -- the fine-grained E4M3 quantization rule as device code,
// shared by the quantization kernels and the GEMM that quantizes its token
// operand in the producer ("dssusan.co.kr Q&A post 93378", Figure 7(a)
// passage: every group scaled by its own max-abs):
//   s = amax / 448 (binary32 division),  q = E4M3_rn_satfinite(fl32(x / s)),
//   s == 0 -> q = signed zero.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fgf8 {
namespace {

constexpr float kE4M3Max = 448.0f;

// Two binary32 values to two E4M3 codes (round to nearest even, saturate to
// +-448); `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Group divisor: s and its correctly rounded reciprocal.  `fast` is false for
// s == 0 (all-zero group: the elements are +-0 and are encoded as they are),
// for very small s and for s so large that 1/s would be subnormal; those
// groups take the IEEE division.
struct Divisor {
    float s, r;
    bool fast;
};

__device__ __forceinline__ Divisor make_divisor(float s)
{
    Divisor d;
    d.s = s;
    d.fast = s >= 0x1p-90f && s <= 0x1p125f;
    d.r = d.fast ? __frcp_rn(s) : 0.0f;
    return d;
}

// fl32(x / s) by Markstein's final-correction step (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): with r = RN(1/s) and
// q0 = RN(x*r) within one ulp of x/s, the remainder e = x - s*q0 is exact in
// one fused multiply-add and RN(q0 + e*r) is the correctly rounded quotient,
// provided nothing overflows or underflows.  In a `fast` group (s >= 2^-90,
// |x| <= 448 s) that holds for every |x| >= 2^-100; an element below that has
// |x/s| < 2^-10, under the smallest E4M3 rounding midpoint, so it encodes to a
// signed zero whichever binary32 neighbour the step returns.  The remainder is
// formed negated, e' = s*q0 - x, and subtracted, q0 - e'*r: the same values
// for x != 0, and for x = -0 the result keeps its sign (-0 - (+0) = -0).
__device__ __forceinline__ float scaled(float x, const Divisor &d)
{
    if (d.fast) {
        const float q0 = __fmul_rn(x, d.r);
        const float en = __fmaf_rn(q0, d.s, -x);
        return __fmaf_rn(-en, d.r, q0);
    }
    if (x == 0.0f || d.s == 0.0f) return x;     // +-0 / s keeps the sign of x; all-zero group
    return __fdiv_rn(x, d.s);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Channel j (0..7) of 8 packed BF16 values, as binary32.
__device__ __forceinline__ float bf16_lane(const uint4 &v, int j)
{
    const uint32_t w = j < 2 ? v.x : j < 4 ? v.y : j < 6 ? v.z : v.w;
    return __uint_as_float((j & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// Eight codes.  In a `fast` group the quotients come from the same three
// roundings as scaled(), done on value pairs with packed FP32 operations (each
// lane an IEEE multiply or fused multiply-add): the same bits, fewer
// instructions.
__device__ __forceinline__ uint2 encode8(const float (&f)[8], const Divisor &s)
{
    uint2 o;
    if (s.fast) {
        const float2 r2 = make_float2(s.r, s.r), s2 = make_float2(s.s, s.s);
        uint32_t c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 x2 = make_float2(f[2 * i], f[2 * i + 1]);
            const float2 q0 = __fmul2_rn(x2, r2);
            const float2 en = __ffma2_rn(q0, s2, make_float2(-x2.x, -x2.y));
            const float2 q = __ffma2_rn(make_float2(-en.x, -en.y), r2, q0);
            c[i] = cvt_e4m3x2(q.x, q.y);
        }
        o.x = c[0] | (c[1] << 16);
        o.y = c[2] | (c[3] << 16);
        return o;
    }
    o.x = cvt_e4m3x2(scaled(f[0], s), scaled(f[1], s)) | (cvt_e4m3x2(scaled(f[2], s), scaled(f[3], s)) << 16);
    o.y = cvt_e4m3x2(scaled(f[4], s), scaled(f[5], s)) | (cvt_e4m3x2(scaled(f[6], s), scaled(f[7], s)) << 16);
    return o;
}

__device__ __forceinline__ float amax8(const float (&f)[8])
{
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(f[i]));
    return a;
}

}  // namespace
}  // namespace fgf8
