// Quantisation of one 1x128 activation group by a half-warp, shared by the
// activation-quantisation kernels and the fused quantise-and-multiply GEMM
// so that both produce the same codes bit for bit.
//
// Rule (the "W8A8 Block FP8" layer of the dual-L20 Qwen3.8-27B-FP8 tuning
// report, section 8; the pages leave the arithmetic open and this is the
// plain reading of an amax / 448 fp32 scale): s = amax / 448 with one IEEE
// fp32 division (s = 1 for an all-zero group); code = E4M3(x / s), the IEEE
// fp32 quotient rounded to nearest even, saturating.
//
// How it is computed. IEEE divisions were most of the group code's
// instructions (they made the kernel instruction-bound at large M), so for a
// group amax in [2^-70, 2^70] all three quotients come from short fused
// multiply-add sequences that reproduce them exactly:
//  - s = amax / 448: the constant RN(1/448) and one residual correction
//    (Markstein's method: q0 = a * c, r = 448 * q0 - a exactly, s = q0 - r * c);
//  - y = RN(1 / s): the hardware approximate reciprocal and one
//    Newton-Raphson step (e = 1 - s * y0, y = y0 + e * y0);
//  - x / s: q0 = x * y, r = s * q0 - x (exact), q = q0 - r * y.
// s and y equal the IEEE results bit for bit for all 17,921 bf16 amax values
// of the range (checked exhaustively on the GPU). q can differ from the IEEE
// quotient only where that quotient underflows fp32, and its E4M3 code never
// differs: checked exhaustively on the GPU for every bf16 amax in the range
// and every bf16 x with |x| <= amax (582,683,394 pairs, the whole input
// domain of the range, since the group amax bounds every element); the
// parity tests compare the kernel with the IEEE-division oracle over that
// same domain. Groups outside the range (tiny or huge scales, all-zero
// groups) use the IEEE division.
#pragma once

#include "common.cuh"

namespace fp8act {

constexpr float kFastQuotientMinAmax = 0x1p-70f;
constexpr float kFastQuotientMaxAmax = 0x1p70f;

__device__ __forceinline__ float rcp_approx_ftz(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Lane l (0..15) of the half-warp holds elements 8l..8l+7 of the group in
// `v` (8 bf16). Every lane of the half returns the group's scale and its 8
// codes packed little-endian in `codes`. The xor shuffles stay inside the
// half-warp; the whole warp must execute the call.
__device__ __forceinline__ float quant_group_halfwarp(const uint4& v, uint2& codes) {
    float f[8];
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    float s, q[8];
    if (amax >= kFastQuotientMinAmax && amax <= kFastQuotientMaxAmax) {
        constexpr float kInv448 = 1.0f / kE4M3Max;  // RN(1/448)
        const float s0 = __fmul_rn(amax, kInv448);
        s = __fmaf_rn(-__fmaf_rn(kE4M3Max, s0, -amax), kInv448, s0);
        const float y0 = rcp_approx_ftz(s);
        const float y = __fmaf_rn(__fmaf_rn(-s, y0, 1.0f), y0, y0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float q0 = __fmul_rn(f[i], y);
            const float r = __fmaf_rn(s, q0, -f[i]);
            q[i] = __fmaf_rn(-r, y, q0);
        }
    } else {
        s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, kE4M3Max);
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(f[i], s);
    }
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = cvt_e4m3x2(q[2 * i], q[2 * i + 1]);
    codes = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    return s;
}

}  // namespace fp8act
