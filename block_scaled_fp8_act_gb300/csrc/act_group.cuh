// Quantisation of one 1x128 activation group by a half-warp, shared by the
// activation-quantisation kernels and the fused quantise-and-multiply GEMM
// so that both produce the same codes bit for bit.
//
// Rule (the "W8A8 Block FP8" layer of the dual-L20 Qwen3.8-27B-FP8 tuning
// report, section 8; the pages leave the arithmetic open and this is the
// plain reading of an amax / 448 fp32 scale): s = amax / 448 with one IEEE
// fp32 division (s = 1 for an all-zero group); code = E4M3(x / s) with an
// IEEE fp32 division per element, round to nearest even, saturating.
#pragma once

#include "common.cuh"

namespace fp8act {

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
    const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, kE4M3Max);
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = cvt_e4m3x2(__fdiv_rn(f[2 * i], s), __fdiv_rn(f[2 * i + 1], s));
    codes = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    return s;
}

}  // namespace fp8act
