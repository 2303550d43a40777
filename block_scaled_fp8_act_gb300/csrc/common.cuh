// Device helpers shared by the kernels of libfp8act (sm_103a only).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace fp8act {

constexpr int kGroup = 128;       // quantisation group / block edge along K (and N for weights)
constexpr float kE4M3Max = 448.0f;  // largest finite E4M3 value

__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }

// Two fp32 values to two E4M3 codes packed as (lo | hi << 8): round to
// nearest even, saturating to +-448 (PTX cvt.rn.satfinite.e4m3x2.f32 puts its
// first source in the upper byte).
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 values rounded to bf16 (nearest even) and packed as (lo | hi << 16).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// 16-byte load of data read exactly once: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// 32-byte load of data read exactly once (one 256-bit access; `p` must be
// 32-byte aligned): bytes 0..15 to lo, 16..31 to hi.
__device__ __forceinline__ void ld_stream_v8(const void* p, uint4& lo, uint4& hi) {
    asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
        : "l"(p));
}

// 32-byte load of data that many CTAs re-read (kept in L1); `p` 32-byte aligned.
__device__ __forceinline__ void ld_ro_v8(const void* p, uint4& lo, uint4& hi) {
    asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
        : "l"(p));
}

// 8-byte load of data read exactly once.
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// Hint: bring the 128-byte line holding `p` into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// 16-byte load of data that many CTAs re-read (kept in L1).
__device__ __forceinline__ uint4 ld_shared_ro_v4(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

}  // namespace fp8act
