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

// 16-byte load of data read exactly once and never written while any kernel
// of the library runs (the weights): read-only path, no L1 allocation.
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

// Loads of data that the previous grid in the stream may write: activation
// codes, activation scales and bf16 inputs. A kernel launched with
// programmatic dependent launch starts while that grid may still run, and
// reads such data only after griddepcontrol.wait. These loads are volatile
// and clobber memory, so the compiler keeps them after the wait (a plain asm
// load, which it sees as a pure function of the address, or __ldg may be
// hoisted above it), and they take the coherent path (ld.global.nc assumes
// the data cannot change while the kernel runs). The weight loads above stay
// free to move: the weights never change.

// 16 bytes, kept in L1 (re-read by many warps).
__device__ __forceinline__ uint4 ld_dep_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
    return v;
}

// 16 bytes read once (no L1 allocation).
__device__ __forceinline__ uint4 ld_dep_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
    return v;
}

// 32 bytes in one access (`p` 32-byte aligned), kept in L1: bytes 0..15 to lo, 16..31 to hi.
__device__ __forceinline__ void ld_dep_v8(const void* p, uint4& lo, uint4& hi) {
    asm volatile("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                 : "l"(p)
                 : "memory");
}

// One fp32 value.
__device__ __forceinline__ float ld_dep_f32(const float* p) {
    float v;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}

}  // namespace fp8act
