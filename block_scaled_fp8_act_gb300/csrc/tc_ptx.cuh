// Inline-PTX wrappers for the 5th-generation tensor cores (tcgen05): tensor
// memory allocation, UMMA issue / commit, TMEM loads, fences, and the
// shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout that a TMA copy with CU_TENSOR_MAP_SWIZZLE_128B writes.
#pragma once

#include <cstdint>

namespace fp8act {
namespace tc {

// Allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to shared memory at `smem_dst`. Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_dst), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] x B[smem desc]^T, FP8 (kind::f8f6f4) with fp32
// accumulation; `accumulate` = 0 overwrites D.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}

// Load 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape:
// lane i of the warp reads TMEM lane (warp % 4) * 32 + i).
__device__ __forceinline__ void ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void ld_32x32b_x16(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void ld_32x32b_x8(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

// Load kCols (a multiple of 8) consecutive fp32 columns of this thread's TMEM
// lane into r[0 .. kCols): every load is issued before the caller's single
// wait_ld(), so their latencies overlap.
template <int kCols>
__device__ __forceinline__ void ld_cols(uint32_t taddr, uint32_t* r) {
    static_assert(kCols % 8 == 0, "TMEM loads move 8 columns at a time");
#pragma unroll
    for (int c = 0; c + 16 <= kCols; c += 16) ld_32x32b_x16(taddr + c, r + c);
    if constexpr (kCols % 16) ld_32x32b_x8(taddr + (kCols & ~15), r + (kCols & ~15));
}

__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (sm_100 format) of a K-major operand tile
// stored as the 128-byte swizzled layout: rows of 128 bytes, 8-row groups
// 1024 bytes apart (stride byte offset), the K extent of one MMA inside one
// swizzle row (leading byte offset unused, set to 1). `smem_addr` must lie
// in a 1024-byte aligned tile; advancing it by 32 bytes selects the next
// K = 32 slice of FP8 elements.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);  // start address, 16-byte units
    d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version for sm_100
    d |= static_cast<uint64_t>(2) << 61;                    // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::f8f6f4: E4M3 x E4M3 -> fp32, both
// operands K-major, tile M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                                   // D format: fp32
           | (0u << 7) | (0u << 10)                    // A, B format: E4M3
           | (0u << 15) | (0u << 16)                   // A, B K-major
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Warpgroup register reallocation: every warp of the warpgroup executes it.
// Decrease gives registers back to the CTA's pool; increase waits until the
// pool can cover the new per-thread count.
template <uint32_t kRegs>
__device__ __forceinline__ void regs_decrease() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void regs_increase() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}

}  // namespace tc
}  // namespace fp8act
