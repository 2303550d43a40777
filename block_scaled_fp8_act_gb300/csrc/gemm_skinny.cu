// Weight-streaming block-FP8 GEMM for small M (decode and speculative verify).
//
// At M <= 8 the layer is a pure weight stream: every weight byte is used for
// at most 8 multiply-adds, so the kernel is bound by HBM. The pages put about
// 89% of a decode step into exactly these weight-reading GEMMs and name a
// library kernel that fell off a cliff between M = 1 and M = 2..7
// ("单并发提速73%,多并发能力达原来2.4倍:Qwen3.8-27B性能优化实践", section
// "算子优化"). This kernel has one code path for every M <= 8, so its time does
// not depend on M.
//
// Why tensor cores for a memory-bound kernel: at M = 8 the CUDA cores would
// need 8 fp32 FMAs per weight byte, i.e. ~190 FMA/clk/SM at the HBM rate,
// above the 128 the SM has. One warp-level m16n8k32 e4m3 MMA does 16x8x32
// multiply-adds, so the arithmetic costs a few instructions per 2 KB of
// weights and the loads stay in front.
//
// Layout of the work:
//  - A CTA owns a 16-row tile of W (rows n0..n0+15, all inside one 128-row
//    scale block) and a group of <= 8 tokens. Its warps split the K blocks
//    (kb = warp, warp + nwarps, ...), so each warp's partial sums are for
//    whole 128-wide blocks and the fp32 block scales are applied in registers.
//  - Swap-AB: the 16 weight rows are the MMA's A operand (m16), the tokens its
//    B operand (n8), so tokens past M just cost zero registers.
//  - A dot product inside one 128-wide block does not depend on the order of
//    its terms. Each lane therefore loads 16 contiguous bytes of a weight row
//    straight into its A-fragment registers (no shared-memory staging), and
//    the activation fragment is loaded with the same K permutation:
//    lane (g, t) = (lane/4, lane%4) reads bytes [16t, 16t+16) and
//    [64+16t, 64+16t+16) of the block for weight rows g and g+8 and for token
//    g; MMA i of the block takes words 2i and 2i+1 of those 32 bytes. Over
//    t = 0..3 and i = 0..3 every byte of the block is used exactly once.
//  - Four MMAs (K = 128) accumulate one block's dot in fp32; it is then scaled
//    by sa[m, kb] * sw[n/128, kb] and added into the warp's running sums.
//  - The warps' partial sums meet in shared memory and one pass writes the
//    16 x M outputs (bf16, or fp32 for the error-analysis entry point).
//
// Weight-only mode (kModeA16): the activations stay bf16 (no quantisation
// launch, the job of the weight-only FP8 back-end that the same post uses at
// one request, section "单并发优化"). Each lane widens its 32 weight codes of
// a block to bf16 (E4M3 -> f16 -> f32 -> bf16, exact at every step) and runs
// eight m16n8k16 bf16 MMAs per block, with the same K permutation: MMA i
// takes codes 4i..4i+3 of the lane's 32 and the lane's activations at the
// same positions (64 bytes of bf16 per lane and block). Only the weight
// scale multiplies the block's dot.
//
// Fused mode (kModeFQ): bf16 activations in, the layer's full W8A8 result
// out, in one launch (the quantisation launch per linear layer is what the
// same post's single-request section credits the weight-only back-end with
// saving; here the quantisation stays and moves into the GEMM). Each warp
// quantises exactly the 1x128 groups of the K blocks it multiplies (its <= 8
// tokens), with the activation kernel's own group code (the same codes and
// scales bit for bit), into a private slice of shared memory, once its first
// weight loads are in flight: no warp waits for another. Every CTA repeats
// the quantisation of the same tokens.
//
// Fused, one quantisation per SM (linear_persistent_kernel, M <= 16): one CTA
// per SM whose warps quantise all the tokens once into shared memory and
// then, in groups, stream the weight tiles (16 rows x 8 tokens; above 8
// tokens each row tile twice, the second read mostly from L2, as the
// two-launch grid does) with this file's loop and the two-launch path's
// warp count per tile (so the same sums); it replaces the
// per-CTA quantisation, which a timeline trace showed stalling every CTA's
// weight stream for several microseconds. From two tokens on, a
// thread-block cluster of 2 or 4 CTAs shares the quantisation: each CTA
// quantises every C-th group and stores it into the shared memory of all C
// CTAs (distributed shared memory), so an SM does 1/C of the work for the
// price of two cluster barriers.
#include <atomic>

#include <cuda_fp16.h>

#include "act_group.cuh"
#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace fp8act {
namespace {

constexpr int kMaxWarps = 16;
// Kernel modes: W8A8 (E4M3 activation codes and scales in), weight-only
// (bf16 activations, widened weights) and fused (bf16 activations quantised
// by each warp into shared memory, then the W8A8 loop).
constexpr int kModeW8A8 = 0;
constexpr int kModeA16 = 1;
constexpr int kModeFQ = 2;
// Added to kModeW8A8 / kModeFQ: each lane streams 32 contiguous bytes of a
// weight row per block with one 256-bit load (needs 32-byte aligned weights
// and codes) instead of two 16-byte chunks 64 bytes apart.
constexpr int kWideBit = 4;
constexpr int base_mode(int mode) { return mode & 3; }
constexpr bool wide_mode(int mode) { return (mode & kWideBit) != 0; }
// Fused mode: each warp's shared-memory slice holds the codes [J][rows][128]
// and scales [J][rows] of the J = ceil(KB / warps) K blocks it multiplies
// (kb = warp, warp + warps, ...), rows = min(8, M) tokens.
constexpr size_t kFqMaxSmem = 200 * 1024;  // the fused slices of one CTA, at most
__host__ __device__ constexpr int fq_slice_bytes(int KB, int warps, int rows) {
    return ((KB + warps - 1) / warps * rows * (kGroup + 4) + 15) & ~15;
}
// L2 prefetch distance, in warp steps: each warp keeps the weight lines of
// the next steps on their way into L2 (prefetches hold no registers). One
// step measured best: 10% off the five decode shapes at M = 1 against no
// prefetch, while 8 or 16 steps thrash L2 and lose.
constexpr int kL2Ahead = 1;
constexpr int kMaxGroupedProblems = 16;

__device__ __forceinline__ void mma_e4m3_16x8x32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                  uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16_16x8x16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                  uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 codes (code 0 in the low byte) -> bf16x2 (value 0 in the low
// half). Every E4M3 value, subnormals included, is a normal f16 and a normal
// bf16, so each conversion step is exact.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t codes) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(codes & 0xFFFFu)));
    __half2 h;
    memcpy(&h, &h2, 4);
    const float2 f = __half22float2(h);
    return pack_bf16x2(f.x, f.y);
}

// Eight weight words (32 codes, in the lane's K order) -> sixteen bf16x2 words.
__device__ __forceinline__ void widen_row(const uint4& lo, const uint4& hi, uint32_t (&r)[16]) {
    const uint32_t wd[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        r[2 * i] = e4m3x2_to_bf16x2(wd[i]);
        r[2 * i + 1] = e4m3x2_to_bf16x2(wd[i] >> 16);
    }
}

// One CTA's work: output rows n0..n0+15 for tokens m0..m0 + 8 kTG - 1.
// kUnroll = K blocks whose weight loads a warp has in flight at once;
// kTG = groups of 8 tokens a CTA handles (they share the weight fragments);
// kMode: kModeW8A8 (codes in `q`, scales in `sa`), kModeA16 (bf16
// activations in `q`, `sa` unused) or kModeFQ (bf16 activations in `q`,
// quantised by each warp, step by step, into its slice of the dynamic shared
// memory `fq_smem`; `sa` unused; kTG must be 1).
template <bool kF32Out, int kUnroll, int kTG, int kMode>
__device__ __forceinline__ void skinny_tile(const uint8_t* __restrict__ q, const float* __restrict__ sa,
                                            const uint8_t* __restrict__ w, const float* __restrict__ sw, int M,
                                            int N, int K, void* __restrict__ out, int n0, int m0,
                                            float (*red)[16][8 * kTG], uint8_t* fq_smem = nullptr) {
    static_assert(base_mode(kMode) != kModeFQ || kTG == 1, "the fused mode quantises one group of 8 tokens per CTA");
    const int KB = K / kGroup;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int g = lane >> 2;
    const int t = lane & 3;

    const bool ok_r0 = n0 + g < N;
    const bool ok_r1 = n0 + g + 8 < N;
    constexpr bool kWide = wide_mode(kMode);
    static_assert(!kWide || base_mode(kMode) != kModeA16, "the weight-only mode keeps 16-byte chunks");
    // Lane (g, t) takes bytes [16t, 16t+16) and [64+16t, 64+16t+16) of each
    // 128-byte block, or with kWide the 32 contiguous bytes [32t, 32t+32).
    // Either way the K positions depend on t only, the same for every weight
    // row and token, so A and B fragments pair up the same K elements.
    const int lane_off = kWide ? 32 * t : 16 * t;
    const uint8_t* w_r0 = w + static_cast<int64_t>(n0 + g) * K + lane_off;
    const uint8_t* w_r1 = w + static_cast<int64_t>(n0 + g + 8) * K + lane_off;
    const float* sw_r = sw + static_cast<int64_t>(n0 / kGroup) * KB;

    float acc[kTG][4];
#pragma unroll
    for (int j = 0; j < kTG; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    const uint4 zero = make_uint4(0, 0, 0, 0);

    // Programmatic dependent launch: the weights never depend on the previous
    // grid, so the first weight loads go out before waiting for it; the
    // activations, scales and output are touched only after the wait.
    ptx::griddep_launch_dependents();
    // Lanes 0..15 prefetch the 128-byte line of weight row n0 + lane for the
    // blocks kL2Ahead warp steps ahead; the first steps' lines go out before
    // the wait, so the weight stream starts while the previous grid finishes.
    const int stride = nwarps * kUnroll;
    const bool pf_lane = lane < 16 && n0 + lane < N;
    const uint8_t* w_pf = w + static_cast<int64_t>(n0 + lane) * K;
    if (pf_lane) {
#pragma unroll
        for (int s = 1; s <= kL2Ahead; ++s)
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int kb = warp + s * stride + u * nwarps;
                if (kb < KB) prefetch_l2(w_pf + static_cast<int64_t>(kb) * kGroup);
            }
    }
    bool waited = false;
    // Fused mode: this warp's private slice of the dynamic shared memory holds
    // the codes and scales of the K blocks it multiplies (slot j: block
    // warp + j * nwarps), quantised by the warp itself once its first weight
    // loads are in flight.
    const int fq8 = M < 8 ? M : 8;  // token rows of every slot (the slice size is per launch)
    const int fq_rows = M - m0 < 8 ? M - m0 : 8;
    const int fq_slots = (KB + nwarps - 1) / nwarps;
    uint8_t* const q_s = fq_smem + static_cast<int64_t>(warp) * fq_slice_bytes(KB, nwarps, fq8);
    float* const sa_s = reinterpret_cast<float*>(q_s + fq_slots * fq8 * kGroup);
    for (int kb0 = warp; kb0 < KB; kb0 += stride) {
        if (pf_lane) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int kb = kb0 + (kL2Ahead + 1) * stride + u * nwarps;
                if (kb < KB) prefetch_l2(w_pf + static_cast<int64_t>(kb) * kGroup);
            }
        }
        uint4 r0lo[kUnroll], r0hi[kUnroll], r1lo[kUnroll], r1hi[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int kb = kb0 + u * nwarps;
            const bool ok_k = kb < KB;
            const int64_t off = static_cast<int64_t>(kb) * kGroup;
            if constexpr (kWide) {
                r0lo[u] = r0hi[u] = r1lo[u] = r1hi[u] = zero;
                if (ok_k && ok_r0) ld_stream_v8(w_r0 + off, r0lo[u], r0hi[u]);
                if (ok_k && ok_r1) ld_stream_v8(w_r1 + off, r1lo[u], r1hi[u]);
            } else {
                r0lo[u] = (ok_k && ok_r0) ? ld_stream_v4(w_r0 + off) : zero;
                r0hi[u] = (ok_k && ok_r0) ? ld_stream_v4(w_r0 + off + 64) : zero;
                r1lo[u] = (ok_k && ok_r1) ? ld_stream_v4(w_r1 + off) : zero;
                r1hi[u] = (ok_k && ok_r1) ? ld_stream_v4(w_r1 + off + 64) : zero;
            }
        }
        if (!waited) {
            ptx::griddep_wait();
            waited = true;
            if constexpr (base_mode(kMode) == kModeFQ) {
                // Quantise every 1x128 group (token r, block kb) this warp will multiply,
                // with the activation kernel's group code (the same codes and scales bit
                // for bit): half-warp h takes groups 2 p + h of pass p, and the whole warp
                // runs every pass because the group code shuffles. The first step's
                // weight loads are already in flight and no other warp waits for it.
                const int half = lane >> 4;
                const int hl = lane & 15;
                const int groups = fq_slots * fq_rows;
                for (int base_g = 0; base_g < groups; base_g += 2) {
                    const int gi = base_g + half;
                    const int j = gi / fq_rows, r = gi % fq_rows;
                    const int kb = warp + j * nwarps;
                    const bool ok = gi < groups && kb < KB;
                    const uint4 v = ok ? ld_dep_stream_v4(q + (static_cast<int64_t>(m0 + r) * K + kb * kGroup + 8 * hl) * 2)
                                       : zero;
                    uint2 codes;
                    const float sg = quant_group_halfwarp(v, codes);
                    if (ok) {
                        *reinterpret_cast<uint2*>(q_s + (j * fq8 + r) * kGroup + 8 * hl) = codes;
                        if (hl == 0) sa_s[j * fq8 + r] = sg;
                    }
                }
                __syncwarp();
            }
        }
        if constexpr (base_mode(kMode) == kModeA16) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int kb = kb0 + u * nwarps;
                if (kb >= KB) continue;
                uint32_t wa[16], wb[16];  // rows g and g + 8, bf16x2
                widen_row(r0lo[u], r0hi[u], wa);
                widen_row(r1lo[u], r1hi[u], wb);
                const float s_w = __ldg(sw_r + kb);
                const int64_t off = static_cast<int64_t>(kb) * kGroup * 2;
#pragma unroll
                for (int j = 0; j < kTG; ++j) {
                    const int m = m0 + 8 * j + g;
                    const bool ok_x = m < M;
                    const uint8_t* x_r = q + (static_cast<int64_t>(m) * K + 16 * t) * 2 + off;
                    const uint4 x0 = ok_x ? ld_dep_v4(x_r) : zero;
                    const uint4 x1 = ok_x ? ld_dep_v4(x_r + 16) : zero;
                    const uint4 x2 = ok_x ? ld_dep_v4(x_r + 128) : zero;
                    const uint4 x3 = ok_x ? ld_dep_v4(x_r + 144) : zero;
                    const uint32_t xw[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                                             x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        mma_bf16_16x8x16(d, wa[2 * i], wb[2 * i], wa[2 * i + 1], wb[2 * i + 1], xw[2 * i],
                                         xw[2 * i + 1]);
                    const int c0 = m0 + 8 * j + 2 * t;
                    const float s0 = c0 < M ? s_w : 0.f;
                    const float s1 = c0 + 1 < M ? s_w : 0.f;
                    acc[j][0] = fmaf(d[0], s0, acc[j][0]);
                    acc[j][1] = fmaf(d[1], s1, acc[j][1]);
                    acc[j][2] = fmaf(d[2], s0, acc[j][2]);
                    acc[j][3] = fmaf(d[3], s1, acc[j][3]);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < kTG; ++j) {
                const int m = m0 + 8 * j + g;  // this lane's token for the B fragment
                const bool ok_x = m < M;
                const uint8_t* x_r = base_mode(kMode) == kModeFQ ? q_s + g * kGroup + lane_off
                                                                 : q + static_cast<int64_t>(m) * K + lane_off;
                const int j0 = (kb0 - warp) / nwarps;  // fused mode: slot of this step's first block
                constexpr int kHiOff = kWide ? 16 : 64;  // byte offset of the lane's second 16 bytes
                const int c0 = m0 + 8 * j + 2 * t;  // token columns of this lane's accumulators
                uint4 xlo[kUnroll], xhi[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int kb = kb0 + u * nwarps;
                    const bool ok_k = kb < KB;
                    const int64_t off = static_cast<int64_t>(kb) * kGroup;
                    if constexpr (base_mode(kMode) == kModeFQ) {
                        const int so = (j0 + u) * fq8 * kGroup;  // slot of block u of this step
                        xlo[u] = (ok_k && ok_x) ? *reinterpret_cast<const uint4*>(x_r + so) : zero;
                        xhi[u] = (ok_k && ok_x) ? *reinterpret_cast<const uint4*>(x_r + so + kHiOff) : zero;
                    } else if constexpr (kWide) {
                        xlo[u] = xhi[u] = zero;
                        if (ok_k && ok_x) ld_dep_v8(x_r + off, xlo[u], xhi[u]);
                    } else {
                        xlo[u] = (ok_k && ok_x) ? ld_dep_v4(x_r + off) : zero;
                        xhi[u] = (ok_k && ok_x) ? ld_dep_v4(x_r + off + 64) : zero;
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int kb = kb0 + u * nwarps;
                    if (kb < KB) {
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_e4m3_16x8x32(d, r0lo[u].x, r1lo[u].x, r0lo[u].y, r1lo[u].y, xlo[u].x, xlo[u].y);
                        mma_e4m3_16x8x32(d, r0lo[u].z, r1lo[u].z, r0lo[u].w, r1lo[u].w, xlo[u].z, xlo[u].w);
                        mma_e4m3_16x8x32(d, r0hi[u].x, r1hi[u].x, r0hi[u].y, r1hi[u].y, xhi[u].x, xhi[u].y);
                        mma_e4m3_16x8x32(d, r0hi[u].z, r1hi[u].z, r0hi[u].w, r1hi[u].w, xhi[u].z, xhi[u].w);
                        const float s_w = __ldg(sw_r + kb);
                        float sa0 = 0.f, sa1 = 0.f;
                        if constexpr (base_mode(kMode) == kModeFQ) {
                            if (c0 < M) sa0 = sa_s[(j0 + u) * fq8 + (c0 - m0)];
                            if (c0 + 1 < M) sa1 = sa_s[(j0 + u) * fq8 + (c0 + 1 - m0)];
                        } else {
                            if (c0 < M) sa0 = ld_dep_f32(sa + static_cast<int64_t>(c0) * KB + kb);
                            if (c0 + 1 < M) sa1 = ld_dep_f32(sa + static_cast<int64_t>(c0 + 1) * KB + kb);
                        }
                        const float s0 = sa0 * s_w;
                        const float s1 = sa1 * s_w;
                        acc[j][0] = fmaf(d[0], s0, acc[j][0]);
                        acc[j][1] = fmaf(d[1], s1, acc[j][1]);
                        acc[j][2] = fmaf(d[2], s0, acc[j][2]);
                        acc[j][3] = fmaf(d[3], s1, acc[j][3]);
                    }
                }
            }
        }
    }
    if (!waited) ptx::griddep_wait();

#pragma unroll
    for (int j = 0; j < kTG; ++j) {
        red[warp][g][8 * j + 2 * t] = acc[j][0];
        red[warp][g][8 * j + 2 * t + 1] = acc[j][1];
        red[warp][g + 8][8 * j + 2 * t] = acc[j][2];
        red[warp][g + 8][8 * j + 2 * t + 1] = acc[j][3];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 16 * 8 * kTG; i += blockDim.x) {
        const int r = i & 15;  // consecutive threads write consecutive n
        const int c = i >> 4;
        float v = 0.f;
        for (int ww = 0; ww < nwarps; ++ww) v += red[ww][r][c];
        const int n = n0 + r;
        if (n < N && m0 + c < M) {
            const int64_t o = static_cast<int64_t>(m0 + c) * N + n;
            if constexpr (kF32Out) {
                static_cast<float*>(out)[o] = v;
            } else {
                static_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(v);
            }
        }
    }
}

template <bool kF32Out, int kUnroll, int kTG, int kMode = kModeW8A8>
__global__ void __launch_bounds__(kMaxWarps * 32) gemm_skinny_kernel(
    const uint8_t* __restrict__ q, const float* __restrict__ sa, const uint8_t* __restrict__ w,
    const float* __restrict__ sw, int M, int N, int K, void* __restrict__ out) {
    __shared__ float red[kMaxWarps][16][8 * kTG];
    extern __shared__ __align__(16) uint8_t fq_smem[];
    // CTA b: token group b % ty of weight-row tile b / ty (the token groups of
    // one row tile on adjacent CTAs, so the rows' second read hits L2)
    const int ty = (M + 8 * kTG - 1) / (8 * kTG);
    skinny_tile<kF32Out, kUnroll, kTG, kMode>(q, sa, w, sw, M, N, K, out, (blockIdx.x / ty) * 16,
                                              (blockIdx.x % ty) * 8 * kTG, red, fq_smem);
}

// Several independent problems in one grid: CTA b belongs to the problem p
// with begin[p] <= b < begin[p + 1] and takes its tile (b - begin[p]) %
// tiles_n (16 weight rows) for token group (b - begin[p]) / tiles_n.
struct GroupedProblem {
    const uint8_t* q;
    const float* sa;
    const uint8_t* w;
    const float* sw;
    void* out;
    int M, N, K;
    int begin;    // first CTA of this problem
    int tiles_n;  // 16-row weight tiles
};
struct GroupedArgs {
    GroupedProblem p[kMaxGroupedProblems];
    int count;
};

template <bool kF32Out, int kUnroll>
__global__ void __launch_bounds__(kMaxWarps * 32) gemm_skinny_grouped_kernel(const __grid_constant__ GroupedArgs a) {
    __shared__ float red[kMaxWarps][16][8];
    const int b = static_cast<int>(blockIdx.x);
    int i = 0;
    while (i + 1 < a.count && b >= a.p[i + 1].begin) ++i;
    const GroupedProblem& p = a.p[i];
    const int local = b - p.begin;
    skinny_tile<kF32Out, kUnroll, 1, kModeW8A8>(p.q, p.sa, p.w, p.sw, p.M, p.N, p.K, p.out, (local % p.tiles_n) * 16,
                                            (local / p.tiles_n) * 8, red);
}

// CTAs per SM for a (load depth, token groups, mode, warps) configuration
// without dynamic shared memory, from the occupancy API (cached per device).
template <bool kF32Out, int kUnroll, int kTG, int kMode>
int ctas_per_sm(int wv) {
    static std::atomic<int> cache[64][kMaxWarps + 1];  // 0 = unknown, else 1 + CTAs per SM
    int dev = 0;
    cudaGetDevice(&dev);
    int cached = cache[dev & 63][wv].load(std::memory_order_relaxed);
    if (cached == 0) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_skinny_kernel<kF32Out, kUnroll, kTG, kMode>,
                                                          32 * wv, 0) != cudaSuccess) {
            cudaGetLastError();
            per_sm = 0;
        }
        cached = per_sm + 1;
        cache[dev & 63][wv].store(cached, std::memory_order_relaxed);
    }
    return cached - 1;
}

// CTAs per SM that the SM's shared memory allows with `smem` dynamic bytes
// per CTA (and the 1 KB the runtime reserves per CTA).
int smem_ctas_per_sm(size_t smem) {
    if (smem == 0) return 1 << 20;
    static std::atomic<int> per_sm_bytes[64];
    int dev = 0;
    cudaGetDevice(&dev);
    int b = per_sm_bytes[dev & 63].load(std::memory_order_relaxed);
    if (b == 0) {
        if (cudaDeviceGetAttribute(&b, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) {
            cudaGetLastError();
            b = 228 * 1024;
        }
        per_sm_bytes[dev & 63].store(b, std::memory_order_relaxed);
    }
    return static_cast<int>(static_cast<size_t>(b) / (smem + 1024));
}

// Dynamic shared memory of a CTA with wv warps: the fused mode's slices.
template <int kMode>
size_t cta_smem(int KB, int wv, int M) {
    return base_mode(kMode) == kModeFQ ? static_cast<size_t>(wv) * fq_slice_bytes(KB, wv, M < 8 ? M : 8) : 0;
}

// Warps per CTA for a load depth: among the warp counts whose K groups split
// evenly to within 10% (every warp finishes at about the same time) and for
// which the whole grid is resident in one wave, the one with the most weight
// bytes in flight (capped where HBM saturates, ~20 MB on GB300); 0 if none.
template <bool kF32Out, int kUnroll, int kTG, int kMode = kModeW8A8>
int pick_warps(int64_t ctas, int KB, int num_sms, int64_t* inflight_out, int M = 1) {
    constexpr int64_t kSaturate = int64_t(20) << 20;
    int best = 0;
    int64_t best_inflight = -1;
    for (int wv = 1; wv <= kMaxWarps && wv <= KB; ++wv) {
        const int per_warp = (KB + wv - 1) / wv;
        if (10 * KB < 9 * wv * per_warp) continue;  // warps would finish more than 10% apart
        const size_t smem = cta_smem<kMode>(KB, wv, M);
        if (smem > kFqMaxSmem) continue;
        int per_sm = ctas_per_sm<kF32Out, kUnroll, kTG, kMode>(wv);
        const int by_smem = smem_ctas_per_sm(smem);
        if (by_smem < per_sm) per_sm = by_smem;
        if (ctas > static_cast<int64_t>(per_sm) * num_sms) continue;
        int64_t inflight = ctas * wv * (per_warp < kUnroll ? per_warp : kUnroll) * (16 * kGroup);
        if (inflight > kSaturate) inflight = kSaturate;
        if (inflight > best_inflight || (inflight == best_inflight && wv < best)) {
            best = wv;
            best_inflight = inflight;
        }
    }
    if (inflight_out) *inflight_out = best_inflight;
    return best;
}

template <bool kF32Out, int kUnroll, int kTG, int kMode = kModeW8A8>
cudaError_t launch_typed(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw, int M, int N, int K,
                         void* out, int num_sms, cudaStream_t stream) {
    const int KB = K / kGroup;
    const int64_t ctas = static_cast<int64_t>((N + 15) / 16) * ((M + 8 * kTG - 1) / (8 * kTG));
    if (ctas > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(ctas));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    // The fused mode gives each warp a slice of dynamic shared memory.
    if constexpr (base_mode(kMode) == kModeFQ) {
        static std::atomic<uint64_t> configured{0};  // one bit per device
        int dev = 0;
        cudaGetDevice(&dev);
        const uint64_t bit = 1ull << (dev & 63);
        if (!(configured.load(std::memory_order_acquire) & bit)) {
            const cudaError_t e = cudaFuncSetAttribute(gemm_skinny_kernel<kF32Out, kUnroll, kTG, kMode>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(kFqMaxSmem));
            if (e != cudaSuccess) return e;
            configured.fetch_or(bit, std::memory_order_release);
        }
    }
    int wv = pick_warps<kF32Out, kUnroll, kTG, kMode>(ctas, KB, num_sms, nullptr, M);
    if (wv == 0) wv = KB < 4 ? KB : 4;  // grid larger than one wave: plain 4-warp CTAs
    // the fused slices of very long K at wide M: more warps, smaller slices
    while (cta_smem<kMode>(KB, wv, M) > kFqMaxSmem && wv < kMaxWarps && wv < KB) ++wv;
    if (cta_smem<kMode>(KB, wv, M) > kFqMaxSmem) return cudaErrorInvalidValue;
    cfg.blockDim = dim3(32 * wv);
    cfg.dynamicSmemBytes = cta_smem<kMode>(KB, wv, M);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<kF32Out, kUnroll, kTG, kMode>, q, sa, w, sw, M, N, K, out);
}

// ------------------------------------------------------------------------
// Fused mode with one quantisation per SM (M <= 16). One CTA per SM, up to 32
// warps in groups of `wg`; tile t (16 weight rows x 8 tokens) runs on CTA
// t % gridDim.x, group (t / gridDim.x) % groups, and each group runs the
// two-launch kernel's loop on its tiles (the same warp count per tile, so the
// same K order and sums), reading the activation codes and scales from
// shared memory, where the CTA's warps (or, with a cluster, the cluster's
// CTAs) put them once, after the programmatic-launch wait, with the
// activation kernel's group code. The first weight steps of every group's
// first tile go to L2 before the wait.
constexpr int kPqMaxWarps = 32;
constexpr int kPqMaxGroups = 15;  // named barriers 1..15 (0 is __syncthreads)
// activation groups per half-warp slot and quantisation pass: 4 where the
// prologue holds no weight registers (depth 1), 2 where it does (depth 4)
template <int kUnroll>
constexpr int pq_quant_unroll() { return kUnroll > 1 ? 2 : 4; }
template <int kUnroll>
constexpr int pq_max_warps() { return kUnroll == 1 ? kPqMaxWarps : kPqMaxWarps / 2; }  // 64 / 128 registers
// CTAs per cluster sharing the quantisation: 1 for one token; otherwise the
// smallest of 2 and 4 that leaves each SM at most kPqGroupsPerSm of the
// M x KB activation groups, 4 at most. Measured on the five decode
// projections at M = 1, 2, 4, 8, alone and in the mixed five-shape step,
// against every size: an SM quantises ~256 groups per microsecond, a load
// round trip per pass comes on top, and a cluster costs two cluster barriers
// and the remote stores (0.5-1.5 us at 4 CTAs); 8 CTAs never beat 4, and at
// one token (at most ~one group per half-warp) no cluster paid.
constexpr int kPqGroupsPerSm = 40;
constexpr int kPqMaxCluster = 4;
inline int pq_cluster_size(int M, int KB) {
    if (M <= 1) return 1;
    int c = 2;
    while (c < kPqMaxCluster && M * KB > kPqGroupsPerSm * c) c *= 2;
    return c;
}

struct PqArgs {
    const uint8_t* x;  // bf16 activations [M][K]
    const uint8_t* w;
    const float* sw;
    void* out;
    int M, N, K, KB, tiles;
    int tg;       // groups of 8 tokens (1 or 2); tile t = weight rows 16 (t / tg), tokens 8 (t % tg)
    int wg;       // warps per tile
    int groups;   // warp groups per CTA
    int cluster;  // CTAs per thread-block cluster sharing the quantisation (1, 2, 4 or 8)
};

__host__ __device__ inline int pq_codes_stride(int K) { return K + 16; }  // padded rows
__host__ __device__ inline int pq_sa_offset(int M, int K) { return (M * pq_codes_stride(K) + 15) & ~15; }
__host__ __device__ inline int pq_red_offset(int M, int K, int KB) { return pq_sa_offset(M, K) + ((M * KB * 4 + 15) & ~15); }
inline size_t pq_smem_bytes(int M, int K, int groups, int wg) {
    return static_cast<size_t>(pq_red_offset(M, K, K / kGroup)) + static_cast<size_t>(groups) * wg * 16 * 8 * 4;
}

// One tile (16 weight rows x 8 tokens) by the warps of one group: the W8A8
// loop of skinny_tile (same load depth, K permutation, MMA order, scale
// products and warp-order sum), with the codes and scales read from shared
// memory.
template <bool kF32Out, int kUnroll, bool kWide, class Prologue>
__device__ __forceinline__ void pq_tile(const PqArgs& a, const uint8_t* __restrict__ q_s, const float* __restrict__ sa_s,
                                        float (*red)[16][8], int tile, int gw, uint32_t bar_id, bool run_prologue,
                                        const Prologue& prologue) {
    const int KB = a.KB, K = a.K, M = a.M, N = a.N, wg = a.wg;
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int n0 = (tile / a.tg) * 16, m0 = (tile % a.tg) * 8;
    const bool ok_r0 = n0 + g < N, ok_r1 = n0 + g + 8 < N;
    const int lane_off = kWide ? 32 * t : 16 * t;
    constexpr int kHiOff = kWide ? 16 : 64;
    const uint8_t* w_r0 = a.w + static_cast<int64_t>(n0 + g) * K + lane_off;
    const uint8_t* w_r1 = a.w + static_cast<int64_t>(n0 + g + 8) * K + lane_off;
    const float* sw_r = a.sw + static_cast<int64_t>(n0 / kGroup) * KB;
    const int stride = wg * kUnroll;
    const bool pf_lane = lane < 16 && n0 + lane < N;
    const uint8_t* w_pf = a.w + static_cast<int64_t>(n0 + lane) * K;
    if (pf_lane) {
#pragma unroll
        for (int s = 1; s <= kL2Ahead; ++s)
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int kb = gw + s * stride + u * wg;
                if (kb < KB) prefetch_l2(w_pf + static_cast<int64_t>(kb) * kGroup);
            }
    }
    const bool ok_x = m0 + g < M;
    const uint8_t* x_r = q_s + (m0 + g) * pq_codes_stride(K) + lane_off;
    const int c0 = m0 + 2 * t;  // token columns of this lane's accumulators: c0, c0 + 1
    const uint4 zero = make_uint4(0, 0, 0, 0);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kb0 = gw; kb0 < KB; kb0 += stride) {
        if (pf_lane) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int kb = kb0 + (kL2Ahead + 1) * stride + u * wg;
                if (kb < KB) prefetch_l2(w_pf + static_cast<int64_t>(kb) * kGroup);
            }
        }
        uint4 r0lo[kUnroll], r0hi[kUnroll], r1lo[kUnroll], r1hi[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int kb = kb0 + u * wg;
            const bool ok_k = kb < KB;
            const int64_t off = static_cast<int64_t>(kb) * kGroup;
            if constexpr (kWide) {
                r0lo[u] = r0hi[u] = r1lo[u] = r1hi[u] = zero;
                if (ok_k && ok_r0) ld_stream_v8(w_r0 + off, r0lo[u], r0hi[u]);
                if (ok_k && ok_r1) ld_stream_v8(w_r1 + off, r1lo[u], r1hi[u]);
            } else {
                r0lo[u] = (ok_k && ok_r0) ? ld_stream_v4(w_r0 + off) : zero;
                r0hi[u] = (ok_k && ok_r0) ? ld_stream_v4(w_r0 + off + 64) : zero;
                r1lo[u] = (ok_k && ok_r1) ? ld_stream_v4(w_r1 + off) : zero;
                r1hi[u] = (ok_k && ok_r1) ? ld_stream_v4(w_r1 + off + 64) : zero;
            }
        }
        if (run_prologue) {  // the first tile: its first weight loads are in flight
            prologue();
            run_prologue = false;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int kb = kb0 + u * wg;
            if (kb < KB) {
                const uint4 xlo = ok_x ? *reinterpret_cast<const uint4*>(x_r + kb * kGroup) : zero;
                const uint4 xhi = ok_x ? *reinterpret_cast<const uint4*>(x_r + kb * kGroup + kHiOff) : zero;
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma_e4m3_16x8x32(d, r0lo[u].x, r1lo[u].x, r0lo[u].y, r1lo[u].y, xlo.x, xlo.y);
                mma_e4m3_16x8x32(d, r0lo[u].z, r1lo[u].z, r0lo[u].w, r1lo[u].w, xlo.z, xlo.w);
                mma_e4m3_16x8x32(d, r0hi[u].x, r1hi[u].x, r0hi[u].y, r1hi[u].y, xhi.x, xhi.y);
                mma_e4m3_16x8x32(d, r0hi[u].z, r1hi[u].z, r0hi[u].w, r1hi[u].w, xhi.z, xhi.w);
                const float s_w = __ldg(sw_r + kb);
                const float sa0 = c0 < M ? sa_s[c0 * KB + kb] : 0.f;
                const float sa1 = c0 + 1 < M ? sa_s[(c0 + 1) * KB + kb] : 0.f;
                const float s0 = sa0 * s_w;
                const float s1 = sa1 * s_w;
                acc[0] = fmaf(d[0], s0, acc[0]);
                acc[1] = fmaf(d[1], s1, acc[1]);
                acc[2] = fmaf(d[2], s0, acc[2]);
                acc[3] = fmaf(d[3], s1, acc[3]);
            }
        }
    }
    red[gw][g][2 * t] = acc[0];
    red[gw][g][2 * t + 1] = acc[1];
    red[gw][g + 8][2 * t] = acc[2];
    red[gw][g + 8][2 * t + 1] = acc[3];
    ptx::named_bar_sync(bar_id, wg * 32);
    for (int i = gw * 32 + lane; i < 16 * 8; i += wg * 32) {
        const int r = i & 15, c = i >> 4;
        float v = 0.f;
        for (int ww = 0; ww < wg; ++ww) v += red[ww][r][c];
        const int n = n0 + r;
        if (n < N && m0 + c < M) {
            const int64_t o = static_cast<int64_t>(m0 + c) * N + n;
            if constexpr (kF32Out)
                static_cast<float*>(a.out)[o] = v;
            else
                static_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(v);
        }
    }
    ptx::named_bar_sync(bar_id, wg * 32);  // the partial sums are read before the next tile writes them
}

template <bool kF32Out, int kUnroll, bool kWide>
__global__ void __launch_bounds__(pq_max_warps<kUnroll>() * 32, 1) linear_persistent_kernel(const __grid_constant__ PqArgs a) {
    extern __shared__ __align__(16) uint8_t pq_smem[];
    uint8_t* const q_s = pq_smem;
    float* const sa_s = reinterpret_cast<float*>(pq_smem + pq_sa_offset(a.M, a.K));
    float(*const red_all)[16][8] = reinterpret_cast<float(*)[16][8]>(pq_smem + pq_red_offset(a.M, a.K, a.KB));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int group = warp / a.wg, gw = warp % a.wg;
    const int step = gridDim.x * a.groups;

    ptx::griddep_launch_dependents();
    const int csize = a.cluster;
    if (csize > 1) ptx::cluster_arrive_relaxed();  // this CTA has started (its shared memory takes peer stores)
    // Everything that needs the previous grid's output, run by every thread
    // exactly once: the wait, the quantisation of the 1x128 groups of the M
    // tokens with the activation kernel's group code, and the barrier after
    // which the codes are read. In a cluster of C CTAs, CTA r quantises
    // groups r, r + C, ... and stores each group's codes and scale into the
    // shared memory of every CTA of the cluster (itself included), so each
    // SM does 1/C of the work; the cluster barrier then orders those stores
    // before any read. Within a CTA, its i-th group goes to half-warp slot
    // i % (2 nwarps), so every warp shares the work, and a slot's groups of
    // one pass (pq_quant_unroll) have their loads issued together.
    auto prologue = [&]() {
        const int rank = csize > 1 ? static_cast<int>(ptx::cluster_ctarank()) : 0;
        const int half = lane >> 4, hl = lane & 15;
        const int ngroups = a.M * a.KB;
        const int mine = (ngroups - rank + csize - 1) / csize;  // groups rank, rank + C, ... < ngroups
        const int slots = 2 * nwarps;
        const int slot = 2 * warp + half;
        const uint4 zero = make_uint4(0, 0, 0, 0);
        constexpr int kQU = pq_quant_unroll<kUnroll>();
        // The x lines of the slot's first pass go to L2 before the wait (a
        // cache hint only: the previous grid's writes land in L2, so the
        // loads after the wait still see them), which takes the DRAM round
        // trip of an x that has left L2 off the start of the weight stream.
        if ((hl & 7) == 0) {
#pragma unroll
            for (int u = 0; u < kQU; ++u) {
                const int li = u * slots + slot;
                if (li < mine) {
                    const int gi = rank + li * csize;
                    prefetch_l2(a.x + (static_cast<int64_t>(gi / a.KB) * a.K + (gi % a.KB) * kGroup + 8 * hl) * 2);
                }
            }
        }
        ptx::griddep_wait();
        if (csize > 1) ptx::cluster_wait();  // every peer has started
        for (int base = 0; base < mine; base += kQU * slots) {
            uint4 v[kQU];
#pragma unroll
            for (int u = 0; u < kQU; ++u) {
                const int li = base + u * slots + slot;
                const bool ok = li < mine;
                const int gi = rank + li * csize;
                const int r = ok ? gi / a.KB : 0, kb = ok ? gi % a.KB : 0;
                v[u] = ok ? ld_dep_stream_v4(a.x + (static_cast<int64_t>(r) * a.K + kb * kGroup + 8 * hl) * 2) : zero;
            }
#pragma unroll
            for (int u = 0; u < kQU; ++u) {
                if (base + u * slots + 2 * warp >= mine) break;  // warp-uniform: the group code shuffles
                const int li = base + u * slots + slot;
                const bool ok = li < mine;
                const int gi = rank + li * csize;
                const int r = ok ? gi / a.KB : 0, kb = ok ? gi % a.KB : 0;
                uint2 codes;
                const float sg = quant_group_halfwarp(v[u], codes);
                if (ok) {
                    uint8_t* const qd = q_s + r * pq_codes_stride(a.K) + kb * kGroup + 8 * hl;
                    float* const sd = sa_s + r * a.KB + kb;
                    if (csize == 1) {
                        *reinterpret_cast<uint2*>(qd) = codes;
                        if (hl == 0) *sd = sg;
                    } else {
                        const uint32_t qa = ptx::smem_u32(qd), sda = ptx::smem_u32(sd);
                        for (int c = 0; c < csize; ++c) {
                            ptx::st_shared_cluster_v2(ptx::mapa_shared(qa, c), codes);
                            if (hl == 0) ptx::st_shared_cluster_f32(ptx::mapa_shared(sda, c), sg);
                        }
                    }
                }
            }
        }
        if (csize > 1)
            ptx::cluster_sync();
        else
            __syncthreads();
    };
    float(*const red)[16][8] = red_all + group * a.wg;
    // tiles dealt round-robin over the CTAs, then the groups: tile t runs on
    // CTA t % gridDim.x, so every SM of the grid streams
    const int first = blockIdx.x + group * gridDim.x;
    // Depth 4 (short K): the first tile issues its first weight loads (four
    // K blocks per warp) before the prologue, as the two-launch kernel does
    // before its wait. Depth 1: the first tile's lines are only prefetched to
    // L2 before the prologue; holding the loads across it measured slower
    // there (64 registers: the prologue's own registers crowd them).
    constexpr bool kLoadsFirst = kUnroll > 1;
    if (!kLoadsFirst || first >= a.tiles) {  // a group without tiles still takes part in the prologue
        if (!kLoadsFirst && first < a.tiles && lane < 16 && (first / a.tg) * 16 + lane < a.N) {
            const uint8_t* w_pf = a.w + static_cast<int64_t>((first / a.tg) * 16 + lane) * a.K;
#pragma unroll
            for (int st = 0; st <= kL2Ahead; ++st) {
                const int kb = gw + st * a.wg;
                if (kb < a.KB) prefetch_l2(w_pf + static_cast<int64_t>(kb) * kGroup);
            }
        }
        prologue();
        if (first >= a.tiles) return;
    }
    pq_tile<kF32Out, kUnroll, kWide>(a, q_s, sa_s, red, first, gw, 1 + group, kLoadsFirst, prologue);
    for (int tile = first + step; tile < a.tiles; tile += step)
        pq_tile<kF32Out, kUnroll, kWide>(a, q_s, sa_s, red, tile, gw, 1 + group, false, prologue);
}

template <bool kF32Out, int kUnroll, bool kWide>
cudaError_t configure_persistent() {
    static std::atomic<uint64_t> configured{0};  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        const cudaError_t e = cudaFuncSetAttribute(linear_persistent_kernel<kF32Out, kUnroll, kWide>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_release);
    }
    return cudaSuccess;
}

// Clusters of `csize` CTAs of the per-SM fused kernel that the device holds
// at once (one CTA per SM; a cluster's CTAs share a GPC, so for csize > 2
// some SMs may stay out), from the occupancy API, cached per device.
template <bool kF32Out, int kUnroll, bool kWide>
int persistent_clusters(int csize) {
    static std::atomic<int> cache[64][4];  // csize 1, 2, 4, 8; 1 + clusters, 0 = unknown
    const int ci = csize >= 8 ? 3 : csize >= 4 ? 2 : csize >= 2 ? 1 : 0;
    int dev = 0;
    cudaGetDevice(&dev);
    int cached = cache[dev & 63][ci].load(std::memory_order_relaxed);
    if (cached == 0) {
        int n = 0;
        if (configure_persistent<kF32Out, kUnroll, kWide>() == cudaSuccess) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(csize);
            q.blockDim = dim3(pq_max_warps<kUnroll>() * 32);
            q.dynamicSmemBytes = 227 * 1024;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = csize;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, linear_persistent_kernel<kF32Out, kUnroll, kWide>, &q) !=
                cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
        } else {
            cudaGetLastError();
        }
        cached = n + 1;
        cache[dev & 63][ci].store(cached, std::memory_order_relaxed);
    }
    return cached - 1;
}

template <bool kF32Out, int kUnroll, bool kWide>
cudaError_t launch_persistent(const PqArgs& a, int grid, size_t smem, cudaStream_t stream) {
    const cudaError_t e = configure_persistent<kF32Out, kUnroll, kWide>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(a.groups * a.wg * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = a.cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.cluster > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, linear_persistent_kernel<kF32Out, kUnroll, kWide>, a);
}

}  // namespace

cudaError_t launch_gemm_skinny_unroll(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw, int M,
                                      int N, int K, void* out, bool out_f32, int num_sms, int unroll,
                                      cudaStream_t stream) {
    // Above M = 8 the grid gets a CTA per 8 tokens and row tile, the token
    // groups of a row tile on adjacent CTAs (each re-reads the weights, the
    // second read mostly from L2); for 9..16 tokens this measured faster than
    // CTAs that hold 16 tokens against one weight fragment.
    // 256-bit weight and code loads on the depth-4 (short K) path when both
    // start on 32-byte boundaries (rows are K bytes apart, K a multiple of
    // 128, so every lane's 32-byte chunk then is aligned too; the API
    // guarantees only 16). Measured: 3.8 against 4.1 us on (5120, 3072) at
    // M = 1; on the depth-1 path they were slower (16.2 against 14.6 us on
    // (17408, 5120)), so it keeps 16-byte chunks.
    constexpr int kW = kModeW8A8 | kWideBit;
    const bool wide = ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(w)) & 31) == 0;
    if (unroll >= 4) {
        if (wide)
            return out_f32 ? launch_typed<true, 4, 1, kW>(q, sa, w, sw, M, N, K, out, num_sms, stream)
                           : launch_typed<false, 4, 1, kW>(q, sa, w, sw, M, N, K, out, num_sms, stream);
        return out_f32 ? launch_typed<true, 4, 1>(q, sa, w, sw, M, N, K, out, num_sms, stream)
                       : launch_typed<false, 4, 1>(q, sa, w, sw, M, N, K, out, num_sms, stream);
    }
    if (unroll >= 2)
        return out_f32 ? launch_typed<true, 2, 1>(q, sa, w, sw, M, N, K, out, num_sms, stream)
                       : launch_typed<false, 2, 1>(q, sa, w, sw, M, N, K, out, num_sms, stream);
    return out_f32 ? launch_typed<true, 1, 1>(q, sa, w, sw, M, N, K, out, num_sms, stream)
                   : launch_typed<false, 1, 1>(q, sa, w, sw, M, N, K, out, num_sms, stream);
}

cudaError_t launch_gemm_skinny(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw, int M,
                               int N, int K, void* out, bool out_f32, int num_sms, cudaStream_t stream) {
    // Load depth per warp step. Long K (>= 32 blocks): one block per step,
    // which takes the fewest registers (64) and so leaves room for the most
    // warps while the whole grid stays resident; it measured fastest on every
    // long-K projection at M = 1..16. Short K: four blocks per step; the loop
    // is only a few steps long, so most of each warp's weights are requested
    // before the programmatic-launch wait and overlap the previous kernel.
    const int KB = K / kGroup;
    const int unroll = KB >= 32 ? 1 : 4;
    return launch_gemm_skinny_unroll(q, sa, w, sw, M, N, K, out, out_f32, num_sms, unroll, stream);
}

cudaError_t launch_gemm_w8a16(const void* x, const uint8_t* w, const float* sw, int M, int N, int K, void* out,
                              bool out_f32, int num_sms, cudaStream_t stream) {
    // One K block per warp step: the widened weights and the bf16
    // activations make each block in flight cost more registers than in the
    // W8A8 mode, and with the whole grid resident in one wave the register
    // count per thread sets how many warps (and so how many weight bytes)
    // each SM keeps in flight. Depth 1 measured fastest at M = 1, 8 and 16.
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    if (M > 8)  // two token groups per CTA share the widened weights
        return out_f32 ? launch_typed<true, 1, 2, kModeA16>(xb, nullptr, w, sw, M, N, K, out, num_sms, stream)
                       : launch_typed<false, 1, 2, kModeA16>(xb, nullptr, w, sw, M, N, K, out, num_sms, stream);
    return out_f32 ? launch_typed<true, 1, 1, kModeA16>(xb, nullptr, w, sw, M, N, K, out, num_sms, stream)
                   : launch_typed<false, 1, 1, kModeA16>(xb, nullptr, w, sw, M, N, K, out, num_sms, stream);
}

cudaError_t launch_gemm_skinny_grouped(const GemmProblem* probs, int count, bool out_f32, cudaStream_t stream) {
    if (count <= 0) return cudaSuccess;
    if (count > kMaxGroupedProblems) return cudaErrorInvalidValue;
    // Largest problems first: their CTAs start in the first wave, the small
    // ones fill in behind them.
    int order[kMaxGroupedProblems];
    for (int i = 0; i < count; ++i) order[i] = i;
    for (int i = 1; i < count; ++i)
        for (int j = i; j > 0; --j) {
            const GemmProblem& a = probs[order[j - 1]];
            const GemmProblem& b = probs[order[j]];
            if (static_cast<int64_t>(a.N) * a.K >= static_cast<int64_t>(b.N) * b.K) break;
            const int tmp = order[j];
            order[j] = order[j - 1];
            order[j - 1] = tmp;
        }
    GroupedArgs args = {};
    int64_t ctas = 0;
    int min_kb = 1 << 30;
    for (int i = 0; i < count; ++i) {
        const GemmProblem& src = probs[order[i]];
        GroupedProblem& d = args.p[i];
        d.q = src.q;
        d.sa = src.sa;
        d.w = src.w;
        d.sw = src.sw;
        d.out = src.out;
        d.M = src.M;
        d.N = src.N;
        d.K = src.K;
        d.begin = static_cast<int>(ctas);
        d.tiles_n = (src.N + 15) / 16;
        ctas += static_cast<int64_t>(d.tiles_n) * ((src.M + 7) / 8);
        if (ctas > 0x7FFFFFFF) return cudaErrorInvalidValue;
        if (src.K / kGroup < min_kb) min_kb = src.K / kGroup;
    }
    args.count = count;
    // The grid spans several waves, so CTAs take the 4-warp shape that
    // measured best for multi-wave grids, one K block per warp step.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(32 * (min_kb < 4 ? min_kb : 4));
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return out_f32 ? cudaLaunchKernelEx(&cfg, gemm_skinny_grouped_kernel<true, 1>, args)
                   : cudaLaunchKernelEx(&cfg, gemm_skinny_grouped_kernel<false, 1>, args);
}

bool fused_fits(int M, int K) {
    // the slices of any warp count hold every block once, plus at most 15
    // bytes of rounding per warp
    const int KB = K / kGroup;
    return static_cast<size_t>(KB) * (M < 8 ? M : 8) * (kGroup + 4) + 15 * kMaxWarps <= kFqMaxSmem;
}

namespace {

// The fused kernel with one quantisation per SM, M <= 16; cudaErrorNotSupported
// (nothing launched) when the codes do not fit shared memory.
template <bool kF32Out, int kUnroll, bool kWide>
cudaError_t launch_persistent_typed(const void* x, const uint8_t* w, const float* sw, int M, int N, int K, void* out,
                                    int num_sms, cudaStream_t stream) {
    PqArgs a;
    a.x = static_cast<const uint8_t*>(x);
    a.w = w;
    a.sw = sw;
    a.out = out;
    a.M = M;
    a.N = N;
    a.K = K;
    a.KB = K / kGroup;
    // tiles of 16 weight rows x 8 tokens, the token groups of one row tile
    // adjacent (neighbouring CTAs, so the second read of the rows hits L2)
    a.tg = (M + 7) / 8;
    a.tiles = (N + 15) / 16 * a.tg;
    // warps per tile: the two-launch kernel's choice for this shape, whose
    // grid has as many CTAs as these tiles (same K order, same sums)
    constexpr int kMode = kWide ? (kModeW8A8 | kWideBit) : kModeW8A8;
    int wv = pick_warps<kF32Out, kUnroll, 1, kMode>(a.tiles, a.KB, num_sms, nullptr, M);
    if (wv == 0) wv = a.KB < 4 ? a.KB : 4;
    a.wg = wv;
    int groups = pq_max_warps<kUnroll>() / wv;
    if (groups > kPqMaxGroups) groups = kPqMaxGroups;
    const int per_sm = (a.tiles + num_sms - 1) / num_sms;
    if (groups > per_sm) groups = per_sm;
    if (groups < 1) return cudaErrorNotSupported;
    a.groups = groups;
    const size_t smem = pq_smem_bytes(M, K, groups, wv);
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    // one CTA per SM (or per tile, if fewer), each taking every grid-th tile
    int grid = a.tiles < num_sms ? a.tiles : num_sms;
    // Share the quantisation over a cluster when each SM would otherwise
    // quantise many groups. The grid becomes whole clusters, all resident at
    // once (CTAs past the last tile only quantise their share): rounded up,
    // or down to the resident clusters when that leaves no CTA group more
    // tiles than before; otherwise a smaller cluster.
    a.cluster = 1;
    const int64_t per_cta = static_cast<int64_t>(groups);
    const int64_t rounds = (a.tiles + grid * per_cta - 1) / (grid * per_cta);
    for (int c = pq_cluster_size(M, a.KB); c > 1; c /= 2) {
        const int resident = persistent_clusters<kF32Out, kUnroll, kWide>(c) * c;
        const int up = (grid + c - 1) / c * c;
        const int g = up <= resident ? up : resident;
        if (g < c || (a.tiles + g * per_cta - 1) / (g * per_cta) > rounds) continue;
        a.cluster = c;
        grid = g;
        break;
    }
    return launch_persistent<kF32Out, kUnroll, kWide>(a, grid, smem, stream);
}

template <bool kF32Out>
cudaError_t launch_persistent_any(const void* x, const uint8_t* w, const float* sw, int M, int N, int K, void* out,
                                  int num_sms, cudaStream_t stream) {
    if (K / kGroup >= 32) return launch_persistent_typed<kF32Out, 1, false>(x, w, sw, M, N, K, out, num_sms, stream);
    if ((reinterpret_cast<uintptr_t>(w) & 31) == 0)
        return launch_persistent_typed<kF32Out, 4, true>(x, w, sw, M, N, K, out, num_sms, stream);
    return launch_persistent_typed<kF32Out, 4, false>(x, w, sw, M, N, K, out, num_sms, stream);
}

}  // namespace

cudaError_t launch_linear_fused(const void* x, const uint8_t* w, const float* sw, int M, int N, int K, void* out,
                                bool out_f32, int num_sms, cudaStream_t stream) {
    if (M <= 16) {
        const cudaError_t e = out_f32 ? launch_persistent_any<true>(x, w, sw, M, N, K, out, num_sms, stream)
                                      : launch_persistent_any<false>(x, w, sw, M, N, K, out, num_sms, stream);
        if (e != cudaErrorNotSupported) return e;
    }
    // The W8A8 loop with the same load depth rule as launch_gemm_skinny, so
    // that at equal launch geometry the two paths sum in the same order.
    // 256-bit weight loads on the depth-4 path as in launch_gemm_skinny_unroll
    // (the codes come from shared memory here, so only the weights' alignment
    // matters).
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    constexpr int kW = kModeFQ | kWideBit;
    const bool wide = (reinterpret_cast<uintptr_t>(w) & 31) == 0;
    if (K / kGroup >= 32) {
        return out_f32 ? launch_typed<true, 1, 1, kModeFQ>(xb, nullptr, w, sw, M, N, K, out, num_sms, stream)
                       : launch_typed<false, 1, 1, kModeFQ>(xb, nullptr, w, sw, M, N, K, out, num_sms, stream);
    }
    if (wide)
        return out_f32 ? launch_typed<true, 4, 1, kW>(xb, nullptr, w, sw, M, N, K, out, num_sms, stream)
                       : launch_typed<false, 4, 1, kW>(xb, nullptr, w, sw, M, N, K, out, num_sms, stream);
    return out_f32 ? launch_typed<true, 4, 1, kModeFQ>(xb, nullptr, w, sw, M, N, K, out, num_sms, stream)
                   : launch_typed<false, 4, 1, kModeFQ>(xb, nullptr, w, sw, M, N, K, out, num_sms, stream);
}

}  // namespace fp8act
