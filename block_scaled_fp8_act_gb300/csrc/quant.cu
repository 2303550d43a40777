// Activation (1x128) and weight (128x128) quantisation to E4M3 with fp32 scales.
//
// Both follow one rule per group: s = amax / 448 (IEEE fp32 division),
// s = 1 for an all-zero group, code = E4M3(x / s), the IEEE fp32 quotient
// rounded to nearest even, saturating. This is the "W8A8 Block FP8" layer of
// the dual-L20 Qwen3.8-27B-FP8 tuning report (section 8); the pages do not
// spell out the arithmetic, and the rule above is the plain reading of an
// amax/448 fp32 scale. A plain multiply by 1/s is not enough: it changes a
// code whenever the quotient sits within an ulp or two of an E4M3 rounding
// midpoint, which bf16 inputs hit often (their short significands make many
// quotients exact midpoints). The activation path forms the scale, the
// reciprocal and the quotients from short fused multiply-add sequences that
// give the IEEE results' scales and codes for every input (act_group.cuh
// says how that was established); the offline weight path keeps the plain
// IEEE division.
#include <atomic>

#include "act_group.cuh"
#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace fp8act {
namespace {

// Each half-warp quantises one 128-element group: lane l of the half holds
// elements 8l..8l+7 (one 16-byte load), the amax is reduced over the 16
// lanes with xor shuffles, and each lane stores its 8 codes (8 bytes).
// Groups are contiguous in memory because K % 128 == 0, so group g of the
// flattened [M*K/128] index starts at element 128 g and its scale is sa[g].
// A warp takes 2 * kActUnroll groups per iteration and issues the loads of
// its next iteration before quantising the current one, so every warp keeps
// two iterations of loads in flight. At large M the kernel is bound by the
// instruction issue and the latency of each group's chain (loads, shuffles,
// scale, reciprocal, quotients); measured at M = 4096, K = 5120 / 8704:
// 5 CTAs of 256 threads per SM (the launch bound below) with two groups per
// half-warp and a grid of exactly the resident CTAs beat deeper unrolls,
// 4, 6 or 8 CTAs per SM (8 spill, and a grid of 8 per SM with 5 resident
// runs in 1.6 waves) and a TMA bulk-copy ring feeding shared memory.
constexpr int kActUnroll = 2;
constexpr int kActThreads = 256;
constexpr int kActMinCtas = 5;
constexpr int kMaxActProblems = 16;

// Where group g of one problem lives.
struct ActSingle {
    const uint4* x;
    uint2* q;
    float* sa;
    __device__ __forceinline__ void at(int64_t g, const uint4*& xg, uint2*& qg, float*& sg) const {
        xg = x + g * 16;
        qg = q + g * 16;
        sg = sa + g;
    }
};

// Several problems in one launch: problem i owns the CTAs [cta_begin_i,
// cta_begin_{i+1}), in proportion to its groups, and they run the
// single-problem loop over it (a per-group lookup of the problem, even with
// a cursor, made the grouped launch slower than separate launches at
// M = 4096: measured 86 / 71 us against 61 us for the five projections).
struct ActGroupedProblem {
    const uint4* x;
    uint2* q;
    float* sa;
    int64_t groups;
    int cta_begin;
};
struct ActGroupedArgs {
    ActGroupedProblem p[kMaxActProblems];
    int count;
};

template <class Map>
__device__ __forceinline__ void act_quant_body(const Map& map, int64_t groups, int block, int nblocks) {
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;
    const int hl = lane & 15;
    const int64_t warp = (static_cast<int64_t>(block) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (static_cast<int64_t>(nblocks) * blockDim.x) >> 5;
    const int64_t per_iter = 2 * kActUnroll;  // groups one warp handles per iteration
    const int64_t step = nwarp * per_iter;
    auto load = [&](int64_t base, uint4 (&v)[kActUnroll]) {
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) {
            const int64_t g = base + 2 * u + half;
            const uint4* xg = nullptr;
            uint2* qg;
            float* sg;
            if (g < groups) map.at(g, xg, qg, sg);
            v[u] = g < groups ? ld_dep_stream_v4(xg + hl) : make_uint4(0, 0, 0, 0);
        }
    };

    // Programmatic dependent launch: let the next kernel (the GEMM, whose
    // weight stream does not depend on us) start launching now, then wait for
    // the grid that produced x (and may still read q / sa) to finish. Before
    // the wait, the two 128-byte lines of each of this warp's first groups
    // are prefetched to L2. A prefetch is only a cache hint and L2 is where
    // the previous grid's writes land, so the loads after the wait still see
    // them; what it saves is the DRAM round trip of an x that has left L2.
    ptx::griddep_launch_dependents();
    if ((hl & 7) == 0) {
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) {
            const int64_t g = warp * per_iter + 2 * u + half;
            if (g < groups) {
                const uint4* xg;
                uint2* qg;
                float* sg;
                map.at(g, xg, qg, sg);
                prefetch_l2(xg + hl);
            }
        }
    }
    ptx::griddep_wait();
    uint4 v[kActUnroll];
    load(warp * per_iter, v);
    for (int64_t base = warp * per_iter; base < groups; base += step) {
        uint4 next[kActUnroll];
        load(base + step, next);
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) {
            const int64_t g = base + 2 * u + half;
            uint2 codes;
            const float s = quant_group_halfwarp(v[u], codes);
            if (g < groups) {
                const uint4* xg;
                uint2* qg;
                float* sg;
                map.at(g, xg, qg, sg);
                qg[hl] = codes;
                if (hl == 0) *sg = s;
            }
        }
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) v[u] = next[u];
    }
}

__global__ void __launch_bounds__(kActThreads, kActMinCtas) act_quant_kernel(const uint4* __restrict__ x, int64_t groups,
                                                        uint2* __restrict__ q, float* __restrict__ sa) {
    act_quant_body(ActSingle{x, q, sa}, groups, blockIdx.x, gridDim.x);
}

__global__ void __launch_bounds__(kActThreads, kActMinCtas) act_quant_grouped_kernel(const __grid_constant__ ActGroupedArgs a) {
    int i = 0;
    while (i + 1 < a.count && static_cast<int>(blockIdx.x) >= a.p[i + 1].cta_begin) ++i;
    const int end = i + 1 < a.count ? a.p[i + 1].cta_begin : static_cast<int>(gridDim.x);
    const ActGroupedProblem& p = a.p[i];
    act_quant_body(ActSingle{p.x, p.q, p.sa}, p.groups, static_cast<int>(blockIdx.x) - p.cta_begin, end - p.cta_begin);
}

// One CTA of 256 threads per 128x128 weight block. Warp w holds rows
// w, w+8, ..., w+120 of the block; lane l holds columns 4l..4l+3 of each.
// The block amax is reduced across the warp, then across the 8 warps in
// shared memory. Rows past N are neither read nor written.
__global__ void __launch_bounds__(256) weight_quant_kernel(const uint16_t* __restrict__ W, int N, int K,
                                                           uint8_t* __restrict__ w, float* __restrict__ sw) {
    __shared__ float warp_max[8];
    const int KB = K / kGroup;
    const int nb = blockIdx.x / KB;
    const int kb = blockIdx.x % KB;
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int col = kb * kGroup + 4 * lane;

    uint2 v[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int row = nb * kGroup + wid + 8 * i;
        v[i] = row < N ? ld_stream_v2(W + static_cast<int64_t>(row) * K + col) : make_uint2(0, 0);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v[i].x)), fabsf(bf16_hi(v[i].x))),
                                 fmaxf(fabsf(bf16_lo(v[i].y)), fabsf(bf16_hi(v[i].y)))));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) warp_max[wid] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, warp_max[i]);
    const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, kE4M3Max);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int row = nb * kGroup + wid + 8 * i;
        if (row < N) {
            const uint32_t lo = cvt_e4m3x2(__fdiv_rn(bf16_lo(v[i].x), s), __fdiv_rn(bf16_hi(v[i].x), s));
            const uint32_t hi = cvt_e4m3x2(__fdiv_rn(bf16_lo(v[i].y), s), __fdiv_rn(bf16_hi(v[i].y), s));
            *reinterpret_cast<uint32_t*>(w + static_cast<int64_t>(row) * K + col) = lo | (hi << 16);
        }
    }
    if (threadIdx.x == 0) sw[static_cast<int64_t>(nb) * KB + kb] = s;
}

}  // namespace

// Resident CTAs per SM of an activation kernel (occupancy API, cached per
// device); the grid never exceeds one wave of them.
static int act_ctas_per_sm(const void* kernel, std::atomic<int> (&cache)[64]) {
    int dev = 0;
    cudaGetDevice(&dev);
    int v = cache[dev & 63].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, kActThreads, 0) != cudaSuccess || v < 1) {
            cudaGetLastError();
            v = kActMinCtas;
        }
        cache[dev & 63].store(v, std::memory_order_relaxed);
    }
    return v;
}

static void act_quant_config(int64_t groups, int num_sms, int per_sm, cudaStream_t stream, cudaLaunchConfig_t& cfg,
                             cudaLaunchAttribute (&attr)[1]) {
    const int64_t groups_per_block = (kActThreads / 32) * 2 * kActUnroll;
    int64_t blocks = (groups + groups_per_block - 1) / groups_per_block;
    const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
    if (blocks > cap) blocks = cap;
    cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kActThreads);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
}

cudaError_t launch_act_quant_grouped(const ActQuantProblem* probs, int count, int num_sms, cudaStream_t stream) {
    if (count <= 0) return cudaSuccess;
    if (count > kMaxActProblems) return cudaErrorInvalidValue;
    int64_t total = 0;
    for (int i = 0; i < count; ++i) total += probs[i].M * (probs[i].K / kGroup);
    if (total == 0) return cudaSuccess;
    static std::atomic<int> per_sm[64];
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    act_quant_config(total, num_sms, act_ctas_per_sm(reinterpret_cast<const void*>(act_quant_grouped_kernel), per_sm),
                     stream, cfg, attr);
    // The grid the single-problem rule gives for all the groups, shared in
    // proportion to each problem's groups (at least one CTA each, and no CTA
    // without a group).
    const int64_t blocks = cfg.gridDim.x;
    constexpr int64_t kGroupsPerBlock = (kActThreads / 32) * 2 * kActUnroll;
    ActGroupedArgs a = {};
    int begin = 0;
    for (int i = 0; i < count; ++i) {
        const int64_t g = probs[i].M * (probs[i].K / kGroup);
        int64_t nb = g == 0 ? 0 : blocks * g / total;
        const int64_t useful = (g + kGroupsPerBlock - 1) / kGroupsPerBlock;
        if (nb > useful) nb = useful;
        if (g > 0 && nb < 1) nb = 1;
        a.p[i].x = static_cast<const uint4*>(probs[i].x);
        a.p[i].q = static_cast<uint2*>(probs[i].q);
        a.p[i].sa = probs[i].sa;
        a.p[i].groups = g;
        a.p[i].cta_begin = begin;
        begin += static_cast<int>(nb);
    }
    a.count = count;
    cfg.gridDim = dim3(static_cast<unsigned>(begin));
    return cudaLaunchKernelEx(&cfg, act_quant_grouped_kernel, a);
}

cudaError_t launch_act_quant(const void* x, int64_t M, int64_t K, void* q, float* sa, int num_sms,
                             cudaStream_t stream) {
    const int64_t groups = M * (K / kGroup);
    static std::atomic<int> per_sm[64];
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    act_quant_config(groups, num_sms, act_ctas_per_sm(reinterpret_cast<const void*>(act_quant_kernel), per_sm), stream,
                     cfg, attr);
    return cudaLaunchKernelEx(&cfg, act_quant_kernel, static_cast<const uint4*>(x), groups,
                              static_cast<uint2*>(q), sa);
}

cudaError_t launch_weight_quant(const void* W, int64_t N, int64_t K, void* w, float* sw, cudaStream_t stream) {
    const int64_t blocks = ((N + kGroup - 1) / kGroup) * (K / kGroup);
    weight_quant_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(W), static_cast<int>(N), static_cast<int>(K), static_cast<uint8_t*>(w), sw);
    return cudaGetLastError();
}

}  // namespace fp8act
