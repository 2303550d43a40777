// Activation (1x128) and weight (128x128) quantisation to E4M3 with fp32 scales.
//
// Both follow one rule per group: s = amax / 448 (IEEE fp32 division),
// s = 1 for an all-zero group, code = E4M3(x / s) with an IEEE fp32 division
// per element and a round-to-nearest-even, saturating conversion. The
// division is kept (not a multiply by 1/s) because the two differ in the last
// bit often enough to change codes. This is the "W8A8 Block FP8" layer of the
// dual-L20 Qwen3.8-27B-FP8 tuning report (section 8); the pages do not spell
// out the arithmetic, and the rule above is the plain reading of an amax/448
// fp32 scale.
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
constexpr int kActUnroll = 2;
constexpr int kMaxActProblems = 16;

// Where group g of the flattened index lives: one problem ...
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

// ... or several, concatenated: problem i owns groups [begin_i, begin_{i+1}).
struct ActGroupedProblem {
    const uint4* x;
    uint2* q;
    float* sa;
    int64_t begin;
};
struct ActGroupedArgs {
    ActGroupedProblem p[kMaxActProblems];
    int count;
    int64_t groups;
};
struct ActGrouped {
    const ActGroupedArgs* a;
    __device__ __forceinline__ void at(int64_t g, const uint4*& xg, uint2*& qg, float*& sg) const {
        int i = 0;
        while (i + 1 < a->count && g >= a->p[i + 1].begin) ++i;
        const int64_t l = g - a->p[i].begin;
        xg = a->p[i].x + l * 16;
        qg = a->p[i].q + l * 16;
        sg = a->p[i].sa + l;
    }
};

template <class Map>
__device__ __forceinline__ void act_quant_body(const Map& map, int64_t groups) {
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;
    const int hl = lane & 15;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t per_iter = 2 * kActUnroll;  // groups one warp handles per iteration

    // Programmatic dependent launch: let the next kernel (the GEMM, whose
    // weight stream does not depend on us) start launching now, then wait for
    // the grid that produced x (and may still read q / sa) to finish.
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    for (int64_t base = warp * per_iter; base < groups; base += nwarp * per_iter) {
        uint4 v[kActUnroll];
        uint2* qg[kActUnroll];
        float* sg[kActUnroll];
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) {
            const int64_t g = base + 2 * u + half;
            const uint4* xg = nullptr;
            qg[u] = nullptr;
            sg[u] = nullptr;
            if (g < groups) map.at(g, xg, qg[u], sg[u]);
            v[u] = g < groups ? ld_dep_stream_v4(xg + hl) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) {
            const int64_t g = base + 2 * u + half;
            uint2 codes;
            const float s = quant_group_halfwarp(v[u], codes);
            if (g < groups) {
                qg[u][hl] = codes;
                if (hl == 0) *sg[u] = s;
            }
        }
    }
}

__global__ void __launch_bounds__(256) act_quant_kernel(const uint4* __restrict__ x, int64_t groups,
                                                        uint2* __restrict__ q, float* __restrict__ sa) {
    act_quant_body(ActSingle{x, q, sa}, groups);
}

__global__ void __launch_bounds__(256) act_quant_grouped_kernel(const __grid_constant__ ActGroupedArgs a) {
    act_quant_body(ActGrouped{&a}, a.groups);
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

static cudaError_t act_quant_config(int64_t groups, int num_sms, cudaStream_t stream, cudaLaunchConfig_t& cfg,
                             cudaLaunchAttribute (&attr)[1]) {
    const int threads = 256;
    const int64_t groups_per_block = (threads / 32) * 2 * kActUnroll;
    int64_t blocks = (groups + groups_per_block - 1) / groups_per_block;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaSuccess;
}

cudaError_t launch_act_quant_grouped(const ActQuantProblem* probs, int count, int num_sms, cudaStream_t stream) {
    if (count <= 0) return cudaSuccess;
    if (count > kMaxActProblems) return cudaErrorInvalidValue;
    ActGroupedArgs a = {};
    int64_t groups = 0;
    for (int i = 0; i < count; ++i) {
        a.p[i].x = static_cast<const uint4*>(probs[i].x);
        a.p[i].q = static_cast<uint2*>(probs[i].q);
        a.p[i].sa = probs[i].sa;
        a.p[i].begin = groups;
        groups += probs[i].M * (probs[i].K / kGroup);
    }
    a.count = count;
    a.groups = groups;
    if (groups == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    act_quant_config(groups, num_sms, stream, cfg, attr);
    return cudaLaunchKernelEx(&cfg, act_quant_grouped_kernel, a);
}

cudaError_t launch_act_quant(const void* x, int64_t M, int64_t K, void* q, float* sa, int num_sms,
                             cudaStream_t stream) {
    const int64_t groups = M * (K / kGroup);
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    act_quant_config(groups, num_sms, stream, cfg, attr);
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
