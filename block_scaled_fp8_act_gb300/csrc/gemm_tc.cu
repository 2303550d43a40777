// Tensor-memory (tcgen05) block-FP8 GEMM for batched decode and prefill (M > 16).
//
// At prefill sizes (M = 4096) the layer is a dense contraction: 2MNK =
// 129..730 GFLOP per call against 36..110 MB of operands, far above the FP8
// ridge point, so the kernel is built around the 5th-generation tensor cores.
// The pages saw exactly this shape regress when served by a kernel tuned for
// M = 1 ("双 NVIDIA L20 上 Qwen3.8-27B-FP8 + MTP 调优测试报告", sections 五 and 八):
// prefill gets its own tile kernel.
//
// One CTA computes a 128 x 256 output tile (128 tokens x 256 weight rows):
//  * warp 0, one thread: TMA producer. A 4-stage ring of shared-memory
//    stages, each one 128-wide K group: the 128 x 128 activation tile and the
//    256 x 128 weight tile, both in the 128-byte swizzled K-major layout. The
//    weight copies of the first stages go out before the kernel waits on the
//    previous grid (programmatic dependent launch).
//  * warp 1: allocates 512 TMEM columns (two 128 x 256 fp32 accumulators);
//    one thread issues, per K group, four tcgen05.mma kind::f8f6f4
//    (M = 128, N = 256, K = 32) into one accumulator, then commits to the
//    stage's "empty" barrier (frees the smem) and the accumulator's "full"
//    barrier.
//  * warps 2..9: epilogue. The block scales change every 128-wide K group,
//    so each group's tensor-core result is promoted to a register
//    accumulator: tcgen05.ld the 128 x 256 fp32 block, multiply by
//    sa[m, kb] * sw[n / 128, kb] (one value per row and column half) and add,
//    while the MMA warp fills the other TMEM accumulator. Warp w reads TMEM
//    lanes 32 (w % 4) .. 32 (w % 4) + 31; warps 2..5 take columns 0..127 and
//    warps 6..9 columns 128..255, so each thread owns one output row segment
//    of 128 columns. After the last K group the registers are rounded to
//    bf16 (or kept fp32) and stored.
// Every wait is bounded; a timeout sets the error word read by
// fp8act_check_status() and the kernel runs to completion on whatever data
// it has (never a hang).
#include <atomic>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"
#include "sm100_ptx.cuh"
#include "tc_ptx.cuh"

namespace fp8act {

__device__ unsigned int g_tc_error = 0;

namespace {

constexpr int BM = 128;  // tokens per tile (TMEM lanes)
constexpr int BN = 256;  // weight rows per tile (TMEM columns per accumulator)
constexpr int kStages = 4;
constexpr int kABytes = BM * kGroup;  // 16 KB
constexpr int kBBytes = BN * kGroup;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr uint32_t kTmemCols = 2 * BN;
constexpr int kSmem = 1024 + kStages * kStageBytes + 256;

struct TcArgs {
    const float* sa;
    const float* sw;
    void* out;
    int M, N, K, KB, NB;
};

__device__ __forceinline__ void flag_error(bool& failed, unsigned int code) {
    if (!failed) {
        failed = true;
        atomicOr(&g_tc_error, code);
    }
}

template <bool kF32Out>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                              const __grid_constant__ CUtensorMap tmap_b,
                                                              const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - ptx::smem_u32(smem_raw));
    const uint32_t bar0 = base + kStages * kStageBytes;
    const uint32_t full0 = bar0;                      // [kStages] TMA landed
    const uint32_t empty0 = full0 + 8 * kStages;      // [kStages] MMAs done reading
    const uint32_t tfull0 = empty0 + 8 * kStages;     // [2] accumulator ready
    const uint32_t tempty0 = tfull0 + 16;             // [2] accumulator drained
    const uint32_t tmem_slot = tempty0 + 16;
    volatile uint32_t* const tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM;
    const int n0 = blockIdx.y * BN;
    const int KB = a.KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull0 + 8 * b, 1);
            ptx::mbar_init(tempty0 + 8 * b, kEpiWarps);
        }
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot_ptr;

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            ptx::griddep_launch_dependents();
            ptx::prefetch_tensormap(&tmap_a);
            ptx::prefetch_tensormap(&tmap_b);
            const uint64_t policy = ptx::policy_evict_last();  // both operands are re-read by other tiles
            bool failed = false;
            const int pre = KB < kStages ? KB : kStages;
            for (int i = 0; i < pre; ++i) {  // weights: independent of the previous grid
                ptx::mbar_arrive_expect_tx(full0 + 8 * i, kStageBytes);
                ptx::tma_load_2d(base + i * kStageBytes + kABytes, &tmap_b, full0 + 8 * i, i * kGroup, n0, policy);
            }
            ptx::griddep_wait();  // activations are the previous grid's output
            for (int i = 0; i < pre; ++i)
                ptx::tma_load_2d(base + i * kStageBytes, &tmap_a, full0 + 8 * i, i * kGroup, m0, policy);
            for (int i = pre; i < KB; ++i) {
                const int s = i % kStages;
                if (!failed && !ptx::mbar_wait(empty0 + 8 * s, ((i / kStages) - 1) & 1)) flag_error(failed, 1u);
                ptx::mbar_arrive_expect_tx(full0 + 8 * s, kStageBytes);
                ptx::tma_load_2d(base + s * kStageBytes + kABytes, &tmap_b, full0 + 8 * s, i * kGroup, n0, policy);
                ptx::tma_load_2d(base + s * kStageBytes, &tmap_a, full0 + 8 * s, i * kGroup, m0, policy);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_e4m3_f32(BM, BN);
            bool failed = false;
            for (int i = 0; i < KB; ++i) {
                const int s = i % kStages;
                const int b = i & 1;
                if (!failed && !ptx::mbar_wait(full0 + 8 * s, (i / kStages) & 1)) flag_error(failed, 2u);
                if (i >= 2 && !failed && !ptx::mbar_wait(tempty0 + 8 * b, ((i >> 1) - 1) & 1)) flag_error(failed, 4u);
                tc::fence_after_sync();
                const uint32_t a_tile = base + s * kStageBytes;
                const uint32_t b_tile = a_tile + kABytes;
#pragma unroll
                for (int k = 0; k < kGroup / 32; ++k)
                    tc::mma_f8f6f4(tmem_base + b * BN, tc::desc_kmajor_sw128(a_tile + 32 * k),
                                   tc::desc_kmajor_sw128(b_tile + 32 * k), idesc, k > 0 ? 1u : 0u);
                tc::commit(empty0 + 8 * s);   // the stage's smem may be refilled once these MMAs finish
                tc::commit(tfull0 + 8 * b);   // the accumulator holds this K group's product
            }
        }
    } else {
        // ------------------------------------------------------- epilogue
        ptx::griddep_wait();  // scales come from the previous grid; it may still read `out`
        const int qd = warp & 3;               // TMEM lane quadrant this warp may access
        const int hf = (warp - 2) >> 2;        // column half: 0 for warps 2..5, 1 for warps 6..9
        const int row = qd * 32 + lane;
        const int m = m0 + row;
        const int nb = n0 / kGroup + hf;
        const bool row_ok = m < a.M && nb < a.NB;
        const float* sa_row = a.sa + static_cast<int64_t>(row_ok ? m : 0) * KB;
        const float* sw_row = a.sw + static_cast<int64_t>(row_ok ? nb : 0) * KB;
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(qd * 32) << 16) + hf * 128;
        float acc[128];
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = 0.f;
        bool failed = false;
        for (int i = 0; i < KB; ++i) {
            const int b = i & 1;
            const float scale = row_ok ? __ldg(sa_row + i) * __ldg(sw_row + i) : 0.f;
            if (!failed && !ptx::mbar_wait(tfull0 + 8 * b, (i >> 1) & 1)) flag_error(failed, 8u);
            tc::fence_after_sync();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tc::ld_32x32b_x32(t_row + b * BN + c * 32, r);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[c * 32 + j] = fmaf(__uint_as_float(r[j]), scale, acc[c * 32 + j]);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty0 + 8 * b);
        }
        // store this thread's 128-column row segment
        if (m < a.M) {
            const int nstart = n0 + hf * 128;
            if constexpr (kF32Out) {
                float* dst = static_cast<float*>(a.out) + static_cast<int64_t>(m) * a.N + nstart;
                if ((a.N & 3) == 0 && nstart + 128 <= a.N) {
#pragma unroll
                    for (int j = 0; j < 128; j += 4)
                        *reinterpret_cast<float4*>(dst + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 128; ++j)
                        if (nstart + j < a.N) dst[j] = acc[j];
                }
            } else {
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + static_cast<int64_t>(m) * a.N + nstart;
                if ((a.N & 7) == 0 && nstart + 128 <= a.N) {
#pragma unroll
                    for (int j = 0; j < 128; j += 8) {
                        uint4 v;
                        v.x = pack_bf16x2(acc[j], acc[j + 1]);
                        v.y = pack_bf16x2(acc[j + 2], acc[j + 3]);
                        v.z = pack_bf16x2(acc[j + 4], acc[j + 5]);
                        v.w = pack_bf16x2(acc[j + 6], acc[j + 7]);
                        *reinterpret_cast<uint4*>(dst + j) = v;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 128; ++j)
                        if (nstart + j < a.N) dst[j] = __float2bfloat16_rn(acc[j]);
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem_base, kTmemCols);
}

template <bool kF32Out>
cudaError_t launch_typed(const CUtensorMap& ta, const CUtensorMap& tb, const TcArgs& args, cudaStream_t stream) {
    auto kernel = gemm_tc_kernel<kF32Out>;
    static std::atomic<uint64_t> configured{0};  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((args.M + BM - 1) / BM, (args.N + BN - 1) / BN);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, ta, tb, args);
}

}  // namespace

unsigned int read_and_clear_tc_error() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (v) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(zero));
    }
    return v;
}

cudaError_t launch_gemm_tc(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw, int M, int N, int K,
                           void* out, bool out_f32, cudaStream_t stream) {
    TcArgs a;
    a.sa = sa;
    a.sw = sw;
    a.out = out;
    a.M = M;
    a.N = N;
    a.K = K;
    a.KB = K / kGroup;
    a.NB = (N + kGroup - 1) / kGroup;
    CUtensorMap ta, tb;
    if (!encode_tmap_2d_u8(&ta, q, static_cast<uint64_t>(K), static_cast<uint64_t>(M), static_cast<uint64_t>(K),
                           kGroup, BM, true) ||
        !encode_tmap_2d_u8(&tb, w, static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(K),
                           kGroup, BN, true))
        return cudaErrorInvalidValue;
    return out_f32 ? launch_typed<true>(ta, tb, a, stream) : launch_typed<false>(ta, tb, a, stream);
}

}  // namespace fp8act
