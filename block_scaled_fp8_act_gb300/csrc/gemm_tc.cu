// Tensor-memory (tcgen05) block-FP8 GEMM for batched decode and prefill (M > 16).
//
// At prefill sizes (M = 4096) the layer is a dense contraction: 2MNK =
// 129..730 GFLOP per call against 36..110 MB of operands, far above the FP8
// ridge point, so the kernel is built around the 5th-generation tensor cores.
// The pages saw exactly this shape regress when served by a kernel tuned for
// M = 1 ("双 NVIDIA L20 上 Qwen3.8-27B-FP8 + MTP 调优测试报告", sections 五 and 八):
// batched decode and prefill get their own tile kernel.
//
// A CTA computes 128 x BN output tiles (128 tokens x BN weight rows). Without
// split K the grid is persistent (at most one CTA per SM) and each CTA walks
// tiles blockIdx.x, blockIdx.x + gridDim.x, ... in m-fastest order (a wave
// shares its weight tiles through L2); the stage ring and the two TMEM
// accumulators run on across tile boundaries, so one tile's store overlaps the
// next tile's first MMAs. Per CTA:
//  * warp 0, one thread: TMA producer. A ring of shared-memory stages, each
//    one 128-wide K group: the 128 x 128 activation tile and the BN x 128
//    weight tile, both in the 128-byte swizzled K-major layout. The weight
//    copies of the first stages go out before the kernel waits on the
//    previous grid (programmatic dependent launch).
//  * warp 1: allocates 2 BN TMEM columns (two 128 x BN fp32 accumulators);
//    one thread issues, per K group, four tcgen05.mma kind::f8f6f4
//    (M = 128, N = BN, K = 32) into one accumulator, then commits to the
//    stage's "empty" barrier (frees the smem) and the accumulator's "full"
//    barrier.
//  * warps 2..9: epilogue. The block scales change every 128-wide K group,
//    so each group's tensor-core result is promoted to a register
//    accumulator: tcgen05.ld the group's fp32 block, multiply by
//    sa[m, kb] * sw[n / 128, kb] and add, while the MMA warp fills the other
//    TMEM accumulator. Warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31;
//    warps 2..5 take the first BN / 2 columns and warps 6..9 the rest, so
//    each thread owns one output row segment of BN / 2 columns.
//
// Split K: when the output tiles alone cannot fill the SMs (batched decode on
// N = 5120 projections has 40 tiles of 128 rows), a cluster of S CTAs shares
// a tile, each taking a contiguous slice of the K groups. At the end every CTA
// parks its fp32 partial tile in its own (now idle) stage memory, the cluster
// synchronises once, and CTA r adds its share of the tile's real token rows
// of all S partials through distributed shared memory, in rank order
// (deterministic), and stores them. No global scratch, no atomics.
//
// Grouped calls (gemm_tc_grouped_kernel, further down): the tiles of up to 8
// problems in one persistent launch, dealt evenly over the CTAs, K never
// split.
//
// Failure handling: every wait is bounded (the bound is a launch argument).
// The first wait that gives up sets the device error word read by
// fp8act_check_status() and a CTA-wide abort flag; every role then stops
// issuing work, the producer waits (bounded) for the copies it already
// issued, the MMA thread for the MMAs it already issued, and only then is
// TMEM freed and the CTA leaves (never a hang, no copy or MMA in flight at exit).
#include <algorithm>
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
constexpr int kABytes = BM * kGroup;  // 16 KB
constexpr int kEpiWarps = 8;

template <int BN>
struct TcCfg {
    // Warp roles: warp 0 TMA producer, warp 1 MMA issuer, then the eight
    // epilogue warps. The 256-wide tile runs 12 warps (three warpgroups) so
    // that warpgroup 0 (producer, MMA, two idle warps) can hand registers to
    // the two epilogue warpgroups with setmaxnreg: 128 x 24 + 256 x 240 =
    // 64512 = 384 x 168, exactly the launch's registers. The producer and MMA
    // loops fit in 24 registers; the epilogue's 128 accumulators, 64 staged
    // TMEM values and packed FMAs need the 240 (no spills).
    static constexpr int kCtrlWarps = BN == 256 ? 4 : 2;
    static constexpr int kThreads = (kCtrlWarps + kEpiWarps) * 32;
    static constexpr int kRegsLaunch = 168;  // per thread at launch (ptxas, __launch_bounds__)
    static constexpr int kRegsCtrl = 24;
    static constexpr int kRegsEpi = 240;
    static_assert(BN != 256 || 128 * kRegsCtrl + 256 * kRegsEpi <= kThreads * kRegsLaunch,
                  "register split exceeds the launch's registers");
    static constexpr int kBBytes = BN * kGroup;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = BN == 256 ? 4 : 6;    // ~192 KB of stages either way
    static constexpr uint32_t kTmemCols = 2 * BN;          // two accumulators
    static constexpr int kCols = BN / 2;                   // output columns per epilogue thread
    static constexpr int kRedStride = BN + 4;  // row stride (floats) of the parked partial tile: 16-byte
                                               // aligned rows, rows 4 banks apart (conflict-free v4)
    static constexpr int kSmem = 1024 + kStages * kStageBytes + 256;  // + barriers, TMEM slot, abort flag
    static_assert(16 * kStages + 32 + 8 + 8 + 4 <= 256, "barrier area");
    static_assert(BM * kRedStride * 4 <= kStages * kStageBytes, "partial tile must fit in the stages");
};

struct TcArgs {
    const float* sa;
    const float* sw;
    void* out;
    int M, N, K, KB, NB;
    int ldo;  // output row stride (elements): N, or the full width when `out` is a column slice
    unsigned long long wait_ns;  // bound of every wait that can give up (test hook shortens it)
    int withhold;                // test hook: the producer never issues the CTA's first K group
};

__device__ __forceinline__ void fail(volatile int* abort, unsigned int code) {
    *abort = 1;
    atomicOr(&g_tc_error, code);
}

// d0 += a0 * s and d1 += a1 * s as one packed two-lane fp32 FMA: two
// independent IEEE round-to-nearest FMAs, the same bits as two fmaf calls in
// half the instructions.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float s) {
    const float2 r = __ffma2_rn(make_float2(a0, a1), make_float2(s, s), make_float2(d0, d1));
    d0 = r.x;
    d1 = r.y;
}

template <bool kF32Out>
__device__ __forceinline__ void store_one(void* out, int64_t idx, float v) {
    if constexpr (kF32Out)
        static_cast<float*>(out)[idx] = v;
    else
        static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
}

// One CTA per SM. Ten warps share the SM's four register-file partitions
// (three warps on two of them), which caps a thread at 168 registers.
template <int BN, bool kF32Out>
__global__ void __launch_bounds__(TcCfg<BN>::kThreads, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                              const __grid_constant__ CUtensorMap tmap_b,
                                                              const TcArgs a) {
    using C = TcCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - ptx::smem_u32(smem_raw));
    const uint32_t bar0 = base + C::kStages * C::kStageBytes;
    const uint32_t full0 = bar0;                       // [kStages] TMA landed
    const uint32_t empty0 = full0 + 8 * C::kStages;    // [kStages] MMAs done reading
    const uint32_t tfull0 = empty0 + 8 * C::kStages;   // [2] accumulator ready
    const uint32_t tempty0 = tfull0 + 16;              // [2] accumulator drained
    const uint32_t drain = tempty0 + 16;               // MMA thread: every issued MMA has completed
    const uint32_t tmem_slot = drain + 8;
    volatile uint32_t* const tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
    volatile int* const abort = reinterpret_cast<volatile int*>(base_ptr + (tmem_slot - base) + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int mtiles = (a.M + BM - 1) / BM;
    const int tiles = mtiles * ((a.N + BN - 1) / BN);
    const int splits = gridDim.z;
    const int split = blockIdx.z;  // == cluster rank when splits > 1 (cluster dims 1 x 1 x splits)
    const int kb_begin = static_cast<int>(static_cast<int64_t>(split) * a.KB / splits);
    const int kb_end = static_cast<int>(static_cast<int64_t>(split + 1) * a.KB / splits);
    const int nk = kb_end - kb_begin;
    // tiles of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ... (one when splitting K)
    const int my_tiles = blockIdx.x < tiles ? (tiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
    const int total = my_tiles * nk;  // K groups this CTA streams

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull0 + 8 * b, 1);
            ptx::mbar_init(tempty0 + 8 * b, kEpiWarps);
        }
        ptx::mbar_init(drain, 1);
        *abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, C::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot_ptr;

    // epilogue geometry (warps kCtrlWarps .. kCtrlWarps + 7)
    const bool epi = warp >= C::kCtrlWarps;
    const int qd = warp & 3;                          // TMEM lane quadrant this warp may access
    const int hf = (warp - C::kCtrlWarps) >> 2;       // column half
    const int row = qd * 32 + lane;
    float acc[C::kCols];
    int m0 = (blockIdx.x % mtiles) * BM;   // tile of a split-K CTA (its only tile)
    int n0 = (blockIdx.x / mtiles) * BN;

    if (!epi) {
    if constexpr (BN == 256) tc::regs_decrease<C::kRegsCtrl>();
    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            ptx::griddep_launch_dependents();
            ptx::prefetch_tensormap(&tmap_a);
            ptx::prefetch_tensormap(&tmap_b);
            const uint64_t policy = ptx::policy_evict_last();  // both operands are re-read by other tiles
            const bool skip0 = a.withhold != 0;
            // stage use i -> tile blockIdx.x + (i / nk) * gridDim.x, K group kb_begin + i % nk
            auto tile_mn = [&](int i, int& m0_, int& n0_) {
                const int tile = blockIdx.x + (i / nk) * gridDim.x;
                m0_ = (tile % mtiles) * BM;
                n0_ = (tile / mtiles) * BN;
            };
            const int pre = total < C::kStages ? total : C::kStages;
            for (int i = skip0 ? 1 : 0; i < pre; ++i) {  // weights: independent of the previous grid
                int m0_, n0_;
                tile_mn(i, m0_, n0_);
                ptx::mbar_arrive_expect_tx(full0 + 8 * i, C::kStageBytes);
                ptx::tma_load_2d(base + i * C::kStageBytes + kABytes, &tmap_b, full0 + 8 * i,
                                 (kb_begin + i % nk) * kGroup, n0_, policy);
            }
            ptx::griddep_wait();  // activations are the previous grid's output
            for (int i = skip0 ? 1 : 0; i < pre; ++i) {
                int m0_, n0_;
                tile_mn(i, m0_, n0_);
                ptx::tma_load_2d(base + i * C::kStageBytes, &tmap_a, full0 + 8 * i, (kb_begin + i % nk) * kGroup, m0_,
                                 policy);
            }
            int issued = pre;
            for (int i = pre; i < total; ++i) {
                const int s = i % C::kStages;
                int m0_, n0_;
                tile_mn(i, m0_, n0_);
                if (!ptx::mbar_wait_or_abort(empty0 + 8 * s, ((i / C::kStages) - 1) & 1, a.wait_ns, abort)) {
                    fail(abort, 1u);
                    break;
                }
                ptx::mbar_arrive_expect_tx(full0 + 8 * s, C::kStageBytes);
                ptx::tma_load_2d(base + s * C::kStageBytes + kABytes, &tmap_b, full0 + 8 * s,
                                 (kb_begin + i % nk) * kGroup, n0_, policy);
                ptx::tma_load_2d(base + s * C::kStageBytes, &tmap_a, full0 + 8 * s, (kb_begin + i % nk) * kGroup, m0_,
                                 policy);
                issued = i + 1;
            }
            // Every copy issued must land before the CTA may leave: wait for
            // the last use of each stage (the MMA thread has usually seen it).
            for (int i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i)
                if (!(skip0 && i == 0) && !ptx::mbar_wait(full0 + 8 * (i % C::kStages), (i / C::kStages) & 1))
                    fail(abort, 16u);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_e4m3_f32(BM, BN);
            for (int i = 0; i < total; ++i) {
                const int s = i % C::kStages;
                const int b = i & 1;
                if (!ptx::mbar_wait_or_abort(full0 + 8 * s, (i / C::kStages) & 1, a.wait_ns, abort)) {
                    fail(abort, 2u);
                    break;
                }
                if (i >= 2 && !ptx::mbar_wait_or_abort(tempty0 + 8 * b, ((i >> 1) - 1) & 1, a.wait_ns, abort)) {
                    fail(abort, 4u);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t a_tile = base + s * C::kStageBytes;
                const uint32_t b_tile = a_tile + kABytes;
#pragma unroll
                for (int k = 0; k < kGroup / 32; ++k)
                    tc::mma_f8f6f4(tmem_base + b * BN, tc::desc_kmajor_sw128(a_tile + 32 * k),
                                   tc::desc_kmajor_sw128(b_tile + 32 * k), idesc, k > 0 ? 1u : 0u);
                tc::commit(empty0 + 8 * s);   // the stage's smem may be refilled once these MMAs finish
                tc::commit(tfull0 + 8 * b);   // the accumulator holds this K group's product
            }
            // No MMA may still run when TMEM is freed or the CTA leaves.
            tc::commit(drain);
            if (!ptx::mbar_wait(drain, 0)) fail(abort, 32u);
        }
    }
    } else {
        // ------------------------------------------------------- epilogue
        if constexpr (BN == 256) tc::regs_increase<C::kRegsEpi>();
        ptx::griddep_wait();  // scales come from the previous grid; it may still read `out`
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(qd * 32) << 16) + hf * C::kCols;
        bool failed = false;
        int i = 0;  // accumulator uses so far
        for (int t = 0; t < my_tiles && !failed; ++t) {
            const int tile = blockIdx.x + t * gridDim.x;
            m0 = (tile % mtiles) * BM;
            n0 = (tile / mtiles) * BN;
            const int m = m0 + row;
            const int nb = (n0 + hf * C::kCols) / kGroup;
            const bool row_ok = m < a.M && nb < a.NB;
            const float* sa_row = a.sa + static_cast<int64_t>(row_ok ? m : 0) * a.KB;
            const float* sw_row = a.sw + static_cast<int64_t>(row_ok ? nb : 0) * a.KB;
#pragma unroll
            for (int j = 0; j < C::kCols; ++j) acc[j] = 0.f;
            for (int k = 0; k < nk; ++k, ++i) {
                const int b = i & 1;
                const int kb = kb_begin + k;
                const float scale = row_ok ? ld_dep_f32(sa_row + kb) * __ldg(sw_row + kb) : 0.f;
                // the whole warp decides together (tcgen05.ld is warp-collective)
                if (!__all_sync(0xffffffffu, ptx::mbar_wait_or_abort(tfull0 + 8 * b, (i >> 1) & 1, a.wait_ns, abort))) {
                    if (lane == 0) fail(abort, 8u);
                    failed = true;
                    break;
                }
                tc::fence_after_sync();
                if constexpr (C::kCols == 64) {
                    // both 32-column halves in flight, one wait; packed FMAs (7% off the
                    // batched-decode GEMM)
                    uint32_t r0[32], r1[32];
                    tc::ld_32x32b_x32(t_row + b * BN, r0);
                    tc::ld_32x32b_x32(t_row + b * BN + 32, r1);
                    tc::wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        fma2(acc[j], acc[j + 1], __uint_as_float(r0[j]), __uint_as_float(r0[j + 1]), scale);
                        fma2(acc[32 + j], acc[33 + j], __uint_as_float(r1[j]), __uint_as_float(r1[j + 1]), scale);
                    }
                } else {
                    // two rounds of 64 columns, both 32-column loads of a round in flight;
                    // packed FMAs (13% off the prefill GEMM; they need the 240-register
                    // epilogue, at 224 ptxas spilled and they lost 7.5%)
                    const float2 s2 = make_float2(scale, scale);
#pragma unroll
                    for (int c = 0; c < C::kCols / 64; ++c) {
                        uint32_t r0[32], r1[32];
                        tc::ld_32x32b_x32(t_row + b * BN + c * 64, r0);
                        tc::ld_32x32b_x32(t_row + b * BN + c * 64 + 32, r1);
                        tc::wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            float2 x = __ffma2_rn(make_float2(__uint_as_float(r0[j]), __uint_as_float(r0[j + 1])), s2,
                                                  make_float2(acc[c * 64 + j], acc[c * 64 + j + 1]));
                            acc[c * 64 + j] = x.x;
                            acc[c * 64 + j + 1] = x.y;
                        }
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            float2 x = __ffma2_rn(make_float2(__uint_as_float(r1[j]), __uint_as_float(r1[j + 1])), s2,
                                                  make_float2(acc[c * 64 + 32 + j], acc[c * 64 + 33 + j]));
                            acc[c * 64 + 32 + j] = x.x;
                            acc[c * 64 + 33 + j] = x.y;
                        }
                    }
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(tempty0 + 8 * b);
            }
            if (splits == 1 && m < a.M && !failed) {
                // store this thread's row segment directly
                const int nstart = n0 + hf * C::kCols;
                if constexpr (kF32Out) {
                    float* dst = static_cast<float*>(a.out) + static_cast<int64_t>(m) * a.ldo + nstart;
                    if ((a.ldo & 3) == 0 && nstart + C::kCols <= a.N) {
#pragma unroll
                        for (int j = 0; j < C::kCols; j += 4)
                            *reinterpret_cast<float4*>(dst + j) =
                                make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < C::kCols; ++j)
                            if (nstart + j < a.N) dst[j] = acc[j];
                    }
                } else {
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + static_cast<int64_t>(m) * a.ldo + nstart;
                    if ((a.ldo & 7) == 0 && nstart + C::kCols <= a.N) {
#pragma unroll
                        for (int j = 0; j < C::kCols; j += 8) {
                            uint4 v;
                            v.x = pack_bf16x2(acc[j], acc[j + 1]);
                            v.y = pack_bf16x2(acc[j + 2], acc[j + 3]);
                            v.z = pack_bf16x2(acc[j + 4], acc[j + 5]);
                            v.w = pack_bf16x2(acc[j + 6], acc[j + 7]);
                            *reinterpret_cast<uint4*>(dst + j) = v;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < C::kCols; ++j)
                            if (nstart + j < a.N) dst[j] = __float2bfloat16_rn(acc[j]);
                    }
                }
            }
        }
    }

    if constexpr (BN == 128) {  // split K is only chosen with 128-wide tiles
    if (splits > 1) {
        // Park the partial tile in the idle stage memory once every role has
        // left its loop (every issued copy has landed, every issued MMA has
        // completed), then reduce a slice of rows across the cluster.
        __syncthreads();
        float* red = reinterpret_cast<float*>(base_ptr);
        const bool ok = *abort == 0;
        const int vrows = a.M - m0 < BM ? a.M - m0 : BM;  // token rows of the tile that exist
        if (epi && row < vrows) {
#pragma unroll
            for (int j = 0; j < C::kCols; j += 4)
                *reinterpret_cast<float4*>(red + row * C::kRedStride + hf * C::kCols + j) =
                    make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
        }
        __syncwarp();  // barrier.cluster.*.aligned: the whole warp arrives together
        ptx::cluster_sync();
        {
            // CTA r sums rows [vrows r / S, vrows (r + 1) / S) of every peer's partial (the
            // tile's real token rows only), 4 consecutive columns per element, in rank order.
            // Distributed shared memory moves ~15 B per clock per SM whatever the access
            // style (loads, bulk copies or st.async, measured with every SM busy), so the
            // bytes that cross it set the time: vrows x BN x 4 per CTA. Every thread of the
            // CTA takes part, two elements at a time with every peer's load in flight.
            constexpr int kMaxSplits = 8;
            constexpr int kBatch = 2;
            const int r_begin = split * vrows / splits;
            const int r_end = (split + 1) * vrows / splits;
            const int elems = (r_end - r_begin) * (BN / 4);
#pragma unroll 1
            for (int e0 = threadIdx.x; e0 < elems; e0 += kBatch * C::kThreads) {
                float4 part[kBatch][kMaxSplits];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int e = e0 + u * C::kThreads < elems ? e0 + u * C::kThreads : e0;
                    const int r = r_begin + e / (BN / 4);
                    const int col = 4 * (e % (BN / 4));
                    const uint32_t local = ptx::smem_u32(red + r * C::kRedStride + col);
#pragma unroll
                    for (int c = 0; c < kMaxSplits; ++c)
                        if (c < splits) part[u][c] = ptx::ld_shared_cluster_v4(ptx::mapa_shared(local, c));
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int e = e0 + u * C::kThreads;
                    if (e >= elems) continue;
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < kMaxSplits; ++c)
                        if (c < splits) {
                            v.x += part[u][c].x;
                            v.y += part[u][c].y;
                            v.z += part[u][c].z;
                            v.w += part[u][c].w;
                        }
                    const int r = r_begin + e / (BN / 4);
                    const int col = 4 * (e % (BN / 4));
                    const int m = m0 + r, n = n0 + col;
                    if (!ok) continue;
                    const int64_t o = static_cast<int64_t>(m) * a.ldo + n;
                    if (n + 3 < a.N && (a.ldo & 3) == 0) {
                        if constexpr (kF32Out) {
                            *reinterpret_cast<float4*>(static_cast<float*>(a.out) + o) = v;
                        } else {
                            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + o) =
                                make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
                        }
                    } else {
                        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (n + i < a.N) store_one<kF32Out>(a.out, o + i, vv[i]);
                    }
                }
            }
        }
        __syncwarp();
        ptx::cluster_sync();  // no CTA leaves while its peers still read its shared memory
    }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem_base, C::kTmemCols);
}

template <int BN, bool kF32Out>
cudaError_t launch_typed(const CUtensorMap& ta, const CUtensorMap& tb, const TcArgs& args, int num_sms,
                         cudaStream_t stream) {
    using C = TcCfg<BN>;
    auto kernel = gemm_tc_kernel<BN, kF32Out>;
    static std::atomic<uint64_t> configured{0};   // one bit per device
    static std::atomic<int> max_clusters[64][9];  // per device and cluster size: 1 + clusters resident
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        if constexpr (BN == 256) {
            // setmaxnreg.inc waits for registers the block does not have if the
            // compiler allocated fewer than the split assumes: refuse to launch.
            cudaFuncAttributes fa{};
            e = cudaFuncGetAttributes(&fa, kernel);
            if (e != cudaSuccess) return e;
            if (fa.numRegs < C::kRegsLaunch) return cudaErrorInvalidConfiguration;
        }
        configured.fetch_or(bit, std::memory_order_release);
    }
    const int mt = (args.M + BM - 1) / BM;
    const int nt = (args.N + BN - 1) / BN;
    const int tiles = mt * nt;

    // Split K over a cluster when the tiles leave SMs idle (128-wide tiles
    // only): the largest S in 8..2 with at least 2 K groups per CTA, tiles * S
    // CTAs within the SM count, and every cluster resident at once.
    int splits = 1;
    for (int s = 8; s >= 2 && BN == 128; --s) {
        if (tiles * s > num_sms || args.KB < 2 * s) continue;
        int cached = max_clusters[dev & 63][s].load(std::memory_order_relaxed);
        if (cached == 0) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(1, 1, s);
            q.blockDim = dim3(C::kThreads);
            q.dynamicSmemBytes = C::kSmem;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = 1;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = s;
            q.attrs = qa;
            q.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kernel, &q) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
            cached = n + 1;
            max_clusters[dev & 63][s].store(cached, std::memory_order_relaxed);
        }
        if (tiles <= cached - 1) {
            splits = s;
            break;
        }
    }

    cudaLaunchConfig_t cfg = {};
    // split K: one CTA per (tile, split); otherwise persistent, one CTA per SM at most
    cfg.gridDim = dim3(splits > 1 ? tiles : (tiles < num_sms ? tiles : num_sms), 1, splits);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = splits;
    cfg.attrs = attr;
    cfg.numAttrs = splits > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, ta, tb, args);
}

// ------------------------------------------------------------------------
// Grouped calls: several problems in one persistent launch of the tile
// kernel. BN = 128 when every problem has one token tile (16 < M <= 128,
// batched decode), BN = 256 otherwise (prefill widths, with the 12-warp
// register split of gemm_tc_kernel<256>); a problem's token tiles are walked
// fastest within a weight column group, so a wave shares its weight tiles
// through L2. The problems' tiles form one list, problems in order of falling
// K (a tile costs its K groups). With G CTAs the list runs in whole rounds of
// G tiles, CTA b taking position r G + b in even rounds r and r G + G - 1 - b
// in odd ones (a snake, so the costly first tiles spread over all CTAs); the
// tiles of the last, partial round go, largest first, to the CTAs with the
// fewest K groups so far (the host works that out; the kernel gets each
// CTA's leftover tile). The tiles of several projections fill the grid
// without splitting K, so there is no cross-CTA reduction (on one N = 5120
// projection alone at batched widths that reduction is a third of the
// launch) and no last partial wave per problem, and the stage ring and the
// two accumulators run on across the tiles of different problems. Each
// problem has its own tensor maps in the kernel parameters. Roles, barriers,
// bounded waits and the drain are those of gemm_tc_kernel.
constexpr int kMaxTcGroup = 8;        // problems per launch (their tensor maps travel in the parameters)
constexpr int kMaxTcGroupCtas = 256;  // grid limit of the grouped launch

struct TcGroupProblem {
    const float* sa;
    const float* sw;
    void* out;
    int M, N, KB;
    int mtiles;      // 128-token tiles (walked fastest within a weight column group)
    int tile_begin;  // list position of this problem's first tile
};

struct TcGroupedArgs {
    CUtensorMap ta[kMaxTcGroup];  // activation codes [M, K], 128 x 128 boxes
    CUtensorMap tb[kMaxTcGroup];  // weight codes [N, K], 128 x BN boxes
    TcGroupProblem p[kMaxTcGroup];
    int count;
    int tiles;                   // list length
    int full_rounds;             // tiles / G
    unsigned long long wait_ns;  // bound of every wait that can give up (test hook shortens it)
    int withhold;                // test hook: the producer never issues the CTA's first K group
    short leftover[kMaxTcGroupCtas];  // CTA b's tile of the partial last round, or -1
};

__host__ __device__ __forceinline__ int grouped_position(int round, int b, int G) {
    return round * G + ((round & 1) ? G - 1 - b : b);
}

// The j-th tile of CTA b, or -1 past its last.
__device__ __forceinline__ int grouped_tile(const TcGroupedArgs& a, int j, int b, int G) {
    if (j < a.full_rounds) return grouped_position(j, b, G);
    return j == a.full_rounds ? a.leftover[b] : -1;
}

__device__ __forceinline__ int grouped_problem(const TcGroupedArgs& a, int t) {
    int p = 0;
    while (p + 1 < a.count && t >= a.p[p + 1].tile_begin) ++p;
    return p;
}

// The producer's walk over this CTA's (tile, K group) units.
struct GroupedCursor {
    int j, t, p, kb;
    __device__ __forceinline__ void start(const TcGroupedArgs& a, int b, int G) {
        j = 0;
        t = grouped_tile(a, 0, b, G);
        p = t >= 0 ? grouped_problem(a, t) : 0;
        kb = 0;
    }
    __device__ __forceinline__ void next(const TcGroupedArgs& a, int b, int G) {
        if (++kb == a.p[p].KB) {
            kb = 0;
            t = grouped_tile(a, ++j, b, G);
            if (t >= 0) p = grouped_problem(a, t);
        }
    }
    __device__ __forceinline__ int m0(const TcGroupedArgs& a) const {
        return (t - a.p[p].tile_begin) % a.p[p].mtiles * BM;
    }
    __device__ __forceinline__ int n0(const TcGroupedArgs& a, int bn) const {
        return (t - a.p[p].tile_begin) / a.p[p].mtiles * bn;
    }
};

template <int BN, bool kF32Out>
__global__ void __launch_bounds__(TcCfg<BN>::kThreads, 1)
    gemm_tc_grouped_kernel(const __grid_constant__ TcGroupedArgs a) {
    using C = TcCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - ptx::smem_u32(smem_raw));
    const uint32_t bar0 = base + C::kStages * C::kStageBytes;
    const uint32_t full0 = bar0;                       // [kStages] TMA landed
    const uint32_t empty0 = full0 + 8 * C::kStages;    // [kStages] MMAs done reading
    const uint32_t tfull0 = empty0 + 8 * C::kStages;   // [2] accumulator ready
    const uint32_t tempty0 = tfull0 + 16;              // [2] accumulator drained
    const uint32_t drain = tempty0 + 16;               // MMA thread: every issued MMA has completed
    const uint32_t tmem_slot = drain + 8;
    volatile uint32_t* const tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
    volatile int* const abort = reinterpret_cast<volatile int*>(base_ptr + (tmem_slot - base) + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x);
    const int b = static_cast<int>(blockIdx.x);
    int total = 0;  // K groups this CTA streams
    for (int j = 0;; ++j) {
        const int t = grouped_tile(a, j, b, G);
        if (t < 0) break;
        total += a.p[grouped_problem(a, t)].KB;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(tfull0 + 8 * i, 1);
            ptx::mbar_init(tempty0 + 8 * i, kEpiWarps);
        }
        ptx::mbar_init(drain, 1);
        *abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, C::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot_ptr;

    const bool epi = warp >= C::kCtrlWarps;
    if (!epi) {
    if constexpr (BN == 256) tc::regs_decrease<C::kRegsCtrl>();
    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            ptx::griddep_launch_dependents();
            for (int p = 0; p < a.count; ++p) {
                ptx::prefetch_tensormap(&a.ta[p]);
                ptx::prefetch_tensormap(&a.tb[p]);
            }
            // one token tile: every weight tile is read once; several: the token tiles of a
            // weight column group run together and share it through L2
            const uint64_t pol_w = BN == 128 ? ptx::policy_evict_first() : ptx::policy_evict_last();
            const uint64_t pol_q = ptx::policy_evict_last();  // a problem's codes are re-read by its tiles
            const bool skip0 = a.withhold != 0;
            const int pre = total < C::kStages ? total : C::kStages;
            GroupedCursor cw;  // weights: independent of the previous grid
            cw.start(a, b, G);
            for (int i = 0; i < pre; ++i, cw.next(a, b, G)) {
                if (skip0 && i == 0) continue;
                ptx::mbar_arrive_expect_tx(full0 + 8 * i, C::kStageBytes);
                ptx::tma_load_2d(base + i * C::kStageBytes + kABytes, &a.tb[cw.p], full0 + 8 * i, cw.kb * kGroup,
                                 cw.n0(a, BN), pol_w);
            }
            ptx::griddep_wait();  // the activation codes are the previous grid's output
            GroupedCursor ca;
            ca.start(a, b, G);
            for (int i = 0; i < pre; ++i, ca.next(a, b, G)) {
                if (skip0 && i == 0) continue;
                ptx::tma_load_2d(base + i * C::kStageBytes, &a.ta[ca.p], full0 + 8 * i, ca.kb * kGroup, ca.m0(a),
                                 pol_q);
            }
            int issued = pre;
            for (int i = pre; i < total; ++i, cw.next(a, b, G)) {
                const int s = i % C::kStages;
                if (!ptx::mbar_wait_or_abort(empty0 + 8 * s, ((i / C::kStages) - 1) & 1, a.wait_ns, abort)) {
                    fail(abort, 1u);
                    break;
                }
                ptx::mbar_arrive_expect_tx(full0 + 8 * s, C::kStageBytes);
                ptx::tma_load_2d(base + s * C::kStageBytes + kABytes, &a.tb[cw.p], full0 + 8 * s, cw.kb * kGroup,
                                 cw.n0(a, BN), pol_w);
                ptx::tma_load_2d(base + s * C::kStageBytes, &a.ta[cw.p], full0 + 8 * s, cw.kb * kGroup, cw.m0(a),
                                 pol_q);
                issued = i + 1;
            }
            // Every copy issued must land before the CTA may leave.
            for (int i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i)
                if (!(skip0 && i == 0) && !ptx::mbar_wait(full0 + 8 * (i % C::kStages), (i / C::kStages) & 1))
                    fail(abort, 16u);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_e4m3_f32(BM, BN);
            for (int i = 0; i < total; ++i) {
                const int s = i % C::kStages;
                const int acc_b = i & 1;
                if (!ptx::mbar_wait_or_abort(full0 + 8 * s, (i / C::kStages) & 1, a.wait_ns, abort)) {
                    fail(abort, 2u);
                    break;
                }
                if (i >= 2 && !ptx::mbar_wait_or_abort(tempty0 + 8 * acc_b, ((i >> 1) - 1) & 1, a.wait_ns, abort)) {
                    fail(abort, 4u);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t a_tile = base + s * C::kStageBytes;
                const uint32_t b_tile = a_tile + kABytes;
#pragma unroll
                for (int k = 0; k < kGroup / 32; ++k)
                    tc::mma_f8f6f4(tmem_base + acc_b * BN, tc::desc_kmajor_sw128(a_tile + 32 * k),
                                   tc::desc_kmajor_sw128(b_tile + 32 * k), idesc, k > 0 ? 1u : 0u);
                tc::commit(empty0 + 8 * s);       // the stage's smem may be refilled once these MMAs finish
                tc::commit(tfull0 + 8 * acc_b);   // the accumulator holds this K group's product
            }
            // No MMA may still run when TMEM is freed or the CTA leaves.
            tc::commit(drain);
            if (!ptx::mbar_wait(drain, 0)) fail(abort, 32u);
        }
    }
    } else {
        // ------------------------------------------------------- epilogue
        if constexpr (BN == 256) tc::regs_increase<C::kRegsEpi>();
        ptx::griddep_wait();  // scales come from the previous grid; it may still read `out`
        const int qd = warp & 3;                     // TMEM lane quadrant this warp may access
        const int hf = (warp - C::kCtrlWarps) >> 2;  // column half
        const int row = qd * 32 + lane;              // token within the tile
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(qd * 32) << 16) + hf * C::kCols;
        float acc[C::kCols];
        bool failed = false;
        int i = 0;  // accumulator uses so far
        for (int j = 0; !failed; ++j) {
            const int t = grouped_tile(a, j, b, G);
            if (t < 0) break;
            const TcGroupProblem& pr = a.p[grouped_problem(a, t)];
            const int local = t - pr.tile_begin;
            const int m = local % pr.mtiles * BM + row;
            const int n0 = local / pr.mtiles * BN;
            const int nb = (n0 + hf * C::kCols) / kGroup;
            const bool row_ok = m < pr.M && n0 + hf * C::kCols < pr.N;
            const float* sa_row = pr.sa + static_cast<int64_t>(row_ok ? m : 0) * pr.KB;
            const float* sw_row = pr.sw + static_cast<int64_t>(row_ok ? nb : 0) * pr.KB;
#pragma unroll
            for (int jj = 0; jj < C::kCols; ++jj) acc[jj] = 0.f;
            for (int k = 0; k < pr.KB; ++k, ++i) {
                const int acc_b = i & 1;
                const float scale = row_ok ? ld_dep_f32(sa_row + k) * __ldg(sw_row + k) : 0.f;
                // the whole warp decides together (tcgen05.ld is warp-collective)
                if (!__all_sync(0xffffffffu,
                                ptx::mbar_wait_or_abort(tfull0 + 8 * acc_b, (i >> 1) & 1, a.wait_ns, abort))) {
                    if (lane == 0) fail(abort, 8u);
                    failed = true;
                    break;
                }
                tc::fence_after_sync();
                // rounds of 64 columns, both 32-column loads of a round in flight; packed FMAs
#pragma unroll
                for (int c = 0; c < C::kCols / 64; ++c) {
                    uint32_t r0[32], r1[32];
                    tc::ld_32x32b_x32(t_row + acc_b * BN + c * 64, r0);
                    tc::ld_32x32b_x32(t_row + acc_b * BN + c * 64 + 32, r1);
                    tc::wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 2) {
                        fma2(acc[c * 64 + jj], acc[c * 64 + jj + 1], __uint_as_float(r0[jj]),
                             __uint_as_float(r0[jj + 1]), scale);
                        fma2(acc[c * 64 + 32 + jj], acc[c * 64 + 33 + jj], __uint_as_float(r1[jj]),
                             __uint_as_float(r1[jj + 1]), scale);
                    }
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(tempty0 + 8 * acc_b);
            }
            if (m < pr.M && !failed) {
                const int nstart = n0 + hf * C::kCols;
                if constexpr (kF32Out) {
                    float* dst = static_cast<float*>(pr.out) + static_cast<int64_t>(m) * pr.N + nstart;
                    if ((pr.N & 3) == 0 && nstart + C::kCols <= pr.N) {
#pragma unroll
                        for (int jj = 0; jj < C::kCols; jj += 4)
                            *reinterpret_cast<float4*>(dst + jj) =
                                make_float4(acc[jj], acc[jj + 1], acc[jj + 2], acc[jj + 3]);
                    } else {
#pragma unroll
                        for (int jj = 0; jj < C::kCols; ++jj)
                            if (nstart + jj < pr.N) dst[jj] = acc[jj];
                    }
                } else {
                    __nv_bfloat16* dst =
                        static_cast<__nv_bfloat16*>(pr.out) + static_cast<int64_t>(m) * pr.N + nstart;
                    if ((pr.N & 7) == 0 && nstart + C::kCols <= pr.N) {
#pragma unroll
                        for (int jj = 0; jj < C::kCols; jj += 8) {
                            uint4 v;
                            v.x = pack_bf16x2(acc[jj], acc[jj + 1]);
                            v.y = pack_bf16x2(acc[jj + 2], acc[jj + 3]);
                            v.z = pack_bf16x2(acc[jj + 4], acc[jj + 5]);
                            v.w = pack_bf16x2(acc[jj + 6], acc[jj + 7]);
                            *reinterpret_cast<uint4*>(dst + jj) = v;
                        }
                    } else {
#pragma unroll
                        for (int jj = 0; jj < C::kCols; ++jj)
                            if (nstart + jj < pr.N) dst[jj] = __float2bfloat16_rn(acc[jj]);
                    }
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem_base, C::kTmemCols);
}

template <int BN, bool kF32Out>
cudaError_t launch_grouped_typed(const TcGroupedArgs& args, int grid, cudaStream_t stream) {
    using C = TcCfg<BN>;
    auto kernel = gemm_tc_grouped_kernel<BN, kF32Out>;
    static std::atomic<uint64_t> configured{0};  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        if constexpr (BN == 256) {
            // setmaxnreg.inc waits for registers the block does not have if the
            // compiler allocated fewer than the split assumes: refuse to launch.
            cudaFuncAttributes fa{};
            e = cudaFuncGetAttributes(&fa, kernel);
            if (e != cudaSuccess) return e;
            if (fa.numRegs < C::kRegsLaunch) return cudaErrorInvalidConfiguration;
        }
        configured.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args);
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
                           void* out, bool out_f32, int num_sms, cudaStream_t stream) {
    TcArgs a;
    a.sa = sa;
    a.sw = sw;
    a.out = out;
    a.M = M;
    a.N = N;
    a.K = K;
    a.KB = K / kGroup;
    a.NB = (N + kGroup - 1) / kGroup;
    a.ldo = N;
    a.wait_ns = tile_wait_limit_ns();
    a.withhold = tile_withhold_first_load() ? 1 : 0;
    // 256-wide weight tiles when the grid is large (prefill: fewer operand
    // re-reads per FLOP); 128-wide ones otherwise (twice the tiles to spread
    // a batched-decode weight stream over the SMs).
    const int mt = (M + BM - 1) / BM;
    const bool wide = static_cast<int64_t>(mt) * ((N + 255) / 256) >= 2 * num_sms;
    CUtensorMap ta;
    if (!encode_tmap_2d_u8(&ta, q, static_cast<uint64_t>(K), static_cast<uint64_t>(M), static_cast<uint64_t>(K),
                           kGroup, BM, true))
        return cudaErrorInvalidValue;
    // One launch over the output columns [n_begin, n_begin + cols) of `out`.
    auto launch_cols = [&](int bn, int n_begin, int cols) -> cudaError_t {
        TcArgs s = a;
        s.N = cols;
        s.NB = (cols + kGroup - 1) / kGroup;
        s.sw = sw + static_cast<int64_t>(n_begin / kGroup) * a.KB;
        s.out = out_f32 ? static_cast<void*>(static_cast<float*>(out) + n_begin)
                        : static_cast<void*>(static_cast<__nv_bfloat16*>(out) + n_begin);
        CUtensorMap tb;
        if (!encode_tmap_2d_u8(&tb, w + static_cast<int64_t>(n_begin) * K, static_cast<uint64_t>(K),
                               static_cast<uint64_t>(cols), static_cast<uint64_t>(K), kGroup, bn, true))
            return cudaErrorInvalidValue;
        if (bn == 256)
            return out_f32 ? launch_typed<256, true>(ta, tb, s, num_sms, stream)
                           : launch_typed<256, false>(ta, tb, s, num_sms, stream);
        return out_f32 ? launch_typed<128, true>(ta, tb, s, num_sms, stream)
                       : launch_typed<128, false>(ta, tb, s, num_sms, stream);
    };
    if (!wide) return launch_cols(128, 0, N);
    // Split tail wave: the persistent 256-wide launch takes the whole column
    // groups that fit in its whole waves; the rest (at most half a wave of
    // 128-wide tiles) runs as a second launch of 128-wide tiles, which splits
    // K over a cluster of CTAs (the tiles leave SMs idle). Both launches write
    // column slices of the same output. On the N = 5120 prefill shapes (640
    // tiles = 4.2 waves) this replaces a fifth wave run by 32 of the 152 CTAs.
    const int tiles = mt * ((N + 255) / 256);
    const int waves = tiles / num_sms;
    const int n_split = (waves * num_sms / mt) * 256;
    const int tail_tiles = mt * ((N - n_split + 127) / 128);
    // only where the tail launch can split K at least two ways (measured: an
    // unsplit 128-wide tail launch did not beat the persistent kernel's own tail)
    if (waves >= 1 && n_split > 0 && n_split < N && 2 * tail_tiles <= num_sms && a.KB >= 4) {
        const cudaError_t e = launch_cols(256, 0, n_split);
        if (e != cudaSuccess) return e;
        return launch_cols(128, n_split, N - n_split);
    }
    return launch_cols(256, 0, N);
}

int gemm_tc_grouped_capacity() { return kMaxTcGroup; }

cudaError_t launch_gemm_tc_grouped(const GemmProblem* probs, int count, bool out_f32, int num_sms,
                                   cudaStream_t stream) {
    if (count <= 0) return cudaSuccess;
    if (count > kMaxTcGroup) return cudaErrorInvalidValue;
    // One token tile everywhere (batched decode): 128-wide weight tiles. Otherwise
    // (prefill widths) 256-wide ones, the token tiles of a column group walked
    // together, as in the single-problem kernel.
    bool one_token_tile = true;
    for (int i = 0; i < count; ++i) one_token_tile = one_token_tile && probs[i].M <= BM;
    const int bn = one_token_tile ? 128 : 256;
    // problems in order of falling K: a tile's cost is its K groups
    int order[kMaxTcGroup];
    for (int i = 0; i < count; ++i) order[i] = i;
    for (int i = 1; i < count; ++i)
        for (int j = i; j > 0 && probs[order[j - 1]].K < probs[order[j]].K; --j) {
            const int tmp = order[j];
            order[j] = order[j - 1];
            order[j - 1] = tmp;
        }
    TcGroupedArgs a = {};
    int64_t tiles = 0;
    for (int i = 0; i < count; ++i) {
        const GemmProblem& src = probs[order[i]];
        if (src.M < 1 || src.N < 1) return cudaErrorInvalidValue;
        if (!encode_tmap_2d_u8(&a.ta[i], src.q, static_cast<uint64_t>(src.K), static_cast<uint64_t>(src.M),
                               static_cast<uint64_t>(src.K), kGroup, BM, true) ||
            !encode_tmap_2d_u8(&a.tb[i], src.w, static_cast<uint64_t>(src.K), static_cast<uint64_t>(src.N),
                               static_cast<uint64_t>(src.K), kGroup, bn, true))
            return cudaErrorInvalidValue;
        TcGroupProblem& d = a.p[i];
        d.sa = src.sa;
        d.sw = src.sw;
        d.out = src.out;
        d.M = src.M;
        d.N = src.N;
        d.KB = src.K / kGroup;
        d.mtiles = (src.M + BM - 1) / BM;
        d.tile_begin = static_cast<int>(tiles);
        tiles += static_cast<int64_t>(d.mtiles) * ((src.N + bn - 1) / bn);
        if (tiles > 32767) return cudaErrorNotSupported;  // leftover tiles are recorded as 16-bit positions
    }
    a.count = count;
    a.tiles = static_cast<int>(tiles);
    a.wait_ns = tile_wait_limit_ns();
    a.withhold = tile_withhold_first_load() ? 1 : 0;
    int grid = a.tiles < num_sms ? a.tiles : num_sms;
    if (grid > kMaxTcGroupCtas) grid = kMaxTcGroupCtas;
    // Whole snake rounds, then the partial round's tiles (largest first) to
    // the CTAs with the fewest K groups after the whole rounds.
    a.full_rounds = a.tiles / grid;
    const int partial = a.tiles - a.full_rounds * grid;
    auto cost = [&](int t) {
        int i = 0;
        while (i + 1 < count && t >= a.p[i + 1].tile_begin) ++i;
        return a.p[i].KB;
    };
    int load[kMaxTcGroupCtas], by_load[kMaxTcGroupCtas];
    for (int c = 0; c < grid; ++c) {
        load[c] = 0;
        for (int r = 0; r < a.full_rounds; ++r) load[c] += cost(grouped_position(r, c, grid));
        by_load[c] = c;
        a.leftover[c] = -1;
    }
    std::stable_sort(by_load, by_load + grid, [&](int x, int y) { return load[x] < load[y]; });
    for (int i = 0; i < partial; ++i) a.leftover[by_load[i]] = static_cast<short>(a.full_rounds * grid + i);
    if (bn == 128)
        return out_f32 ? launch_grouped_typed<128, true>(a, grid, stream)
                       : launch_grouped_typed<128, false>(a, grid, stream);
    return out_f32 ? launch_grouped_typed<256, true>(a, grid, stream) : launch_grouped_typed<256, false>(a, grid, stream);
}

}  // namespace fp8act
