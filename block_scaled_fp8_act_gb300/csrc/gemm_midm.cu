// Weight-streaming tcgen05 block-FP8 GEMM for small batched decode (16 < M <= 48
// in the library's dispatch; the kernel itself handles up to 128 tokens).
//
// At M = 64..128 tokens the layer is still bound by the weight stream (about
// 2M flop per weight byte, far below the FP8 ridge point), but there are too
// many tokens for the mma.sync weight-streaming kernel. This is the regime of
// the high-concurrency section of "单并发提速73%,多并发能力达原来2.4倍:
// Qwen3.8-27B性能优化实践" (smartx.com), "高并发优化:重新平衡算力与显存容量",
// where a weight-only kernel lost 24% at 64 concurrent requests and the FP8
// W8A8 GEMM was restored, and of its 34-sequence, 3-token verify load.
//
// Swap-AB tiles: the 128 weight rows of one 128 x 128 scale block are the
// MMA's A operand (M = 128, one TMEM lane per weight row) and the tokens its
// B operand (N = MT = M rounded up to 16, rows past M zero-filled by TMA), so
// no tensor-core row is spent on padding beyond the next multiple of 16 and
// the weight block's scale is one number per (tile, K group). A "unit" is one
// (tile, 128-wide K group): 16 KB of weights and MT x 128 activation codes.
//
// Per CTA (one per SM at most, 10 warps):
//  * warp 0, one thread: TMA producer. A ring of shared-memory stages, each
//    one unit (weights and activation codes, both 128-byte swizzled K-major),
//    refilled as soon as the unit's MMAs have completed. The weight copies of
//    the first stages go out before the kernel waits on the previous grid
//    (programmatic dependent launch).
//  * warp 1: allocates 512 TMEM columns (four 128 x MT fp32 accumulators);
//    one thread issues four tcgen05.mma kind::f8f6f4 (M = 128, N = MT,
//    K = 32) per unit, commits the stage back to the producer and the
//    accumulator to the epilogue.
//  * warps 2..9: epilogue. The block scales change every K group, so each
//    unit's product is promoted in registers: every thread issues all of its
//    TMEM loads for the unit before one wait (the loads' latencies overlap),
//    then adds value * sa[token, kb] * sw[tile, kb] into its running sums.
//    Warp w reads TMEM lanes 32 (w % 4) .. +31 (weight rows) and one half of
//    the MT columns (tokens). The scales of each window of 8 units are
//    copied asynchronously (cp.async) two windows ahead into a ring in shared
//    memory and multiplied there, so no thread waits on an L2 round trip
//    (two named barriers per window).
//
// Split K: the weight stream must cover the SMs. When the 128-row tiles are
// fewer than the SMs (40 tiles on the N = 5120 projections), a thread-block
// cluster of S CTAs shares a tile, each taking a contiguous slice of the K
// groups; the partial tiles are parked in the (idle) stage memory and summed
// across the cluster through distributed shared memory in rank order
// (deterministic). No global scratch, no atomics. Without split K the grid
// is persistent: CTA b walks tiles b, b + gridDim.x, ...
//
// Failure handling: every wait is bounded (the bound is a launch argument).
// The first wait that gives up sets the device error word read by
// fp8act_check_status() and a CTA-wide abort flag; every role then stops
// issuing work, the producer waits (bounded) for the copies it already
// issued, the MMA thread for the MMAs it already issued, and only then is
// TMEM freed and the CTA leaves.
#include <atomic>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"
#include "sm100_ptx.cuh"
#include "tc_ptx.cuh"

namespace fp8act {

__device__ unsigned int g_midm_error = 0;

namespace {

constexpr int kRows = 128;        // weight rows per tile: MMA M, TMEM lanes
constexpr int kAccs = 4;          // TMEM accumulators of 128 columns
constexpr int kCtrlWarps = 2;     // producer, MMA issuer
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = (kCtrlWarps + kEpiWarps) * 32;
constexpr int kABytes = kRows * kGroup;  // 16 KB of weights per unit
constexpr int kMaxSplits = 8;
constexpr int kMaxSmem = 227 * 1024;
constexpr uint32_t kEpiBarrier = 1;  // named barrier id of the epilogue warps (0 = __syncthreads)
constexpr int kMaxStages = 8;
constexpr int kMinStages = 4;


template <int MT>
struct MidCfg {
    static_assert(MT % 16 == 0 && MT >= 16 && MT <= 128, "token tile: a multiple of 16 up to 128");
    // One ring: each stage holds one unit's weight tile and activation-code
    // tile, issued together. (The codes are L2 resident, but under a full
    // weight stream their L2 latency is as long as the weights' DRAM latency,
    // so a shallower ring of codes stalls the MMAs: measured.) The number of
    // stages is set per launch: as many as fit next to the CTA's scale table.
    static constexpr int kBBytes = ((MT * kGroup + 1023) / 1024) * 1024;  // 1024-aligned stages
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kCols = MT / 2;  // columns (tokens) per epilogue thread
    static constexpr int kBarBytes = 8 * (2 * kMaxStages + 2 * kAccs + 1) + 16;
    static_assert(kRows * MT * 4 <= kMinStages * kStageBytes, "the parked partial tile must fit in the stages");
};

// Bytes of the scale table a CTA holds: sa for its K groups and all tokens
// of the tile (MT columns), sw for its K groups and each of its tiles.
inline int64_t table_bytes(int MT, int nk, int my_tiles) {
    return 4 * static_cast<int64_t>(nk) * (MT + my_tiles);
}

struct MidArgs {
    const float* sa;
    const float* sw;
    void* out;
    int M, N, K, KB, tiles;
    unsigned long long wait_ns;  // bound of every wait that can give up (test hook shortens it)
    int withhold;                // test hook: the producer never issues the CTA's first unit
    int stages;       // ring depth (kMinStages .. kMaxStages)
    int table_bytes;  // shared memory of the scale table (multiple of 16)
};

__device__ __forceinline__ void fail(volatile int* abort, unsigned int code) {
    *abort = 1;
    atomicOr(&g_midm_error, code);
}

template <int MT, bool kF32Out>
__global__ void __launch_bounds__(kThreads, 1) gemm_midm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                                                const __grid_constant__ CUtensorMap tmap_q,
                                                                const MidArgs a) {
    using C = MidCfg<MT>;
    const int S = a.stages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - ptx::smem_u32(smem_raw));
    float* const sa_tab = reinterpret_cast<float*>(base_ptr + S * C::kStageBytes);  // [nk][MT], then sw [tiles][nk]
    const uint32_t bar0 = base + S * C::kStageBytes + a.table_bytes;
    const uint32_t full0 = bar0;                   // [S] unit landed
    const uint32_t empty0 = full0 + 8 * S;         // [S] MMAs done reading it
    const uint32_t tfull0 = empty0 + 8 * S;        // [kAccs] accumulator ready
    const uint32_t tempty0 = tfull0 + 8 * kAccs;   // [kAccs] accumulator drained
    const uint32_t drain = tempty0 + 8 * kAccs;    // MMA thread: every issued MMA has completed
    const uint32_t tmem_slot = drain + 8;
    volatile uint32_t* const tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
    volatile int* const abort = reinterpret_cast<volatile int*>(base_ptr + (tmem_slot - base) + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int splits = gridDim.z;
    const int split = blockIdx.z;  // == cluster rank when splits > 1 (cluster dims 1 x 1 x splits)
    const int kb_begin = static_cast<int>(static_cast<int64_t>(split) * a.KB / splits);
    const int kb_end = static_cast<int>(static_cast<int64_t>(split + 1) * a.KB / splits);
    const int nk = kb_end - kb_begin;
    const int my_tiles =
        static_cast<int>(blockIdx.x) < a.tiles ? (a.tiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
    const int total = my_tiles * nk;  // units of this CTA: tile-major, K group minor

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < kAccs; ++b) {
            ptx::mbar_init(tfull0 + 8 * b, 1);
            ptx::mbar_init(tempty0 + 8 * b, kEpiWarps);
        }
        ptx::mbar_init(drain, 1);
        *abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot_ptr;

    float acc[C::kCols];
    int tile0 = blockIdx.x;  // the tile of a split-K CTA (its only one)

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            ptx::griddep_launch_dependents();
            ptx::prefetch_tensormap(&tmap_w);
            ptx::prefetch_tensormap(&tmap_q);
            const uint64_t pol_w = ptx::policy_evict_first();  // every weight byte is read once
            const uint64_t pol_q = ptx::policy_evict_last();   // the codes are re-read by every tile
            auto unit = [&](int i, int& n0, int& kx) {
                n0 = (static_cast<int>(blockIdx.x) + (i / nk) * static_cast<int>(gridDim.x)) * kRows;
                kx = (kb_begin + i % nk) * kGroup;
            };
            const int first = a.withhold != 0 ? 1 : 0;  // test hook: unit 0 is never issued
            const int pre = total < S ? total : S;
            for (int i = first; i < pre; ++i) {  // weights: independent of the previous grid
                int n0, kx;
                unit(i, n0, kx);
                ptx::mbar_arrive_expect_tx(full0 + 8 * i, kABytes + MT * kGroup);
                ptx::tma_load_2d(base + i * C::kStageBytes, &tmap_w, full0 + 8 * i, kx, n0, pol_w);
            }
            ptx::griddep_wait();  // the activation codes are the previous grid's output
            for (int i = first; i < pre; ++i) {
                int n0, kx;
                unit(i, n0, kx);
                ptx::tma_load_2d(base + i * C::kStageBytes + kABytes, &tmap_q, full0 + 8 * i, kx, 0, pol_q);
            }
            int issued = pre;
            // stage and phase of use i advance incrementally (S is a launch
            // argument: no division in the loop)
            int s = 0;
            uint32_t ph = 0;  // parity of the pass over the ring that use i belongs to
            for (int i = pre; i < total; ++i) {
                if (!ptx::mbar_wait_or_abort(empty0 + 8 * s, ph, a.wait_ns, abort)) {  // use i - S done
                    fail(abort, 1u);
                    break;
                }
                int n0, kx;
                unit(i, n0, kx);
                ptx::mbar_arrive_expect_tx(full0 + 8 * s, kABytes + MT * kGroup);
                ptx::tma_load_2d(base + s * C::kStageBytes, &tmap_w, full0 + 8 * s, kx, n0, pol_w);
                ptx::tma_load_2d(base + s * C::kStageBytes + kABytes, &tmap_q, full0 + 8 * s, kx, 0, pol_q);
                issued = i + 1;
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // Every copy issued must land before the CTA may leave: wait for
            // the last use of each stage (the MMA thread has usually seen it).
            for (int i = issued > S ? issued - S : 0; i < issued; ++i)
                if (i >= first && !ptx::mbar_wait(full0 + 8 * (i % S), (i / S) & 1)) fail(abort, 16u);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_e4m3_f32(kRows, MT);
            int s = 0;
            uint32_t ph = 0;
            for (int i = 0; i < total; ++i, s = (s + 1 == S) ? 0 : s + 1, ph ^= (s == 0) ? 1u : 0u) {
                const int b = i % kAccs;
                if (!ptx::mbar_wait_or_abort(full0 + 8 * s, ph, a.wait_ns, abort)) {
                    fail(abort, 2u);
                    break;
                }
                if (i >= kAccs &&
                    !ptx::mbar_wait_or_abort(tempty0 + 8 * b, ((i / kAccs) - 1) & 1, a.wait_ns, abort)) {
                    fail(abort, 4u);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t a_tile = base + s * C::kStageBytes;
                const uint32_t b_tile = a_tile + kABytes;
#pragma unroll
                for (int k = 0; k < kGroup / 32; ++k)
                    tc::mma_f8f6f4(tmem_base + b * 128, tc::desc_kmajor_sw128(a_tile + 32 * k),
                                   tc::desc_kmajor_sw128(b_tile + 32 * k), idesc, k > 0 ? 1u : 0u);
                tc::commit(empty0 + 8 * s);  // the stage may be refilled once these MMAs finish
                tc::commit(tfull0 + 8 * b);  // the accumulator holds this unit's product
            }
            // No MMA may still run when TMEM is freed or the CTA leaves.
            tc::commit(drain);
            if (!ptx::mbar_wait(drain, 0)) fail(abort, 32u);
        }
    } else {
        // ------------------------------------------------------- epilogue
        const int et = threadIdx.x - kCtrlWarps * 32;  // 0 .. 255
        const int qd = warp & 3;                       // TMEM lane quadrant this warp may access
        const int hf = (warp - kCtrlWarps) >> 2;       // column half
        const int row = qd * 32 + lane;                // weight row within the tile
        const int col0 = hf * C::kCols;                // first token of this thread
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(qd * 32) << 16) + col0;
        ptx::griddep_wait();  // scales come from the previous grid; it may still read `out`
        // The CTA's scale table, loaded once: while the weight stream runs, the
        // SM's memory-request slots are held by the TMA copies and any global
        // load from these warps waits for thousands of clocks (measured), so
        // the loop below reads shared memory only. sa_tab[kk][m] = sa[m,
        // kb_begin + kk] (0 past M), sw_tab[t][kk] = sw[tile t, kb_begin + kk].
        float* const sw_tab = sa_tab + nk * MT;
        for (int idx = et; idx < MT * nk; idx += kEpiThreads) {  // consecutive threads: consecutive kb
            const int m = idx / nk, kk = idx % nk;
            sa_tab[kk * MT + m] = m < a.M ? ld_dep_f32(a.sa + static_cast<int64_t>(m) * a.KB + kb_begin + kk) : 0.f;
        }
        for (int idx = et; idx < my_tiles * nk; idx += kEpiThreads) {
            const int t = idx / nk, kk = idx % nk;
            const int tile = static_cast<int>(blockIdx.x) + t * static_cast<int>(gridDim.x);
            sw_tab[idx] = ld_dep_f32(a.sw + static_cast<int64_t>(tile) * a.KB + kb_begin + kk);
        }
        ptx::named_bar_sync(kEpiBarrier, kEpiThreads);
        {
            int k = 0, t = 0;  // K group within the tile and tile index of unit i (no division)
#pragma unroll 1
            for (int i = 0; i < total; ++i, k = (k + 1 == nk) ? 0 : k + 1, t += (k == 0) ? 1 : 0) {
                const int b = i % kAccs;
                if (!__all_sync(0xffffffffu,
                                ptx::mbar_wait_or_abort(tfull0 + 8 * b, (i / kAccs) & 1, a.wait_ns, abort))) {
                    if (lane == 0) fail(abort, 8u);
                    break;
                }
                tc::fence_after_sync();
                uint32_t v[C::kCols];
                tc::ld_cols<C::kCols>(t_row + b * 128, v);
                tc::wait_ld();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(tempty0 + 8 * b);  // TMEM values are in registers now
                if (k == 0) {
#pragma unroll
                    for (int j = 0; j < C::kCols; ++j) acc[j] = 0.f;
                }
                // scale of token m for this unit: sa[m, kb] * sw[tile, kb] (one fp32 product)
                const float* sc = sa_tab + k * MT + col0;
                const float s_w = sw_tab[t * nk + k];
                const float2 sw2 = make_float2(s_w, s_w);
#pragma unroll
                for (int j = 0; j < C::kCols; j += 4) {
                    const float4 s4 = *reinterpret_cast<const float4*>(sc + j);
                    const float2 c0 = __fmul2_rn(make_float2(s4.x, s4.y), sw2);
                    const float2 c1 = __fmul2_rn(make_float2(s4.z, s4.w), sw2);
                    float2 r0 = __ffma2_rn(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), c0,
                                           make_float2(acc[j], acc[j + 1]));
                    float2 r1 = __ffma2_rn(make_float2(__uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])), c1,
                                           make_float2(acc[j + 2], acc[j + 3]));
                    acc[j] = r0.x;
                    acc[j + 1] = r0.y;
                    acc[j + 2] = r1.x;
                    acc[j + 3] = r1.y;
                }
                if (k == nk - 1 && splits == 1) {
                    // the tile's sum is complete: token-major rows, consecutive lanes write
                    // consecutive weight rows (coalesced); a running pointer keeps one
                    // address live at a time
                    const int tile = static_cast<int>(blockIdx.x) + t * static_cast<int>(gridDim.x);
                    const int n = tile * kRows + row;
                    if (n < a.N) {
                        const int jn = a.M - col0 < C::kCols ? a.M - col0 : C::kCols;  // tokens < M
                        if constexpr (kF32Out) {
                            float* dst = static_cast<float*>(a.out) + static_cast<int64_t>(col0) * a.N + n;
#pragma unroll
                            for (int j = 0; j < C::kCols; ++j, dst += a.N)
                                if (j < jn) *dst = acc[j];
                        } else {
                            __nv_bfloat16* dst =
                                static_cast<__nv_bfloat16*>(a.out) + static_cast<int64_t>(col0) * a.N + n;
#pragma unroll
                            for (int j = 0; j < C::kCols; ++j, dst += a.N)
                                if (j < jn) *dst = __float2bfloat16_rn(acc[j]);
                        }
                    }
                }
            }
        }
    }

    // Every role has left its loop; the producer's copies have landed and
    // the MMA thread's MMAs have completed (both waited, bounded).
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem_base, 512);

    if (splits > 1) {
        // Park the partial tile column-major ([token][weight row]) in the idle
        // stage memory; then CTA r sums the 4-row groups [32 r / S, 32 (r + 1) / S)
        // of every peer's partial in rank order (all loads in flight first)
        // and stores them.
        float* red = reinterpret_cast<float*>(base_ptr);
        const bool ok = *abort == 0;
        if (warp >= kCtrlWarps) {
            const int qd = warp & 3;
            const int hf = (warp - kCtrlWarps) >> 2;
            const int row = qd * 32 + lane;
#pragma unroll
            for (int j = 0; j < C::kCols; ++j) red[(hf * C::kCols + j) * kRows + row] = ok ? acc[j] : 0.f;
        }
        __syncwarp();  // barrier.cluster.*.aligned: the whole warp arrives together
        ptx::cluster_sync();
        const int q_begin = split * (kRows / 4) / splits;
        const int q_end = (split + 1) * (kRows / 4) / splits;
        const int nq = q_end - q_begin;
        const int elems = nq * a.M;  // (token, 4-row group) pairs
        const int n0 = tile0 * kRows;
        constexpr int kBatch = 2;
#pragma unroll 1
        for (int e0 = threadIdx.x; e0 < elems; e0 += kBatch * kThreads) {
            float4 part[kBatch][kMaxSplits];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int e = e0 + u * kThreads;
                const int m = e < elems ? e / nq : 0;
                const int r = 4 * (q_begin + (e < elems ? e % nq : 0));
                const uint32_t local = ptx::smem_u32(red + m * kRows + r);
#pragma unroll
                for (int c = 0; c < kMaxSplits; ++c)
                    if (c < splits) part[u][c] = ptx::ld_shared_cluster_v4(ptx::mapa_shared(local, c));
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int e = e0 + u * kThreads;
                if (e >= elems) continue;
                const int m = e / nq;
                const int n = n0 + 4 * (q_begin + e % nq);
                float4 v = part[u][0];
#pragma unroll
                for (int c = 1; c < kMaxSplits; ++c)
                    if (c < splits) {
                        v.x += part[u][c].x;
                        v.y += part[u][c].y;
                        v.z += part[u][c].z;
                        v.w += part[u][c].w;
                    }
                if (!ok) continue;
                const int64_t o = static_cast<int64_t>(m) * a.N + n;
                if ((a.N & 3) == 0 && n + 3 < a.N) {
                    if constexpr (kF32Out)
                        *reinterpret_cast<float4*>(static_cast<float*>(a.out) + o) = v;
                    else
                        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + o) =
                            make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
                } else {
                    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        if (n + t >= a.N) break;
                        if constexpr (kF32Out)
                            static_cast<float*>(a.out)[o + t] = vv[t];
                        else
                            static_cast<__nv_bfloat16*>(a.out)[o + t] = __float2bfloat16_rn(vv[t]);
                    }
                }
            }
        }
        __syncwarp();
        ptx::cluster_sync();  // no CTA leaves while its peers still read its shared memory
    }
}

// Largest cluster count of S CTAs that can be resident at once (cached per
// device, kernel instance and S; the query uses the largest shared-memory
// size, which keeps one CTA per SM like every launch).
template <int MT, bool kF32Out>
int max_clusters(int s) {
    static std::atomic<int> cache[64][kMaxSplits + 1];  // 1 + clusters resident; 0 = unknown
    int dev = 0;
    cudaGetDevice(&dev);
    int cached = cache[dev & 63][s].load(std::memory_order_relaxed);
    if (cached == 0) {
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(1, 1, s);
        q.blockDim = dim3(kThreads);
        q.dynamicSmemBytes = kMaxSmem;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = 1;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = s;
        q.attrs = qa;
        q.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_midm_kernel<MT, kF32Out>, &q) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cached = n + 1;
        cache[dev & 63][s].store(cached, std::memory_order_relaxed);
    }
    return cached - 1;
}

// K splits of a launch: split K over a cluster when the 128-row tiles leave
// SMs idle, the largest S in 8..2 with at least 2 K groups per CTA, tiles * S
// CTAs within the SM count, and every cluster resident at once.
template <int MT, bool kF32Out>
int choose_splits(int tiles, int KB, int num_sms) {
    for (int s = kMaxSplits; s >= 2; --s) {
        if (tiles * s > num_sms || KB < 2 * s) continue;
        if (tiles > max_clusters<MT, kF32Out>(s)) continue;
        return s;
    }
    return 1;
}

template <int MT, bool kF32Out>
cudaError_t launch_typed(const CUtensorMap& tw, const CUtensorMap& tq, MidArgs args, int num_sms,
                         cudaStream_t stream) {
    using C = MidCfg<MT>;
    auto kernel = gemm_midm_kernel<MT, kF32Out>;
    static std::atomic<uint64_t> configured{0};  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_release);
    }
    const int tiles = args.tiles;
    const int splits = choose_splits<MT, kF32Out>(tiles, args.KB, num_sms);
    const int grid_x = splits > 1 ? tiles : (tiles < num_sms ? tiles : num_sms);
    // The CTA's scale table, then as many stages as fit beside it (at least
    // kMinStages; otherwise the caller falls back to the token-tiled kernel).
    const int nk_max = (args.KB + splits - 1) / splits;
    const int64_t table = (table_bytes(MT, nk_max, (tiles + grid_x - 1) / grid_x) + 15) & ~int64_t(15);
    const int64_t room = kMaxSmem - 1024 - C::kBarBytes - table;
    const int64_t fit = room / C::kStageBytes;
    if (fit < kMinStages) return cudaErrorNotSupported;
    args.stages = static_cast<int>(fit < kMaxStages ? fit : kMaxStages);
    args.table_bytes = static_cast<int>(table);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, 1, splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 1024 + args.stages * C::kStageBytes + table + C::kBarBytes;
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
    return cudaLaunchKernelEx(&cfg, kernel, tw, tq, args);
}

template <int MT>
cudaError_t launch_mt(const CUtensorMap& tw, const CUtensorMap& tq, const MidArgs& a, bool out_f32, int num_sms,
                      cudaStream_t stream) {
    return out_f32 ? launch_typed<MT, true>(tw, tq, a, num_sms, stream)
                   : launch_typed<MT, false>(tw, tq, a, num_sms, stream);
}

}  // namespace

unsigned int read_and_clear_midm_error() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_midm_error, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (v) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_midm_error, &zero, sizeof(zero));
    }
    return v;
}

cudaError_t launch_gemm_midm(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw, int M, int N,
                             int K, void* out, bool out_f32, int num_sms, cudaStream_t stream) {
    if (M <= 16 || M > kMidMaxTokens) return cudaErrorInvalidValue;
    MidArgs a;
    a.sa = sa;
    a.sw = sw;
    a.out = out;
    a.M = M;
    a.N = N;
    a.K = K;
    a.KB = K / kGroup;
    a.tiles = (N + kRows - 1) / kRows;
    a.wait_ns = tile_wait_limit_ns();
    a.withhold = tile_withhold_first_load() ? 1 : 0;
    a.stages = kMinStages;
    a.table_bytes = 0;
    const int MT = (M + 15) & ~15;
    CUtensorMap tw, tq;
    if (!encode_tmap_2d_u8(&tw, w, static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(K),
                           kGroup, kRows, true) ||
        !encode_tmap_2d_u8(&tq, q, static_cast<uint64_t>(K), static_cast<uint64_t>(M), static_cast<uint64_t>(K),
                           kGroup, static_cast<uint32_t>(MT), true))
        return cudaErrorInvalidValue;
    switch (MT) {
        case 32: return launch_mt<32>(tw, tq, a, out_f32, num_sms, stream);
        case 48: return launch_mt<48>(tw, tq, a, out_f32, num_sms, stream);
        case 64: return launch_mt<64>(tw, tq, a, out_f32, num_sms, stream);
        case 80: return launch_mt<80>(tw, tq, a, out_f32, num_sms, stream);
        case 96: return launch_mt<96>(tw, tq, a, out_f32, num_sms, stream);
        case 112: return launch_mt<112>(tw, tq, a, out_f32, num_sms, stream);
        default: return launch_mt<128>(tw, tq, a, out_f32, num_sms, stream);
    }
}

}  // namespace fp8act
