// Diagnostic: a plain streaming read of a device buffer, the floor a
// weight-streaming GEMM of the same bytes can reach. Launched exactly like
// the GEMM kernels (programmatic dependent launch: the reads start before the
// previous kernel on the stream has finished), one CTA per SM streaming a
// contiguous share of the buffer through a ring of 32 KB TMA bulk copies into
// shared memory (the deepest read pipeline an SM offers); the consumer warps
// fold every landed chunk into one word per CTA, XORed into `sink`, so that
// the data is used as a GEMM would use it. Every wait is bounded; a wait that
// gives up stops the producer and drains its copies before the CTA leaves.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace fp8act {

__device__ unsigned int g_read_error = 0;

namespace {

constexpr int kChunk = 32 * 1024;   // bytes per bulk copy
constexpr int kRing = 6;            // copies in flight per CTA
constexpr int kConsumerWarps = 8;
constexpr int kReadThreads = (1 + kConsumerWarps) * 32;
constexpr int kReadSmem = 1024 + kRing * kChunk + 2 * kRing * 8;

__global__ void __launch_bounds__(kReadThreads, 1) stream_read_kernel(const uint8_t* __restrict__ src, int64_t bytes,
                                                                       unsigned int* __restrict__ sink) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - ptx::smem_u32(smem_raw));
    const uint32_t full0 = base + kRing * kChunk, empty0 = full0 + 8 * kRing;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's share: whole chunks, the last one possibly short (16-byte multiple)
    const int64_t chunks = (bytes + kChunk - 1) / kChunk;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * chunks / gridDim.x;
    const int64_t c1 = static_cast<int64_t>(blockIdx.x + 1) * chunks / gridDim.x;
    const int n = static_cast<int>(c1 - c0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();
    uint32_t acc = 0;
    if (warp == 0) {
        if (lane == 0) {
            ptx::griddep_launch_dependents();
            int issued = 0;
            for (int i = 0; i < n; ++i) {
                const int s = i % kRing;
                if (i >= kRing && !ptx::mbar_wait(empty0 + 8 * s, ((i / kRing) - 1) & 1)) {
                    atomicOr(&g_read_error, 1u);
                    break;
                }
                const int64_t off = (c0 + i) * kChunk;
                const uint32_t len = static_cast<uint32_t>(bytes - off < kChunk ? bytes - off : kChunk);
                ptx::mbar_arrive_expect_tx(full0 + 8 * s, len);
                ptx::bulk_load_g2s(base + s * kChunk, src + off, len, full0 + 8 * s);
                issued = i + 1;
            }
            for (int i = issued > kRing ? issued - kRing : 0; i < issued; ++i)  // nothing in flight at exit
                if (!ptx::mbar_wait(full0 + 8 * (i % kRing), (i / kRing) & 1)) atomicOr(&g_read_error, 2u);
        }
    } else {
        const int ct = threadIdx.x - 32;  // consumer thread 0 .. 255
        for (int i = 0; i < n; ++i) {
            const int s = i % kRing;
            if (!ptx::mbar_wait(full0 + 8 * s, (i / kRing) & 1)) {
                atomicOr(&g_read_error, 4u);
                break;
            }
            const int64_t off = (c0 + i) * kChunk;
            const int len = static_cast<int>(bytes - off < kChunk ? bytes - off : kChunk);
            const uint4* chunk = reinterpret_cast<const uint4*>(base_ptr + s * kChunk);
            for (int j = ct; j < len / 16; j += kConsumerWarps * 32) {
                const uint4 v = chunk[j];
                acc ^= v.x ^ v.y ^ v.z ^ v.w;
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty0 + 8 * s);
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    ptx::griddep_wait();  // the previous kernel may still use `sink`
    if (lane == 0 && warp > 0) atomicXor(sink, acc);
}

}  // namespace

cudaError_t launch_stream_read(const void* src, int64_t bytes, unsigned int* sink, int num_sms, cudaStream_t stream) {
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configured[dev & 63]) {
        const cudaError_t e =
            cudaFuncSetAttribute(stream_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kReadSmem);
        if (e != cudaSuccess) return e;
        configured[dev & 63] = true;
    }
    const int64_t chunks = (bytes + kChunk - 1) / kChunk;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(chunks < num_sms ? chunks : num_sms));
    cfg.blockDim = dim3(kReadThreads);
    cfg.dynamicSmemBytes = kReadSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stream_read_kernel, static_cast<const uint8_t*>(src), bytes, sink);
}

unsigned int read_and_clear_read_error() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_read_error, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (v) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_read_error, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace fp8act
