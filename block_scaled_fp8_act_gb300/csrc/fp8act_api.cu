// C ABI of libfp8act: argument checks, device checks, dispatch on M.
// The contract of every function is documented in include/fp8act.h.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/fp8act.h"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kGroup = 128;
constexpr int kSkinnyMaxM = 16;  // M up to this streams weights through mma.sync; above, tcgen05 kernels
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // the tcgen05 kernels' default wait bound (2 s)

// Failure-path test hook (fp8act_set_wait_limit): < 0 = the default bound.
std::atomic<long long> g_wait_limit_ns{-1};
std::atomic<int> g_withhold_first_load{0};

// Per-device facts looked up once: -1 = unknown, 0 = unsupported, else SM count.
std::atomic<int> g_device_sms[kMaxDevices];
std::atomic<bool> g_device_init[kMaxDevices];

// SM count of the current device if it is a compute-capability 10.3 part, 0 otherwise.
int current_device_sms(int* status) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        *status = FP8ACT_ERR_DEVICE;
        return 0;
    }
    if (!g_device_init[dev].load(std::memory_order_acquire)) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaGetLastError();
        g_device_sms[dev].store((major == 10 && minor == 3) ? sms : 0, std::memory_order_relaxed);
        g_device_init[dev].store(true, std::memory_order_release);
    }
    const int sms = g_device_sms[dev].load(std::memory_order_relaxed);
    *status = sms > 0 ? FP8ACT_OK : FP8ACT_ERR_DEVICE;
    return sms;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int launch_status(cudaError_t e) {
    if (e == cudaSuccess) return FP8ACT_OK;
    return FP8ACT_ERR_LAUNCH;
}

// K: positive multiple of 128; rows*K must fit in int64 and each of M, N, K in int.
int check_k(int K) { return (K <= 0 || K % kGroup) ? FP8ACT_ERR_SHAPE : FP8ACT_OK; }

// The GEMM kernel for M tokens: weight streaming through mma.sync up to 16,
// the swap-AB tcgen05 weight-streaming kernel up to 128, token-tiled tcgen05
// tiles above (prefill).
cudaError_t launch_gemm_any(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw, int M, int N,
                            int K, void* out, bool out_f32, int sms, cudaStream_t s) {
    if (M <= kSkinnyMaxM) return fp8act::launch_gemm_skinny(q, sa, w, sw, M, N, K, out, out_f32, sms, s);
    if (M <= fp8act::kMidMaxM) {
        // cudaErrorNotSupported: the CTA's scale table would not fit (very long K
        // on few tiles); the token-tiled kernel below handles any shape.
        const cudaError_t e = fp8act::launch_gemm_midm(q, sa, w, sw, M, N, K, out, out_f32, sms, s);
        if (e != cudaErrorNotSupported) return e;
    }
    return fp8act::launch_gemm_tc(q, sa, w, sw, M, N, K, out, out_f32, sms, s);
}

int gemm_common(const void* q, const float* sa, const void* w, const float* sw, int M, int N, int K, void* out,
                bool out_f32, void* stream) {
    if (M < 0 || N < 0) return FP8ACT_ERR_SHAPE;
    if (int st = check_k(K)) return st;
    if (M == 0 || N == 0) return FP8ACT_OK;
    if (!q || !sa || !w || !sw || !out) return FP8ACT_ERR_NULL;
    if (!aligned(q, 16) || !aligned(w, 16) || !aligned(out, 16) || !aligned(sa, 4) || !aligned(sw, 4))
        return FP8ACT_ERR_ALIGN;
    int st = FP8ACT_OK;
    const int sms = current_device_sms(&st);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint8_t* q8 = static_cast<const uint8_t*>(q);
    const uint8_t* w8 = static_cast<const uint8_t*>(w);
    return launch_status(launch_gemm_any(q8, sa, w8, sw, M, N, K, out, out_f32, sms, s));
}

constexpr int kMaxGrouped = 16;
constexpr int kTileGroupMaxM = 128;  // one token tile: the grouped tile launch takes these

// The single-call checks of one GEMM problem (no launch); OK for an empty one.
int check_gemm(const fp8act_gemm_problem& p) {
    if (p.M < 0 || p.N < 0) return FP8ACT_ERR_SHAPE;
    if (int st = check_k(p.K)) return st;
    if (p.M == 0 || p.N == 0) return FP8ACT_OK;
    if (!p.q_e4m3 || !p.sa || !p.w_e4m3 || !p.sw || !p.out) return FP8ACT_ERR_NULL;
    if (!aligned(p.q_e4m3, 16) || !aligned(p.w_e4m3, 16) || !aligned(p.out, 16) || !aligned(p.sa, 4) ||
        !aligned(p.sw, 4))
        return FP8ACT_ERR_ALIGN;
    return FP8ACT_OK;
}

int gemm_grouped_common(const fp8act_gemm_problem* problems, int count, bool out_f32, void* stream) {
    if (count < 0 || count > kMaxGrouped) return FP8ACT_ERR_SHAPE;
    if (count == 0) return FP8ACT_OK;
    if (!problems) return FP8ACT_ERR_NULL;
    bool any = false;
    for (int i = 0; i < count; ++i) {
        if (int st = check_gemm(problems[i])) return st;
        any = any || (problems[i].M > 0 && problems[i].N > 0);
    }
    if (!any) return FP8ACT_OK;
    int st = FP8ACT_OK;
    const int sms = current_device_sms(&st);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    fp8act::GemmProblem skinny[kMaxGrouped];
    int n_skinny = 0;
    for (int i = 0; i < count; ++i) {
        const fp8act_gemm_problem& p = problems[i];
        if (p.M == 0 || p.N == 0 || p.M > kSkinnyMaxM) continue;
        skinny[n_skinny++] = {static_cast<const uint8_t*>(p.q_e4m3), p.sa, static_cast<const uint8_t*>(p.w_e4m3),
                              p.sw, p.out, p.M, p.N, p.K};
    }
    if (int e = launch_status(fp8act::launch_gemm_skinny_grouped(skinny, n_skinny, out_f32, s))) return e;
    auto one = [&](const fp8act::GemmProblem& p) {
        return launch_status(launch_gemm_any(p.q, p.sa, p.w, p.sw, p.M, p.N, p.K, p.out, out_f32, sms, s));
    };
    // Problems of the tile kernel, grouped by width: one token tile each (16 < M
    // <= 128: 128-wide weight tiles, a chunk is worth one launch once its tiles
    // fill the SMs) and several (M > 128: 256-wide tiles, once they fill two
    // waves, the single-problem kernel's own rule for wide tiles). One grouped
    // persistent launch per chunk of up to gemm_tc_grouped_capacity()
    // problems; a chunk with fewer tiles, one launch per problem.
    fp8act::GemmProblem narrow[kMaxGrouped], wide[kMaxGrouped];
    int n_narrow = 0, n_wide = 0;
    for (int i = 0; i < count; ++i) {
        const fp8act_gemm_problem& p = problems[i];
        if (p.M <= kSkinnyMaxM || p.N == 0) continue;
        const fp8act::GemmProblem g = {static_cast<const uint8_t*>(p.q_e4m3), p.sa,
                                       static_cast<const uint8_t*>(p.w_e4m3), p.sw, p.out, p.M, p.N, p.K};
        if (p.M <= kTileGroupMaxM)
            narrow[n_narrow++] = g;
        else
            wide[n_wide++] = g;
    }
    const int cap = fp8act::gemm_tc_grouped_capacity();
    auto run_chunks = [&](const fp8act::GemmProblem* list, int n_list, int bn, int64_t min_tiles) -> int {
        for (int c0 = 0; c0 < n_list; c0 += cap) {
            const int n = n_list - c0 < cap ? n_list - c0 : cap;
            int64_t tiles = 0;
            for (int j = 0; j < n; ++j)
                tiles += static_cast<int64_t>((list[c0 + j].M + 127) / 128) * ((list[c0 + j].N + bn - 1) / bn);
            const cudaError_t g = tiles >= min_tiles
                                      ? fp8act::launch_gemm_tc_grouped(list + c0, n, out_f32, sms, s)
                                      : cudaErrorNotSupported;
            if (g == cudaErrorNotSupported) {  // too few tiles to fill the grid (or too many to list)
                for (int j = 0; j < n; ++j)
                    if (int e = one(list[c0 + j])) return e;
            } else if (int e = launch_status(g)) {
                return e;
            }
        }
        return FP8ACT_OK;
    };
    if (int e = run_chunks(narrow, n_narrow, 128, sms)) return e;
    if (int e = run_chunks(wide, n_wide, 256, 2 * static_cast<int64_t>(sms))) return e;
    return FP8ACT_OK;
}

int linear_common(const void* x, const void* w, const float* sw, int M, int N, int K, void* out, bool out_f32,
                  void* stream) {
    if (M < 0 || N < 0) return FP8ACT_ERR_SHAPE;
    if (int st = check_k(K)) return st;
    if (M == 0 || N == 0) return FP8ACT_OK;
    if (!fp8act::fused_fits(M, K)) return FP8ACT_ERR_SHAPE;
    if (!x || !w || !sw || !out) return FP8ACT_ERR_NULL;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(out, 16) || !aligned(sw, 4)) return FP8ACT_ERR_ALIGN;
    int st = FP8ACT_OK;
    const int sms = current_device_sms(&st);
    if (st) return st;
    return launch_status(fp8act::launch_linear_fused(x, static_cast<const uint8_t*>(w), sw, M, N, K, out, out_f32,
                                                     sms, static_cast<cudaStream_t>(stream)));
}

int w8a16_common(const void* x, const void* w, const float* sw, int M, int N, int K, void* out, bool out_f32,
                 void* stream) {
    if (M < 0 || N < 0) return FP8ACT_ERR_SHAPE;
    if (int st = check_k(K)) return st;
    if (M == 0 || N == 0) return FP8ACT_OK;
    if (!x || !w || !sw || !out) return FP8ACT_ERR_NULL;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(out, 16) || !aligned(sw, 4)) return FP8ACT_ERR_ALIGN;
    int st = FP8ACT_OK;
    const int sms = current_device_sms(&st);
    if (st) return st;
    return launch_status(fp8act::launch_gemm_w8a16(x, static_cast<const uint8_t*>(w), sw, M, N, K, out, out_f32, sms,
                                                   static_cast<cudaStream_t>(stream)));
}

}  // namespace

namespace fp8act {
unsigned long long tile_wait_limit_ns() {
    const long long v = g_wait_limit_ns.load(std::memory_order_relaxed);
    return v < 0 ? kDefaultWaitNs : static_cast<unsigned long long>(v);
}
bool tile_withhold_first_load() { return g_withhold_first_load.load(std::memory_order_relaxed) != 0; }
}  // namespace fp8act

extern "C" {

int fp8_act_quant(const void* x_bf16, int M, int K, void* q_e4m3, float* sa, void* stream) {
    if (M < 0) return FP8ACT_ERR_SHAPE;
    if (int st = check_k(K)) return st;
    if (M == 0) return FP8ACT_OK;
    if (!x_bf16 || !q_e4m3 || !sa) return FP8ACT_ERR_NULL;
    if (!aligned(x_bf16, 16) || !aligned(q_e4m3, 16) || !aligned(sa, 4)) return FP8ACT_ERR_ALIGN;
    int st = FP8ACT_OK;
    const int sms = current_device_sms(&st);
    if (st) return st;
    return launch_status(fp8act::launch_act_quant(x_bf16, M, K, q_e4m3, sa, sms, static_cast<cudaStream_t>(stream)));
}

int fp8_weight_quant(const void* w_bf16, int N, int K, void* w_e4m3, float* sw, void* stream) {
    if (N < 0) return FP8ACT_ERR_SHAPE;
    if (int st = check_k(K)) return st;
    if (N == 0) return FP8ACT_OK;
    if (!w_bf16 || !w_e4m3 || !sw) return FP8ACT_ERR_NULL;
    if (!aligned(w_bf16, 16) || !aligned(w_e4m3, 16) || !aligned(sw, 4)) return FP8ACT_ERR_ALIGN;
    int st = FP8ACT_OK;
    current_device_sms(&st);
    if (st) return st;
    return launch_status(fp8act::launch_weight_quant(w_bf16, N, K, w_e4m3, sw, static_cast<cudaStream_t>(stream)));
}

int fp8_block_gemm(const void* q_e4m3, const float* sa, const void* w_e4m3, const float* sw, int M, int N, int K,
                   void* out_bf16, void* stream) {
    return gemm_common(q_e4m3, sa, w_e4m3, sw, M, N, K, out_bf16, false, stream);
}

int fp8_block_gemm_f32(const void* q_e4m3, const float* sa, const void* w_e4m3, const float* sw, int M, int N,
                       int K, float* out_f32, void* stream) {
    return gemm_common(q_e4m3, sa, w_e4m3, sw, M, N, K, out_f32, true, stream);
}

int fp8_block_gemm_w8a16(const void* x_bf16, const void* w_e4m3, const float* sw, int M, int N, int K,
                         void* out_bf16, void* stream) {
    return w8a16_common(x_bf16, w_e4m3, sw, M, N, K, out_bf16, false, stream);
}

int fp8_block_gemm_w8a16_f32(const void* x_bf16, const void* w_e4m3, const float* sw, int M, int N, int K,
                             float* out_f32, void* stream) {
    return w8a16_common(x_bf16, w_e4m3, sw, M, N, K, out_f32, true, stream);
}

int fp8_linear(const void* x_bf16, const void* w_e4m3, const float* sw, int M, int N, int K, void* out_bf16,
               void* stream) {
    return linear_common(x_bf16, w_e4m3, sw, M, N, K, out_bf16, false, stream);
}

int fp8_linear_f32(const void* x_bf16, const void* w_e4m3, const float* sw, int M, int N, int K, float* out_f32,
                   void* stream) {
    return linear_common(x_bf16, w_e4m3, sw, M, N, K, out_f32, true, stream);
}

int fp8_act_quant_grouped(const fp8act_quant_problem* problems, int count, void* stream) {
    if (count < 0 || count > kMaxGrouped) return FP8ACT_ERR_SHAPE;
    if (count == 0) return FP8ACT_OK;
    if (!problems) return FP8ACT_ERR_NULL;
    fp8act::ActQuantProblem probs[kMaxGrouped];
    int n = 0;
    for (int i = 0; i < count; ++i) {
        const fp8act_quant_problem& p = problems[i];
        if (p.M < 0) return FP8ACT_ERR_SHAPE;
        if (int st = check_k(p.K)) return st;
        if (p.M == 0) continue;
        if (!p.x_bf16 || !p.q_e4m3 || !p.sa) return FP8ACT_ERR_NULL;
        if (!aligned(p.x_bf16, 16) || !aligned(p.q_e4m3, 16) || !aligned(p.sa, 4)) return FP8ACT_ERR_ALIGN;
        probs[n++] = {p.x_bf16, p.q_e4m3, p.sa, p.M, p.K};
    }
    if (n == 0) return FP8ACT_OK;
    int st = FP8ACT_OK;
    const int sms = current_device_sms(&st);
    if (st) return st;
    return launch_status(fp8act::launch_act_quant_grouped(probs, n, sms, static_cast<cudaStream_t>(stream)));
}

int fp8_block_gemm_grouped(const fp8act_gemm_problem* problems, int count, void* stream) {
    return gemm_grouped_common(problems, count, false, stream);
}

int fp8_block_gemm_grouped_f32(const fp8act_gemm_problem* problems, int count, void* stream) {
    return gemm_grouped_common(problems, count, true, stream);
}

const char* fp8act_strerror(int status) {
    switch (status) {
        case FP8ACT_OK: return "ok";
        case FP8ACT_ERR_NULL: return "a required pointer is NULL";
        case FP8ACT_ERR_SHAPE:
            return "bad shape: M, N must be >= 0 and K a positive multiple of 128 (grouped calls: at most 16 "
                   "problems; fp8_linear: min(8, M) rows of K codes and scales must fit in 200 KiB)";
        case FP8ACT_ERR_ALIGN: return "misaligned pointer: tensors need 16-byte, scales 4-byte alignment";
        case FP8ACT_ERR_LAUNCH: return "kernel launch failed";
        case FP8ACT_ERR_TIMEOUT: return "a kernel gave up a bounded wait (device-side timeout)";
        case FP8ACT_ERR_DEVICE: return "no current CUDA device of compute capability 10.3 (GB300)";
        case FP8ACT_ERR_CUDA: return "CUDA runtime error";
        default: return "unknown fp8act status";
    }
}

int fp8act_check_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return FP8ACT_ERR_CUDA;
    }
    const unsigned int tc = fp8act::read_and_clear_tc_error();
    const unsigned int mid = fp8act::read_and_clear_midm_error();
    const unsigned int rd = fp8act::read_and_clear_read_error();
    return (tc | mid | rd) ? FP8ACT_ERR_TIMEOUT : FP8ACT_OK;
}

int fp8act_set_wait_limit(long long limit_ns, int withhold_first_load) {
    g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
    g_withhold_first_load.store(withhold_first_load ? 1 : 0, std::memory_order_relaxed);
    return FP8ACT_OK;
}

int fp8act_stream_read(const void* src, size_t bytes, unsigned int* sink, void* stream) {
    if (bytes == 0) return FP8ACT_OK;
    if (!src || !sink) return FP8ACT_ERR_NULL;
    if (!aligned(src, 16) || !aligned(sink, 4) || bytes % 16) return FP8ACT_ERR_ALIGN;
    int st = FP8ACT_OK;
    const int sms = current_device_sms(&st);
    if (st) return st;
    return launch_status(fp8act::launch_stream_read(src, static_cast<int64_t>(bytes), sink, sms,
                                                    static_cast<cudaStream_t>(stream)));
}

int fp8act_version(void) { return 200; }

}  // extern "C"
