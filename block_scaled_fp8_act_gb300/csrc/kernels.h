// Host-side launchers of libfp8act's kernels (internal; the public API is include/fp8act.h).
// Arguments are validated by the C-ABI layer before any of these is called.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fp8act {

// Activation quantisation, x bf16 [M, K] -> q E4M3 [M, K], sa fp32 [M, K/128].
cudaError_t launch_act_quant(const void* x, int64_t M, int64_t K, void* q, float* sa, int num_sms,
                             cudaStream_t stream);

// One activation-quantisation problem: x bf16 [M, K] -> q [M, K], sa [M, K/128].
struct ActQuantProblem {
    const void* x;
    void* q;
    float* sa;
    int64_t M, K;
};
// Up to 16 of them in one launch (their 128-wide groups concatenated).
cudaError_t launch_act_quant_grouped(const ActQuantProblem* probs, int count, int num_sms, cudaStream_t stream);

// Weight quantisation, W bf16 [N, K] -> w E4M3 [N, K], sw fp32 [ceil(N/128), K/128].
cudaError_t launch_weight_quant(const void* W, int64_t N, int64_t K, void* w, float* sw, cudaStream_t stream);

// Weight-streaming GEMM for small M (tensor-core mma.sync, 16-row tiles,
// K split across the warps of a CTA, programmatic dependent launch). Any M
// works (a CTA per 8 tokens and 16-row tile) but every token group re-reads
// the weights, so it is the M <= 16 path.
cudaError_t launch_gemm_skinny(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw, int M,
                               int N, int K, void* out, bool out_f32, int num_sms, cudaStream_t stream);
// The same with an explicit load depth per warp (1, 2 or 4 K blocks per step).
cudaError_t launch_gemm_skinny_unroll(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw, int M,
                                      int N, int K, void* out, bool out_f32, int num_sms, int unroll,
                                      cudaStream_t stream);

// Weight-only variant of the same kernel: bf16 activations x [M, K], no
// activation scales (E4M3 weights widened to bf16, bf16 MMAs).
cudaError_t launch_gemm_w8a16(const void* x, const uint8_t* w, const float* sw, int M, int N, int K, void* out,
                              bool out_f32, int num_sms, cudaStream_t stream);

// One block-FP8 GEMM problem (device pointers, row-major, as fp8_block_gemm).
struct GemmProblem {
    const uint8_t* q;
    const float* sa;
    const uint8_t* w;
    const float* sw;
    void* out;
    int M, N, K;
};

// Up to 16 independent problems with M <= 16 in one launch of the
// weight-streaming kernel (each CTA finds its problem from its index).
cudaError_t launch_gemm_skinny_grouped(const GemmProblem* probs, int count, bool out_f32, cudaStream_t stream);

// Several problems (M > 16) in one persistent launch of the tcgen05 tile
// kernel: 128 x 128 tiles when every M <= 128 (one token tile each), 128 x
// 256 tiles otherwise; all their tiles in one list dealt evenly over the
// CTAs, K never split. At most gemm_tc_grouped_capacity() problems per
// launch; worth it when their tiles fill the SMs (two waves for 256-wide
// ones). cudaErrorNotSupported (nothing launched) past 32767 tiles.
int gemm_tc_grouped_capacity();
cudaError_t launch_gemm_tc_grouped(const GemmProblem* probs, int count, bool out_f32, int num_sms,
                                   cudaStream_t stream);

// Fused activation quantisation + block GEMM for small M: bf16 x [M, K] in,
// out [M, N] as fp8_block_gemm(fp8_act_quant(x)) would give. M <= 8: one
// CTA per SM quantises all the tokens once into shared memory (from M = 2 a
// cluster of 2 or 4 CTAs splits that work), then warp groups stream
// the tiles; otherwise (or when the codes do not fit) each
// warp quantises the groups of the K blocks it multiplies into its
// shared-memory slice; fused_fits() tells whether min(8, M) rows of every
// block fit that kernel's shared-memory ceiling.
bool fused_fits(int M, int K);
cudaError_t launch_linear_fused(const void* x, const uint8_t* w, const float* sw, int M, int N, int K, void* out,
                                bool out_f32, int num_sms, cudaStream_t stream);

// Tensor-memory (tcgen05) GEMM: 128 x 256 (prefill) or 128 x 128 output
// tiles, TMA-fed ring, per-K-group promotion of the fp32 block scales in the
// epilogue, split K over a thread-block cluster when the tiles are too few.
cudaError_t launch_gemm_tc(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw, int M, int N, int K,
                           void* out, bool out_f32, int num_sms, cudaStream_t stream);

// Weight-streaming tcgen05 GEMM for small batched decode, kMidMaxM >= M > 16:
// 128 weight rows x round16(M) tokens per tile (swap-AB), TMA-fed ring, the
// block scales promoted per K group, split K over a thread-block cluster
// when the tiles are fewer than the SMs. Returns cudaErrorNotSupported
// (launching nothing) when a CTA's scale table would not fit its shared
// memory (very long K on few tiles).
constexpr int kMidMaxM = 48;   // measured: ahead of the token-tiled kernel up to 48 tokens, behind above 64
constexpr int kMidMaxTokens = 128;  // the kernel itself handles up to 128
cudaError_t launch_gemm_midm(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw, int M, int N,
                             int K, void* out, bool out_f32, int num_sms, cudaStream_t stream);

// Diagnostic streaming read of `bytes` (a multiple of 16) from `src`: one CTA
// per SM, a ring of TMA bulk copies, launched like the GEMMs; folds the data
// into *sink.
cudaError_t launch_stream_read(const void* src, int64_t bytes, unsigned int* sink, int num_sms, cudaStream_t stream);

// Device-side error words of the tcgen05 kernels (non-zero after a bounded
// wait gave up); reading one synchronises with the device and clears it.
unsigned int read_and_clear_tc_error();
unsigned int read_and_clear_midm_error();
unsigned int read_and_clear_read_error();  // the streaming-read diagnostic

// Launch arguments of the tcgen05 kernels' failure path, set process-wide by
// the fp8act_set_wait_limit() test hook: the wall-time bound of every wait
// that may give up, and whether each CTA withholds its first operand copy.
unsigned long long tile_wait_limit_ns();
bool tile_withhold_first_load();

}  // namespace fp8act
