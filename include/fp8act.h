/*
 * fp8act.h - C ABI of libfp8act.so, the W8A8 block-FP8 linear layer for GB300 (sm_103a).
 *
 * The layer: y = x W^T with x [M, K] quantised per token in 1x128 K groups and
 * W [N, K] quantised per 128x128 block, both to FP8 E4M3 with one fp32 scale
 * per group / block, multiplied with fp32 accumulation and stored as bf16.
 * "W8A8 Block FP8" is the layer type of the five projection shapes in
 * "双 NVIDIA L20 上 Qwen3.8-27B-FP8 + MTP 调优测试报告" (ownding.com), section 八
 * (L20 FP8 kernel tuning). The run-time activation quantisation is the step
 * that "单并发提速73%,多并发能力达原来2.4倍:Qwen3.8-27B性能优化实践"
 * (smartx.com), section "单并发优化", credits the weight-only Marlin back-end
 * with skipping. Neither page fixes the arithmetic; this library implements:
 *
 *   s      = amax / 448 over the group (fp32, IEEE division); s = 1 if amax = 0
 *   code   = E4M3(x / s): IEEE fp32 division, round to nearest even,
 *            saturated to +-448 (largest finite E4M3), sign of zero kept
 *   y[m,n] = sum_kb sa[m,kb] * sw[n/128,kb] * sum_{k in block kb} q[m,k] w[n,k]
 *   out    = bf16(y), round to nearest even
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Pointers are DEVICE pointers on the current CUDA device, owned by the
 *   caller (the one exception: the `problems` arrays of the grouped calls
 *   live in host memory and are read during the call only). The library
 *   never allocates, frees or synchronises inside these calls and reads no
 *   device data on the host, so every call can be captured in a CUDA graph.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is
 *   enqueued asynchronously; the returned status covers argument checks and
 *   the launch only. Kernel-side timeouts are reported by
 *   fp8act_check_status().
 * - Layouts are row-major and contiguous: x, q [M, K]; sa [M, K/128];
 *   W, w [N, K] (K contiguous); sw [ceil(N/128), K/128]; out [M, N].
 * - K must be a positive multiple of 128. M and N may be any value >= 0; a
 *   call with M == 0 (or N == 0) does nothing and returns FP8ACT_OK.
 * - x, q, W, w and out must be 16-byte aligned; sa and sw 4-byte aligned.
 * - Behaviour on NaN or infinite inputs is unspecified (no error is raised).
 * - The library runs only on compute capability 10.3 (GB300); on any other
 *   device every compute call returns FP8ACT_ERR_DEVICE.
 */
#ifndef FP8ACT_H
#define FP8ACT_H

#if defined(__GNUC__)
#define FP8ACT_API __attribute__((visibility("default")))
#else
#define FP8ACT_API
#endif

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8ACT_OK = 0,
    FP8ACT_ERR_NULL = 1,     /* a required pointer is NULL                         */
    FP8ACT_ERR_SHAPE = 2,    /* M, N < 0; K <= 0 or K % 128 != 0; size overflow;
                                more than 16 grouped problems; fp8_linear K too large */
    FP8ACT_ERR_ALIGN = 3,    /* a pointer violates the alignment rule above       */
    FP8ACT_ERR_LAUNCH = 4,   /* the kernel launch failed (cudaGetLastError)       */
    FP8ACT_ERR_TIMEOUT = 5,  /* a kernel's bounded wait gave up (see check_status) */
    FP8ACT_ERR_DEVICE = 6,   /* no current device, or not compute capability 10.3 */
    FP8ACT_ERR_CUDA = 7      /* another CUDA runtime error                         */
} fp8act_status;

/*
 * Activation quantisation, one scale per token and 128-wide K group.
 *   x_bf16  [M, K] bf16 in
 *   q_e4m3  [M, K] E4M3 codes out (1 byte each)
 *   sa      [M, K/128] fp32 scales out
 * Bit-exact with the definition above.
 */
FP8ACT_API int fp8_act_quant(const void* x_bf16, int M, int K, void* q_e4m3, float* sa, void* stream);

/*
 * Weight quantisation, one scale per 128x128 block (an offline step: the
 * served checkpoint stores w and sw). A partial block at the N edge takes its
 * amax over the rows that exist.
 *   w_bf16  [N, K] bf16 in
 *   w_e4m3  [N, K] E4M3 codes out
 *   sw      [ceil(N/128), K/128] fp32 scales out
 */
FP8ACT_API int fp8_weight_quant(const void* w_bf16, int N, int K, void* w_e4m3, float* sw, void* stream);

/*
 * Block-scaled GEMM: out[M, N] = bf16(y) with y as defined above, fp32
 * accumulation. Dispatches on M:
 *   M <= 16      a weight-streaming kernel over 16-row weight tiles on the
 *                warp-level tensor-core MMA (decode and speculative verify);
 *   16 < M <= 48 a weight-streaming tcgen05 kernel: 128 weight rows x
 *                round16(M) tokens per tile (swap-AB), K split over a
 *                thread-block cluster when the tiles are fewer than the SMs;
 *   M > 48       tcgen05 tiles of 128 tokens x 128 / 256 weight rows (batched
 *                decode, "高并发优化" of the smartx.com Qwen3.8-27B post, and
 *                prefill), K split over a cluster when the tiles are few.
 *   (The boundary at 48 is measured: ahead below it, behind from 64.)
 * Every M >= 1 is supported and every kernel sums in a fixed order, so
 * results are bit-reproducible for a given M, N, K.
 *
 * Ordering (programmatic dependent launch): each kernel may start while the
 * kernel before it on the stream is still running; it reads the activation
 * codes and scales, and writes `out`, only after that kernel has completed,
 * but it starts reading w and sw at once. The weights and weight scales must
 * therefore be complete before the previous kernel on the stream starts (an
 * fp8_act_quant launch lets the GEMM after it start immediately): write them
 * on another stream or earlier and synchronise (an event or
 * cudaStreamSynchronize) before the chain that reads them, as a served
 * model's loaded checkpoint is.
 *   q_e4m3, sa : activation codes [M, K] and scales [M, K/128]
 *   w_e4m3, sw : weight codes [N, K] and scales [ceil(N/128), K/128]
 *   out_bf16   : [M, N] bf16 out
 */
FP8ACT_API int fp8_block_gemm(const void* q_e4m3, const float* sa, const void* w_e4m3, const float* sw,
                   int M, int N, int K, void* out_bf16, void* stream);

/*
 * The same kernels as fp8_block_gemm with an fp32 store in place of the
 * bf16 cast (for error analysis of the accumulation before rounding).
 */
FP8ACT_API int fp8_block_gemm_f32(const void* q_e4m3, const float* sa, const void* w_e4m3, const float* sw,
                       int M, int N, int K, float* out_f32, void* stream);

/*
 * Weight-only block-FP8 GEMM (W8A16): the bf16 activations times the same
 * block-scaled E4M3 weights, with no activation quantisation:
 *   out[m, n] = bf16( sum_kb sw[n/128, kb] * sum_{k in block kb} x[m, k] * w[n, k] ),
 * each E4M3 weight widened exactly to bf16, bf16 x bf16 products, fp32
 * accumulation. This is the role of the weight-only FP8 back-end (Marlin)
 * that "单并发提速73%,多并发能力达原来2.4倍:Qwen3.8-27B性能优化实践"
 * (smartx.com), section "单并发优化", picks at one request: it saves the
 * quantisation launch per linear layer. The kernel is the weight-streaming
 * one of fp8_block_gemm; it reads the weights once per 16 tokens, so it is
 * meant for decode (M <= 16). Every M >= 1 is supported.
 *   x_bf16     : [M, K] bf16 activations (16-byte aligned)
 *   w_e4m3, sw : weight codes [N, K] and scales [ceil(N/128), K/128]
 *   out_bf16   : [M, N] bf16 out (out_f32: [M, N] fp32, the value before the cast)
 * Errors as for fp8_block_gemm.
 */
FP8ACT_API int fp8_block_gemm_w8a16(const void* x_bf16, const void* w_e4m3, const float* sw, int M, int N, int K,
                                    void* out_bf16, void* stream);
FP8ACT_API int fp8_block_gemm_w8a16_f32(const void* x_bf16, const void* w_e4m3, const float* sw, int M, int N,
                                        int K, float* out_f32, void* stream);

/*
 * Fused linear layer: fp8_act_quant and fp8_block_gemm in one launch,
 *   out = fp8_block_gemm(fp8_act_quant(x), w, sw),
 * with the same activation codes and scales bit for bit (the kernel
 * quantises with the activation kernel's own group code). The
 * single-RTX-PRO-6000 Qwen3.8-27B post (smartx.com), section "单并发优化",
 * counts the quantisation launch per linear layer among the costs of the
 * W8A8 path at one request, and the zskr.cn Qwen3-27B decode article,
 * section 3.3, fuses the quantisation op into the preceding computation.
 * For M <= 16 one CTA per SM quantises all the tokens once into shared
 * memory after the wait for the previous kernel (from M = 2 on, a
 * thread-block cluster of 2 or 4 CTAs splits that work and each CTA stores
 * its groups into every peer's shared memory), then its warp groups stream
 * the weight tiles (16 rows x 8 tokens) with the two-launch kernel's loop
 * and warp count (the same sums: the result equals the two-launch path bit
 * for bit). Above M = 16, or where the M x K codes do not fit the CTA's
 * shared memory (about K <= 13000 at 16 tokens), every warp of the
 * weight-streaming kernel quantises the 1x128 groups of the K blocks it
 * multiplies (for its at most 8 tokens) into shared memory, which repeats
 * the activation work in every CTA and is several times slower. The call is
 * meant for decode and speculative verify: on the five projection shapes it
 * is ~5% faster than the two launches at one token, level at 4 and 9
 * tokens, and 7-8% slower at 8 and 16. The codes and scales of min(8, M)
 * tokens take min(8, M) * K * 33 / 32 bytes of shared memory per CTA in the
 * per-warp kernel, at most 200 KiB (K <= 24576 once M >= 8); larger K
 * returns FP8ACT_ERR_SHAPE.
 *   x_bf16     : [M, K] bf16 activations (16-byte aligned)
 *   w_e4m3, sw : weight codes [N, K] and scales [ceil(N/128), K/128]
 *   out_bf16   : [M, N] bf16 out (out_f32: [M, N] fp32, the value before the cast)
 */
FP8ACT_API int fp8_linear(const void* x_bf16, const void* w_e4m3, const float* sw, int M, int N, int K,
                          void* out_bf16, void* stream);
FP8ACT_API int fp8_linear_f32(const void* x_bf16, const void* w_e4m3, const float* sw, int M, int N, int K,
                              float* out_f32, void* stream);

/*
 * Grouped calls: several independent problems in one kernel launch.
 * The zskr.cn decode-optimisation article on Qwen3-27B, section 3.3
 * ("第三板斧"), merges the Q, K and V matmuls into one operator to save
 * launches, and the single-RTX-PRO-6000 Qwen3.8-27B post counts about 176
 * launches per decode step. A single launch also streams the problems'
 * weights back to back, with no ramp-up or tail between them.
 * (Projections that share their input can also be concatenated along N
 * into one ordinary call: weight rows of each part must start on a
 * 128-row block boundary so that the scale blocks do not straddle parts.)
 *
 * `problems` is a HOST array of `count` entries (0 <= count <= 16), read
 * during the call only. Each entry follows the rules of the single call
 * (pointers, alignment, K % 128 == 0); entries with M == 0 or N == 0 are
 * skipped. Problems must not write overlapping outputs. Errors: the first
 * invalid entry's status, before anything is launched; FP8ACT_ERR_SHAPE for
 * count < 0 or count > 16; FP8ACT_ERR_NULL for problems == NULL with
 * count > 0.
 */
typedef struct {
    const void* x_bf16; /* [M, K] bf16 in           */
    void* q_e4m3;       /* [M, K] E4M3 codes out    */
    float* sa;          /* [M, K/128] fp32 scales out */
    int M, K;
} fp8act_quant_problem;

typedef struct {
    const void* q_e4m3; /* [M, K] activation codes               */
    const float* sa;    /* [M, K/128] activation scales          */
    const void* w_e4m3; /* [N, K] weight codes                   */
    const float* sw;    /* [ceil(N/128), K/128] weight scales    */
    void* out;          /* [M, N] bf16 (fp32 for the _f32 call)  */
    int M, N, K;
} fp8act_gemm_problem;

/* fp8_act_quant over every problem, one launch. Bit-exact with it. */
FP8ACT_API int fp8_act_quant_grouped(const fp8act_quant_problem* problems, int count, void* stream);

/*
 * fp8_block_gemm over every problem (concatenated projections such as QKV,
 * or several layers' independent problems; the zskr.cn Qwen3-27B decode
 * article, section 3.3, fuses such projections). The problems with M <= 16
 * share one launch of the weight-streaming kernel (largest weights first).
 * Those with 16 < M <= 128 share one persistent launch of the tcgen05 tile
 * kernel per 8 problems when their 128-row weight tiles at least fill the
 * SMs, those with M > 128 one per 8 problems when their 256-row tiles fill
 * two waves (the tiles of all problems dealt evenly over the CTAs, K never
 * split); a chunk with fewer tiles runs one tile-kernel launch per problem.
 * All on the same stream; the results equal fp8_block_gemm's within its
 * tolerance.
 */
FP8ACT_API int fp8_block_gemm_grouped(const fp8act_gemm_problem* problems, int count, void* stream);
FP8ACT_API int fp8_block_gemm_grouped_f32(const fp8act_gemm_problem* problems, int count, void* stream);

/* A static English description of a status code (never NULL). */
FP8ACT_API const char* fp8act_strerror(int status);

/*
 * Synchronises `stream` and reports whether any kernel of this library on the
 * current device gave up a bounded wait since the last call (FP8ACT_ERR_TIMEOUT),
 * then clears the flag. The flag is one word per device, shared by every
 * stream: a timeout in a kernel on another stream is reported here too (and
 * cleared), and work still running on other streams may set it after the
 * call returns. Returns FP8ACT_ERR_CUDA if the stream itself failed.
 * Not capturable (it synchronises); meant for tests and health checks.
 */
FP8ACT_API int fp8act_check_status(void* stream);

/*
 * Test hook for the failure path of the tcgen05 kernels (M > 16). Every wait
 * of those kernels on a barrier that another role completes is bounded by
 * wall time (2 s by default); on expiry the CTA stops issuing work, waits for
 * the copies and MMAs it has already issued, frees its tensor memory, leaves,
 * and fp8act_check_status() reports FP8ACT_ERR_TIMEOUT.
 *   limit_ns            bound of those waits for launches issued after this
 *                       call; a negative value restores the 2 s default
 *   withhold_first_load non-zero: every CTA of those launches skips its first
 *                       operand copy, so that its first wait runs out
 *                       (the GEMM's output is then undefined)
 * Process-wide; not for production use (a CUDA graph captured meanwhile
 * keeps the values it was captured with). Always returns FP8ACT_OK.
 */
FP8ACT_API int fp8act_set_wait_limit(long long limit_ns, int withhold_first_load);

/*
 * Diagnostic: the floor of a weight stream. Reads `bytes` bytes of device
 * memory at `src` once, one CTA per SM streaming a contiguous share through a
 * ring of 32 KB TMA bulk copies, launched exactly like the GEMMs above
 * (programmatic dependent launch: the reads start before the previous kernel
 * on the stream has finished), and XORs a fold of the data into *sink. Its
 * waits are bounded like the tcgen05 kernels' (fp8act_check_status). A chain of these calls over buffers the size
 * of a layer's weights times the plain streaming read the GEMM's weight
 * stream is compared against. The section "算子优化" of the smartx.com
 * Qwen3.8-27B post puts the decode step's weight-reading GEMMs "near the
 * bandwidth lower bound"; this call measures that bound on the device.
 *   src   16-byte aligned device pointer; bytes a multiple of 16
 *   sink  4-byte aligned device word (read-modify-written)
 * Errors: FP8ACT_ERR_NULL, FP8ACT_ERR_ALIGN (also for bytes % 16 != 0),
 * FP8ACT_ERR_DEVICE, FP8ACT_ERR_LAUNCH.
 */
FP8ACT_API int fp8act_stream_read(const void* src, size_t bytes, unsigned int* sink, void* stream);

/* Library version, major * 10000 + minor * 100 + patch. */
FP8ACT_API int fp8act_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8ACT_H */
