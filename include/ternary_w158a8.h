/*
 * ternary_w158a8.h -- C ABI of libtw.so: the W1.58A8 ternary-weight product
 * (2-bit packed weights in {-1, 0, +1} times int8 activations) on one NVIDIA
 * B300 (sm_103a).
 *
 * Sources (web pages on ternary-weight LLM inference, cited by title and section):
 *   "1bit-systems：在AMD Strix Halo上实现纯Rust本地三值权重LLM推理"
 *       section 三值量化 (weights take only -1, 0, +1; 1.58 bit each),
 *       section 技术架构 (hand-written ternary GEMV and RMSNorm kernels),
 *       section 性能实测 (the GEMV is bound by memory bandwidth),
 *       section 系统组件全景 (a thin FFI boundary between the host runtime and the kernels).
 *   "BitNet-rs：Rust实现的高效1比特大语言模型推理引擎", section 技术实现细节
 *       (activations are quantised to 8 bit).
 *   bitnet.cpp CPU tutorial (m.qwbw.cn/news/64613), section 1.1 (ternary weights
 *       stored 2-bit aligned; the product needs only a sign check and an add),
 *       section 3.2 (conversion absmean-quantises all weights onto the ternary set).
 *   "BitNet 1 位 LLM 独立推理引擎：位串行 GEMM 内核与 LUT 优化工程实践", 正文
 *       paragraph 4 (I2_S, the plain 2-bit weight format).
 *   "1-bit 大模型官方推理框架：低显存低功耗 LLM 部署方案", FAQ 2 (weights are
 *       restored to a wider type for accumulation).
 *
 * Definitions used throughout (the pages give no formulas; these are the readings):
 *   absmean   gamma = (float)(S / (N*K)), S = exact sum of |W| rounded once to double.
 *   ternary   t = clamp(round_half_even(fl32(W / gamma)), -1, 1); gamma == 0 -> t = 0.
 *   packing   byte b of row n holds (t[n][4b+j] + 1) in bits 2j..2j+1, j = 0..3
 *             (code 0 = -1, 1 = 0, 2 = +1; 3 never written); rows are contiguous,
 *             K/4 bytes each.
 *   act quant per token m: a = max_k |x[m][k]|; x_q = clamp(round_half_even(
 *             fl32(fl32(x * 127) / a)), -128, 127); s_x[m] = a; a == 0 -> x_q = 0, s_x = 0;
 *             x_sum[m] = sum_k x_q[m][k].
 *   RMSNorm   r = exact sum of x^2 rounded once to double; ms = (float)(r / K);
 *             inv = 1 / sqrtf(ms + eps) (IEEE fp32); u = fl32(fl32(x * inv) * g[k]);
 *             then the activation quantisation of u.
 *   product   acc[m][n] = sum_k t[n][k] * x_q[m][k], exact in int32;
 *             y[m][n] = acc * gamma * s_x[m] / 127 in fp32 (within 1e-6 relative of
 *             the value computed in double).
 *
 * Conventions for every call:
 *   - All data pointers are DEVICE pointers owned by the caller (cudaMalloc'd or
 *     managed memory); the library allocates nothing and never synchronises
 *     (tw_device_status excepted).
 *   - The quantisation and product calls are launched with programmatic dependent
 *     launch: a kernel of this library may start while the kernel enqueued just before
 *     it on `stream` is still running, if that kernel lets its dependents start early
 *     (griddepcontrol.launch_dependents: this library's quantisation and product
 *     kernels do; its packing kernels and ordinary kernels do not).  Before that kernel
 *     has finished it reads only its parameters -- the packed weights, w_scale and the
 *     RMSNorm gain -- never the activations, and writes nothing.  So do not let the
 *     kernel just before a product call write that call's weights, scale or gain while
 *     allowing early starts (weights packed at load time are always fine).
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and runs
 *     asynchronously; results are valid once the stream reaches that point.
 *   - Arguments are checked on the host before anything is enqueued: a failed
 *     check returns its status and enqueues nothing.  A failed launch returns
 *     TW_ERR_CUDA.  No call aborts, throws or prints.
 *   - W is [N][K] row-major fp32 (out x in), x is [M][K] row-major, y is [M][N].
 *   - Inputs must be finite; results for NaN or infinite inputs are unspecified
 *     (no out-of-range memory access is made for them).
 *   - Calls are thread-safe; calls that share output buffers on different streams
 *     race on those buffers like any CUDA work.
 */
#ifndef TERNARY_W158A8_H
#define TERNARY_W158A8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define TW_API __declspec(dllexport)
#else
#define TW_API __attribute__((visibility("default")))
#endif

/* Same type as cudaStream_t, declared here so the header needs no CUDA include. */
typedef struct CUstream_st *tw_stream_t;

typedef enum {
  TW_OK = 0,
  TW_ERR_NULL = 1,           /* a required pointer is NULL */
  TW_ERR_SHAPE = 2,          /* M, N or K out of range, K % 4 != 0, or size overflow */
  TW_ERR_ALIGN = 3,          /* a pointer lacks the alignment stated for it */
  TW_ERR_NOT_DEVICE_PTR = 4, /* a pointer is not device-accessible memory */
  TW_ERR_CUDA = 5,           /* the CUDA runtime reported an error (launch or query) */
  TW_ERR_UNSUPPORTED = 6,    /* no sm_103a device, or a case this build does not handle */
  TW_ERR_TIMEOUT = 7,        /* a bounded device-side wait gave up */
  TW_ERR_WORKSPACE = 8       /* workspace missing or smaller than tw_pack_workspace_bytes() */
} tw_status;

/* Human-readable name of a status code (static string, never NULL). */
TW_API const char *tw_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
TW_API int tw_version(void);

/* Upper bounds accepted by the calls below. */
#define TW_MAX_K 65532            /* K <= 65532 and K % 4 == 0 */
#define TW_MAX_NK (1LL << 40)     /* N * K < 2^40 */
#define TW_GEMV_MAX_M 16          /* tw_ternary_gemv: 1 <= M <= 16 */
#define TW_QUANT_GEMV_MAX_M 4     /* tw_quant_gemv: 1 <= M <= 4 */

/*
 * Workspace (bytes) that tw_pack_ternary needs for an N x K tensor: an exact
 * 256-bucket histogram of |W| plus a completion counter.  Returns 0 for shapes
 * tw_pack_ternary would reject.
 */
TW_API size_t tw_pack_workspace_bytes(int64_t N, int64_t K);

/*
 * Absmean ternarisation and 2-bit packing of one weight tensor
 * (bitnet.cpp tutorial section 3.2; I2_S 2-bit format, "BitNet 1 位 LLM 独立推理引擎" 正文 para 4).
 *   W          [N][K] fp32, 16-byte aligned.
 *   packed     [N][K/4] uint8 output, 4-byte aligned.
 *   w_scale    one fp32 output: gamma.
 *   workspace  device scratch of at least tw_pack_workspace_bytes(N, K) bytes,
 *              8-byte aligned; its contents on entry do not matter (it is cleared
 *              on `stream`); it must not be used by other work until this call's
 *              work on `stream` has finished.
 * Requires 1 <= N, 4 <= K <= TW_MAX_K, K % 4 == 0, N*K < TW_MAX_NK.
 * gamma is the same bit pattern whatever the launch configuration: the sum of
 * |W| is accumulated exactly before its single rounding.
 */
TW_API tw_status tw_pack_ternary(const float *W, int64_t N, int64_t K, uint8_t *packed,
                                 float *w_scale, void *workspace, size_t ws_bytes,
                                 tw_stream_t stream);

/*
 * tw_pack_ternary without a workspace argument, for callers that cannot allocate
 * device memory at the point of the call: a plug-in running inside a host
 * framework that owns every device allocation, a service whose memory pools are
 * fixed at start-up, or a loop that must not allocate after initialisation.  The
 * pages have no counterpart of this call; it is a convenience of this library.
 *   Arguments, requirements, results and errors as tw_pack_ternary (minus the
 *   workspace), so N*K < TW_MAX_NK is the size limit (TW_ERR_SHAPE beyond it).
 *   Scratch: a 2304-byte array in the library's device memory (a file-scope
 *   __device__ variable), which every GPU that loads the library holds until the
 *   process exits.  The call allocates nothing, frees nothing and calls no
 *   allocating routine; it clears the scratch on `stream` before use.
 *   Every call looks up the scratch address afresh (cudaGetSymbolAddress, in the
 *   current device's current context), so the call stays correct after
 *   cudaDeviceReset or with another driver context made current; nothing from an
 *   earlier call is reused.  The first call in a context loads the library's device
 *   code there; make that first call before any stream capture.
 *   All calls share the one scratch array per device: calls whose work overlaps on
 *   the GPU (different streams, or other threads) race on it and may produce a wrong
 *   w_scale.  Serialise them, e.g. on one stream.
 */
TW_API tw_status tw_pack_ternary_noalloc(const float *W, int64_t N, int64_t K, uint8_t *packed,
                                         float *w_scale, tw_stream_t stream);

/*
 * Per-token absmax int8 activation quantisation ("BitNet-rs" page, 技术实现细节).
 *   x      [M][K] fp32, 16-byte aligned.
 *   x_q    [M][K] int8 output, 4-byte aligned.
 *   s_x    [M] fp32 output: max|x| per token (the dequantisation uses s_x / 127).
 *   x_sum  [M] int32 output (sum of x_q per token), or NULL.
 * Requires 1 <= M <= 2^20, 4 <= K <= TW_MAX_K, K % 4 == 0.
 * One CTA per token; for 2 to 16 tokens with K >= 6144, each token is shared by a thread-block
 * cluster of 2, 4 or 8 CTAs (K < 8192, < 16384, above) that exchange their chunks' partial
 * results through distributed shared memory (the same bits).  Launched with programmatic
 * dependent launch; x is read only after the previous kernel on `stream` has finished.
 */
TW_API tw_status tw_quant_act(const float *x, int64_t M, int64_t K, int8_t *x_q, float *s_x,
                              int32_t *x_sum, tw_stream_t stream);

/*
 * RMSNorm followed by the quantisation above, in one kernel ("1bit-systems" page,
 * 技术架构: an RMSNorm kernel feeds the ternary GEMV).
 *   g      [K] fp32 gain, 16-byte aligned.   eps: added to the mean square.
 *   other arguments as tw_quant_act.  The mean square is exact up to its one
 *   rounding (see the definitions above), so x_q is independent of launch shape.
 */
TW_API tw_status tw_rmsnorm_quant_act(const float *x, const float *g, float eps, int64_t M,
                                      int64_t K, int8_t *x_q, float *s_x, int32_t *x_sum,
                                      tw_stream_t stream);

/*
 * Ternary matrix-vector product for a small token batch (bitnet.cpp tutorial
 * section 1.1: a sign check and an add per weight; "1bit-systems" page 性能实测:
 * bound by streaming the packed weights).
 *   packed   [N][K/4] uint8 from tw_pack_ternary.   w_scale: device pointer to gamma.
 *   x_q      [M][K] int8.   s_x: [M] fp32.
 *   x_sum    [M] int32 sums of x_q per token, or NULL (then computed in the kernel);
 *            when given it must equal the true sums.
 *   y        [M][N] fp32 output.
 *   acc_out  [M][N] int32 output of the exact accumulators, or NULL.
 * Requires 1 <= M <= TW_GEMV_MAX_M, N >= 1, 4 <= K <= TW_MAX_K, K % 4 == 0.  The fast
 * paths need K % 64 == 0 and packed and x_q 16-byte aligned: up to 4 tokens the
 * streaming kernel (integer dp4a), from 5 to 16 -- and from 3 for rows of at most 8192
 * weights that one CTA block per SM holds -- the tensor cores through mma.sync with f16
 * operands and fp32 accumulation, exact (the 2-bit codes enter as f16 bit patterns
 * c 4^s 2^-24, the activations scaled by 4^-s; every partial sum is a multiple of 2^-24
 * below 1).  Other cases take a slower exact path (dp4a).
 */
TW_API tw_status tw_ternary_gemv(const uint8_t *packed, const float *w_scale, const int8_t *x_q,
                                 const float *s_x, const int32_t *x_sum, int64_t M, int64_t N,
                                 int64_t K, float *y, int32_t *acc_out, tw_stream_t stream);

/*
 * Decode step in one launch: per-token activation quantisation (after RMSNorm when
 * g != NULL) fused in front of the ternary GEMV -- the RMSNorm kernel feeding the
 * ternary GEMV of the "1bit-systems" page (技术架构), with the int8 quantisation of
 * the "BitNet-rs" page (技术实现细节).  Results are bit-identical to
 * tw_rmsnorm_quant_act / tw_quant_act followed by tw_ternary_gemv.
 *   x        [M][K] fp32, 16-byte aligned.   g: [K] fp32 gain or NULL (no RMSNorm).
 *   packed   [N][K/4] uint8, 16-byte aligned.   w_scale: device pointer to gamma.
 *   y        [M][N] fp32 output.
 *   x_q_out  [M][K] int8, s_x_out [M] fp32, x_sum_out [M] int32: optional outputs of
 *            the quantised activations (NULL to skip); x_q_out 16-byte aligned.
 *   acc_out  [M][N] int32 accumulators, or NULL.
 * Requires 1 <= M <= TW_QUANT_GEMV_MAX_M, N >= 1, K % 64 == 0, 64 <= K <= TW_MAX_K;
 * TW_ERR_UNSUPPORTED when the shape does not fit the kernel's shared memory.
 * Launched with programmatic dependent launch: the kernel starts loading
 * `packed` into registers before the previous kernel on `stream` has finished,
 * and reads x (and writes every output) only after it has (x is only prefetched
 * into the coherent L2 before that point).  So the packed weights must not be
 * written by the kernel enqueued immediately before this call on `stream`
 * (weights packed at load time, with any later synchronisation or any other
 * kernel in between, are fine).  The same holds for w_scale and the RMSNorm gain
 * g, which are also read before that point.
 * From K = 12288 (8192 with RMSNorm), when more than one CTA runs (rows that the one-token kernel's shared
 * memory does not hold), the CTAs are launched in thread-block clusters of 4 (2 where too
 * few clusters of 4 can be resident) and each CTA quantises only its share of K, exchanging
 * the partial statistics and the quantised groups through distributed shared memory; the
 * results are the same bits.
 */
TW_API tw_status tw_quant_gemv(const float *x, const float *g, float eps, const uint8_t *packed,
                               const float *w_scale, int64_t M, int64_t N, int64_t K, float *y,
                               int8_t *x_q_out, float *s_x_out, int32_t *x_sum_out, int32_t *acc_out,
                               tw_stream_t stream);

/*
 * Device scratch (bytes) that tw_ternary_gemm / tw_ternary_matmul can use for an M x K
 * activation block: a bf16 copy of x_q in the tensor cores' K order.  0 for shapes the
 * calls would reject.
 */
TW_API size_t tw_gemm_workspace_bytes(int64_t M, int64_t K);

/*
 * The same product for larger token batches on the tensor cores ("1-bit 大模型官方推理框架"
 * page, FAQ 2: ternary weights restored to a wider type for the accumulation).
 * Weights are unpacked to bf16 {-1, 0, +1} and activations to bf16 integers in
 * shared memory; tcgen05.mma accumulates in fp32 in tensor memory, exact because
 * every partial sum is an integer below 2^24 (|acc| <= 128 * K).
 * Arguments as tw_ternary_gemv; M >= 1 (any size), K % 16 == 0, packed and x_q
 * 16-byte aligned (other K: TW_ERR_SHAPE).
 *   workspace  NULL, or device scratch of at least tw_gemm_workspace_bytes(M, K) bytes,
 *              256-byte aligned (TW_ERR_WORKSPACE / TW_ERR_ALIGN otherwise).  With it, and
 *              K % 64 == 0, the activations are widened once per call into the scratch
 *              and the tensor-memory-access unit loads them already in the operand
 *              layout; without it every CTA widens its own activation tiles (slower).
 *              Its contents on entry do not matter; it must not be used by other work
 *              until this call's work on `stream` has finished.
 * Tiles: up to 128 tokens (with the workspace) x 256 weight rows, the tokens on the
 * MMA's M side; otherwise 128 weight rows x up to 256 tokens.  K is split over a
 * thread-block cluster (up to 8 CTAs, partial sums combined through distributed shared
 * memory) when the tile grid alone would leave SMs idle.  With the workspace the GEMM
 * kernel is launched with programmatic dependent launch behind the widening kernel (its
 * weight fetches overlap that kernel; everything enqueued before this call has
 * finished by then, so no extra condition applies to the caller).
 */
TW_API tw_status tw_ternary_gemm(const uint8_t *packed, const float *w_scale, const int8_t *x_q,
                                 const float *s_x, const int32_t *x_sum, int64_t M, int64_t N,
                                 int64_t K, float *y, int32_t *acc_out, void *workspace,
                                 size_t ws_bytes, tw_stream_t stream);

/*
 * The product for any M: tw_ternary_gemv below the measured crossover (M <= 16; M <= 11
 * for matrices of 2^24 weights or more with K > 16384, or with N < 4096 and K >= 6912, when
 * a large enough workspace is given, K % 64 == 0),
 * tw_ternary_gemm above it (when K % 16 == 0 and packed / x_q are 16-byte aligned; an
 * exact CUDA-core kernel otherwise).  Arguments as tw_ternary_gemm; the workspace is
 * used only on the tensor-core path and may be NULL.
 */
TW_API tw_status tw_ternary_matmul(const uint8_t *packed, const float *w_scale, const int8_t *x_q,
                                   const float *s_x, const int32_t *x_sum, int64_t M, int64_t N,
                                   int64_t K, float *y, int32_t *acc_out, void *workspace,
                                   size_t ws_bytes, tw_stream_t stream);

/*
 * Fused epilogues for one decode token ("1-bit 大模型官方推理框架：低显存低功耗 LLM 部署方案",
 * its summary on kernel fusion and FAQ 2 on how the dequantised values are used): the
 * residual add after a layer's output projections, and the partial statistics of the
 * following RMSNorm, formed where the GEMV writes its outputs, so that the next quantisation
 * starts from them instead of reducing over its input first.
 *
 * Workspace (bytes) that carries those statistics from tw_quant_gemv_residual to
 * tw_quant_gemv_stats: one 16-byte partial per CTA of the writing launch.  Its contents on
 * entry to tw_quant_gemv_residual do not matter.
 */
TW_API size_t tw_epilogue_workspace_bytes(void);

/*
 * tw_quant_gemv for one token (M = 1; RMSNorm when g != NULL) with the residual epilogue:
 *   y       = acc * gamma * s_x / 127 as the definitions state it (in double, one rounding
 *             to fp32: bit-identical to that expression), written when y != NULL;
 *   h_out   = fl32(h + y) for each of the N outputs (h_out may be h);
 *   workspace: the partial statistics of h_out for the RMSNorm with gain g_next that reads
 *             it next (tw_quant_gemv_stats): per CTA a float-float sum of squares of its
 *             outputs and the output with the largest fl(|h_out g_next|).
 *   x, g, eps, packed, w_scale, acc_out: as tw_quant_gemv.   h, h_out: [N] fp32, 16-byte
 *   aligned.   g_next: [N] fp32.   workspace: tw_epilogue_workspace_bytes() bytes, 16-byte
 *   aligned.
 * Requires 64 <= N <= 8192 and N % 64 == 0, 64 <= K <= 8192 and K % 64 == 0;
 * TW_ERR_UNSUPPORTED when the one-token kernel's shared memory does not hold the CTA's
 * share of the weights.  Launched with programmatic dependent launch as tw_quant_gemv (g_next
 * is also read before the previous kernel has finished).
 */
TW_API tw_status tw_quant_gemv_residual(const float *x, const float *g, float eps, const uint8_t *packed,
                                        const float *w_scale, int64_t N, int64_t K, const float *h,
                                        float *h_out, const float *g_next, float *y, int32_t *acc_out,
                                        void *workspace, size_t ws_bytes, tw_stream_t stream);

/*
 * tw_quant_gemv for one token with RMSNorm, its statistics taken from the workspace that the
 * tw_quant_gemv_residual which wrote x left: every CTA folds the partials (float-float sum
 * of squares; 1 / rms decided exactly as the RMSNorm definition states, from x itself when
 * the sum cannot decide the rounding) and takes the candidate scale from the output with the
 * largest fl(|x g|); the quantisation checks every |u| against it and takes the true largest
 * |u| when one exceeds it.  The results equal tw_quant_gemv(x, g, eps, ...) exactly.
 *   x: [K] fp32 (the h_out of that call), 16-byte aligned.   g: [K] gain (its g_next).
 *   workspace: as that call left it (for x with K = its N), 16-byte aligned.
 *   Other arguments as tw_quant_gemv.
 * Requires N >= 1, 64 <= K <= 8192, K % 64 == 0; TW_ERR_UNSUPPORTED as above.  The workspace
 * is read after the previous kernel on `stream` has finished (programmatic dependent launch).
 */
TW_API tw_status tw_quant_gemv_stats(const float *x, const float *g, float eps, const void *workspace,
                                     const uint8_t *packed, const float *w_scale, int64_t N, int64_t K,
                                     float *y, int8_t *x_q_out, float *s_x_out, int32_t *x_sum_out,
                                     int32_t *acc_out, tw_stream_t stream);

/*
 * The denser weight layout: five trits per byte, 1.6 bits per weight ("BitNet 1 位 LLM
 * 独立推理引擎：位串行 GEMM 内核与 LUT 优化工程实践", 正文 paragraph 3: TL2 packs several
 * ternary weights into one small table index so that fewer weight bytes are loaded; the
 * "1bit-systems" page, 性能实测: the bandwidth-bound GEMV only gets faster by reading
 * fewer bytes).  The pages fix no byte layout; this library's reading:
 *   a row takes RB = 16 * ceil(K / 80) bytes (tw_t5_row_bytes(K); ceil(K / 5) rounded up
 *   to whole 16-byte chunks, exactly K / 5 when K % 80 == 0); byte i of a row holds the
 *   weights 4i, 4i+1, 4i+2, 4i+3 as base-3 digits 0..3 and the weight 4 RB + i as digit 4,
 *   each digit t + 1 (byte = sum_j digit_j 3^j <= 242); weights at k >= K are 0.
 * Returns 0 for K the calls below reject.
 */
TW_API size_t tw_t5_row_bytes(int64_t K);

/*
 * Absmean ternarisation (the same gamma and t as tw_pack_ternary) stored five trits per
 * byte.
 *   W          [N][K] fp32, 16-byte aligned.
 *   packed5    [N][tw_t5_row_bytes(K)] uint8 output, 16-byte aligned.
 *   w_scale, workspace, ws_bytes: as tw_pack_ternary (the same workspace size).
 * Requires 1 <= N, 4 <= K <= TW_MAX_K, K % 4 == 0, N*K < TW_MAX_NK.
 */
TW_API tw_status tw_pack_ternary_t5(const float *W, int64_t N, int64_t K, uint8_t *packed5,
                                    float *w_scale, void *workspace, size_t ws_bytes,
                                    tw_stream_t stream);

/*
 * The ternary GEMV over rows stored five trits per byte: the same acc and y as
 * tw_ternary_gemv on the same weights (exact int32 accumulators).  A 256-entry table in
 * shared memory turns each byte into its five weights.
 *   packed5  [N][tw_t5_row_bytes(K)] uint8 from tw_pack_ternary_t5, 16-byte aligned.
 *   x_q      [M][K] int8, 16-byte aligned.   w_scale, s_x, y, acc_out: as tw_ternary_gemv.
 * Requires 1 <= M <= 2, N >= 1, 16 <= K <= 40960, K % 16 == 0, N*K < TW_MAX_NK.  Bytes
 * above 242 never come out of tw_pack_ternary_t5; the kernel reads them as zero weights.
 * Launched with programmatic dependent launch: it builds its table before the previous
 * kernel on `stream` has finished and reads x_q and s_x only after it has.
 */
TW_API tw_status tw_ternary_gemv_t5(const uint8_t *packed5, const float *w_scale, const int8_t *x_q,
                                    const float *s_x, int64_t M, int64_t N, int64_t K, float *y,
                                    int32_t *acc_out, tw_stream_t stream);

/*
 * Reads and clears the library's device status word: 0, or TW_ERR_TIMEOUT when a
 * kernel gave up a bounded wait (it then left its outputs unwritten).  Synchronises
 * the current device; meant for diagnostics after a failed step, not the hot path.
 */
TW_API tw_status tw_device_status(int32_t *status);

/*
 * Test switch for the failure handling of the tensor-core GEMM (diagnostics; synchronises
 * the current device).  With on != 0, every tw_ternary_gemm launch that follows on this
 * device starts with its abort flag raised, as if one of its bounded waits had given up
 * before it issued any copy or product: it releases its tensor memory, waits for nothing
 * that is not in flight, writes no output and records TW_ERR_TIMEOUT for tw_device_status.
 * on = 0 restores normal operation.  No other call is affected.
 */
TW_API tw_status tw_debug_gemm_abort(int on);

#ifdef __cplusplus
}
#endif

#endif /* TERNARY_W158A8_H */
