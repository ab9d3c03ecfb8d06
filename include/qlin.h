/*
 * qlin -- quantized linear layers Y = X . deq(W)^T for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libqlin.so.  Two variants of the linear layer of LLM serving:
 *
 *  W4A16  INT4 weights, q = clamp(round(w/s) + z, 0, 15), one FP16 scale s
 *         and one 4-bit zero-point z per group of G = 128 weights along K
 *         (4.125 bits/weight for codes + scales; G = 32 and 64 are also
 *         taken, at 4.5 and 4.25 bits); BF16 activations; the
 *         dequantisation x_hat = s (q - z) happens inside the GEMM kernel.
 *  W8A8   FP8 E4M3 weights with one FP32 scale for the whole tensor and E4M3
 *         activations with one FP32 scale per token (row), both "current"
 *         scales amax / 448; FP32 accumulation, BF16 output.
 *
 * Sources (web pages, cited by title and section):
 *  [LP] "Low-precision LLM inference: FP8/INT8/INT4/FP4 kernels and
 *        calibration" (blog.ruahverce.com): S1 precision manifest, S2 uniform
 *        integer quantisation, S3 symmetric/asymmetric, S4 scale granularity,
 *        S5 effective bits, S7 FP8 formats, S8 FP8 scale recipes, S11 W4A16
 *        pipeline, S22 accumulator precision, S23 fused kernels, S24 kernel
 *        eligibility checklist, S25 padding, S28 CUDA graphs and dynamic scale,
 *        S31 artifact manifest (fail-closed fallback policy).
 *  [TP] "Quantization throughput by batch size: why W4A16 is overtaken by
 *        W8A8" (hrletsgo.me): small batches are bound by weight bytes, large
 *        batches by tensor-core throughput.
 *
 * Conventions for every call
 *  - X is [M][K] row-major, W is [N][K] row-major (the nn.Linear layout),
 *    Y is [M][N] row-major.  BF16/FP16 buffers hold raw 16-bit patterns.
 *  - Every pointer is a DEVICE pointer owned by the caller, 16-byte aligned;
 *    `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - Every call is asynchronous on `stream`, allocates nothing, never reads a
 *    device value on the host, and can be captured in a CUDA graph ([LP] S28).
 *  - Arguments are validated before anything is launched; a call that returns
 *    an error launched nothing and wrote nothing.  There is no fallback path,
 *    no CPU path and no silent padding ([LP] S24, S25, S31 "fail-closed").
 *  - Errors found by a kernel while it runs (a scale that overflows FP16, a
 *    pipeline wait that gave up) are recorded in a per-device error word read
 *    by qlin_get_device_error().
 *  - M = 0 is a valid empty call: it returns QLIN_OK and launches nothing.
 *
 * Eligibility ([LP] S24): device sm_103 (compute capability 10.3);
 * G in {32, 64, 128}, or G == K for per-channel scales (one group spanning
 * the row, [LP] S4 "per-channel"); the CUDA-core GEMV that serves small M
 * when K % 256 != 0, qlin_w4a16_gemv_noalloc and qlin_w4a8_gemm take G = 128
 * only; N % 128 == 0; K % 128 == 0;
 * 1 <= N, K; 0 <= M <= 2^24, and M <= 262140 (4 x 65535 token blocks of its
 * launch grid) wherever a call runs the CUDA-core GEMV (QLIN_PATH_GEMV with
 * K % 256 != 0, and qlin_w4a16_gemv_noalloc in that case); larger M returns
 * QLIN_ERR_UNSUPPORTED_SHAPE there.
 */
#ifndef QLIN_H
#define QLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QLIN_OK = 0,
  QLIN_ERR_INVALID_VALUE = 1,      /* null pointer, bad flag, bad value found on device */
  QLIN_ERR_UNSUPPORTED_SHAPE = 2,  /* M/N/K/G outside the eligibility rules above */
  QLIN_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned */
  QLIN_ERR_WORKSPACE_TOO_SMALL = 4,
  QLIN_ERR_ARCH = 5,               /* current device is not compute capability 10.3 */
  QLIN_ERR_CUDA = 6,               /* a CUDA runtime call or a launch failed */
  QLIN_ERR_TIMEOUT = 7             /* a kernel's bounded pipeline wait gave up */
} qlin_status_t;

/* Version of the packed INT4 tile layout written by qlin_pack_w4 ([LP] S31
 * "kernel_pack_format").  A consumer must reject any other version. */
#define QLIN_PACK_FORMAT_VERSION 2

/* Operation ids for qlin_workspace_size. */
#define QLIN_OP_W4A16_GEMM 1
#define QLIN_OP_W8A8_GEMM 2
#define QLIN_OP_QUANT_W_FP8 3
#define QLIN_OP_W8A8_BLOCK_GEMM 4
#define QLIN_OP_MXFP8_GEMM 5
#define QLIN_OP_W4A8_GEMM 6
#define QLIN_OP_MXFP4_GEMM 7
#define QLIN_OP_NVFP4_GEMM 8

/* Activation of the fused output epilogue (qlin_*_gemm_fused, every GEMM). */
#define QLIN_ACT_NONE 0
#define QLIN_ACT_RELU 1 /* max(v, 0)                                   */
#define QLIN_ACT_SILU 2 /* v / (1 + exp(-v))                           */
#define QLIN_ACT_GELU 3 /* v * Phi(v) = 0.5 v (1 + erf(v / sqrt 2))    */

/* Kernel selection for the *_ex GEMM calls (measurement and ablation). */
#define QLIN_PATH_AUTO 0   /* choose by M (the default of the plain calls) */
#define QLIN_PATH_GEMV 1   /* small-M split-K kernel (see qlin_w4a16_gemm)  */
#define QLIN_PATH_TC 2     /* TMA + tcgen05 tensor-core kernel             */

/* Human-readable name of a status code (static string, never NULL). */
const char* qlin_status_string(qlin_status_t status);

/* QLIN_PACK_FORMAT_VERSION of the library that is loaded. */
int qlin_pack_format_version(void);

/* The cudaError_t (as int) behind the most recent QLIN_ERR_CUDA returned by a
 * call on the calling thread; 0 if there was none.  A call that returns
 * QLIN_ERR_CUDA has also cleared the runtime's last-error state, so a failed
 * launch is not reported again by a later, unrelated call. */
int qlin_last_cuda_error(void);

/* The CUDA runtime's name for an error code (static string, never NULL). */
const char* qlin_cuda_error_name(int code);

/* Byte sizes of the three packed-weight buffers for an [N][K] weight.
 * codes = N*K/2, scales = 2*N*K/G, zeros = N*K/(2G) ([LP] S5: codes + scales
 * give exactly 4 + 16/G bits per weight; the zeros add 4/G). */
qlin_status_t qlin_w4_packed_sizes(int64_t N, int64_t K, int G, size_t* codes, size_t* scales, size_t* zeros);

/* Scratch bytes a call of `op` needs for these sizes (0 if none).  G is the
 * W4A16 quantisation group (checked as qlin_w4a16_gemm checks it) for
 * QLIN_OP_W4A16_GEMM and ignored by the other operations.  The
 * workspace must be zero-filled before its first use with this library and
 * is left zero-filled by every call that completes (split-K counters, the
 * small-M kernel's work-queue word and the partial sums are all cleared by the
 * call that used them), so one workspace may serve calls of any shapes in
 * turn; calls that share one workspace must not overlap in time (use one per
 * stream).  After a call whose kernel reported a device error (see
 * qlin_get_device_error) its contents are undefined: zero it again. */
qlin_status_t qlin_workspace_size(int op, int64_t M, int64_t N, int64_t K, int G, size_t* bytes);

/*
 * Quantise and pack BF16 weights W[N][K] ([LP] S2-S5, run once at load).
 *  Per row n and group g (columns gG .. gG+G-1), in IEEE binary32:
 *   asymmetric (symmetric = 0): lo = min(min w, 0), hi = max(max w, 0),
 *     s = fp16(( hi - lo) / 15), z = clamp(rint(-lo / s), 0, 15),
 *     q = clamp(rint(w / s) + z, 0, 15);
 *   symmetric (symmetric = 1): s = fp16(max|w| / 7), q = clamp(rint(w/s),-8,7)
 *     stored offset-binary as q + 8 with stored zero-point 8 (logical z = 0).
 *   rint rounds half to even; a group whose scale rounds to 0 stores s = 1,
 *   z = 0 (symmetric: 8).  A scale that overflows FP16 sets the device error
 *   word to QLIN_ERR_INVALID_VALUE.
 *  Outputs, in tile layout version 2 (tiles of 128 rows x 64 columns):
 *   codes  (N*K/2 bytes): tile (n/128, k/64) is 4096 bytes at
 *          ((n/128)*(K/64) + k/64) * 4096; in it, half h = (k%64)/32 of row
 *          r = n%128 is the 16 bytes at h*2048 + r*16: four little-endian
 *          32-bit words.  Writing the column within the half as
 *          c = k%32 = 16a + 8b + 2t + e (a, b, e in {0,1}; t in 0..3), column
 *          c is in word t at nibble position p = 2a + b + 4e, i.e. bits
 *          4p..4p+3.  Word t thus holds what lane t of an mma.sync quad needs
 *          for two 16-column k-steps, and the pair (c, c+1) is the two halves
 *          of (word >> 4(2a + b)) & 0x000F000F.
 *   scales (2*N*K/G bytes): FP16 of (n, g) at element
 *          ((n/128)*(K/G) + g) * 128 + n%128.
 *   zeros  (N*K/(2G) bytes): nibble of (n, g) in byte
 *          ((n/128)*(K/G) + g) * 64 + (n%128)/2, low nibble for even n.
 *  Requires G in {32, 64, 128} or G == K (per-channel: K/G = 1 scale and
 *  zero-point per row, found from the row's range over all of K), N % 128 ==
 *  0, K % 128 == 0.
 */
qlin_status_t qlin_pack_w4(const void* W_bf16, int64_t N, int64_t K, int G, int symmetric, void* codes,
                 void* scales_f16, void* zeros_u4, void* stream);

/*
 * W4A16 linear layer ([LP] S11, S23): Y = bf16( sum_k X[m][k] s (q - z) ),
 * accumulated in FP32 ([LP] S22), from the packed buffers of qlin_pack_w4.
 * Kernel choice by M ([LP] S24 "different kernels for small batch and
 * large prefill"): for M <= qlin_gemv_max_m (32) a split-K kernel that
 * unpacks the nibbles in registers and multiplies on the tensor cores with
 * register-level MMA (M <= 32 and K % 256 == 0; a CUDA-core GEMV otherwise on
 * QLIN_PATH_GEMV), above it a TMA + tcgen05 BF16 tensor-core kernel (weights
 * dequantised to BF16 in tensor or shared memory).  Split-K partial sums are reduced in a fixed order, so results
 * are deterministic.  workspace: qlin_workspace_size(QLIN_OP_W4A16_GEMM, ...)
 * bytes (may be NULL when that is 0).
 */
qlin_status_t qlin_w4a16_gemm(const void* X_bf16, const void* codes, const void* scales_f16, const void* zeros_u4,
                    void* Y_bf16, int64_t M, int64_t N, int64_t K, int G, void* workspace, size_t ws_bytes,
                    void* stream);

/* Same, with the kernel path forced (QLIN_PATH_*). */
qlin_status_t qlin_w4a16_gemm_ex(const void* X_bf16, const void* codes, const void* scales_f16, const void* zeros_u4,
                       void* Y_bf16, int64_t M, int64_t N, int64_t K, int G, void* workspace, size_t ws_bytes,
                       int path, void* stream);

/* W4A16 with a fused output epilogue ([LP] S23 "fused epilogue ... write
 * output once", S24 "bias / activation epilogue"):
 *     Y[m][n] = bf16( act( acc[m][n] + bias[n] ) )
 * acc the FP32 result of qlin_w4a16_gemm, bias BF16 [N] (NULL: none, else
 * 16-byte aligned), act one of QLIN_ACT_*; bias and activation are applied in
 * FP32 and Y is rounded once.  Every kernel path applies it where it writes Y
 * (also after a split-K reduction), so no extra pass over Y is made. */
qlin_status_t qlin_w4a16_gemm_fused(const void* X_bf16, const void* codes, const void* scales_f16, const void* zeros_u4,
                          void* Y_bf16, int64_t M, int64_t N, int64_t K, int G, const void* bias_bf16, int act,
                          void* workspace, size_t ws_bytes, int path, void* stream);

/*
 * Per-token FP8 activation quantisation ([LP] S4 per-token, S8 current
 * scaling), one fused kernel: for each row m, amax_m = max_k |X[m][k]|,
 * sx[m] = amax_m / 448 (1 if amax_m = 0), Xq[m][k] = e4m3_rn_satfinite(
 * X[m][k] / sx[m]) with an IEEE binary32 division.  Outputs: Xq [M][K] E4M3
 * bytes, sx [M] FP32.  The scale never leaves the device ([LP] S28).
 */
qlin_status_t qlin_quant_act_fp8(const void* X_bf16, int64_t M, int64_t K, void* Xq_e4m3, float* sx, void* stream);

/*
 * Per-tensor FP8 weight quantisation ([LP] S4 per-tensor, S8), run once at
 * load: sw = amax(W)/448 (1 if 0), Wq = e4m3_rn_satfinite(W / sw).
 * Outputs Wq [N][K] E4M3 bytes and *sw (one FP32, device memory).
 * workspace: qlin_workspace_size(QLIN_OP_QUANT_W_FP8, ...) bytes (holds the
 * grid-wide amax).
 */
qlin_status_t qlin_quant_w_fp8(const void* W_bf16, int64_t N, int64_t K, void* Wq_e4m3, float* sw, void* workspace,
                     size_t ws_bytes, void* stream);

/*
 * W8A8 FP8 linear layer ([LP] S8, S9, S22): Y[m][n] = bf16( acc[m][n] *
 * sx[m] * sw ) with acc = sum_k e4m3(Xq[m][k]) e4m3(Wq[n][k]) in FP32.
 * Kernel choice by M: for M <= qlin_gemv_max_m (16) a split-K kernel on
 * register-level E4M3 MMA (mma.sync m16n8k32, K % 256 == 0; a CUDA-core GEMV
 * otherwise on QLIN_PATH_GEMV), above it TMA + tcgen05 kind::f8f6f4.
 * workspace: qlin_workspace_size(QLIN_OP_W8A8_GEMM, ...) bytes.
 */
qlin_status_t qlin_w8a8_fp8_gemm(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3, const float* sw,
                       void* Y_bf16, int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                       void* stream);

qlin_status_t qlin_w8a8_fp8_gemm_ex(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3, const float* sw,
                          void* Y_bf16, int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                          int path, void* stream);

/* W8A8 with the fused output epilogue of qlin_w4a16_gemm_fused:
 * Y[m][n] = bf16( act( (acc[m][n] * sx[m]) * sw + bias[n] ) ). */
qlin_status_t qlin_w8a8_fp8_gemm_fused(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3, const float* sw,
                             void* Y_bf16, int64_t M, int64_t N, int64_t K, const void* bias_bf16, int act,
                             void* workspace, size_t ws_bytes, int path, void* stream);

/* ---- FP8 block scaling ([LP] S8 "Block Scaling": each block of the tensor
 * has its own scale, x ~ x_fp8 * scale_block, scale_block = amax_block /
 * max_fp8).  The pages leave the block shape and scale type open: here
 * activations use 1 x 128 blocks (one token, 128 columns) and weights 128 x 128
 * blocks, with FP32 scales computed exactly as the per-token recipe does
 * (amax / 448, 1 for an all-zero block; E4M3 RNE with saturation of x / scale,
 * binary32 division). */

/* X [M][K] BF16 -> Xq [M][K] E4M3 and sx [K/128][M] FP32 (block-major: the
 * scales of one K block of all tokens are contiguous).  K % 128 == 0.  sx
 * 4-byte aligned, X and Xq 16-byte aligned.  Asynchronous, no workspace. */
qlin_status_t qlin_quant_act_fp8_blocks(const void* X_bf16, int64_t M, int64_t K, void* Xq_e4m3, float* sx, void* stream);

/* W [N][K] BF16 -> Wq [N][K] E4M3 and sw [N/128][K/128] FP32 (row-block major).
 * N % 128 == 0, K % 128 == 0.  Asynchronous, no workspace. */
qlin_status_t qlin_quant_w_fp8_blocks(const void* W_bf16, int64_t N, int64_t K, void* Wq_e4m3, float* sw, void* stream);

/* Block-scaled W8A8: Y[m][n] = bf16( sum_b sx[b][m] * sw[n/128][b] *
 * sum_{k in block b} Xq[m][k] * Wq[n][k] ), every block's product accumulated
 * in FP32 on the tensor cores and promoted with its two scales into an FP32
 * sum in block order.  Shapes and alignment as qlin_w8a8_fp8_gemm;
 * workspace: qlin_workspace_size(QLIN_OP_W8A8_BLOCK_GEMM, ...) bytes (0 when the
 * K range is not split), zero-filled, left zero-filled.  Deterministic. */
qlin_status_t qlin_w8a8_fp8_block_gemm(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3, const float* sw,
                             void* Y_bf16, int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                             void* stream);

/* Block-scaled FP8 with the fused output epilogue: Y[m][n] = bf16( act(
 * y[m][n] + bias[n] ) ), y the FP32 value qlin_w8a8_fp8_block_gemm rounds;
 * bias and act as in qlin_w4a16_gemm_fused. */
qlin_status_t qlin_w8a8_fp8_block_gemm_fused(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3,
                                             const float* sw, void* Y_bf16, int64_t M, int64_t N, int64_t K,
                                             const void* bias_bf16, int act, void* workspace, size_t ws_bytes,
                                             void* stream);

/*
 * W4A8 linear layer ([LP] S1 precision manifest "W4A8: INT4 weights, INT8/FP8
 * activations -> accumulate FP32 -> output BF16"; S20 QServe W4A8): the packed
 * INT4 weights of qlin_pack_w4 (G = 128) times the per-token E4M3 activations
 * of qlin_quant_act_fp8,
 *     Y[m][n] = bf16( sx[m] * sum_g s[n][g] * sum_{k in g} e4m3(Xq[m][k]) (q[n][k] - z[n][g]) ),
 * the inner sums accumulated in FP32 on the tensor cores (tcgen05
 * kind::f8f6f4; q - z, an integer in [-15, 15], is exact in E4M3) and each
 * group's partial product promoted with its FP16 scale in FP32.
 * Requires G == 128; shapes and alignment as qlin_w4a16_gemm (sx 4-byte
 * aligned); workspace: qlin_workspace_size(QLIN_OP_W4A8_GEMM, ...) bytes (0
 * when the K range is not split), zero-filled, left zero-filled.  Deterministic.
 */
qlin_status_t qlin_w4a8_gemm(const void* Xq_e4m3, const float* sx, const void* codes, const void* scales_f16,
                             const void* zeros_u4, void* Y_bf16, int64_t M, int64_t N, int64_t K, int G,
                             void* workspace, size_t ws_bytes, void* stream);

/* W4A8 with the fused output epilogue of qlin_w4a16_gemm_fused ([LP] S23,
 * S24): Y[m][n] = bf16( act( y[m][n] + bias[n] ) ), y the FP32 value that
 * qlin_w4a8_gemm rounds; bias BF16 [N] (NULL: none, else 16-byte aligned),
 * act one of QLIN_ACT_*.  Everything else as qlin_w4a8_gemm. */
qlin_status_t qlin_w4a8_gemm_fused(const void* Xq_e4m3, const float* sx, const void* codes, const void* scales_f16,
                                   const void* zeros_u4, void* Y_bf16, int64_t M, int64_t N, int64_t K, int G,
                                   const void* bias_bf16, int act, void* workspace, size_t ws_bytes, void* stream);

/* ---- MXFP8 (the OCP Microscaling format that [LP] S10 names; [VQ] S2: the
 * MXFP8 W8A8 path runs on Blackwell only): E4M3 elements in blocks of 32
 * consecutive values along K, each block with one power-of-two scale 2^e
 * stored as an E8M0 byte e + 127.  e = floor(log2 amax) - 8 (8 being the
 * exponent of E4M3's largest normal, 448 = 1.75 x 2^8), clamped to
 * [-127, 127]; an all-zero block takes e = -127; elements are
 * E4M3(v / 2^e), round to nearest even, saturating at +-448.  The product
 * applies both block scales on the tensor cores (tcgen05 kind::mxf8f6f4 with
 * hardware block scaling): no promotion pass.
 *
 * Scale layout ("scale atoms", the form the tensor cores take them in):
 * for a tensor of R rows, ceil(R/128) x (K/128) atoms of 512 bytes, atom
 * (R0, c) at byte ((R0 * (K/128)) + c) * 512 covering rows 128 R0 .. +127
 * and columns 128 c .. +127.  Row r of the atom (r = row % 128) holds the
 * scales of its four 32-column blocks kk = 0..3 in the four bytes
 * 16 (r % 32) + 4 (r / 32) + kk.  Atom rows past R are 0. */

/* Bytes of the scale atoms of an R x K tensor: ceil(R/128) * 128 * K / 32.
 * K % 128 == 0, R >= 0. */
qlin_status_t qlin_mx_scale_bytes(int64_t R, int64_t K, size_t* bytes);

/* Quantise X [R][K] BF16 to MXFP8: codes [R][K] E4M3 (16-byte aligned) and
 * scales in the atom layout above (qlin_mx_scale_bytes bytes, 16-byte aligned).
 * Used for the weights (R = N, once at load) and the activations (R = M, per
 * call).  K % 128 == 0.  Asynchronous, no workspace. */
qlin_status_t qlin_quant_mxfp8(const void* X_bf16, int64_t R, int64_t K, void* codes_e4m3, void* scales_e8m0,
                               void* stream);

/* MXFP8 linear layer: Y[m][n] = bf16( sum_b 2^(xs[m][b]-127) 2^(ws[n][b]-127)
 * sum_{k in block b} e4m3(Xq[m][k]) e4m3(Wq[n][k]) ), b over the 32-column
 * blocks, accumulated in FP32 on the tensor cores.  Xq / xs from
 * qlin_quant_mxfp8 of the activations, Wq / ws of the weights.  Shapes as
 * qlin_w8a8_fp8_gemm (N % 128 == 0, K % 128 == 0); workspace:
 * qlin_workspace_size(QLIN_OP_MXFP8_GEMM, ...) bytes (0 when the K range is
 * not split), zero-filled, left zero-filled.  Deterministic. */
qlin_status_t qlin_mxfp8_gemm(const void* Xq_e4m3, const void* xs_e8m0, const void* Wq_e4m3, const void* ws_e8m0,
                              void* Y_bf16, int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                              void* stream);

/* MXFP8 with the fused output epilogue: Y[m][n] = bf16( act( y[m][n] +
 * bias[n] ) ), y the FP32 value qlin_mxfp8_gemm rounds; bias and act as in
 * qlin_w4a16_gemm_fused.  Everything else as qlin_mxfp8_gemm. */
qlin_status_t qlin_mxfp8_gemm_fused(const void* Xq_e4m3, const void* xs_e8m0, const void* Wq_e4m3,
                                    const void* ws_e8m0, void* Y_bf16, int64_t M, int64_t N, int64_t K,
                                    const void* bias_bf16, int act, void* workspace, size_t ws_bytes, void* stream);

/* ---- FP4 ([LP] S10: the E2M1 element -- 1 sign, 2 exponent and 1 mantissa
 * bit, magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 -- in the two block formats that
 * page tells apart).  Codes are packed two per byte along K, column 2i in the
 * low nibble, so an [R][K] tensor takes R * K / 2 bytes.  Conversion to E2M1
 * rounds to nearest even and saturates at +-6.  K % 256 == 0 in every FP4
 * call; R (and M) need not be a multiple of anything.
 *
 * MXFP4 (the OCP MX specification's FP4 format): blocks of 32 along K share
 * an E8M0 scale 2^e, e = floor(log2 amax) - 2 (2 being the exponent of E2M1's
 * largest normal, 6 = 1.5 x 2^2), clamped to [-127, 127], -127 for an all-zero
 * block; elements E2M1(v / 2^e).  Scales in the MXFP8 atom layout above
 * (qlin_mx_scale_bytes(R, K) bytes).
 *
 * NVFP4 (the vendor's two-level recipe on the same element): one FP32 scale
 * per tensor, sg = amax(|X|) / (6 x 448) (1 when that is 0); blocks of 16
 * along K with an E4M3 scale sb = E4M3(amax_b / (6 sg)) (nearest even,
 * saturating); elements E2M1(v / (sb sg)), each step one binary32 operation;
 * a block whose scale is 0 stores code 0 in every element.  Scales in atoms
 * of four 16-column blocks: for R rows, ceil(R/128) x (K/64) atoms of 512
 * bytes, atom (R0, c) at byte ((R0 * (K/64)) + c) * 512 covering rows
 * 128 R0 .. +127 and columns 64 c .. +63, row r's scales kk = 0..3 at bytes
 * 16 (r % 32) + 4 ((r % 128) / 32) + kk; atom rows past R are 0. */

/* Bytes of the NVFP4 scale atoms of an R x K tensor: ceil(R/128) * 128 * K / 16.
 * K % 256 == 0, R >= 0. */
qlin_status_t qlin_nvfp4_scale_bytes(int64_t R, int64_t K, size_t* bytes);

/* Quantise X [R][K] BF16 to MXFP4: codes [R][K/2] packed E2M1 (16-byte
 * aligned) and scales in the MXFP8 atom layout (qlin_mx_scale_bytes(R, K)
 * bytes, 16-byte aligned).  Weights once at load (R = N), activations per call
 * (R = M).  Asynchronous, no workspace. */
qlin_status_t qlin_quant_mxfp4(const void* X_bf16, int64_t R, int64_t K, void* codes_e2m1, void* scales_e8m0,
                               void* stream);

/* NVFP4 per-tensor scale of the n BF16 values at X (16-byte aligned,
 * n % 8 == 0, n >= 1) into the device float *sg (4-byte aligned): a memset, an
 * amax reduction and a one-thread kernel on `stream`; nothing is copied to the
 * host. */
qlin_status_t qlin_nvfp4_tensor_scale(const void* X_bf16, int64_t n, float* sg, void* stream);

/* Quantise X [R][K] BF16 to NVFP4 with the per-tensor scale at device address
 * sg (read by the kernel, so it may come from qlin_nvfp4_tensor_scale on the
 * same stream): codes [R][K/2] packed E2M1, scales in the NVFP4 atom layout
 * (qlin_nvfp4_scale_bytes(R, K) bytes); all 16-byte aligned.  Asynchronous. */
qlin_status_t qlin_quant_nvfp4(const void* X_bf16, int64_t R, int64_t K, const float* sg, void* codes_e2m1,
                               void* scales_e4m3, void* stream);

/* MXFP4 linear layer: Y[m][n] = bf16( sum_b 2^(xs[m][b]-127) 2^(ws[n][b]-127)
 * sum_{k in block b} e2m1(Xq[m][k]) e2m1(Wq[n][k]) ), b over the 32-column
 * blocks, accumulated in FP32 on the tensor cores (tcgen05 kind::mxf4 with
 * hardware block scaling).  Xq / xs from qlin_quant_mxfp4 of the activations,
 * Wq / ws of the weights.  N % 128 == 0, K % 256 == 0; workspace:
 * qlin_workspace_size(QLIN_OP_MXFP4_GEMM, ...) bytes (0 when the K range is
 * not split), zero-filled, left zero-filled.  Deterministic. */
qlin_status_t qlin_mxfp4_gemm(const void* Xq_e2m1, const void* xs_e8m0, const void* Wq_e2m1, const void* ws_e8m0,
                              void* Y_bf16, int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                              void* stream);

/* MXFP4 with the fused output epilogue (bias and act as in
 * qlin_w4a16_gemm_fused, applied to the FP32 value qlin_mxfp4_gemm rounds). */
qlin_status_t qlin_mxfp4_gemm_fused(const void* Xq_e2m1, const void* xs_e8m0, const void* Wq_e2m1,
                                    const void* ws_e8m0, void* Y_bf16, int64_t M, int64_t N, int64_t K,
                                    const void* bias_bf16, int act, void* workspace, size_t ws_bytes, void* stream);

/* NVFP4 linear layer: Y[m][n] = bf16( sgx sgw sum_b e4m3(xs[m][b]) e4m3(ws[n][b])
 * sum_{k in block b} e2m1(Xq[m][k]) e2m1(Wq[n][k]) ), b over the 16-column
 * blocks; the block scales are applied by the tensor cores (tcgen05
 * kind::mxf4nvf4), the FP32 product sgx * sgw in the epilogue.  sgx / sgw are
 * device pointers to the two per-tensor scales, read by the kernel.  Shapes,
 * workspace (QLIN_OP_NVFP4_GEMM) and determinism as qlin_mxfp4_gemm. */
qlin_status_t qlin_nvfp4_gemm(const void* Xq_e2m1, const void* xs_e4m3, const float* sgx, const void* Wq_e2m1,
                              const void* ws_e4m3, const float* sgw, void* Y_bf16, int64_t M, int64_t N, int64_t K,
                              void* workspace, size_t ws_bytes, void* stream);

/* NVFP4 with the fused output epilogue: Y[m][n] = bf16( act( y[m][n] +
 * bias[n] ) ), y the FP32 value qlin_nvfp4_gemm rounds (after sgx * sgw);
 * bias and act as in qlin_w4a16_gemm_fused. */
qlin_status_t qlin_nvfp4_gemm_fused(const void* Xq_e2m1, const void* xs_e4m3, const float* sgx, const void* Wq_e2m1,
                                    const void* ws_e4m3, const float* sgw, void* Y_bf16, int64_t M, int64_t N,
                                    int64_t K, const void* bias_bf16, int act, void* workspace, size_t ws_bytes,
                                    void* stream);

/* Synchronises `stream`, then reads and clears the current device's error
 * word: QLIN_OK, or the first error a kernel recorded since the last call. */
qlin_status_t qlin_get_device_error(void* stream);

/* Failure-detection self-test: launches one CTA that waits, with the same
 * bounded mbarrier wait the tensor-core kernels use, on a barrier that nothing
 * completes.  After `limit_us` microseconds of device time the wait gives up
 * and records QLIN_ERR_TIMEOUT in the error word, and the kernel returns; the
 * context stays usable.  Returns the launch status; read the recorded error
 * with qlin_get_device_error().  limit_us must be in 1..1000000. */
qlin_status_t qlin_selftest_wait_timeout(uint32_t limit_us, void* stream);

/*
 * W4A16 split-K GEMV that allocates nothing (no counterpart on the pages: it
 * exists for callers that cannot allocate device memory when they run the
 * layer -- code inside a memory pool it does not own, a runtime that forbids
 * allocation after start-up, a host that must keep a fixed footprint).
 * Same arguments and result as qlin_w4a16_gemm_ex(..., QLIN_PATH_GEMV, ...)
 * but without a workspace: the split-K partial sums live in one scratch array
 * of 8 MiB inside the library image (a file-scope __device__ array that every
 * GPU which loads the library holds until the process exits).
 *  - Sizes whose split-K partial sums need more than 8 MiB are rejected with
 *    QLIN_ERR_WORKSPACE_TOO_SMALL before anything is launched.  With the
 *    current split choice this accepts every M <= 32 on the Llama-3-8B and
 *    Llama-3-70B layer shapes (their split-K sums stay in on-chip memory).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - Every call shares the one array and it keeps the last call's contents:
 *    the call clears the per-tile counters itself (an asynchronous memset on
 *    `stream`), so calls that overlap on the GPU -- on different streams, or
 *    from different threads -- race and must not be issued.
 *  - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
qlin_status_t qlin_w4a16_gemv_noalloc(const void* X_bf16, const void* codes, const void* scales_f16, const void* zeros_u4,
                            void* Y_bf16, int64_t M, int64_t N, int64_t K, int G, void* stream);

/* The M at or below which the AUTO path of each GEMM uses the GEMV kernel. */
int qlin_gemv_max_m(int op);

/* Kernels a GEMM call can launch (qlin_plan_info, info[0]). */
#define QLIN_KERNEL_W4A16_MMA 1   /* small-M W4A16: register dequantisation + mma.sync, split-K in a cluster */
#define QLIN_KERNEL_W4A16_GEMV 2  /* small-M W4A16 on the CUDA cores (K % 256 != 0), split-K in the workspace */
#define QLIN_KERNEL_W4A16_TC 3    /* W4A16 TMA + tcgen05 BF16 MMA */
#define QLIN_KERNEL_W8A8_MMA 4    /* small-M W8A8: E4M3 mma.sync, split-K in a cluster */
#define QLIN_KERNEL_W8A8_GEMV 5   /* small-M W8A8 on the CUDA cores (K % 256 != 0) */
#define QLIN_KERNEL_W8A8_TC 6     /* W8A8 TMA + tcgen05 kind::f8f6f4 */
#define QLIN_KERNEL_W8A8_BLOCK_TC 7 /* block-scaled W8A8 on tcgen05 with FP32 promotion */
#define QLIN_KERNEL_MXFP8_TC 8    /* MXFP8 on tcgen05 kind::mxf8f6f4 with hardware block scaling */
#define QLIN_KERNEL_W4A8_TC 9     /* W4A8: INT4 -> E4M3 dequantisation, tcgen05 kind::f8f6f4, group promotion */
#define QLIN_KERNEL_MXFP4_TC 10   /* MXFP4 on tcgen05 kind::mxf4 with hardware block scaling */
#define QLIN_KERNEL_NVFP4_TC 11   /* NVFP4 on tcgen05 kind::mxf4nvf4 with hardware block scaling */

/*
 * Dispatch query (for tests and measurement tools; launches nothing, reads
 * no device memory): the kernel and tiling a call of `op`
 * (QLIN_OP_W4A16_GEMM, QLIN_OP_W8A8_GEMM, QLIN_OP_W8A8_BLOCK_GEMM,
 * QLIN_OP_MXFP8_GEMM, QLIN_OP_W4A8_GEMM, QLIN_OP_MXFP4_GEMM or
 * QLIN_OP_NVFP4_GEMM) with these sizes and `path` (QLIN_PATH_*; ignored by
 * the block-scaled, MX, FP4 and W4A8 GEMMs)
 * would launch.  num_sms is the SM count to plan for, 0 for the current
 * device's (the small-M kernels always read the current device's cluster
 * occupancy).  Writes 8 values:
 *   info[0] kernel (QLIN_KERNEL_*)
 *   info[1] tokens per tile (the MMA's N side; 8 x n8 blocks for mma.sync)
 *   info[2] weight rows per tile
 *   info[3] K blocks per pipeline stage (tcgen05 kernels; 1 otherwise)
 *   info[4] split-K ranges per output tile
 *   info[5] workspace bytes of that launch
 *   info[6] 1 when the tcgen05 W4A16 kernel keeps its dequantised BF16 tile in
 *           tensor memory, 0 when in shared memory (0 for other kernels)
 *   info[7] token blocks (tiles along M)
 * The returned status is the one the GEMM call would return for the sizes
 * (shape, group and path checks); pointers are not checked.
 */
qlin_status_t qlin_plan_info(int op, int64_t M, int64_t N, int64_t K, int G, int path, int num_sms, int64_t* info);

#ifdef __cplusplus
}
#endif

#endif /* QLIN_H */
