// Declarations shared by the translation units of libqlin (host side).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/qlin.h"

namespace qlin {

constexpr int kTileN = 128;   // weight rows per tile
constexpr int kTileK = 64;    // columns per tile (one 128-byte BF16 row)
constexpr int kGroup = 128;   // quantisation group along K

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

// Device error word: first error wins.
__device__ __forceinline__ void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Output epilogue of the GEMMs ([LP] S23 "fused epilogue", S24 "bias /
// activation epilogue fused"): Y = bf16(act(acc + bias[n])), acc the FP32
// result after the quantisation scales; bias BF16 [N] or null, act QLIN_ACT_*.
struct Epi {
  const uint16_t* bias = nullptr;
  int act = QLIN_ACT_NONE;
};
// bias[n] as FP32 (0 without a bias); load it early, it is needed only at the end
__device__ __forceinline__ float epi_bias(const Epi& e, int64_t n) {
  return e.bias ? __uint_as_float(static_cast<uint32_t>(__ldg(e.bias + n)) << 16) : 0.0f;
}
// SiLU as v / (1 + e^-v) with the hardware exponential and the fast divide
// (relative error ~2^-21, far below the BF16 output's 2^-9; 0 once e^-v
// overflows, i.e. for v < -88, where |silu(v)| < 2^-120); GELU as v * Phi(v)
// with CUDA's normcdff.
__device__ __forceinline__ float epi_silu(float v) { return __fdividef(v, 1.0f + __expf(-v)); }
__device__ __forceinline__ float epi_gelu(float v) { return v * normcdff(v); }
// act(v + b)
__device__ __forceinline__ float epi_act(int act, float v, float b) {
  v += b;
  switch (act) {
    case QLIN_ACT_RELU: return fmaxf(v, 0.0f);
    case QLIN_ACT_SILU: return epi_silu(v);
    case QLIN_ACT_GELU: return epi_gelu(v);
    default: return v;
  }
}
__device__ __forceinline__ float epi_apply(const Epi& e, float v, int64_t n) { return epi_act(e.act, v, epi_bias(e, n)); }
// act(v + b) as a called function, for epilogue loops that are unrolled over
// many outputs (the block-format, block-scaled and W4A8 kernels): one copy of
// each activation's code serves every output, where inlining it per output
// would multiply the kernel's code many times over
static __device__ __noinline__ float epi_act_call(int act, float v) { return epi_act(act, v, 0.0f); }
// act(v + b) with the addition inline and the activation called only when one is set
__device__ __forceinline__ float epi_sparse(int act, float v, float b) {
  v += b;
  return act == QLIN_ACT_NONE ? v : epi_act_call(act, v);
}
// the same for output column n
__device__ __forceinline__ float epi_cols(const Epi& e, float v, int64_t n) { return epi_sparse(e.act, v, epi_bias(e, n)); }
// act(o[i] + b) for a run of values of one output column: one branch on the
// activation for the whole run, so that each loop stays straight-line code
template <int L>
__device__ __forceinline__ void epi_run(int act, float (&o)[L], float b) {
  switch (act) {
    case QLIN_ACT_RELU:
#pragma unroll
      for (int i = 0; i < L; ++i) o[i] = epi_act(QLIN_ACT_RELU, o[i], b);
      break;
    case QLIN_ACT_SILU:
#pragma unroll
      for (int i = 0; i < L; ++i) o[i] = epi_act(QLIN_ACT_SILU, o[i], b);
      break;
    case QLIN_ACT_GELU:
#pragma unroll
      for (int i = 0; i < L; ++i) o[i] = epi_act(QLIN_ACT_GELU, o[i], b);
      break;
    default:
#pragma unroll
      for (int i = 0; i < L; ++i) o[i] += b;
  }
}

// Split-K workspace: [counters: one uint32 per output tile, padded to 256 B]
// [partials: splits x M x N float].
struct SplitPlan {
  int splits = 1;        // K ranges per output tile
  int kb_per_split = 0;  // 64-column blocks per range (last range may be shorter)
  int64_t tiles = 0;     // output tiles (m blocks x n tiles)
  size_t ws_bytes = 0;   // workspace needed (0 when splits == 1)
  size_t zero_bytes = 0; // leading workspace bytes (counters) that must be zero at launch
};

// cudaFuncSetAttribute once per (kernel, device), so that no such call is made
// while a stream is being captured into a CUDA graph.  Keyed by the kernel's
// address: template instantiations share a type but not an address.
cudaError_t set_smem_once_impl(const void* kernel, int bytes, bool wide_clusters);
// QLIN_OK for cudaSuccess; otherwise records e for qlin_last_cuda_error(),
// clears the runtime's last-error state and returns QLIN_ERR_CUDA.
qlin_status_t cuda_status(cudaError_t e);
// wide_clusters: also allow thread-block clusters of up to 16 CTAs.
template <typename F>
inline cudaError_t set_smem_once(F* kernel, int bytes, bool wide_clusters = false) {
  return set_smem_once_impl(reinterpret_cast<const void*>(kernel), bytes, wide_clusters);
}

inline size_t counters_bytes(int64_t tiles) { return static_cast<size_t>((tiles * 4 + 255) / 256 * 256); }

// ---- launchers (return cudaError_t of the launch)
cudaError_t launch_pack_w4(const uint16_t* W, int64_t N, int64_t K, int G, int symmetric, uint8_t* codes,
                           uint16_t* scales, uint8_t* zeros, int* err, int num_sms, cudaStream_t st);
cudaError_t launch_quant_act_fp8(const uint16_t* X, int64_t M, int64_t K, uint8_t* Xq, float* sx,
                                 cudaStream_t st);
cudaError_t launch_quant_w_fp8(const uint16_t* W, int64_t N, int64_t K, uint8_t* Wq, float* sw, uint32_t* amax_ws,
                               int num_sms, cudaStream_t st);

SplitPlan plan_w4a16_gemv(int64_t M, int64_t N, int64_t K, int num_sms);
// The CUDA-core GEMVs launch one grid row per block of up to four tokens:
// at most 65535 of them.
bool gemv_m_ok(int64_t M);
cudaError_t launch_w4a16_gemv(const uint16_t* X, const uint8_t* codes, const uint16_t* scales, const uint8_t* zeros,
                              uint16_t* Y, int64_t M, int64_t N, int64_t K, const SplitPlan& plan, void* ws,
                              cudaStream_t st, const Epi& epi = Epi{});

// W4A16 small-M kernel with register-level dequantisation feeding mma.sync
// (M <= 32, K % 256 == 0); kb_per_split counts 256-column stages.
bool mma_path_ok(int64_t M, int64_t K);
SplitPlan plan_w4a16_mma(int64_t M, int64_t N, int64_t K, int num_sms, int G = 128);
cudaError_t launch_w4a16_mma(const uint16_t* X, const uint8_t* codes, const uint16_t* scales, const uint8_t* zeros,
                             uint16_t* Y, int64_t M, int64_t N, int64_t K, int G, const SplitPlan& plan, void* ws,
                             int* err, cudaStream_t st, const Epi& epi = Epi{});

// W8A8 small-M kernel on register-level E4M3 mma.sync (M <= 16, K % 256 == 0);
// kb_per_split counts 256-column stages.
bool mma8_path_ok(int64_t M, int64_t K);
SplitPlan plan_w8a8_mma(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_w8a8_mma(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, uint16_t* Y,
                            int64_t M, int64_t N, int64_t K, const SplitPlan& plan, int* err, cudaStream_t st,
                            const Epi& epi = Epi{});
SplitPlan plan_w8a8_gemv(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_w8a8_gemv(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, uint16_t* Y,
                             int64_t M, int64_t N, int64_t K, const SplitPlan& plan, void* ws, cudaStream_t st,
                             const Epi& epi = Epi{});

// tcgen05 kernels: swap-AB (weights are the 128-row MMA operand, tokens the N
// side), except block-scaled FP8 with 128-token tiles, which is token-major
struct TcPlan {
  int bn = 16;           // tokens per tile (MMA N)
  int wn = 128;          // weight rows per tile (256: block-scaled token-major tiles)
  int kps = 1;           // K blocks per pipeline stage
  int64_t mblocks = 1;   // token blocks
  SplitPlan split;
};
TcPlan plan_w4a16_tc(int64_t M, int64_t N, int64_t K, int num_sms);
TcPlan plan_w8a8_tc(int64_t M, int64_t N, int64_t K, int num_sms);
TcPlan plan_w8a8_block_tc(int64_t M, int64_t N, int64_t K, int num_sms);

cudaError_t launch_w4a16_tc(const uint16_t* X, const uint8_t* codes, const uint16_t* scales, const uint8_t* zeros,
                            uint16_t* Y, int64_t M, int64_t N, int64_t K, int G, const TcPlan& plan, void* ws,
                            int* err, int num_sms, cudaStream_t st, const Epi& epi = Epi{});
cudaError_t launch_w8a8_tc(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, uint16_t* Y,
                           int64_t M, int64_t N, int64_t K, const TcPlan& plan, void* ws, int* err, int num_sms,
                           cudaStream_t st, const Epi& epi = Epi{});
// FP8 block scaling: sx = [K/128][M], sw = [N/128][K/128] FP32 block scales.
cudaError_t launch_w8a8_block_tc(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, uint16_t* Y,
                                 int64_t M, int64_t N, int64_t K, const TcPlan& plan, void* ws, int* err, int num_sms,
                                 cudaStream_t st, const Epi& epi);
// W4A8: packed INT4 weights (G = 128) dequantised to E4M3, times per-token E4M3 activations.
TcPlan plan_w4a8_tc(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_w4a8_tc(const uint8_t* Xq, const float* sx, const uint8_t* codes, const uint16_t* scales,
                           const uint8_t* zeros, uint16_t* Y, int64_t M, int64_t N, int64_t K, const TcPlan& plan,
                           void* ws, int* err, int num_sms, cudaStream_t st, const Epi& epi);
// MXFP8: E4M3 operands with E8M0 scales per 32 columns, in scale atoms
// [rows / 128][K / 128][512 B] (see qlin_quant_mxfp8).
TcPlan plan_mxfp8_tc(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_mxfp8_tc(const uint8_t* Xq, const uint8_t* xs, const uint8_t* Wq, const uint8_t* ws_sf,
                            uint16_t* Y, int64_t M, int64_t N, int64_t K, const TcPlan& plan, void* ws, int* err,
                            int num_sms, cudaStream_t st, const Epi& epi);
cudaError_t launch_quant_mxfp8(const uint16_t* X, int64_t R, int64_t K, uint8_t* codes, uint8_t* scales,
                               cudaStream_t st);
// FP4: packed E2M1 operands (two per byte, K / 2 bytes per row) with MXFP4
// (E8M0 per 32 columns) or NVFP4 (E4M3 per 16 columns and an FP32 per-tensor
// scale sgx / sgw) scale atoms; see qlin_quant_mxfp4 / qlin_quant_nvfp4.
TcPlan plan_fp4_tc(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_fp4_tc(const uint8_t* Xq, const uint8_t* xs, const float* sgx, const uint8_t* Wq,
                          const uint8_t* ws_sf, const float* sgw, uint16_t* Y, int64_t M, int64_t N, int64_t K,
                          bool nv, const TcPlan& plan, void* ws, int* err, int num_sms, cudaStream_t st,
                          const Epi& epi);
cudaError_t launch_quant_mxfp4(const uint16_t* X, int64_t R, int64_t K, uint8_t* codes, uint8_t* scales,
                               cudaStream_t st);
cudaError_t launch_nvfp4_tensor_scale(const uint16_t* X, int64_t n, float* sg, int num_sms, cudaStream_t st);
cudaError_t launch_quant_nvfp4(const uint16_t* X, int64_t R, int64_t K, const float* sg, uint8_t* codes,
                               uint8_t* scales, cudaStream_t st);
cudaError_t launch_quant_act_fp8_blocks(const uint16_t* X, int64_t M, int64_t K, uint8_t* Xq, float* sx,
                                        cudaStream_t st);
cudaError_t launch_quant_w_fp8_blocks(const uint16_t* W, int64_t N, int64_t K, uint8_t* Wq, float* sw,
                                      cudaStream_t st);

cudaError_t launch_wait_timeout(uint64_t limit_ns, int* err, cudaStream_t st);

// SM count of the current device after the library's device checks
// (returns a qlin status).
qlin_status_t device_num_sms(int* out);
// Device address of the current device's error word (valid after device_num_sms succeeded).
int* device_error_word();

// Tensor-map encoding through the driver entry point (no libcuda link).
// swizzle128: 128-byte swizzled shared-memory tiles (MMA operands), else a plain row-major box.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                    bool swizzle128 = true);

}  // namespace qlin
