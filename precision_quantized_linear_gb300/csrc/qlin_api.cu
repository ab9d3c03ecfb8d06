// Host side of libqlin: argument validation ([LP] S24 eligibility checklist,
// S31 fail-closed), kernel choice by M ([LP] S24, [TP] small vs large batch),
// tensor-map encoding and the per-device error word.  Nothing here allocates
// per call, synchronises (except qlin_get_device_error) or reads device data.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <unordered_map>

#include "qlin_internal.cuh"

namespace qlin {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxM = int64_t(1) << 24;
constexpr int64_t kFp4K = 256;  // K granularity of the FP4 calls

// Error word of each device (first error wins; cleared by qlin_get_device_error).
__device__ int g_error_word;

struct DeviceState {
  bool ready = false;
  qlin_status_t status = QLIN_OK;
  int num_sms = 0;
  int* err = nullptr;  // device address of g_error_word on this device
};

static DeviceState g_dev[kMaxDevices];
static std::mutex g_mu;
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static qlin_status_t device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QLIN_ERR_CUDA;
  DeviceState& d = g_dev[dev];
  if (d.ready) {
    *out = &d;
    return d.status;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      d.status = QLIN_ERR_CUDA;
    } else if (major != 10 || minor != 3) {
      d.status = QLIN_ERR_ARCH;  // the library holds sm_103a code only
    } else if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_error_word) != cudaSuccess) {
      d.status = QLIN_ERR_CUDA;
    } else {
      if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
          d.status = QLIN_ERR_CUDA;
        } else {
          g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
      }
    }
    d.ready = true;
  }
  *out = &d;
  return d.status;
}

qlin_status_t device_num_sms(int* out) {
  DeviceState* d = nullptr;
  const qlin_status_t st = device_state(&d);
  if (st == QLIN_OK) *out = d->num_sms;
  return st;
}

int* device_error_word() {
  DeviceState* d = nullptr;
  return device_state(&d) == QLIN_OK ? d->err : nullptr;
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                    bool swizzle128) {
  (void)elem_bytes;
  if (!g_encode) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t set_smem_once_impl(const void* kernel, int bytes, bool wide_clusters) {
  static std::mutex mu;
  static std::unordered_map<const void*, unsigned long long> done;  // kernel -> bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  std::lock_guard<std::mutex> lk(mu);
  auto it = done.find(kernel);
  if (it != done.end() && (it->second & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && wide_clusters) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done[kernel] |= bit;
  return e;
}

// M at or below which the GEMV kernels are chosen (measured crossover).
static int g_gemv_max_m_w4 = 32;
static int g_gemv_max_m_w8 = 16;  // the E4M3 mma.sync kernel beats the tcgen05 path up to M = 16

}  // namespace qlin

using namespace qlin;

static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static qlin_status_t check_shape(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || M > kMaxM || N <= 0 || K <= 0) return QLIN_ERR_UNSUPPORTED_SHAPE;
  if (N % kTileN != 0 || K % kGroup != 0) return QLIN_ERR_UNSUPPORTED_SHAPE;
  if (N > (int64_t(1) << 31) || K > (int64_t(1) << 31)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  return QLIN_OK;
}

// The CUDA error behind the last QLIN_ERR_CUDA returned on this thread.
static thread_local int g_last_cuda_error = 0;

namespace qlin {
qlin_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return QLIN_OK;
  g_last_cuda_error = static_cast<int>(e);
  (void)cudaGetLastError();  // a launch error must not be reported again by the next call
  return QLIN_ERR_CUDA;
}
}  // namespace qlin

static qlin_status_t launch_status(cudaError_t e) { return cuda_status(e); }

// W4A16 quantisation groups the kernels take ([LP] S4 per-group, S5 b_eff =
// 4 + 16 / G): 32, 64 or 128 columns, or G == K, one group per row ([LP] S4
// "per-channel")
static bool group_ok(int G, int64_t K) { return G == 32 || G == 64 || G == 128 || (G > 0 && G == K); }

// Validated output epilogue of the *_fused calls.
static qlin_status_t make_epi(const void* bias_bf16, int act, Epi* epi) {
  if (act < QLIN_ACT_NONE || act > QLIN_ACT_GELU) return QLIN_ERR_INVALID_VALUE;
  if (bias_bf16 && !aligned16(bias_bf16)) return QLIN_ERR_MISALIGNED;
  epi->bias = static_cast<const uint16_t*>(bias_bf16);
  epi->act = act;
  return QLIN_OK;
}

extern "C" {

const char* qlin_status_string(qlin_status_t status) {
  switch (status) {
    case QLIN_OK: return "QLIN_OK";
    case QLIN_ERR_INVALID_VALUE: return "QLIN_ERR_INVALID_VALUE";
    case QLIN_ERR_UNSUPPORTED_SHAPE: return "QLIN_ERR_UNSUPPORTED_SHAPE";
    case QLIN_ERR_MISALIGNED: return "QLIN_ERR_MISALIGNED";
    case QLIN_ERR_WORKSPACE_TOO_SMALL: return "QLIN_ERR_WORKSPACE_TOO_SMALL";
    case QLIN_ERR_ARCH: return "QLIN_ERR_ARCH";
    case QLIN_ERR_CUDA: return "QLIN_ERR_CUDA";
    case QLIN_ERR_TIMEOUT: return "QLIN_ERR_TIMEOUT";
    default: return "QLIN_ERR_UNKNOWN";
  }
}

int qlin_pack_format_version(void) { return QLIN_PACK_FORMAT_VERSION; }

int qlin_last_cuda_error(void) { return g_last_cuda_error; }

const char* qlin_cuda_error_name(int code) { return cudaGetErrorName(static_cast<cudaError_t>(code)); }

int qlin_gemv_max_m(int op) { return op == QLIN_OP_W8A8_GEMM ? g_gemv_max_m_w8 : g_gemv_max_m_w4; }

qlin_status_t qlin_w4_packed_sizes(int64_t N, int64_t K, int G, size_t* codes, size_t* scales, size_t* zeros) {
  if (!codes || !scales || !zeros) return QLIN_ERR_INVALID_VALUE;
  if (!group_ok(G, K)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  qlin_status_t st = check_shape(0, N, K);
  if (st != QLIN_OK) return st;
  *codes = static_cast<size_t>(N * K / 2);
  *scales = static_cast<size_t>(N * (K / G) * 2);
  *zeros = static_cast<size_t>(N * (K / G) / 2);
  return QLIN_OK;
}

// Which kernel and plan a W4A16 / W8A8 GEMM call launches.  The launch path
// and qlin_plan_info both use these, so that the query reports what runs.
struct Dispatch {
  int kernel = 0;  // QLIN_KERNEL_*
  SplitPlan sp;    // small-M kernels
  TcPlan tp;       // tcgen05 kernels
  size_t ws = 0;   // workspace bytes of the launch
};

static qlin_status_t dispatch_w4(int64_t M, int64_t N, int64_t K, int G, int path, int sms, Dispatch* d) {
  if (path == QLIN_PATH_AUTO) path = M <= g_gemv_max_m_w4 ? QLIN_PATH_GEMV : QLIN_PATH_TC;
  if (path == QLIN_PATH_GEMV) {
    if (mma_path_ok(M, K)) {
      d->kernel = QLIN_KERNEL_W4A16_MMA;
      d->sp = plan_w4a16_mma(M, N, K, sms, G);
      d->ws = d->sp.ws_bytes;
      return QLIN_OK;
    }
    if (G != kGroup) return QLIN_ERR_UNSUPPORTED_SHAPE;  // the CUDA-core GEMV takes G = 128 only
    if (!gemv_m_ok(M)) return QLIN_ERR_UNSUPPORTED_SHAPE;
    d->kernel = QLIN_KERNEL_W4A16_GEMV;
    d->sp = plan_w4a16_gemv(M, N, K, sms);
    d->ws = d->sp.ws_bytes;
    return QLIN_OK;
  }
  d->kernel = QLIN_KERNEL_W4A16_TC;
  d->tp = plan_w4a16_tc(M, N, K, sms);
  d->ws = d->tp.split.ws_bytes;
  return QLIN_OK;
}

static qlin_status_t dispatch_w8(int64_t M, int64_t N, int64_t K, int path, int sms, Dispatch* d) {
  if (path == QLIN_PATH_AUTO) path = M <= g_gemv_max_m_w8 ? QLIN_PATH_GEMV : QLIN_PATH_TC;
  if (path == QLIN_PATH_GEMV) {
    if (mma8_path_ok(M, K)) {  // register-level E4M3 MMA; split-K inside clusters, no workspace
      d->kernel = QLIN_KERNEL_W8A8_MMA;
      d->sp = plan_w8a8_mma(M, N, K, sms);
      d->ws = 0;
      return QLIN_OK;
    }
    if (!gemv_m_ok(M)) return QLIN_ERR_UNSUPPORTED_SHAPE;
    d->kernel = QLIN_KERNEL_W8A8_GEMV;
    d->sp = plan_w8a8_gemv(M, N, K, sms);
    d->ws = d->sp.ws_bytes;
    return QLIN_OK;
  }
  d->kernel = QLIN_KERNEL_W8A8_TC;
  d->tp = plan_w8a8_tc(M, N, K, sms);
  d->ws = d->tp.split.ws_bytes;
  return QLIN_OK;
}

// Workspace of any path the AUTO or forced calls may take for these sizes.
static size_t ws_w4(int64_t M, int64_t N, int64_t K, int G, int sms) {
  size_t a = mma_path_ok(M, K) ? plan_w4a16_mma(M, N, K, sms, G).ws_bytes : plan_w4a16_gemv(M, N, K, sms).ws_bytes;
  const size_t b = plan_w4a16_tc(M, N, K, sms).split.ws_bytes;
  return a > b ? a : b;
}
static size_t ws_w8(int64_t M, int64_t N, int64_t K, int sms) {
  const size_t a = plan_w8a8_gemv(M, N, K, sms).ws_bytes;
  const size_t b = plan_w8a8_tc(M, N, K, sms).split.ws_bytes;
  return a > b ? a : b;
}

qlin_status_t qlin_workspace_size(int op, int64_t M, int64_t N, int64_t K, int G, size_t* bytes) {
  if (!bytes) return QLIN_ERR_INVALID_VALUE;
  DeviceState* d = nullptr;
  qlin_status_t st = device_state(&d);
  if (st != QLIN_OK) return st;
  st = check_shape(M, N, K);
  if (st != QLIN_OK) return st;
  switch (op) {
    case QLIN_OP_W4A16_GEMM:
      if (!group_ok(G, K)) return QLIN_ERR_UNSUPPORTED_SHAPE;
      *bytes = M == 0 ? 0 : ws_w4(M, N, K, G, d->num_sms);
      return QLIN_OK;
    case QLIN_OP_W8A8_GEMM: *bytes = M == 0 ? 0 : ws_w8(M, N, K, d->num_sms); return QLIN_OK;
    case QLIN_OP_QUANT_W_FP8: *bytes = 256; return QLIN_OK;
    case QLIN_OP_W8A8_BLOCK_GEMM:
      *bytes = M == 0 ? 0 : plan_w8a8_block_tc(M, N, K, d->num_sms).split.ws_bytes;
      return QLIN_OK;
    case QLIN_OP_MXFP8_GEMM: *bytes = M == 0 ? 0 : plan_mxfp8_tc(M, N, K, d->num_sms).split.ws_bytes; return QLIN_OK;
    case QLIN_OP_MXFP4_GEMM:
    case QLIN_OP_NVFP4_GEMM:
      if (K % kFp4K != 0) return QLIN_ERR_UNSUPPORTED_SHAPE;
      *bytes = M == 0 ? 0 : plan_fp4_tc(M, N, K, d->num_sms).split.ws_bytes;
      return QLIN_OK;
    case QLIN_OP_W4A8_GEMM:
      if (G != kGroup) return QLIN_ERR_UNSUPPORTED_SHAPE;
      *bytes = M == 0 ? 0 : plan_w4a8_tc(M, N, K, d->num_sms).split.ws_bytes;
      return QLIN_OK;
    default: return QLIN_ERR_INVALID_VALUE;
  }
}

qlin_status_t qlin_plan_info(int op, int64_t M, int64_t N, int64_t K, int G, int path, int num_sms, int64_t* info) {
  if (!info || num_sms < 0) return QLIN_ERR_INVALID_VALUE;
  if (path < QLIN_PATH_AUTO || path > QLIN_PATH_TC) return QLIN_ERR_INVALID_VALUE;
  qlin_status_t st = check_shape(M, N, K);
  if (st != QLIN_OK) return st;
  if (M == 0) return QLIN_ERR_UNSUPPORTED_SHAPE;  // an empty call launches nothing
  if (num_sms == 0) {
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != QLIN_OK) return st;
    num_sms = d->num_sms;
  }
  Dispatch dp;
  if (op == QLIN_OP_W4A16_GEMM) {
    if (!group_ok(G, K)) return QLIN_ERR_UNSUPPORTED_SHAPE;
    st = dispatch_w4(M, N, K, G, path, num_sms, &dp);
  } else if (op == QLIN_OP_W8A8_GEMM) {
    st = dispatch_w8(M, N, K, path, num_sms, &dp);
  } else if (op == QLIN_OP_W8A8_BLOCK_GEMM) {
    dp.kernel = QLIN_KERNEL_W8A8_BLOCK_TC;
    dp.tp = plan_w8a8_block_tc(M, N, K, num_sms);
    dp.ws = dp.tp.split.ws_bytes;
  } else if (op == QLIN_OP_W4A8_GEMM) {
    if (G != kGroup) return QLIN_ERR_UNSUPPORTED_SHAPE;
    dp.kernel = QLIN_KERNEL_W4A8_TC;
    dp.tp = plan_w4a8_tc(M, N, K, num_sms);
    dp.ws = dp.tp.split.ws_bytes;
  } else if (op == QLIN_OP_MXFP8_GEMM) {
    dp.kernel = QLIN_KERNEL_MXFP8_TC;
    dp.tp = plan_mxfp8_tc(M, N, K, num_sms);
    dp.ws = dp.tp.split.ws_bytes;
  } else if (op == QLIN_OP_MXFP4_GEMM || op == QLIN_OP_NVFP4_GEMM) {
    if (K % kFp4K != 0) return QLIN_ERR_UNSUPPORTED_SHAPE;
    dp.kernel = op == QLIN_OP_MXFP4_GEMM ? QLIN_KERNEL_MXFP4_TC : QLIN_KERNEL_NVFP4_TC;
    dp.tp = plan_fp4_tc(M, N, K, num_sms);
    dp.ws = dp.tp.split.ws_bytes;
  } else {
    return QLIN_ERR_INVALID_VALUE;
  }
  if (st != QLIN_OK) return st;
  for (int i = 0; i < 8; ++i) info[i] = 0;
  info[0] = dp.kernel;
  const bool tc = dp.kernel == QLIN_KERNEL_W4A16_TC || dp.kernel == QLIN_KERNEL_W8A8_TC ||
                  dp.kernel == QLIN_KERNEL_W8A8_BLOCK_TC || dp.kernel == QLIN_KERNEL_MXFP8_TC ||
                  dp.kernel == QLIN_KERNEL_W4A8_TC || dp.kernel == QLIN_KERNEL_MXFP4_TC ||
                  dp.kernel == QLIN_KERNEL_NVFP4_TC;
  if (tc) {
    info[1] = dp.tp.bn;
    info[2] = dp.tp.wn;
    info[3] = dp.tp.kps;
    info[4] = dp.tp.split.splits;
    info[6] = (dp.kernel == QLIN_KERNEL_W4A16_TC && dp.tp.bn <= 128) || dp.kernel == QLIN_KERNEL_W4A8_TC ? 1 : 0;
    info[7] = dp.tp.mblocks;
  } else {
    const int64_t tok = (dp.kernel == QLIN_KERNEL_W4A16_MMA || dp.kernel == QLIN_KERNEL_W8A8_MMA)
                            ? (M <= 8 ? 8 : M <= 16 ? 16 : 32)
                            : (M >= 4 ? 4 : M >= 2 ? 2 : 1);
    info[1] = tok;
    info[2] = kTileN;
    info[3] = 1;
    info[4] = dp.sp.splits;
    info[7] = (M + tok - 1) / tok;
  }
  info[5] = static_cast<int64_t>(dp.ws);
  return QLIN_OK;
}

qlin_status_t qlin_pack_w4(const void* W_bf16, int64_t N, int64_t K, int G, int symmetric, void* codes, void* scales_f16,
                 void* zeros_u4, void* stream) {
  if (!group_ok(G, K)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  qlin_status_t st = check_shape(0, N, K);
  if (st != QLIN_OK) return st;
  if (symmetric != 0 && symmetric != 1) return QLIN_ERR_INVALID_VALUE;
  if (!W_bf16 || !codes || !scales_f16 || !zeros_u4) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(W_bf16) || !aligned16(codes) || !aligned16(scales_f16) || !aligned16(zeros_u4))
    return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != QLIN_OK) return st;
  return launch_status(launch_pack_w4(static_cast<const uint16_t*>(W_bf16), N, K, G, symmetric,
                                      static_cast<uint8_t*>(codes), static_cast<uint16_t*>(scales_f16),
                                      static_cast<uint8_t*>(zeros_u4), d->err, d->num_sms,
                                      static_cast<cudaStream_t>(stream)));
}

static qlin_status_t w4a16_impl(const void* X_bf16, const void* codes, const void* scales_f16, const void* zeros_u4,
                      void* Y_bf16, int64_t M, int64_t N, int64_t K, int G, const Epi& epi, void* workspace,
                      size_t ws_bytes, int path, void* stream) {
  if (!group_ok(G, K)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  qlin_status_t st = check_shape(M, N, K);
  if (st != QLIN_OK) return st;
  if (path < QLIN_PATH_AUTO || path > QLIN_PATH_TC) return QLIN_ERR_INVALID_VALUE;
  if (M == 0) return QLIN_OK;
  if (!X_bf16 || !codes || !scales_f16 || !zeros_u4 || !Y_bf16) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(X_bf16) || !aligned16(codes) || !aligned16(scales_f16) || !aligned16(zeros_u4) ||
      !aligned16(Y_bf16) || (workspace && !aligned16(workspace)))
    return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != QLIN_OK) return st;
  Dispatch dp;
  st = dispatch_w4(M, N, K, G, path, d->num_sms, &dp);
  if (st != QLIN_OK) return st;
  if (dp.ws > 0 && (!workspace || ws_bytes < dp.ws)) return QLIN_ERR_WORKSPACE_TOO_SMALL;
  const auto* X = static_cast<const uint16_t*>(X_bf16);
  const auto* c = static_cast<const uint8_t*>(codes);
  const auto* s = static_cast<const uint16_t*>(scales_f16);
  const auto* z = static_cast<const uint8_t*>(zeros_u4);
  auto* Y = static_cast<uint16_t*>(Y_bf16);
  auto cs = static_cast<cudaStream_t>(stream);
  switch (dp.kernel) {
    case QLIN_KERNEL_W4A16_MMA:
      return launch_status(launch_w4a16_mma(X, c, s, z, Y, M, N, K, G, dp.sp, workspace, d->err, cs, epi));
    case QLIN_KERNEL_W4A16_GEMV:
      return launch_status(launch_w4a16_gemv(X, c, s, z, Y, M, N, K, dp.sp, workspace, cs, epi));
    default:
      return launch_status(launch_w4a16_tc(X, c, s, z, Y, M, N, K, G, dp.tp, workspace, d->err, d->num_sms, cs, epi));
  }
}

qlin_status_t qlin_w4a16_gemm_ex(const void* X_bf16, const void* codes, const void* scales_f16, const void* zeros_u4,
                       void* Y_bf16, int64_t M, int64_t N, int64_t K, int G, void* workspace, size_t ws_bytes,
                       int path, void* stream) {
  return w4a16_impl(X_bf16, codes, scales_f16, zeros_u4, Y_bf16, M, N, K, G, Epi{}, workspace, ws_bytes, path,
                    stream);
}

qlin_status_t qlin_w4a16_gemm_fused(const void* X_bf16, const void* codes, const void* scales_f16, const void* zeros_u4,
                          void* Y_bf16, int64_t M, int64_t N, int64_t K, int G, const void* bias_bf16, int act,
                          void* workspace, size_t ws_bytes, int path, void* stream) {
  Epi epi;
  const qlin_status_t st = make_epi(bias_bf16, act, &epi);
  if (st != QLIN_OK) return st;
  return w4a16_impl(X_bf16, codes, scales_f16, zeros_u4, Y_bf16, M, N, K, G, epi, workspace, ws_bytes, path, stream);
}

qlin_status_t qlin_w4a16_gemm(const void* X_bf16, const void* codes, const void* scales_f16, const void* zeros_u4,
                    void* Y_bf16, int64_t M, int64_t N, int64_t K, int G, void* workspace, size_t ws_bytes,
                    void* stream) {
  return qlin_w4a16_gemm_ex(X_bf16, codes, scales_f16, zeros_u4, Y_bf16, M, N, K, G, workspace, ws_bytes,
                            QLIN_PATH_AUTO, stream);
}

qlin_status_t qlin_quant_act_fp8(const void* X_bf16, int64_t M, int64_t K, void* Xq_e4m3, float* sx, void* stream) {
  if (M < 0 || M > kMaxM || K <= 0 || K % kGroup != 0 || K > (int64_t(1) << 31)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return QLIN_OK;
  if (!X_bf16 || !Xq_e4m3 || !sx) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(X_bf16) || !aligned16(Xq_e4m3) || !aligned16(sx)) return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  qlin_status_t st = device_state(&d);
  if (st != QLIN_OK) return st;
  return launch_status(launch_quant_act_fp8(static_cast<const uint16_t*>(X_bf16), M, K,
                                            static_cast<uint8_t*>(Xq_e4m3), sx, static_cast<cudaStream_t>(stream)));
}

qlin_status_t qlin_quant_w_fp8(const void* W_bf16, int64_t N, int64_t K, void* Wq_e4m3, float* sw, void* workspace,
                     size_t ws_bytes, void* stream) {
  qlin_status_t st = check_shape(0, N, K);
  if (st != QLIN_OK) return st;
  if (!W_bf16 || !Wq_e4m3 || !sw || !workspace) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(W_bf16) || !aligned16(Wq_e4m3) || !aligned16(sw) || !aligned16(workspace))
    return QLIN_ERR_MISALIGNED;
  if (ws_bytes < 256) return QLIN_ERR_WORKSPACE_TOO_SMALL;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != QLIN_OK) return st;
  return launch_status(launch_quant_w_fp8(static_cast<const uint16_t*>(W_bf16), N, K, static_cast<uint8_t*>(Wq_e4m3),
                                          sw, static_cast<uint32_t*>(workspace), d->num_sms,
                                          static_cast<cudaStream_t>(stream)));
}

static qlin_status_t w8a8_impl(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3, const float* sw, void* Y_bf16,
                     int64_t M, int64_t N, int64_t K, const Epi& epi, void* workspace, size_t ws_bytes, int path,
                     void* stream) {
  qlin_status_t st = check_shape(M, N, K);
  if (st != QLIN_OK) return st;
  if (path < QLIN_PATH_AUTO || path > QLIN_PATH_TC) return QLIN_ERR_INVALID_VALUE;
  if (M == 0) return QLIN_OK;
  if (!Xq_e4m3 || !sx || !Wq_e4m3 || !sw || !Y_bf16) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(Xq_e4m3) || !aligned16(Wq_e4m3) || !aligned16(Y_bf16) || (workspace && !aligned16(workspace)) ||
      (reinterpret_cast<uintptr_t>(sx) & 3u) || (reinterpret_cast<uintptr_t>(sw) & 3u))
    return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != QLIN_OK) return st;
  Dispatch dp;
  st = dispatch_w8(M, N, K, path, d->num_sms, &dp);
  if (st != QLIN_OK) return st;
  if (dp.ws > 0 && (!workspace || ws_bytes < dp.ws)) return QLIN_ERR_WORKSPACE_TOO_SMALL;
  const auto* xq = static_cast<const uint8_t*>(Xq_e4m3);
  const auto* wq = static_cast<const uint8_t*>(Wq_e4m3);
  auto* Y = static_cast<uint16_t*>(Y_bf16);
  auto cs = static_cast<cudaStream_t>(stream);
  switch (dp.kernel) {
    case QLIN_KERNEL_W8A8_MMA: return launch_status(launch_w8a8_mma(xq, sx, wq, sw, Y, M, N, K, dp.sp, d->err, cs, epi));
    case QLIN_KERNEL_W8A8_GEMV:
      return launch_status(launch_w8a8_gemv(xq, sx, wq, sw, Y, M, N, K, dp.sp, workspace, cs, epi));
    default:
      return launch_status(launch_w8a8_tc(xq, sx, wq, sw, Y, M, N, K, dp.tp, workspace, d->err, d->num_sms, cs, epi));
  }
}

qlin_status_t qlin_w8a8_fp8_gemm_ex(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3, const float* sw, void* Y_bf16,
                          int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes, int path,
                          void* stream) {
  return w8a8_impl(Xq_e4m3, sx, Wq_e4m3, sw, Y_bf16, M, N, K, Epi{}, workspace, ws_bytes, path, stream);
}

qlin_status_t qlin_w8a8_fp8_gemm_fused(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3, const float* sw,
                             void* Y_bf16, int64_t M, int64_t N, int64_t K, const void* bias_bf16, int act,
                             void* workspace, size_t ws_bytes, int path, void* stream) {
  Epi epi;
  const qlin_status_t st = make_epi(bias_bf16, act, &epi);
  if (st != QLIN_OK) return st;
  return w8a8_impl(Xq_e4m3, sx, Wq_e4m3, sw, Y_bf16, M, N, K, epi, workspace, ws_bytes, path, stream);
}

qlin_status_t qlin_w8a8_fp8_gemm(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3, const float* sw, void* Y_bf16,
                       int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes, void* stream) {
  return qlin_w8a8_fp8_gemm_ex(Xq_e4m3, sx, Wq_e4m3, sw, Y_bf16, M, N, K, workspace, ws_bytes, QLIN_PATH_AUTO,
                               stream);
}

qlin_status_t qlin_quant_act_fp8_blocks(const void* X_bf16, int64_t M, int64_t K, void* Xq_e4m3, float* sx, void* stream) {
  if (M < 0 || M > kMaxM || K <= 0 || K % kGroup != 0 || K > (int64_t(1) << 31)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return QLIN_OK;
  if (!X_bf16 || !Xq_e4m3 || !sx) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(X_bf16) || !aligned16(Xq_e4m3) || (reinterpret_cast<uintptr_t>(sx) & 3u)) return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  qlin_status_t st = device_state(&d);
  if (st != QLIN_OK) return st;
  return launch_status(launch_quant_act_fp8_blocks(static_cast<const uint16_t*>(X_bf16), M, K,
                                                   static_cast<uint8_t*>(Xq_e4m3), sx,
                                                   static_cast<cudaStream_t>(stream)));
}

qlin_status_t qlin_quant_w_fp8_blocks(const void* W_bf16, int64_t N, int64_t K, void* Wq_e4m3, float* sw, void* stream) {
  qlin_status_t st = check_shape(0, N, K);
  if (st != QLIN_OK) return st;
  if (!W_bf16 || !Wq_e4m3 || !sw) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(W_bf16) || !aligned16(Wq_e4m3) || (reinterpret_cast<uintptr_t>(sw) & 3u)) return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != QLIN_OK) return st;
  return launch_status(launch_quant_w_fp8_blocks(static_cast<const uint16_t*>(W_bf16), N, K,
                                                 static_cast<uint8_t*>(Wq_e4m3), sw, static_cast<cudaStream_t>(stream)));
}

static qlin_status_t w8a8_block_impl(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3, const float* sw,
                                     void* Y_bf16, int64_t M, int64_t N, int64_t K, const Epi& epi, void* workspace,
                                     size_t ws_bytes, void* stream) {
  qlin_status_t st = check_shape(M, N, K);
  if (st != QLIN_OK) return st;
  if (M == 0) return QLIN_OK;
  if (!Xq_e4m3 || !sx || !Wq_e4m3 || !sw || !Y_bf16) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(Xq_e4m3) || !aligned16(Wq_e4m3) || !aligned16(Y_bf16) || (workspace && !aligned16(workspace)) ||
      (reinterpret_cast<uintptr_t>(sx) & 3u) || (reinterpret_cast<uintptr_t>(sw) & 3u))
    return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != QLIN_OK) return st;
  const TcPlan p = plan_w8a8_block_tc(M, N, K, d->num_sms);
  if (p.split.ws_bytes > 0 && (!workspace || ws_bytes < p.split.ws_bytes)) return QLIN_ERR_WORKSPACE_TOO_SMALL;
  return launch_status(launch_w8a8_block_tc(static_cast<const uint8_t*>(Xq_e4m3), sx,
                                            static_cast<const uint8_t*>(Wq_e4m3), sw, static_cast<uint16_t*>(Y_bf16),
                                            M, N, K, p, workspace, d->err, d->num_sms,
                                            static_cast<cudaStream_t>(stream), epi));
}

qlin_status_t qlin_w8a8_fp8_block_gemm(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3, const float* sw,
                             void* Y_bf16, int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                             void* stream) {
  return w8a8_block_impl(Xq_e4m3, sx, Wq_e4m3, sw, Y_bf16, M, N, K, Epi{}, workspace, ws_bytes, stream);
}

qlin_status_t qlin_w8a8_fp8_block_gemm_fused(const void* Xq_e4m3, const float* sx, const void* Wq_e4m3,
                                             const float* sw, void* Y_bf16, int64_t M, int64_t N, int64_t K,
                                             const void* bias_bf16, int act, void* workspace, size_t ws_bytes,
                                             void* stream) {
  Epi epi;
  const qlin_status_t st = make_epi(bias_bf16, act, &epi);
  if (st != QLIN_OK) return st;
  return w8a8_block_impl(Xq_e4m3, sx, Wq_e4m3, sw, Y_bf16, M, N, K, epi, workspace, ws_bytes, stream);
}

static qlin_status_t w4a8_impl(const void* Xq_e4m3, const float* sx, const void* codes, const void* scales_f16,
                               const void* zeros_u4, void* Y_bf16, int64_t M, int64_t N, int64_t K, int G,
                               const Epi& epi, void* workspace, size_t ws_bytes, void* stream) {
  if (G != kGroup) return QLIN_ERR_UNSUPPORTED_SHAPE;  // one quantisation group per 128-column K block
  qlin_status_t st = check_shape(M, N, K);
  if (st != QLIN_OK) return st;
  if (M == 0) return QLIN_OK;
  if (!Xq_e4m3 || !sx || !codes || !scales_f16 || !zeros_u4 || !Y_bf16) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(Xq_e4m3) || !aligned16(codes) || !aligned16(scales_f16) || !aligned16(zeros_u4) ||
      !aligned16(Y_bf16) || (workspace && !aligned16(workspace)) || (reinterpret_cast<uintptr_t>(sx) & 3u))
    return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != QLIN_OK) return st;
  const TcPlan p = plan_w4a8_tc(M, N, K, d->num_sms);
  if (p.split.ws_bytes > 0 && (!workspace || ws_bytes < p.split.ws_bytes)) return QLIN_ERR_WORKSPACE_TOO_SMALL;
  return launch_status(launch_w4a8_tc(static_cast<const uint8_t*>(Xq_e4m3), sx, static_cast<const uint8_t*>(codes),
                                      static_cast<const uint16_t*>(scales_f16), static_cast<const uint8_t*>(zeros_u4),
                                      static_cast<uint16_t*>(Y_bf16), M, N, K, p, workspace, d->err, d->num_sms,
                                      static_cast<cudaStream_t>(stream), epi));
}

qlin_status_t qlin_w4a8_gemm(const void* Xq_e4m3, const float* sx, const void* codes, const void* scales_f16,
                             const void* zeros_u4, void* Y_bf16, int64_t M, int64_t N, int64_t K, int G,
                             void* workspace, size_t ws_bytes, void* stream) {
  return w4a8_impl(Xq_e4m3, sx, codes, scales_f16, zeros_u4, Y_bf16, M, N, K, G, Epi{}, workspace, ws_bytes, stream);
}

qlin_status_t qlin_w4a8_gemm_fused(const void* Xq_e4m3, const float* sx, const void* codes, const void* scales_f16,
                                   const void* zeros_u4, void* Y_bf16, int64_t M, int64_t N, int64_t K, int G,
                                   const void* bias_bf16, int act, void* workspace, size_t ws_bytes, void* stream) {
  Epi epi;
  const qlin_status_t st = make_epi(bias_bf16, act, &epi);
  if (st != QLIN_OK) return st;
  return w4a8_impl(Xq_e4m3, sx, codes, scales_f16, zeros_u4, Y_bf16, M, N, K, G, epi, workspace, ws_bytes, stream);
}

qlin_status_t qlin_mx_scale_bytes(int64_t R, int64_t K, size_t* bytes) {
  if (!bytes) return QLIN_ERR_INVALID_VALUE;
  if (R < 0 || R > kMaxM * 64 || K <= 0 || K % kGroup != 0 || K > (int64_t(1) << 31)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  *bytes = static_cast<size_t>((R + 127) / 128 * 128 * (K / 32));
  return QLIN_OK;
}

qlin_status_t qlin_quant_mxfp8(const void* X_bf16, int64_t R, int64_t K, void* codes_e4m3, void* scales_e8m0,
                               void* stream) {
  if (R < 0 || R > kMaxM * 64 || K <= 0 || K % kGroup != 0 || K > (int64_t(1) << 31)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  if (R == 0) return QLIN_OK;
  if (!X_bf16 || !codes_e4m3 || !scales_e8m0) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(X_bf16) || !aligned16(codes_e4m3) || !aligned16(scales_e8m0)) return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  qlin_status_t st = device_state(&d);
  if (st != QLIN_OK) return st;
  return launch_status(launch_quant_mxfp8(static_cast<const uint16_t*>(X_bf16), R, K,
                                          static_cast<uint8_t*>(codes_e4m3), static_cast<uint8_t*>(scales_e8m0),
                                          static_cast<cudaStream_t>(stream)));
}

static qlin_status_t mxfp8_impl(const void* Xq_e4m3, const void* xs_e8m0, const void* Wq_e4m3, const void* ws_e8m0,
                                void* Y_bf16, int64_t M, int64_t N, int64_t K, const Epi& epi, void* workspace,
                                size_t ws_bytes, void* stream) {
  qlin_status_t st = check_shape(M, N, K);
  if (st != QLIN_OK) return st;
  if (M == 0) return QLIN_OK;
  if (!Xq_e4m3 || !xs_e8m0 || !Wq_e4m3 || !ws_e8m0 || !Y_bf16) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(Xq_e4m3) || !aligned16(xs_e8m0) || !aligned16(Wq_e4m3) || !aligned16(ws_e8m0) ||
      !aligned16(Y_bf16) || (workspace && !aligned16(workspace)))
    return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != QLIN_OK) return st;
  const TcPlan p = plan_mxfp8_tc(M, N, K, d->num_sms);
  if (p.split.ws_bytes > 0 && (!workspace || ws_bytes < p.split.ws_bytes)) return QLIN_ERR_WORKSPACE_TOO_SMALL;
  return launch_status(launch_mxfp8_tc(static_cast<const uint8_t*>(Xq_e4m3), static_cast<const uint8_t*>(xs_e8m0),
                                       static_cast<const uint8_t*>(Wq_e4m3), static_cast<const uint8_t*>(ws_e8m0),
                                       static_cast<uint16_t*>(Y_bf16), M, N, K, p, workspace, d->err, d->num_sms,
                                       static_cast<cudaStream_t>(stream), epi));
}

qlin_status_t qlin_mxfp8_gemm(const void* Xq_e4m3, const void* xs_e8m0, const void* Wq_e4m3, const void* ws_e8m0,
                              void* Y_bf16, int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                              void* stream) {
  return mxfp8_impl(Xq_e4m3, xs_e8m0, Wq_e4m3, ws_e8m0, Y_bf16, M, N, K, Epi{}, workspace, ws_bytes, stream);
}

qlin_status_t qlin_mxfp8_gemm_fused(const void* Xq_e4m3, const void* xs_e8m0, const void* Wq_e4m3,
                                    const void* ws_e8m0, void* Y_bf16, int64_t M, int64_t N, int64_t K,
                                    const void* bias_bf16, int act, void* workspace, size_t ws_bytes, void* stream) {
  Epi epi;
  const qlin_status_t st = make_epi(bias_bf16, act, &epi);
  if (st != QLIN_OK) return st;
  return mxfp8_impl(Xq_e4m3, xs_e8m0, Wq_e4m3, ws_e8m0, Y_bf16, M, N, K, epi, workspace, ws_bytes, stream);
}

// ---- FP4: packed E2M1, K % 256 == 0 (one 128-byte TMA box = 256 columns per K block)

static bool fp4_rows_ok(int64_t R, int64_t K) {
  return R >= 0 && R <= kMaxM * 64 && K > 0 && K % kFp4K == 0 && K <= (int64_t(1) << 31);
}

qlin_status_t qlin_nvfp4_scale_bytes(int64_t R, int64_t K, size_t* bytes) {
  if (!bytes) return QLIN_ERR_INVALID_VALUE;
  if (!fp4_rows_ok(R, K)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  *bytes = static_cast<size_t>((R + 127) / 128 * 128 * (K / 16));
  return QLIN_OK;
}

qlin_status_t qlin_quant_mxfp4(const void* X_bf16, int64_t R, int64_t K, void* codes_e2m1, void* scales_e8m0,
                               void* stream) {
  if (!fp4_rows_ok(R, K)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  if (R == 0) return QLIN_OK;
  if (!X_bf16 || !codes_e2m1 || !scales_e8m0) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(X_bf16) || !aligned16(codes_e2m1) || !aligned16(scales_e8m0)) return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  qlin_status_t st = device_state(&d);
  if (st != QLIN_OK) return st;
  return launch_status(launch_quant_mxfp4(static_cast<const uint16_t*>(X_bf16), R, K,
                                          static_cast<uint8_t*>(codes_e2m1), static_cast<uint8_t*>(scales_e8m0),
                                          static_cast<cudaStream_t>(stream)));
}

qlin_status_t qlin_nvfp4_tensor_scale(const void* X_bf16, int64_t n, float* sg, void* stream) {
  if (n <= 0 || n % 8 != 0) return QLIN_ERR_UNSUPPORTED_SHAPE;
  if (!X_bf16 || !sg) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(X_bf16) || (reinterpret_cast<uintptr_t>(sg) & 3u) != 0) return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  qlin_status_t st = device_state(&d);
  if (st != QLIN_OK) return st;
  return launch_status(launch_nvfp4_tensor_scale(static_cast<const uint16_t*>(X_bf16), n, sg, d->num_sms,
                                                 static_cast<cudaStream_t>(stream)));
}

qlin_status_t qlin_quant_nvfp4(const void* X_bf16, int64_t R, int64_t K, const float* sg, void* codes_e2m1,
                               void* scales_e4m3, void* stream) {
  if (!fp4_rows_ok(R, K)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  if (R == 0) return QLIN_OK;
  if (!X_bf16 || !sg || !codes_e2m1 || !scales_e4m3) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(X_bf16) || !aligned16(codes_e2m1) || !aligned16(scales_e4m3) ||
      (reinterpret_cast<uintptr_t>(sg) & 3u) != 0)
    return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  qlin_status_t st = device_state(&d);
  if (st != QLIN_OK) return st;
  return launch_status(launch_quant_nvfp4(static_cast<const uint16_t*>(X_bf16), R, K, sg,
                                          static_cast<uint8_t*>(codes_e2m1), static_cast<uint8_t*>(scales_e4m3),
                                          static_cast<cudaStream_t>(stream)));
}

static qlin_status_t fp4_gemm(const void* Xq, const void* xs, const float* sgx, const void* Wq, const void* ws_sf,
                              const float* sgw, bool nv, void* Y_bf16, int64_t M, int64_t N, int64_t K,
                              const Epi& epi, void* workspace, size_t ws_bytes, void* stream) {
  qlin_status_t st = check_shape(M, N, K);
  if (st != QLIN_OK) return st;
  if (K % kFp4K != 0) return QLIN_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return QLIN_OK;
  if (!Xq || !xs || !Wq || !ws_sf || !Y_bf16 || (nv && (!sgx || !sgw))) return QLIN_ERR_INVALID_VALUE;
  if (!aligned16(Xq) || !aligned16(xs) || !aligned16(Wq) || !aligned16(ws_sf) || !aligned16(Y_bf16) ||
      (workspace && !aligned16(workspace)) ||
      (nv && ((reinterpret_cast<uintptr_t>(sgx) & 3u) != 0 || (reinterpret_cast<uintptr_t>(sgw) & 3u) != 0)))
    return QLIN_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != QLIN_OK) return st;
  const TcPlan p = plan_fp4_tc(M, N, K, d->num_sms);
  if (p.split.ws_bytes > 0 && (!workspace || ws_bytes < p.split.ws_bytes)) return QLIN_ERR_WORKSPACE_TOO_SMALL;
  return launch_status(launch_fp4_tc(static_cast<const uint8_t*>(Xq), static_cast<const uint8_t*>(xs), sgx,
                                     static_cast<const uint8_t*>(Wq), static_cast<const uint8_t*>(ws_sf), sgw,
                                     static_cast<uint16_t*>(Y_bf16), M, N, K, nv, p, workspace, d->err, d->num_sms,
                                     static_cast<cudaStream_t>(stream), epi));
}

qlin_status_t qlin_mxfp4_gemm(const void* Xq_e2m1, const void* xs_e8m0, const void* Wq_e2m1, const void* ws_e8m0,
                              void* Y_bf16, int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                              void* stream) {
  return fp4_gemm(Xq_e2m1, xs_e8m0, nullptr, Wq_e2m1, ws_e8m0, nullptr, false, Y_bf16, M, N, K, Epi{}, workspace,
                  ws_bytes, stream);
}

qlin_status_t qlin_mxfp4_gemm_fused(const void* Xq_e2m1, const void* xs_e8m0, const void* Wq_e2m1,
                                    const void* ws_e8m0, void* Y_bf16, int64_t M, int64_t N, int64_t K,
                                    const void* bias_bf16, int act, void* workspace, size_t ws_bytes, void* stream) {
  Epi epi;
  const qlin_status_t st = make_epi(bias_bf16, act, &epi);
  if (st != QLIN_OK) return st;
  return fp4_gemm(Xq_e2m1, xs_e8m0, nullptr, Wq_e2m1, ws_e8m0, nullptr, false, Y_bf16, M, N, K, epi, workspace,
                  ws_bytes, stream);
}

qlin_status_t qlin_nvfp4_gemm(const void* Xq_e2m1, const void* xs_e4m3, const float* sgx, const void* Wq_e2m1,
                              const void* ws_e4m3, const float* sgw, void* Y_bf16, int64_t M, int64_t N, int64_t K,
                              void* workspace, size_t ws_bytes, void* stream) {
  return fp4_gemm(Xq_e2m1, xs_e4m3, sgx, Wq_e2m1, ws_e4m3, sgw, true, Y_bf16, M, N, K, Epi{}, workspace, ws_bytes,
                  stream);
}

qlin_status_t qlin_nvfp4_gemm_fused(const void* Xq_e2m1, const void* xs_e4m3, const float* sgx, const void* Wq_e2m1,
                                    const void* ws_e4m3, const float* sgw, void* Y_bf16, int64_t M, int64_t N,
                                    int64_t K, const void* bias_bf16, int act, void* workspace, size_t ws_bytes,
                                    void* stream) {
  Epi epi;
  const qlin_status_t st = make_epi(bias_bf16, act, &epi);
  if (st != QLIN_OK) return st;
  return fp4_gemm(Xq_e2m1, xs_e4m3, sgx, Wq_e2m1, ws_e4m3, sgw, true, Y_bf16, M, N, K, epi, workspace, ws_bytes,
                  stream);
}

qlin_status_t qlin_selftest_wait_timeout(uint32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return QLIN_ERR_INVALID_VALUE;
  DeviceState* d = nullptr;
  qlin_status_t st = device_state(&d);
  if (st != QLIN_OK) return st;
  return launch_status(launch_wait_timeout(static_cast<uint64_t>(limit_us) * 1000ull, d->err,
                                           static_cast<cudaStream_t>(stream)));
}

qlin_status_t qlin_get_device_error(void* stream) {
  DeviceState* d = nullptr;
  qlin_status_t st = device_state(&d);
  if (st != QLIN_OK) return st;
  auto cs = static_cast<cudaStream_t>(stream);
  st = cuda_status(cudaStreamSynchronize(cs));
  if (st != QLIN_OK) return st;
  int word = 0;
  st = cuda_status(cudaMemcpy(&word, d->err, sizeof(int), cudaMemcpyDeviceToHost));
  if (st != QLIN_OK) return st;
  const int zero = 0;
  st = cuda_status(cudaMemcpy(d->err, &zero, sizeof(int), cudaMemcpyHostToDevice));
  if (st != QLIN_OK) return st;
  return static_cast<qlin_status_t>(word);
}

}  // extern "C"
