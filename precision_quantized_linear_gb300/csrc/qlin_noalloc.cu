// W4A16 split-K GEMV for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run a layer:
// code that runs inside a memory pool it does not own, a runtime that forbids
// allocation after start-up, or a host that must keep its footprint fixed.
// The regular qlin_w4a16_gemm asks them for a split-K workspace; this entry
// point instead uses one fixed scratch array that lives in the library image
// (a file-scope __device__ array), so the call allocates nothing.
#include <mutex>

#include "qlin_internal.cuh"

namespace qlin {

// Fixed scratch of the no-allocation entry point.  Every GPU that loads the
// library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[64] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, called once per device with that device current.
static qlin_status_t noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QLIN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return QLIN_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return QLIN_OK;
}

}  // namespace qlin

using namespace qlin;

extern "C" qlin_status_t qlin_w4a16_gemv_noalloc(const void* X_bf16, const void* codes, const void* scales_f16,
                                       const void* zeros_u4, void* Y_bf16, int64_t M, int64_t N, int64_t K, int G,
                                       void* stream) {
  if (G != kGroup) return QLIN_ERR_UNSUPPORTED_SHAPE;
  if (M < 0 || M > (int64_t(1) << 24) || N <= 0 || K <= 0 || N % kTileN != 0 || K % kGroup != 0 ||
      N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
    return QLIN_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return QLIN_OK;
  if (!X_bf16 || !codes || !scales_f16 || !zeros_u4 || !Y_bf16) return QLIN_ERR_INVALID_VALUE;
  const uintptr_t a = reinterpret_cast<uintptr_t>(X_bf16) | reinterpret_cast<uintptr_t>(codes) |
                      reinterpret_cast<uintptr_t>(scales_f16) | reinterpret_cast<uintptr_t>(zeros_u4) |
                      reinterpret_cast<uintptr_t>(Y_bf16);
  if (a & 15u) return QLIN_ERR_MISALIGNED;
  int num_sms = 0;
  qlin_status_t st = device_num_sms(&num_sms);
  if (st != QLIN_OK) return st;
  // same kernel choice as qlin_w4a16_gemm_ex(..., QLIN_PATH_GEMV, ...)
  const bool mma = mma_path_ok(M, K);
  if (!mma && !gemv_m_ok(M)) return QLIN_ERR_UNSUPPORTED_SHAPE;
  const SplitPlan plan = mma ? plan_w4a16_mma(M, N, K, num_sms) : plan_w4a16_gemv(M, N, K, num_sms);
  if (plan.ws_bytes > kNoAllocScratchBytes) return QLIN_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != QLIN_OK) return st;
  auto cs = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the counters must start at
  // zero, the partial sums are overwritten before they are read.
  if (plan.zero_bytes > 0) {
    st = cuda_status(cudaMemsetAsync(scratch, 0, plan.zero_bytes, cs));
    if (st != QLIN_OK) return st;
  }
  void* ws = plan.ws_bytes > 0 ? scratch : nullptr;
  const auto* Xp = static_cast<const uint16_t*>(X_bf16);
  const auto* cp = static_cast<const uint8_t*>(codes);
  const auto* sp = static_cast<const uint16_t*>(scales_f16);
  const auto* zp = static_cast<const uint8_t*>(zeros_u4);
  auto* Yp = static_cast<uint16_t*>(Y_bf16);
  const cudaError_t e = mma ? launch_w4a16_mma(Xp, cp, sp, zp, Yp, M, N, K, kGroup, plan, ws, device_error_word(), cs)
                            : launch_w4a16_gemv(Xp, cp, sp, zp, Yp, M, N, K, plan, ws, cs);
  return cuda_status(e);
}
