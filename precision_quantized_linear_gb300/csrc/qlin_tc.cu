// Tensor-core kernels for sm_103a: TMA -> shared memory -> tcgen05.mma with
// the accumulator in TMEM -> tcgen05.ld epilogue.
//
// Orientation ("swap AB"): the 128 weight rows of a tile are the MMA's M side
// and the tokens are its N side (16..256), so that a decode batch of a few
// tokens still fills the 128-row MMA and every weight is read once per token
// block.  D[n][m] = sum_k W[n][k] X[m][k] lands in TMEM lane n, column m.
//
// W4A16 ([LP] S11, S23 "fast path"): the packed INT4 tile and its scales /
// zero-points are bulk-copied into shared memory; four dequantisation warps
// turn them into BF16 s (q - z) written straight into the 128-byte-swizzled
// K-major layout the MMA reads; kind::f16 MMA (BF16 x BF16 -> FP32).
// W8A8 ([LP] S8, S9): E4M3 weight and activation tiles by TMA; kind::f8f6f4
// MMA; the epilogue applies sx[m] * sw.
//
// Warp roles (192 threads): warp 0 issues the copies, warp 1 owns TMEM and
// issues the MMAs (one elected lane), warps 2-5 dequantise (W4A16) and run the
// epilogue.  Every wait is bounded in time; on expiry the kernel records
// QLIN_ERR_TIMEOUT, stops issuing work and leaves.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qlin_internal.cuh"
#include "qlin_ptx.cuh"

namespace qlin {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr int kSmemBudget = 225 * 1024;

template <int BN, bool W4>
struct TcCfg {
  static constexpr int kBlkBytes = 128;                      // bytes of one row of a K block
  static constexpr int kCols = W4 ? 64 : 128;                // K columns per block
  static constexpr int kXBytes = BN * kBlkBytes;             // token tile
  static constexpr int kWBytes = W4 ? 4096 : 128 * kBlkBytes;  // packed codes / E4M3 weight tile
  static constexpr int kMetaBytes = W4 ? 1024 : 0;           // scales (256) + zeros (64), padded
  static constexpr int kStage = kXBytes + kWBytes + kMetaBytes;
  static constexpr int kAStage = W4 ? 128 * kBlkBytes : 0;   // dequantised BF16 weight tile
  static constexpr int kAStages = W4 ? 4 : 0;
  static constexpr int kStagesRaw = (kSmemBudget - 2048 - kAStages * kAStage) / kStage;
  static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
  static constexpr int kTmemCols = BN < 32 ? 32 : BN;
  static constexpr int kSmemBytes = 1024 /*align slack*/ + kStages * kStage + kAStages * kAStage + 1024 /*barriers*/;
  static_assert(kStages >= 2, "pipeline too shallow");
  static_assert(kXBytes % 1024 == 0 && kStage % 1024 == 0, "1024-byte alignment of swizzled tiles");
};

__device__ __forceinline__ uint16_t to_bf16(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

__device__ __forceinline__ void named_bar_epi() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }

// Eight columns of one 32-bit code word -> eight BF16 s (q - z), as 16 bytes.
__device__ __forceinline__ uint4 dequant8(uint32_t w, __nv_bfloat162 zoff, __nv_bfloat162 s2) {
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t v = ((w >> (4 * t)) & 0x000F000Fu) | 0x43004300u;  // BF16x2 (128 + q)
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v);
    b = __hmul2(__hsub2(b, zoff), s2);  // (q - z) exact, then one rounding
    o[t] = bf16x2_bits(b);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int BN, bool W4>
__global__ void __launch_bounds__(192, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                   const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                   const uint8_t* __restrict__ zeros, const float* __restrict__ sx, const float* __restrict__ sw,
                   uint16_t* __restrict__ Y, int64_t M, int64_t N, int64_t K, int kb_per_split, int splits,
                   float* partials, uint32_t* counters, int* err) {
  using C = TcCfg<BN, W4>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* aring = ring + C::kStages * C::kStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(aring + C::kAStages * C::kAStage);
  uint64_t* full = bars;
  uint64_t* empty = full + C::kStages;
  uint64_t* a_full = empty + C::kStages;
  uint64_t* a_empty = a_full + (W4 ? C::kAStages : 0);
  uint64_t* tmem_full = a_empty + (W4 ? C::kAStages : 0);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_full + 1);
  __shared__ int s_last;
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x, split = blockIdx.y, mb = blockIdx.z;
  const int64_t KB = K / C::kCols;
  const int kb0 = split * kb_per_split;
  const int kb1 = static_cast<int>(imin64(KB, kb0 + kb_per_split));
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W4 ? 1 + 4 : 1);
    }
    if constexpr (W4) {
      for (int a = 0; a < C::kAStages; ++a) {
        mbar_init(&a_full[a], 4);
        mbar_init(&a_empty[a], 1);
      }
    }
    mbar_init(tmem_full, 1);
    fence_mbar_init();
    s_fail = 0;
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmap_x);
    if constexpr (!W4) prefetch_tensormap(&tmap_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      const int64_t ng = K / kGroup;
      for (int it = 0; it < nkb; ++it) {
        const int s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, kWaitLimitNs)) {
          set_error(err, QLIN_ERR_TIMEOUT);
          break;
        }
        uint8_t* st = ring + s * C::kStage;
        const int kb = kb0 + it;
        mbar_arrive_expect_tx(&full[s], C::kXBytes + (W4 ? 4096 + 256 + 64 : C::kWBytes));
        tma_load_2d_hint(st, &tmap_x, &full[s], kb * C::kCols, mb * BN, pol_keep);
        if constexpr (W4) {
          const int64_t meta = static_cast<int64_t>(nt) * ng + kb / 2;
          bulk_load_hint(st + C::kXBytes, codes + (static_cast<int64_t>(nt) * KB + kb) * 4096, 4096, &full[s],
                         pol_stream);
          bulk_load(st + C::kXBytes + 4096, scales + meta * kTileN, 256, &full[s]);
          bulk_load(st + C::kXBytes + 4096 + 256, zeros + meta * (kTileN / 2), 64, &full[s]);
        } else {
          tma_load_2d_hint(st + C::kXBytes, &tmap_w, &full[s], kb * C::kCols, nt * kTileN, pol_stream);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = W4 ? idesc_make(1, 1, 128, BN) : idesc_make(0, 0, 128, BN);
      bool ok = true;
      for (int it = 0; it < nkb && ok; ++it) {
        const int s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1;
        if (!mbar_wait(&full[s], ph, kWaitLimitNs)) {
          ok = false;
          break;
        }
        uint32_t a_addr;
        const int a = W4 ? it % C::kAStages : 0;
        if constexpr (W4) {
          if (!mbar_wait(&a_full[a], (it / C::kAStages) & 1, kWaitLimitNs)) {
            ok = false;
            break;
          }
          a_addr = smem_u32(aring + a * C::kAStage);
        } else {
          a_addr = smem_u32(ring + s * C::kStage + C::kXBytes);
        }
        tc_fence_after();
        const uint32_t b_addr = smem_u32(ring + s * C::kStage);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 32 bytes of K per MMA
          const uint64_t ad = sdesc_sw128(a_addr + kk * 32);
          const uint64_t bd = sdesc_sw128(b_addr + kk * 32);
          if constexpr (W4)
            mma_f16(tmem_d, ad, bd, idesc, (it | kk) != 0);
          else
            mma_f8(tmem_d, ad, bd, idesc, (it | kk) != 0);
        }
        mma_commit(&empty[s]);
        if constexpr (W4) mma_commit(&a_empty[a]);
      }
      if (!ok) set_error(err, QLIN_ERR_TIMEOUT);
      mma_commit(tmem_full);
    }
  } else {
    // ---------------------------------------------------------------- dequant + epilogue
    const int t = threadIdx.x - 64;  // 0..127
    bool ok = true;
    if constexpr (W4) {
      const int r = t;  // weight row of the tile this thread dequantises
      for (int it = 0; it < nkb; ++it) {
        const int s = it % C::kStages;
        const int a = it % C::kAStages;
        const bool got = mbar_wait(&full[s], (it / C::kStages) & 1, kWaitLimitNs) &&
                         mbar_wait(&a_empty[a], ((it / C::kAStages) & 1) ^ 1, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, got)) {  // leave the loop as a whole warp
          ok = false;
          break;
        }
        const uint8_t* st = ring + s * C::kStage + C::kXBytes;
        const uint4 c0 = *reinterpret_cast<const uint4*>(st + r * 16);
        const uint4 c1 = *reinterpret_cast<const uint4*>(st + 2048 + r * 16);
        const float scale = __half2float(*reinterpret_cast<const __half*>(st + 4096 + r * 2));
        const uint32_t zb = st[4096 + 256 + r / 2];
        const float zq = static_cast<float>((r & 1) ? (zb >> 4) : (zb & 15u));
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // codes are in registers now
        const __nv_bfloat162 zoff = __float2bfloat162_rn(128.0f + zq);
        const __nv_bfloat162 s2 = __float2bfloat162_rn(scale);
        uint8_t* arow = aring + a * C::kAStage + r * 128;
        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 16-byte chunk c holds columns 8c..8c+7
          const uint4 v = dequant8(words[c], zoff, s2);
          *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[a]);
      }
      if (!ok) set_error(err, QLIN_ERR_TIMEOUT);
    }
    // epilogue: TMEM lane quadrant is fixed by the warp's rank modulo 4
    const int quad = warp & 3;
    const int64_t n = static_cast<int64_t>(nt) * kTileN + quad * 32 + lane;
    const bool have = __all_sync(0xffffffffu, ok && mbar_wait(tmem_full, 0, kWaitLimitNs));
    if (!have) {
      set_error(err, QLIN_ERR_TIMEOUT);
      s_fail = 1;
    }
    tc_fence_after();
    const int64_t mbase = static_cast<int64_t>(mb) * BN;
    const float s_w = W4 ? 1.0f : *sw;
    if (have) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem_d + (static_cast<uint32_t>(quad * 32) << 16) + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t m = mbase + c0 + i;
          if (m < M) {
            const float acc = __uint_as_float(v[i]);
            if (splits == 1) {
              Y[m * N + n] = W4 ? to_bf16(acc) : to_bf16((acc * __ldg(sx + m)) * s_w);
            } else {
              __stcg(partials + (static_cast<int64_t>(split) * M + m) * N + n, acc);
            }
          }
        }
      }
    }
    if (splits > 1) {
      __threadfence();
      named_bar_epi();
      const int64_t tile = static_cast<int64_t>(mb) * gridDim.x + nt;
      if (t == 0) s_last = !s_fail && (atomicAdd(counters + tile, 1u) == static_cast<uint32_t>(splits - 1));
      named_bar_epi();
      if (s_last) {
        __threadfence();
        // the last CTA of the tile adds the K ranges in order; row n per thread
        const int64_t mend = imin64(M, mbase + BN);
        for (int64_t m = mbase; m < mend; ++m) {
          float acc = 0.0f;
          for (int s = 0; s < splits; ++s) acc += __ldcg(partials + (static_cast<int64_t>(s) * M + m) * N + n);
          Y[m * N + n] = W4 ? to_bf16(acc) : to_bf16((acc * __ldg(sx + m)) * s_w);
        }
        named_bar_epi();
        if (t == 0) counters[tile] = 0u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_d, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ self-test

// A barrier nobody arrives on: the bounded wait must give up and report.
__global__ void wait_timeout_kernel(uint64_t limit_ns, int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) set_error(err, QLIN_ERR_TIMEOUT);
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, int* err, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(limit_ns, err);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ planning

static int pick_bn(int64_t M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

static TcPlan plan_tc(int64_t M, int64_t N, int64_t K, int num_sms, int cols) {
  TcPlan p;
  p.bn = pick_bn(M);
  p.mblocks = (M + p.bn - 1) / p.bn;
  const int64_t tiles = (N / kTileN) * p.mblocks;
  const int64_t KB = K / cols;
  // One CTA per SM.  Pick the split count whose CTAs fill whole waves best
  // (busy SM-slots / all slots of the waves), with at least 4 blocks of K per
  // CTA; on a tie take fewer splits (less partial-sum traffic).
  int s = 1;
  double best = -1.0;
  const int64_t max_s = KB / 4 > 0 ? (KB / 4 < 32 ? KB / 4 : 32) : 1;
  for (int c = 1; c <= max_s; ++c) {
    const int64_t ctas = tiles * c;
    const int64_t waves = (ctas + num_sms - 1) / num_sms;
    const double eff = static_cast<double>(ctas) / static_cast<double>(waves * num_sms);
    if (eff > best + 0.02) {
      best = eff;
      s = c;
    }
  }
  const int per = static_cast<int>((KB + s - 1) / s);
  s = static_cast<int>((KB + per - 1) / per);
  p.split.splits = s;
  p.split.kb_per_split = per;
  p.split.tiles = tiles;
  p.split.ws_bytes = s > 1 ? counters_bytes(tiles) + sizeof(float) * static_cast<size_t>(s) * M * N : 0;
  return p;
}

TcPlan plan_w4a16_tc(int64_t M, int64_t N, int64_t K, int num_sms) { return plan_tc(M, N, K, num_sms, 64); }
TcPlan plan_w8a8_tc(int64_t M, int64_t N, int64_t K, int num_sms) { return plan_tc(M, N, K, num_sms, 128); }

template <int BN, bool W4>
static cudaError_t launch_tc(const CUtensorMap& tx, const CUtensorMap& tw, const uint8_t* codes,
                             const uint16_t* scales, const uint8_t* zeros, const float* sx, const float* sw,
                             uint16_t* Y, int64_t M, int64_t N, int64_t K, const TcPlan& plan, void* ws, int* err,
                             cudaStream_t st) {
  using C = TcCfg<BN, W4>;
  cudaError_t e = set_smem_once(tc_gemm_kernel<BN, W4>, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  uint32_t* counters = static_cast<uint32_t*>(ws);
  float* partials = ws ? reinterpret_cast<float*>(static_cast<char*>(ws) + counters_bytes(plan.split.tiles)) : nullptr;
  dim3 grid(static_cast<unsigned>(N / kTileN), plan.split.splits, static_cast<unsigned>(plan.mblocks));
  tc_gemm_kernel<BN, W4><<<grid, 192, C::kSmemBytes, st>>>(tx, tw, codes, scales, zeros, sx, sw, Y, M, N, K,
                                                           plan.split.kb_per_split, plan.split.splits, partials,
                                                           counters, err);
  return cudaGetLastError();
}

cudaError_t launch_w4a16_tc(const uint16_t* X, const uint8_t* codes, const uint16_t* scales, const uint8_t* zeros,
                            uint16_t* Y, int64_t M, int64_t N, int64_t K, const TcPlan& plan, void* ws, int* err,
                            cudaStream_t st) {
  CUtensorMap tx, tw;
  if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, K * 2, 64, plan.bn))
    return cudaErrorInvalidValue;
  tw = tx;
  switch (plan.bn) {
    case 16: return launch_tc<16, true>(tx, tw, codes, scales, zeros, nullptr, nullptr, Y, M, N, K, plan, ws, err, st);
    case 32: return launch_tc<32, true>(tx, tw, codes, scales, zeros, nullptr, nullptr, Y, M, N, K, plan, ws, err, st);
    case 64: return launch_tc<64, true>(tx, tw, codes, scales, zeros, nullptr, nullptr, Y, M, N, K, plan, ws, err, st);
    case 128: return launch_tc<128, true>(tx, tw, codes, scales, zeros, nullptr, nullptr, Y, M, N, K, plan, ws, err, st);
    default: return launch_tc<256, true>(tx, tw, codes, scales, zeros, nullptr, nullptr, Y, M, N, K, plan, ws, err, st);
  }
}

cudaError_t launch_w8a8_tc(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, uint16_t* Y,
                           int64_t M, int64_t N, int64_t K, const TcPlan& plan, void* ws, int* err,
                           cudaStream_t st) {
  CUtensorMap tx, tw;
  if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Xq, K, M, K, 128, plan.bn)) return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wq, K, N, K, 128, 128)) return cudaErrorInvalidValue;
  switch (plan.bn) {
    case 16: return launch_tc<16, false>(tx, tw, nullptr, nullptr, nullptr, sx, sw, Y, M, N, K, plan, ws, err, st);
    case 32: return launch_tc<32, false>(tx, tw, nullptr, nullptr, nullptr, sx, sw, Y, M, N, K, plan, ws, err, st);
    case 64: return launch_tc<64, false>(tx, tw, nullptr, nullptr, nullptr, sx, sw, Y, M, N, K, plan, ws, err, st);
    case 128: return launch_tc<128, false>(tx, tw, nullptr, nullptr, nullptr, sx, sw, Y, M, N, K, plan, ws, err, st);
    default: return launch_tc<256, false>(tx, tw, nullptr, nullptr, nullptr, sx, sw, Y, M, N, K, plan, ws, err, st);
  }
}

}  // namespace qlin
