// W8A8 FP8 for small M (decode): split-K kernel whose inner product runs on
// the tensor cores through register-level mma.sync with E4M3 operands.
//
// [LP] S4 per-token / per-tensor scales, S7 E4M3, S8 current scaling, S22
// FP32 accumulation:  Y[m][n] = bf16( (sum_k Xq[m][k] Wq[n][k]) * sx[m] * sw ).
// The weights need no unpacking: an m16n8k32 A fragment is four 32-bit words
// of E4M3 bytes, loaded with ldmatrix from a 128-byte-swizzled tile, and the
// activation rows give the B fragments the same way.  The scales are applied
// once, to the FP32 sums.
//
// One CTA = one 128-row tile x one K range.  Warp 4 brings in, per stage of
// 256 columns, the tile's weights (two TMA boxes of 128 rows x 128 bytes,
// issued before waiting for the previous kernel on the stream) and every
// token's activation bytes (bulk copies).  Warps 0-3 each own 32 rows (two m16
// blocks sharing every B fragment) and every token (one or two n8 blocks).
// The K ranges of one tile run as a thread-block cluster and add their
// partial sums through distributed shared memory, in rank order.
#include <cuda_bf16.h>

#include <array>
#include <mutex>
#include <type_traits>
#include <unordered_map>

#include "qlin_internal.cuh"
#include "qlin_ptx.cuh"

namespace qlin {

constexpr int k8StageCols = 256;                  // K columns (bytes) per stage
constexpr int k8WBytes = kTileN * k8StageCols;    // two 128 x 128 B boxes
constexpr int k8XRow = k8StageCols + 16;          // 272 B per token row (conflict-free ldmatrix)
constexpr int k8RowBlocks = 2;                    // m16 row blocks per consumer warp
constexpr int k8Consumers = kTileN / (16 * k8RowBlocks);
constexpr int k8Producer = k8Consumers;
constexpr int k8Threads = (k8Consumers + 1) * 32;
constexpr uint64_t k8WaitNs = 2000000000ull;
constexpr int k8MaxCluster = 16;
constexpr int k8RedRows = 144;                    // >= splits x ceil(128 / splits) for splits <= 16

template <int NT>
struct Mma8Cfg {
  static constexpr int kTok = 8 * NT;
  static constexpr int kXOff = k8WBytes;
  static constexpr int kStage = ((kXOff + kTok * k8XRow) + 1023) / 1024 * 1024;
  static constexpr int kStages = NT == 1 ? 3 : 2;  // two CTAs per SM
  static constexpr int kRedFloats = kTok * k8RedRows;
  static constexpr int kSmem = 1024 + kStages * kStage + 256 + kRedFloats * 4;
  static_assert(2 * kSmem <= 227 * 1024, "two CTAs per SM");
};

__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <int NT, bool EPI>  // NT: n8 token blocks (M <= 8 NT); EPI: bias / activation epilogue
__global__ void __launch_bounds__(k8Threads, 2) w8a8_mma_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                                               const uint8_t* __restrict__ Xq,
                                                               const float* __restrict__ sx,
                                                               const float* __restrict__ sw,
                                                               uint16_t* __restrict__ Y, int64_t M, int64_t N,
                                                               int64_t K, int stages_per_split, int splits, int* err,
                                                               Epi epi) {
  using C = Mma8Cfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + C::kStages * C::kStage);
  uint64_t* empty = full + C::kStages;
  uint64_t* red_bar = empty + C::kStages;
  float* red = reinterpret_cast<float*>(ring + C::kStages * C::kStage + 256);
  __shared__ volatile int s_abort;

  const int split = blockIdx.x, nt = blockIdx.y;  // the K ranges of a tile form one cluster (rank = split)
  const int64_t KS = K / k8StageCols;
  const int s0 = split * stages_per_split;
  const int nst = static_cast<int>(imin64(KS, s0 + stages_per_split)) - s0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mrows = static_cast<int>(imin64(M, C::kTok));

  auto row_lo = [&](int q) { return q * kTileN / splits; };
  const int r_lo = row_lo(split), r_n = row_lo(split + 1) - r_lo;
  const int rstride = (kTileN + splits - 1) / splits;
  const int groups = NT == 1 ? (mrows + 1) / 2 : 4;

  const uint32_t tx = k8WBytes + mrows * k8StageCols;
  auto issue_w = [&](int i) {  // weights of stage i: two boxes of 128 rows x 128 bytes
    uint8_t* st = ring + (i % C::kStages) * C::kStage;
    uint64_t* bar = &full[i % C::kStages];
    const int k0 = (s0 + i) * k8StageCols;
    mbar_arrive_expect_tx(bar, tx);
    tma_load_2d(st, &tmap_w, bar, k0, nt * kTileN);
    tma_load_2d(st + kTileN * 128, &tmap_w, bar, k0 + 128, nt * kTileN);
  };
  auto issue_x = [&](int i) {  // activation bytes of stage i
    uint8_t* st = ring + (i % C::kStages) * C::kStage;
    const int64_t k0 = static_cast<int64_t>(s0 + i) * k8StageCols;
    for (int m = 0; m < mrows; ++m)
      bulk_load(st + C::kXOff + m * k8XRow, Xq + m * K + k0, k8StageCols, &full[i % C::kStages]);
  };
  if (warp == k8Producer && lane == 0) {
    prefetch_tensormap(&tmap_w);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], k8Consumers);
    }
    mbar_init(red_bar, 1);
    fence_mbar_init();
    if (splits > 1) mbar_arrive_expect_tx(red_bar, static_cast<uint32_t>(splits * r_n * groups * 2 * NT * 4));
    s_abort = 0;
    for (int i = 0; i < nst && i < C::kStages; ++i) issue_w(i);  // weights first: they do not depend on the stream
  }
  // token rows >= M are never copied: zero them once so B fragments need no bounds test
  for (int idx = threadIdx.x; idx < C::kStages * (C::kTok - mrows) * (k8XRow / 16); idx += k8Threads) {
    const int per = (C::kTok - mrows) * (k8XRow / 16);
    const int stg = idx / per, rem = idx % per;
    const int row = mrows + rem / (k8XRow / 16), c16 = rem % (k8XRow / 16);
    *reinterpret_cast<uint4*>(ring + stg * C::kStage + C::kXOff + row * k8XRow + c16 * 16) = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (splits > 1) cluster_arrive_relaxed();
  grid_dep_wait();
  grid_dep_launch();

  const int gq = lane >> 2, tq = lane & 3;
  float acc[k8RowBlocks][NT][4];
#pragma unroll
  for (int rb = 0; rb < k8RowBlocks; ++rb)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[rb][j][e] = 0.0f;

  if (warp == k8Producer) {
    if (lane == 0) {
      for (int i = 0; i < nst && i < C::kStages; ++i) issue_x(i);
      for (int i = C::kStages; i < nst; ++i) {
        if (!mbar_wait(&empty[i % C::kStages], ((i / C::kStages) & 1) ^ 1, k8WaitNs, &s_abort)) {
          set_error(err, QLIN_ERR_TIMEOUT);
          s_abort = 1;
          break;
        }
        issue_w(i);
        issue_x(i);
      }
    }
  } else {
    // consumers: rows 32 warp .. 32 warp + 31 (row blocks rb: 16 rows each)
    if (splits > 1) cluster_wait();
    // ldmatrix lane roles: A: matrix mi = lane / 8 is rows (mi & 1) * 8 + lane % 8 of
    // the row block, bytes (mi >> 1) * 16 of the k-step; B: token row 8j + lane % 8,
    // bytes (lane / 8) * 16 of a pair of k-steps
    const int mi = lane >> 3;
    for (int i = 0; i < nst; ++i) {
      const int slot = i % C::kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (i / C::kStages) & 1, k8WaitNs, &s_abort))) {
        set_error(err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      const uint32_t st = smem_u32(ring + slot * C::kStage);
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {  // pairs of 32-column k-steps
        uint32_t b[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
          ldsm_x4(st + C::kXOff + (j * 8 + (lane & 7)) * k8XRow + kp * 64 + mi * 16, b[j][0], b[j][1], b[j][2],
                  b[j][3]);
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          const int ks = kp * 2 + kh;  // k-step: bytes 32 ks .. 32 ks + 31 of the stage
          const uint32_t box = st + (ks >> 2) * (kTileN * 128);
#pragma unroll
          for (int rb = 0; rb < k8RowBlocks; ++rb) {
            const int row = warp * 32 + rb * 16 + (mi & 1) * 8 + (lane & 7);
            const int chunk = (ks & 3) * 2 + (mi >> 1);  // 16-byte chunk of the 128-byte row
            uint32_t a[4];
            ldsm_x4(box + row * 128 + ((chunk ^ (row & 7)) << 4), a[0], a[1], a[2], a[3]);
#pragma unroll
            for (int j = 0; j < NT; ++j) mma_e4m3_16832(acc[rb][j], a, b[j][2 * kh], b[j][2 * kh + 1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
  }

  // ---------------------------------------------------------------- outputs
  // this thread's outputs: row 32 warp + 16 rb + gq + 8 hr, token 8 j + 2 tq + e
  const float s_w = __ldg(sw);
  if (splits == 1) {
    if (warp < k8Consumers) {
#pragma unroll
      for (int rb = 0; rb < k8RowBlocks; ++rb)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int64_t n = static_cast<int64_t>(nt) * kTileN + warp * 32 + 16 * rb + gq + hr * 8;
          float o[2 * NT];
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int64_t m = j * 8 + 2 * tq + e;
              o[2 * j + e] = m < M ? (acc[rb][j][hr * 2 + e] * __ldg(sx + m)) * s_w : 0.0f;
            }
          if constexpr (EPI) epi_run(epi.act, o, epi_bias(epi, n));
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int64_t m = j * 8 + 2 * tq + e;
              if (m < M) Y[m * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(o[2 * j + e]));
            }
        }
    }
    return;
  }
  // Split K: each CTA sends every row's token sums to the row's owner with
  // asynchronous remote stores that complete on the owner's red_bar; the owner
  // adds the slots in rank order (deterministic) and writes Y.
  __syncwarp();
  if (warp >= k8Consumers) cluster_wait();
  if (warp < k8Consumers && tq < groups) {
    const uint32_t red_u32 = smem_u32(red), bar_u32 = smem_u32(red_bar);
#pragma unroll
    for (int rb = 0; rb < k8RowBlocks; ++rb)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = warp * 32 + 16 * rb + gq + hr * 8;
        const int q = (r * splits + splits - 1) / kTileN;  // owner: the last rank with lo(q) <= r
        const uint32_t dst = cluster_map(red_u32, static_cast<uint32_t>(q)) +
                             static_cast<uint32_t>(((split * rstride + r - row_lo(q)) * C::kTok + tq * 2 * NT) * 4);
        const uint32_t dbar = cluster_map(bar_u32, static_cast<uint32_t>(q));
        if constexpr (NT == 1) {
          st_async_v2(dst, acc[rb][0][hr * 2], acc[rb][0][hr * 2 + 1], dbar);
        } else {
#pragma unroll
          for (int j = 0; j < NT; j += 2)
            st_async_v4(dst + j * 8, acc[rb][j][hr * 2], acc[rb][j][hr * 2 + 1], acc[rb][j + 1][hr * 2],
                        acc[rb][j + 1][hr * 2 + 1], dbar);
        }
      }
  }
  if (!mbar_wait_cluster(red_bar, 0, k8WaitNs)) {
    set_error(err, QLIN_ERR_TIMEOUT);
    return;
  }
  for (int idx = threadIdx.x; idx < r_n * mrows; idx += k8Threads) {
    const int m = idx / r_n, rl = idx % r_n;
    const int slot = NT == 1 ? m : ((m & 7) >> 1) * 2 * NT + (m >> 3) * 2 + (m & 1);
    const float* src = red + rl * C::kTok + slot;
    float v = 0.0f;
    for (int p = 0; p < splits; ++p) v += src[p * rstride * C::kTok];
    const int64_t n = static_cast<int64_t>(nt) * kTileN + r_lo + rl;
    v = (v * __ldg(sx + m)) * s_w;
    if constexpr (EPI) v = epi_apply(epi, v, n);
    Y[static_cast<int64_t>(m) * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

// Clusters of `cs` CTAs of w8a8_mma_kernel<NT, *> that fit at once, per device.
template <int NT>
static int max_active_clusters8(int cs) {
  static std::mutex mu;
  static std::unordered_map<int, std::array<int, k8MaxCluster + 1>> table;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  auto it = table.find(dev);
  if (it == table.end()) {
    std::array<int, k8MaxCluster + 1> t{};
    if (set_smem_once(w8a8_mma_kernel<NT, false>, Mma8Cfg<NT>::kSmem, true) == cudaSuccess) {
      for (int c = 1; c <= k8MaxCluster; ++c) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(c), 1);
        cfg.blockDim = dim3(k8Threads);
        cfg.dynamicSmemBytes = Mma8Cfg<NT>::kSmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(c);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, w8a8_mma_kernel<NT, false>, &cfg) != cudaSuccess) n = 0;
        t[c] = n;
      }
    }
    (void)cudaGetLastError();
    it = table.emplace(dev, t).first;
  }
  return it->second[cs];
}

bool mma8_path_ok(int64_t M, int64_t K) { return M >= 1 && M <= 16 && K % k8StageCols == 0; }

// Split count by the same time model as the W4A16 small-M kernel (waves of
// co-resident clusters x stages per CTA, bandwidth shared by the CTAs of a
// wave, capped by the bytes they keep in flight).
SplitPlan plan_w8a8_mma(int64_t M, int64_t N, int64_t K, int num_sms) {
  (void)num_sms;
  SplitPlan p;
  const int64_t tiles = N / kTileN;
  const int64_t KS = K / k8StageCols;
  const bool nt1 = M <= 8;
  const double bw = 6.5e12, latency = 2.5e-6, startup = 3e-6;
  const int ring = nt1 ? Mma8Cfg<1>::kStages : Mma8Cfg<2>::kStages;
  const double stage_bytes = k8WBytes + static_cast<double>(k8StageCols) * static_cast<double>(M);
  const int64_t cap = KS < k8MaxCluster ? KS : k8MaxCluster;
  int64_t best_s = 1;
  double best_t = 1e30;
  for (int64_t c = 1; c <= cap; ++c) {
    const int64_t per = (KS + c - 1) / c;
    const int64_t s = (KS + per - 1) / per;
    if (s != c) continue;
    const int64_t fit = nt1 ? max_active_clusters8<1>(static_cast<int>(s)) : max_active_clusters8<2>(static_cast<int>(s));
    if (fit <= 0) continue;
    const int64_t waves = (tiles + fit - 1) / fit;
    const double conc = static_cast<double>((tiles < fit ? tiles : fit) * s);
    const double inflight = conc * ring * stage_bytes / latency;
    const double bw_eff = inflight < bw ? inflight : bw;
    const double t = static_cast<double>(waves) * (startup + static_cast<double>(per) * stage_bytes * conc / bw_eff);
    if (t < best_t * 0.98) {
      best_t = t;
      best_s = s;
    }
  }
  const int64_t per = (KS + best_s - 1) / best_s;
  p.splits = static_cast<int>(best_s);
  p.kb_per_split = static_cast<int>(per);  // here: stages of 256 columns per split
  p.tiles = tiles;
  p.ws_bytes = 0;
  return p;
}

template <int NT, bool EPI>
static cudaError_t launch_mma8(const CUtensorMap& tw, const uint8_t* Xq, const float* sx, const float* sw,
                               uint16_t* Y, int64_t M, int64_t N, int64_t K, const SplitPlan& plan, int* err,
                               cudaStream_t st, const Epi& epi) {
  cudaError_t e = set_smem_once(w8a8_mma_kernel<NT, EPI>, Mma8Cfg<NT>::kSmem, true);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.splits), static_cast<unsigned>(N / kTileN));
  cfg.blockDim = dim3(k8Threads);
  cfg.dynamicSmemBytes = Mma8Cfg<NT>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(plan.splits);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, w8a8_mma_kernel<NT, EPI>, tw, Xq, sx, sw, Y, M, N, K, plan.kb_per_split,
                            plan.splits, err, epi);
}

cudaError_t launch_w8a8_mma(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, uint16_t* Y,
                            int64_t M, int64_t N, int64_t K, const SplitPlan& plan, int* err, cudaStream_t st,
                            const Epi& epi) {
  CUtensorMap tw;
  if (!encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wq, K, N, K, 128, kTileN)) return cudaErrorInvalidValue;
  const bool fused = epi.bias != nullptr || epi.act != QLIN_ACT_NONE;
  if (M <= 8)
    return fused ? launch_mma8<1, true>(tw, Xq, sx, sw, Y, M, N, K, plan, err, st, epi)
                 : launch_mma8<1, false>(tw, Xq, sx, sw, Y, M, N, K, plan, err, st, epi);
  return fused ? launch_mma8<2, true>(tw, Xq, sx, sw, Y, M, N, K, plan, err, st, epi)
               : launch_mma8<2, false>(tw, Xq, sx, sw, Y, M, N, K, plan, err, st, epi);
}

}  // namespace qlin
