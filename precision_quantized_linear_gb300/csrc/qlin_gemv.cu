// Small-M (decode) kernels on CUDA cores, split-K over a grid of
// (128-row tile, K range, token chunk) CTAs.  [TP]: at small batch the layer
// is bound by the bytes of the weights, so these kernels stream the packed
// weights once with 128-bit loads and keep the arithmetic per weight small.
//
// Split-K partial sums go to the workspace; the last CTA of a tile (found
// with one atomic counter per tile, no waiting) adds them in split order, so
// results do not depend on scheduling.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qlin_internal.cuh"
#include "qlin_ptx.cuh"

namespace qlin {

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Last-arriver split-K reduction for one 128-row tile and `mcount` tokens.
// Every thread owns one row n (threadIdx.x) and holds `mine[m]`.
template <int MT, typename Epi>
__device__ __forceinline__ void splitk_finish(const float (&mine)[MT], int mcount, int m0, int64_t n, int64_t M,
                                              int64_t N, int split, int splits, int64_t tile, float* partials,
                                              uint32_t* counters, Epi epi) {
  __shared__ int s_last;
  if (splits == 1) {
#pragma unroll
    for (int m = 0; m < MT; ++m)
      if (m < mcount) epi(m0 + m, n, mine[m]);
    return;
  }
#pragma unroll
  for (int m = 0; m < MT; ++m)
    if (m < mcount) __stcg(partials + (static_cast<int64_t>(split) * M + m0 + m) * N + n, mine[m]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(counters + tile, 1u) == static_cast<uint32_t>(splits - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    if (m >= mcount) continue;
    float acc = 0.0f;
    for (int s = 0; s < splits; ++s) {  // read and clear: the workspace is left zero-filled
      float* p = partials + (static_cast<int64_t>(s) * M + m0 + m) * N + n;
      acc += __ldcg(p);
      __stcg(p, 0.0f);
    }
    epi(m0 + m, n, acc);
  }
  if (threadIdx.x == 0) counters[tile] = 0u;
}

// ------------------------------------------------------------------ W4A16

// Two adjacent columns of a word as exact floats 128 + q: the AND/OR puts each
// nibble in the low mantissa bits of a BF16 with exponent 2^7, and a BF16 is
// the top half of an FP32.
__device__ __forceinline__ float2 nib_pair(uint32_t w) {
  const uint32_t v = (w & 0x000F000Fu) | 0x43004300u;
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// [LP] S11: packed INT4 weights -> unpack -> multiply with BF16 activations ->
// accumulate in FP32.  The zero-point and scale are applied once per 64
// columns: sum_k x (q - z) s = s (sum_k x (128 + q) - (128 + z) sum_k x).
template <int MT>
__global__ void __launch_bounds__(128) w4a16_gemv_kernel(const uint16_t* __restrict__ X,
                                                         const uint8_t* __restrict__ codes,
                                                         const uint16_t* __restrict__ scales,
                                                         const uint8_t* __restrict__ zeros, uint16_t* __restrict__ Y,
                                                         int64_t M, int64_t N, int64_t K, int kb_per_split, int splits,
                                                         float* partials, uint32_t* counters, Epi epi) {
  extern __shared__ float4 smem_f4[];
  float* smem = reinterpret_cast<float*>(smem_f4);
  const int nt = blockIdx.x, split = blockIdx.y;
  const int m0 = blockIdx.z * MT;
  const int mcount = static_cast<int>(imin64(MT, M - m0));
  const int64_t KB = K / kTileK;
  const int kb0 = split * kb_per_split;
  const int kb1 = static_cast<int>(imin64(KB, kb0 + kb_per_split));
  const int nkb = kb1 - kb0;
  const int KR = nkb * kTileK;
  float* xs = smem;                 // [MT][KR]
  float* xsum = xs + MT * KR;       // [MT][nkb]
  float* red = xsum + MT * ((nkb + 3) & ~3);  // [4][MT][128]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // the packed weights never depend on the previous kernel on the stream:
  // start streaming them before waiting for it
  const int64_t ng = K / kGroup;
  const uint8_t* tbase = codes + static_cast<int64_t>(nt) * KB * 4096;
  uint4 cn[4][2];
  if (kb0 + warp < kb1) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        cn[i][h] = ldg_stream(tbase + static_cast<int64_t>(kb0 + warp) * 4096 + h * 2048 + (lane + 32 * i) * 16);
  }
  grid_dep_wait();
  grid_dep_launch();

  for (int idx = threadIdx.x; idx < MT * (KR / 8); idx += 128) {
    const int m = idx / (KR / 8), i8 = idx % (KR / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (m < mcount) v = *reinterpret_cast<const uint4*>(X + (m0 + m) * K + static_cast<int64_t>(kb0) * kTileK + i8 * 8);
    float4* d = reinterpret_cast<float4*>(xs + m * KR + i8 * 8);
    d[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                       __uint_as_float(v.y & 0xFFFF0000u));
    d[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u), __uint_as_float(v.w << 16),
                       __uint_as_float(v.w & 0xFFFF0000u));
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < MT * nkb; idx += 128) {
    const int m = idx / nkb, b = idx % nkb;
    const float* p = xs + m * KR + b * kTileK;
    float s = 0.0f;
    for (int i = 0; i < kTileK; ++i) s += p[i];
    xsum[m * ((nkb + 3) & ~3) + b] = s;
  }
  __syncthreads();

  float y[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) y[m][i] = 0.0f;

  for (int kb = kb0 + warp; kb < kb1; kb += 4) {
    uint4 c[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) c[i][h] = cn[i][h];
    if (kb + 4 < kb1) {  // software pipelining: next block's codes are in flight during this block's math
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          cn[i][h] = ldg_stream(tbase + static_cast<int64_t>(kb + 4) * 4096 + h * 2048 + (lane + 32 * i) * 16);
    }
    const int64_t sz = static_cast<int64_t>(nt) * ng + kb / 2;
    float sc[4], cz[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane + 32 * i;
      sc[i] = __half2float(__ushort_as_half(__ldg(scales + sz * kTileN + r)));
      const uint32_t zb = __ldg(zeros + sz * (kTileN / 2) + r / 2);
      cz[i] = 128.0f + static_cast<float>((r & 1) ? (zb >> 4) : (zb & 15u));
    }
    const int kl = (kb - kb0) * kTileK;
    float2 dot[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) dot[m][i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 xv[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m) {  // word j, position pair p: columns 16(p/2) + 8(p%2) + 2j, +1
          const float2* xp = reinterpret_cast<const float2*>(xs + m * KR + kl + h * 32 + j * 2);
#pragma unroll
          for (int p = 0; p < 4; ++p) xv[m][p] = xp[4 * p];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t w = (j == 0) ? c[i][h].x : (j == 1) ? c[i][h].y : (j == 2) ? c[i][h].z : c[i][h].w;
          float2 f[4];
          f[0] = nib_pair(w);
          f[1] = nib_pair(w >> 4);
          f[2] = nib_pair(w >> 8);
          f[3] = nib_pair(w >> 12);
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int t = 0; t < 4; ++t) dot[m][i] = __ffma2_rn(xv[m][t], f[t], dot[m][i]);
        }
      }
    }
    const int xb = kb - kb0;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float d = dot[m][i].x + dot[m][i].y;
        y[m][i] = fmaf(sc[i], fmaf(-cz[i], xsum[m * ((nkb + 3) & ~3) + xb], d), y[m][i]);
      }
  }

#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[(warp * MT + m) * kTileN + lane + 32 * i] = y[m][i];
  __syncthreads();
  float mine[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    float a = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) a += red[(w * MT + m) * kTileN + threadIdx.x];
    mine[m] = a;
  }
  const int64_t n = static_cast<int64_t>(nt) * kTileN + threadIdx.x;
  const int64_t tile = static_cast<int64_t>(blockIdx.z) * gridDim.x + nt;
  splitk_finish<MT>(mine, mcount, m0, n, M, N, split, splits, tile, partials, counters,
                    [&](int64_t m, int64_t nn, float v) { Y[m * N + nn] = f32_to_bf16_rn(epi_apply(epi, v, nn)); });
}

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream finishes; it waits for that kernel (grid
// dependency) before touching activations or outputs.
template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern kernel, dim3 grid, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

static size_t w4_gemv_smem(int mt, int kb_per_split) {
  const int KR = kb_per_split * kTileK;
  return sizeof(float) * (static_cast<size_t>(mt) * KR + mt * ((kb_per_split + 3) & ~3) + 4 * mt * kTileN);
}

static int gemv_mt(int64_t M) { return M >= 4 ? 4 : (M >= 2 ? 2 : 1); }

bool gemv_m_ok(int64_t M) { return (M + gemv_mt(M) - 1) / gemv_mt(M) <= 65535; }

// Split so that about two CTAs per SM stream weights, with x for one K range
// of at most 8192/MT columns in shared memory.
static SplitPlan plan_splits(int64_t tiles_mn, int64_t KB, int num_sms, int max_kb) {
  SplitPlan p;
  int s = static_cast<int>((2LL * num_sms + tiles_mn - 1) / tiles_mn);
  if (s < 1) s = 1;
  const int64_t min_s = (KB + max_kb - 1) / max_kb;
  if (s < min_s) s = static_cast<int>(min_s);
  if (s > KB) s = static_cast<int>(KB);
  if (s > 32) s = s < min_s ? static_cast<int>(min_s) : 32;
  int per = static_cast<int>((KB + s - 1) / s);
  s = static_cast<int>((KB + per - 1) / per);  // no empty ranges
  p.splits = s;
  p.kb_per_split = per;
  p.tiles = tiles_mn;
  return p;
}

SplitPlan plan_w4a16_gemv(int64_t M, int64_t N, int64_t K, int num_sms) {
  const int mt = gemv_mt(M);
  const int64_t tiles = (N / kTileN) * ((M + mt - 1) / mt);
  SplitPlan p = plan_splits(tiles, K / kTileK, num_sms, 8192 / mt / kTileK);
  if (p.splits > 1) {
    p.ws_bytes = counters_bytes(tiles) + sizeof(float) * static_cast<size_t>(p.splits) * M * N;
    p.zero_bytes = counters_bytes(tiles);
  }
  return p;
}

cudaError_t launch_w4a16_gemv(const uint16_t* X, const uint8_t* codes, const uint16_t* scales, const uint8_t* zeros,
                              uint16_t* Y, int64_t M, int64_t N, int64_t K, const SplitPlan& plan, void* ws,
                              cudaStream_t st, const Epi& epi) {
  const int mt = gemv_mt(M);
  dim3 grid(static_cast<unsigned>(N / kTileN), plan.splits, static_cast<unsigned>((M + mt - 1) / mt));
  const size_t smem = w4_gemv_smem(mt, plan.kb_per_split);
  uint32_t* counters = static_cast<uint32_t*>(ws);
  float* partials = ws ? reinterpret_cast<float*>(static_cast<char*>(ws) + counters_bytes(plan.tiles)) : nullptr;
  cudaError_t e = cudaSuccess;
  switch (mt) {
#define QLIN_W4GEMV(MTV)                                                                                 \
  case MTV:                                                                                              \
    e = set_smem_once(w4a16_gemv_kernel<MTV>, 64 * 1024);                                                \
    if (e != cudaSuccess) return e;                                                                      \
    e = launch_pdl(w4a16_gemv_kernel<MTV>, grid, smem, st, X, codes, scales, zeros, Y, M, N, K,            \
                   plan.kb_per_split, plan.splits, partials, counters, epi);                             \
    break;
    QLIN_W4GEMV(1)
    QLIN_W4GEMV(2)
    QLIN_W4GEMV(4)
#undef QLIN_W4GEMV
  }
  return e;
}

// ------------------------------------------------------------------ W8A8 FP8

__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(two)));
  return __half22float2(*reinterpret_cast<__half2*>(&h2));
}

// [LP] S8/S9: E4M3 weights and activations, FP32 accumulation, scales in the
// epilogue.  Rows are row-major here, so a warp streams one row's K range
// (16 columns per lane, 128-bit loads) and reduces with warp shuffles.
template <int MT>
__global__ void __launch_bounds__(128) w8a8_gemv_kernel(const uint8_t* __restrict__ Xq, const float* __restrict__ sx,
                                                        const uint8_t* __restrict__ Wq, const float* __restrict__ sw,
                                                        uint16_t* __restrict__ Y, int64_t M, int64_t N, int64_t K,
                                                        int kb_per_split, int splits, float* partials,
                                                        uint32_t* counters, Epi epi) {
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);  // [MT][KR]
  __shared__ float acc_s[MT][kTileN];
  const int nt = blockIdx.x, split = blockIdx.y;
  const int m0 = blockIdx.z * MT;
  const int mcount = static_cast<int>(imin64(MT, M - m0));
  const int64_t KB = K / kTileK;
  const int kb0 = split * kb_per_split;
  const int kb1 = static_cast<int>(imin64(KB, kb0 + kb_per_split));
  const int KR = (kb1 - kb0) * kTileK;
  const int64_t kbase = static_cast<int64_t>(kb0) * kTileK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_wait();
  grid_dep_launch();

  for (int idx = threadIdx.x; idx < MT * (KR / 8); idx += 128) {
    const int m = idx / (KR / 8), i8 = idx % (KR / 8);
    uint2 v = make_uint2(0, 0);
    if (m < mcount) v = *reinterpret_cast<const uint2*>(Xq + (m0 + m) * K + kbase + i8 * 8);
    float4* d = reinterpret_cast<float4*>(xs + m * KR + i8 * 8);
    const float2 a = e4m3x2_to_f2(v.x), b = e4m3x2_to_f2(v.x >> 16);
    const float2 c = e4m3x2_to_f2(v.y), e = e4m3x2_to_f2(v.y >> 16);
    d[0] = make_float4(a.x, a.y, b.x, b.y);
    d[1] = make_float4(c.x, c.y, e.x, e.y);
  }
  __syncthreads();

  // warp w owns rows 32w .. 32w+31, four at a time
  for (int r0 = warp * 32; r0 < warp * 32 + 32; r0 += 4) {
    float2 acc[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][i] = make_float2(0.0f, 0.0f);
    const uint8_t* wrow = Wq + (static_cast<int64_t>(nt) * kTileN + r0) * K + kbase;
    for (int k = lane * 16; k < KR; k += 512) {
      uint4 w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = ldg_stream(wrow + static_cast<int64_t>(i) * K + k);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float2 xv[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float4 a = *reinterpret_cast<const float4*>(xs + m * KR + k + q * 4);
          xv[m][0] = make_float2(a.x, a.y);
          xv[m][1] = make_float2(a.z, a.w);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t word = (q == 0) ? w[i].x : (q == 1) ? w[i].y : (q == 2) ? w[i].z : w[i].w;
          const float2 f0 = e4m3x2_to_f2(word), f1 = e4m3x2_to_f2(word >> 16);
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            acc[m][i] = __ffma2_rn(xv[m][0], f0, acc[m][i]);
            acc[m][i] = __ffma2_rn(xv[m][1], f1, acc[m][i]);
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v = acc[m][i].x + acc[m][i].y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) acc_s[m][r0 + i] = v;
      }
  }
  __syncthreads();
  float mine[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) mine[m] = acc_s[m][threadIdx.x];
  const float s_w = *sw;
  const int64_t n = static_cast<int64_t>(nt) * kTileN + threadIdx.x;
  const int64_t tile = static_cast<int64_t>(blockIdx.z) * gridDim.x + nt;
  splitk_finish<MT>(mine, mcount, m0, n, M, N, split, splits, tile, partials, counters,
                    [&](int64_t m, int64_t nn, float v) {
                      Y[m * N + nn] = f32_to_bf16_rn(epi_apply(epi, (v * sx[m]) * s_w, nn));
                    });
}

SplitPlan plan_w8a8_gemv(int64_t M, int64_t N, int64_t K, int num_sms) {
  const int mt = gemv_mt(M);
  const int64_t tiles = (N / kTileN) * ((M + mt - 1) / mt);
  SplitPlan p = plan_splits(tiles, K / kTileK, num_sms, 8192 / mt / kTileK);
  if (p.splits > 1) {
    p.ws_bytes = counters_bytes(tiles) + sizeof(float) * static_cast<size_t>(p.splits) * M * N;
    p.zero_bytes = counters_bytes(tiles);
  }
  return p;
}

cudaError_t launch_w8a8_gemv(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, uint16_t* Y,
                             int64_t M, int64_t N, int64_t K, const SplitPlan& plan, void* ws, cudaStream_t st,
                             const Epi& epi) {
  const int mt = gemv_mt(M);
  dim3 grid(static_cast<unsigned>(N / kTileN), plan.splits, static_cast<unsigned>((M + mt - 1) / mt));
  const size_t smem = sizeof(float) * static_cast<size_t>(mt) * plan.kb_per_split * kTileK;
  uint32_t* counters = static_cast<uint32_t*>(ws);
  float* partials = ws ? reinterpret_cast<float*>(static_cast<char*>(ws) + counters_bytes(plan.tiles)) : nullptr;
  cudaError_t e = cudaSuccess;
  switch (mt) {
#define QLIN_W8GEMV(MTV)                                                                                   \
  case MTV:                                                                                                \
    e = set_smem_once(w8a8_gemv_kernel<MTV>, 64 * 1024);                                                   \
    if (e != cudaSuccess) return e;                                                                        \
    e = launch_pdl(w8a8_gemv_kernel<MTV>, grid, smem, st, Xq, sx, Wq, sw, Y, M, N, K, plan.kb_per_split,     \
                   plan.splits, partials, counters, epi);                                                  \
    break;
    QLIN_W8GEMV(1)
    QLIN_W8GEMV(2)
    QLIN_W8GEMV(4)
#undef QLIN_W8GEMV
  }
  return e;
}

}  // namespace qlin
