// Load-time and per-call quantisation kernels:
//  * pack_w4        -- per-group INT4 quantiser + tile-layout packing
//  * quant_act_fp8  -- fused per-token amax + E4M3 cast
//  * quant_w_fp8    -- per-tensor amax (grid reduction) + E4M3 cast
// Rounding follows IEEE binary32 throughout (no fast-math): divisions are
// __fdiv_rn, round() is rintf (half to even), FP16 is __float2half_rn and
// E4M3 is cvt.rn.satfinite.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qlin_internal.cuh"

namespace qlin {

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// min / max over aligned segments of `seg` lanes (seg = 8, 16 or 32)
__device__ __forceinline__ float seg_min(float v, int seg) {
  for (int o = seg >> 1; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float seg_max(float v, int seg) {
  for (int o = seg >> 1; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Packed layout (format version 2): in each 16-byte record (one row, 32
// columns c = 16a + 8b + 2t + e of a 64-column tile) word t holds the eight
// columns a lane t of an mma.sync quad needs for two 16-column k-steps, column
// c in nibble position 2a + b + 4e.  Pair (c, c+1) is then the two halves of
// (word >> 4(2a + b)) & 0x000F000F: one shift by a constant and one logic op.

// [LP] S2-S4: one warp per (pair of rows, chunk of 128 columns).  Lane l owns
// columns 4l..4l+3 of the chunk; a group of G columns (G = 32, 64, 128) is a
// segment of G/4 lanes, and its min/max are segment reductions.
// Lane l = 8R + u covers record R of the group (tile R/2, half R%2); its
// columns 4u, 4u+1 go to word 2(u%2) and 4u+2, 4u+3 to word 2(u%2)+1, both at
// nibble positions u/2 and u/2 + 4, so each word is the OR of the lanes u,
// u^2, u^4, u^6.
// Scale and zero-point of one group from its range ([LP] S2-S3): lo, hi
// include 0; s = fp16((hi - lo) / 15) (symmetric: fp16(amax / 7)); a scale
// that rounds to 0 stores 1 and zero-point 0 (symmetric: 8).
__device__ __forceinline__ void group_params(float lo, float hi, float amax, int symmetric, __half& s16, float& sc,
                                             int& zp) {
  const float s32 = symmetric ? __fdiv_rn(amax, 7.0f) : __fdiv_rn(hi - lo, 15.0f);
  s16 = __float2half_rn(s32);
  sc = __half2float(s16);
  if (sc == 0.0f) {  // degenerate group: s = 1, logical zero-point 0
    s16 = __float2half_rn(1.0f);
    sc = 1.0f;
    zp = symmetric ? 8 : 0;
  } else if (symmetric) {
    zp = 8;
  } else {
    float zf = rintf(__fdiv_rn(-lo, sc));
    zf = fminf(fmaxf(zf, 0.0f), 15.0f);
    zp = static_cast<int>(zf);
  }
}

// Per-channel scales ([LP] S4 "per-channel": one group spanning the row): one
// CTA per pair of rows reduces each row's range over all of K and writes the
// two scales and their zero-point byte (tile layout with K / G = 1).
__global__ void __launch_bounds__(256) row_range_kernel(const uint16_t* __restrict__ W, int64_t K, int symmetric,
                                                        uint16_t* __restrict__ scales, uint8_t* __restrict__ zeros,
                                                        int* err) {
  __shared__ float red[3][8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t zbyte = 0;
  for (int sub = 0; sub < 2; ++sub) {
    const int64_t n = blockIdx.x * 2 + sub;
    const uint2* row = reinterpret_cast<const uint2*>(W + n * K);
    float lo = 0.0f, hi = 0.0f, amax = 0.0f;
    for (int64_t i = threadIdx.x; i < K / 4; i += 256) {
      const uint2 raw = row[i];
      const float v[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        lo = fminf(lo, v[j]);
        hi = fmaxf(hi, v[j]);
        amax = fmaxf(amax, fabsf(v[j]));
      }
    }
    lo = warp_min(lo);
    hi = warp_max(hi);
    amax = warp_max(amax);
    if (lane == 0) {
      red[0][warp] = lo;
      red[1][warp] = hi;
      red[2][warp] = amax;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < 8; ++w) {
        lo = fminf(lo, red[0][w]);
        hi = fmaxf(hi, red[1][w]);
        amax = fmaxf(amax, red[2][w]);
      }
      __half s16;
      float sc;
      int zp;
      group_params(lo, hi, amax, symmetric, s16, sc, zp);
      if (isinf(sc)) set_error(err, QLIN_ERR_INVALID_VALUE);
      scales[(n / kTileN) * kTileN + n % kTileN] = __half_as_ushort(s16);
      zbyte |= static_cast<uint32_t>(zp) << (4 * sub);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) zeros[(blockIdx.x * 2 / kTileN) * (kTileN / 2) + (blockIdx.x * 2 % kTileN) / 2] = zbyte;
}

__global__ void __launch_bounds__(256) pack_w4_kernel(const uint16_t* __restrict__ W, int64_t N, int64_t K,
                                                      int G, int symmetric, uint8_t* __restrict__ codes,
                                                      uint16_t* __restrict__ scales, uint8_t* __restrict__ zeros,
                                                      int* err) {
  const int lane = threadIdx.x & 31;
  // G == K beyond 128 columns: per-channel scales, already written by row_range_kernel
  const bool pc = G > 128;
  const int seg = pc ? 32 : G / 4;          // lanes per group (within a 128-column chunk)
  const int64_t ng = K / 128;               // chunks per row
  const int64_t ngk = K / G;                // groups per row
  const int64_t total = (N / 2) * ng;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; item < total;
       item += nwarps) {
    const int64_t pair = item / ng, g = item % ng;
    uint32_t zbyte = 0;
    const int64_t nb = (pair * 2) / kTileN;
#pragma unroll
    for (int sub = 0; sub < 2; ++sub) {
      const int64_t n = pair * 2 + sub;
      const int r = static_cast<int>(n % kTileN);
      const uint2 raw = *reinterpret_cast<const uint2*>(W + n * K + g * kGroup + 4 * lane);
      const float v[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
      __half s16;
      float sc;
      int zp;
      if (pc) {  // the row's scale and zero-point from the range pass
        s16 = __ushort_as_half(scales[nb * kTileN + r]);
        sc = __half2float(s16);
        zp = static_cast<int>((zeros[nb * (kTileN / 2) + r / 2] >> (4 * (r & 1))) & 15u);
      } else {
        float lo = 0.0f, hi = 0.0f, amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          lo = fminf(lo, v[i]);
          hi = fmaxf(hi, v[i]);
          amax = fmaxf(amax, fabsf(v[i]));
        }
        lo = seg_min(lo, seg);
        hi = seg_max(hi, seg);
        amax = seg_max(amax, seg);
        group_params(lo, hi, amax, symmetric, s16, sc, zp);
        if (isinf(sc) && lane == 0) set_error(err, QLIN_ERR_INVALID_VALUE);
      }
      uint32_t cq[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float rq = rintf(__fdiv_rn(v[i], sc));
        int c;
        if (symmetric) {
          rq = fminf(fmaxf(rq, -8.0f), 7.0f);
          c = static_cast<int>(rq) + 8;
        } else {
          rq = fminf(fmaxf(rq + static_cast<float>(zp), 0.0f), 15.0f);
          c = static_cast<int>(rq);
        }
        cq[i] = static_cast<uint32_t>(c);
      }
      const int u = lane & 7, R = lane >> 3;
      const uint32_t pos = 4u * static_cast<uint32_t>(u >> 1);
      uint32_t wa = (cq[0] << pos) | (cq[1] << (pos + 16));  // word 2(u%2)
      uint32_t wb = (cq[2] << pos) | (cq[3] << (pos + 16));  // word 2(u%2) + 1
      wa |= __shfl_xor_sync(0xffffffffu, wa, 2);
      wb |= __shfl_xor_sync(0xffffffffu, wb, 2);
      wa |= __shfl_xor_sync(0xffffffffu, wa, 4);
      wb |= __shfl_xor_sync(0xffffffffu, wb, 4);
      if (u < 2) {
        const int64_t kb = g * 2 + (R >> 1);
        const int h = R & 1;
        *reinterpret_cast<uint2*>(codes + (nb * (K / kTileK) + kb) * 4096 + h * 2048 + r * 16 + u * 8) =
            make_uint2(wa, wb);
      }
      if (pc) continue;  // scales and zero-points are in place
      const int64_t gg = g * (128 / G) + lane / seg;  // group of this lane's segment
      if (lane % seg == 0) {
        scales[(nb * ngk + gg) * kTileN + r] = __half_as_ushort(s16);
        zbyte |= static_cast<uint32_t>(zp) << (4 * sub);
      }
    }
    if (!pc && lane % seg == 0)
      zeros[(nb * ngk + g * (128 / G) + lane / seg) * (kTileN / 2) + ((pair * 2) % kTileN) / 2] =
          static_cast<uint8_t>(zbyte);
  }
}

cudaError_t launch_pack_w4(const uint16_t* W, int64_t N, int64_t K, int G, int symmetric, uint8_t* codes,
                           uint16_t* scales, uint8_t* zeros, int* err, int num_sms, cudaStream_t st) {
  const int64_t items = (N / 2) * (K / 128);
  const int64_t want = (items + 7) / 8;
  const int blocks = static_cast<int>(want < static_cast<int64_t>(num_sms) * 16 ? want : num_sms * 16);
  if (G > 128) {  // per-channel: the row ranges first
    row_range_kernel<<<static_cast<unsigned>(N / 2), 256, 0, st>>>(W, K, symmetric, scales, zeros, err);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  pack_w4_kernel<<<blocks, 256, 0, st>>>(W, N, K, G, symmetric, codes, scales, zeros, err);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ FP8

// E4M3 pair: `lo` goes to the lower byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int THREADS>
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < THREADS / 32 ? red[lane] : 0.0f;
    v = warp_max(v);
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  const float r = red[0];
  __syncthreads();
  return r;
}

__device__ __forceinline__ uint2 quant8(uint4 v, float s) {
  const uint32_t b0 = e4m3x2(__fdiv_rn(bf16_lo(v.x), s), __fdiv_rn(bf16_hi(v.x), s));
  const uint32_t b1 = e4m3x2(__fdiv_rn(bf16_lo(v.y), s), __fdiv_rn(bf16_hi(v.y), s));
  const uint32_t b2 = e4m3x2(__fdiv_rn(bf16_lo(v.z), s), __fdiv_rn(bf16_hi(v.z), s));
  const uint32_t b3 = e4m3x2(__fdiv_rn(bf16_lo(v.w), s), __fdiv_rn(bf16_hi(v.w), s));
  return make_uint2(b0 | (b1 << 16), b2 | (b3 << 16));
}

__device__ __forceinline__ float amax8(uint4 v, float a) {
  a = fmaxf(a, fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))));
  a = fmaxf(a, fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y))));
  a = fmaxf(a, fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))));
  a = fmaxf(a, fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w))));
  return a;
}

// [LP] S4 per-token, S8 current scaling: one CTA per row; the row is read
// once from HBM (the second pass hits L1/L2), amax is a block reduction.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) quant_act_fp8_kernel(const uint16_t* __restrict__ X, int64_t K,
                                                                uint8_t* __restrict__ Xq, float* __restrict__ sx) {
  __shared__ float red[32];
  const int64_t m = blockIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(X + m * K);
  const int64_t n8 = K / 8;
  float a = 0.0f;
  for (int64_t i = threadIdx.x; i < n8; i += THREADS) a = amax8(row[i], a);
  a = block_max<THREADS>(a, red);
  const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
  if (threadIdx.x == 0) sx[m] = s;
  uint2* out = reinterpret_cast<uint2*>(Xq + m * K);
  for (int64_t i = threadIdx.x; i < n8; i += THREADS) out[i] = quant8(row[i], s);
}

// The same with the row held in registers: each thread loads its ITEMS
// 16-byte pieces of the row at once (K <= THREADS * 8 * ITEMS), so a CTA has
// the whole row in flight, and quantises from registers after the block
// reduction.  Small CTAs let an SM keep many rows in flight.
template <int THREADS, int ITEMS>
__global__ void __launch_bounds__(THREADS) quant_act_fp8_reg_kernel(const uint16_t* __restrict__ X, int64_t K,
                                                                    uint8_t* __restrict__ Xq, float* __restrict__ sx) {
  __shared__ float red[32];
  const int64_t m = blockIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(X + m * K);
  const int n8 = static_cast<int>(K / 8);
  uint4 v[ITEMS];
#pragma unroll
  for (int j = 0; j < ITEMS; ++j) {
    const int i = threadIdx.x + j * THREADS;
    v[j] = i < n8 ? row[i] : make_uint4(0u, 0u, 0u, 0u);
  }
  float a = 0.0f;
#pragma unroll
  for (int j = 0; j < ITEMS; ++j) a = amax8(v[j], a);
  a = block_max<THREADS>(a, red);
  const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
  if (threadIdx.x == 0) sx[m] = s;
  uint2* out = reinterpret_cast<uint2*>(Xq + m * K);
#pragma unroll
  for (int j = 0; j < ITEMS; ++j) {
    const int i = threadIdx.x + j * THREADS;
    if (i < n8) out[i] = quant8(v[j], s);
  }
}

cudaError_t launch_quant_act_fp8(const uint16_t* X, int64_t M, int64_t K, uint8_t* Xq, float* sx, cudaStream_t st) {
  const unsigned g = static_cast<unsigned>(M);
  if (K <= 4096)
    quant_act_fp8_reg_kernel<128, 4><<<g, 128, 0, st>>>(X, K, Xq, sx);
  else if (K <= 8192)
    quant_act_fp8_reg_kernel<128, 8><<<g, 128, 0, st>>>(X, K, Xq, sx);
  else if (K <= 16384)
    quant_act_fp8_reg_kernel<256, 8><<<g, 256, 0, st>>>(X, K, Xq, sx);
  else if (K <= 32768)
    quant_act_fp8_reg_kernel<512, 8><<<g, 512, 0, st>>>(X, K, Xq, sx);
  else
    quant_act_fp8_kernel<512><<<g, 512, 0, st>>>(X, K, Xq, sx);
  return cudaGetLastError();
}

// [LP] S4 per-tensor: grid-wide amax via atomicMax on the IEEE bits of a
// non-negative float (integer order equals float order there).
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* __restrict__ W, int64_t n8,
                                                   uint32_t* __restrict__ amax_bits) {
  __shared__ float red[32];
  float a = 0.0f;
  const uint4* p = reinterpret_cast<const uint4*>(W);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < n8; i += static_cast<int64_t>(gridDim.x) * 256)
    a = amax8(p[i], a);
  a = block_max<256>(a, red);
  if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(a));
}

__global__ void __launch_bounds__(256) cast_w_fp8_kernel(const uint16_t* __restrict__ W, int64_t n8,
                                                         const uint32_t* __restrict__ amax_bits,
                                                         uint8_t* __restrict__ Wq, float* __restrict__ sw) {
  const float a = __uint_as_float(*amax_bits);
  const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *sw = s;
  const uint4* p = reinterpret_cast<const uint4*>(W);
  uint2* out = reinterpret_cast<uint2*>(Wq);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < n8; i += static_cast<int64_t>(gridDim.x) * 256)
    out[i] = quant8(p[i], s);
}

cudaError_t launch_quant_w_fp8(const uint16_t* W, int64_t N, int64_t K, uint8_t* Wq, float* sw, uint32_t* amax_ws,
                               int num_sms, cudaStream_t st) {
  const int64_t n8 = N * K / 8;
  cudaError_t e = cudaMemsetAsync(amax_ws, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  const int64_t want = (n8 + 255) / 256;
  const int blocks = static_cast<int>(want < static_cast<int64_t>(num_sms) * 8 ? want : num_sms * 8);
  amax_kernel<<<blocks, 256, 0, st>>>(W, n8, amax_ws);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cast_w_fp8_kernel<<<blocks, 256, 0, st>>>(W, n8, amax_ws, Wq, sw);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ FP8 block scaling

// [LP] S8 block scaling, 1 x 128 activation blocks: one warp per (token m,
// block b); lanes 0-15 hold eight columns each.  sx is block-major, sx[b][m].
__global__ void __launch_bounds__(256) quant_act_fp8_blocks_kernel(const uint16_t* __restrict__ X, int64_t M,
                                                                   int64_t K, uint8_t* __restrict__ Xq,
                                                                   float* __restrict__ sx) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = K / 128;
  const int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (item >= M * nb) return;  // whole warps only
  const int64_t m = item / nb, b = item % nb;
  const uint4* src = reinterpret_cast<const uint4*>(X + m * K + b * 128);
  uint4 v = make_uint4(0, 0, 0, 0);
  if (lane < 16) v = src[lane];
  const float a = warp_max(amax8(v, 0.0f));
  const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
  if (lane == 0) sx[b * M + m] = s;
  if (lane < 16) reinterpret_cast<uint2*>(Xq + m * K + b * 128)[lane] = quant8(v, s);
}

// 128 x 128 weight blocks: one CTA per block, eight 8-column pieces per thread.
__global__ void __launch_bounds__(256) quant_w_fp8_blocks_kernel(const uint16_t* __restrict__ W, int64_t K,
                                                                 uint8_t* __restrict__ Wq, float* __restrict__ sw) {
  __shared__ float red[32];
  const int64_t nb = K / 128;
  const int64_t i = blockIdx.y, b = blockIdx.x;
  uint4 v[8];
  float a = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int idx = threadIdx.x + 256 * j;  // row idx / 16, columns 8 (idx % 16) ..
    v[j] = reinterpret_cast<const uint4*>(W + (i * 128 + idx / 16) * K + b * 128)[idx % 16];
    a = amax8(v[j], a);
  }
  a = block_max<256>(a, red);
  const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
  if (threadIdx.x == 0) sw[i * nb + b] = s;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int idx = threadIdx.x + 256 * j;
    reinterpret_cast<uint2*>(Wq + (i * 128 + idx / 16) * K + b * 128)[idx % 16] = quant8(v[j], s);
  }
}

cudaError_t launch_quant_act_fp8_blocks(const uint16_t* X, int64_t M, int64_t K, uint8_t* Xq, float* sx,
                                        cudaStream_t st) {
  const int64_t warps = M * (K / 128);
  const int64_t blocks = (warps + 7) / 8;
  quant_act_fp8_blocks_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(X, M, K, Xq, sx);
  return cudaGetLastError();
}

cudaError_t launch_quant_w_fp8_blocks(const uint16_t* W, int64_t N, int64_t K, uint8_t* Wq, float* sw,
                                      cudaStream_t st) {
  quant_w_fp8_blocks_kernel<<<dim3(static_cast<unsigned>(K / 128), static_cast<unsigned>(N / 128)), 256, 0, st>>>(
      W, K, Wq, sw);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ MXFP8

// Eight BF16 columns of one 16-byte load
__device__ __forceinline__ void bf16x8(uint4 raw, float (&v)[8]) {
  v[0] = bf16_lo(raw.x);
  v[1] = bf16_hi(raw.x);
  v[2] = bf16_lo(raw.y);
  v[3] = bf16_hi(raw.y);
  v[4] = bf16_lo(raw.z);
  v[5] = bf16_hi(raw.z);
  v[6] = bf16_lo(raw.w);
  v[7] = bf16_hi(raw.w);
}

// Items (a row's 128- or 256-column chunk) per warp in the MX / FP4
// quantisers: a warp issues all of their loads before the arithmetic, so that
// an SM keeps enough bytes in flight to stream at the HBM rate.
constexpr int kMxItems = 4;

// MX block scale of a 32-element block ([LP] S10, OCP Microscaling v1.0):
// e = floor(log2 amax) - 8 (8: exponent of E4M3's largest normal), clamped to
// [-127, 127]; -127 for an all-zero block.  Read from the exponent field: an
// FP32 subnormal amax (below 2^-126) lies below the clamp.
__device__ __forceinline__ int mx_exponent(float amax) {
  const int eb = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  if (eb == 0) return -127;
  const int e = eb - 127 - 8;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// A warp per kMxItems consecutive (row r, 256 columns) items: lane l holds
// columns 8l .. 8l+7 (one 16-byte load), a block of 32 columns is a segment of
// four lanes, and lanes 16h .. 16h+15 are K block 2c + h.  When K is an odd
// number of 128-column blocks, the last item of a row has only its first half.
// Codes are E4M3(v * 2^-e) -- the power-of-two scaling is exact, so this is
// v / 2^e rounded once, to nearest even with saturation.  The four scale bytes
// of a 128-column block go to one 32-bit word of the scale atom: row r of atom
// (r / 128, k / 128) holds its word at byte 16 (r % 32) + 4 ((r % 128) / 32);
// rows past R (the atom's padding) get 0.
__global__ void __launch_bounds__(256) quant_mxfp8_kernel(const uint16_t* __restrict__ X, int64_t R, int64_t K,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t nkb = K / 128, nc = (nkb + 1) / 2;
  const int64_t total = (R + 127) / 128 * 128 * nc;  // items: (row, 256 columns), padding rows included
  const int64_t item0 = ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * kMxItems;
  if (item0 >= total) return;  // whole warps only
  // all of this warp's loads first, so that kMxItems of them are in flight;
  // item0 + u is row rr[u], chunk cc[u]: one division per warp, then a carry
  // (rows < 2^31 and chunks < 2^23, as the call checks: 32-bit indices keep
  // the warp's state in registers)
  int rr[kMxItems], cc[kMxItems];
  rr[0] = static_cast<int>(item0 / nc);
  cc[0] = static_cast<int>(item0 - static_cast<int64_t>(rr[0]) * nc);
#pragma unroll
  for (int u = 1; u < kMxItems; ++u) {
    const bool wrap = cc[u - 1] + 1 == nc;
    cc[u] = wrap ? 0 : cc[u - 1] + 1;
    rr[u] = wrap ? rr[u - 1] + 1 : rr[u - 1];
  }
  const int half = lane >> 4;
  uint4 raw[kMxItems];
#pragma unroll
  for (int u = 0; u < kMxItems; ++u) {
    const int64_t item = item0 + u, r = rr[u], c = cc[u];
    raw[u] = (item < total && r < R && 2 * c + half < nkb)
                 ? *reinterpret_cast<const uint4*>(X + r * K + c * 256 + 8 * lane)
                 : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < kMxItems; ++u) {
    const int64_t item = item0 + u;
    if (item >= total) break;  // the same for the whole warp
    const int64_t r = rr[u], c = cc[u];
    const bool mine = 2 * c + half < nkb;  // this lane's K block exists
    uint32_t e8 = 0;
    if (r < R) {
      float v[8];
      bf16x8(raw[u], v);
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
      amax = seg_max(amax, 4);
      const int e = amax == 0.0f ? -127 : mx_exponent(amax);
      const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, e in [-127, 119]
      const uint32_t w0 = e4m3x2(v[0] * inv, v[1] * inv) | (e4m3x2(v[2] * inv, v[3] * inv) << 16);
      const uint32_t w1 = e4m3x2(v[4] * inv, v[5] * inv) | (e4m3x2(v[6] * inv, v[7] * inv) << 16);
      if (mine) *reinterpret_cast<uint2*>(codes + r * K + c * 256 + 8 * lane) = make_uint2(w0, w1);
      e8 = static_cast<uint32_t>(e + 127);
    }
    // bytes kk = 0..3 of K block 2c + h's word from lanes 16h, +4, +8, +12
    uint32_t word = (e8 & 0xFFu) << (8 * ((lane >> 2) & 3));
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    word |= __shfl_xor_sync(0xffffffffu, word, 8);
    if ((lane & 15) == 0 && mine) {
      uint8_t* atom = scales + ((r / 128) * nkb + 2 * c + half) * 512;
      *reinterpret_cast<uint32_t*>(atom + 16 * (r % 32) + 4 * ((r % 128) / 32)) = word;
    }
  }
}

cudaError_t launch_quant_mxfp8(const uint16_t* X, int64_t R, int64_t K, uint8_t* codes, uint8_t* scales,
                               cudaStream_t st) {
  const int64_t items = (R + 127) / 128 * 128 * ((K / 128 + 1) / 2);
  const int64_t warps = (items + kMxItems - 1) / kMxItems;
  const int64_t blocks = (warps + 7) / 8;
  quant_mxfp8_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(X, R, K, codes, scales);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ FP4 (E2M1)

// Eight floats -> eight E2M1 codes, rounded to nearest even with saturation
// at +-6 (cvt.rn.satfinite.e2m1x2), two per byte with the even element in the
// low nibble: one 32-bit word.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// MXFP4 ([LP] S10, OCP Microscaling v1.0): a warp per kMxItems consecutive
// (row r, 256 columns) items; lane l holds columns 8l .. 8l+7, a block of 32 columns is a segment of four
// lanes.  e = floor(log2 amax) - 2 (2: exponent of E2M1's largest normal,
// 6 = 1.5 x 2^2), clamped to [-127, 127], -127 for an all-zero block; codes
// E2M1(v * 2^-e) (the power-of-two scaling is exact).  The 256 columns fill
// two scale atoms: the word of atom 2c + h (h = lane / 16) holds the scale
// bytes of lanes 16h, +4, +8, +12; rows past R write only their atom words (0).
__global__ void __launch_bounds__(256) quant_mxfp4_kernel(const uint16_t* __restrict__ X, int64_t R, int64_t K,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t nc = K / 256;
  const int64_t total = (R + 127) / 128 * 128 * nc;  // items: (row, 256 columns), padding rows included
  const int64_t item0 = ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * kMxItems;
  if (item0 >= total) return;  // whole warps only
  // item0 + u is row rr[u], chunk cc[u]: one division per warp, then a carry
  int64_t rr[kMxItems], cc[kMxItems];
  rr[0] = item0 / nc;
  cc[0] = item0 - rr[0] * nc;
#pragma unroll
  for (int u = 1; u < kMxItems; ++u) {
    const bool wrap = cc[u - 1] + 1 == nc;
    cc[u] = wrap ? 0 : cc[u - 1] + 1;
    rr[u] = wrap ? rr[u - 1] + 1 : rr[u - 1];
  }
  uint4 raw[kMxItems];
#pragma unroll
  for (int u = 0; u < kMxItems; ++u) {
    const int64_t item = item0 + u, r = rr[u], c = cc[u];
    raw[u] = (item < total && r < R) ? *reinterpret_cast<const uint4*>(X + r * K + c * 256 + 8 * lane)
                                     : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < kMxItems; ++u) {
    const int64_t item = item0 + u;
    if (item >= total) break;  // the same for the whole warp
    const int64_t r = rr[u], c = cc[u];
    uint32_t e8 = 0;
    if (r < R) {
      float v[8];
      bf16x8(raw[u], v);
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
      amax = seg_max(amax, 4);
      const int eb = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);  // 0: zero or below 2^-126
      int e = eb == 0 ? -127 : eb - 127 - 2;
      e = e < -127 ? -127 : e;
      const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, e in [-127, 125]
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] *= inv;
      *reinterpret_cast<uint32_t*>(codes + r * (K / 2) + c * 128 + 4 * lane) = e2m1x8(v);
      e8 = static_cast<uint32_t>(e + 127);
    }
    uint32_t word = (e8 & 0xFFu) << (8 * ((lane >> 2) & 3));
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    word |= __shfl_xor_sync(0xffffffffu, word, 8);
    if ((lane & 15) == 0) {
      uint8_t* atom = scales + ((r / 128) * (K / 128) + 2 * c + (lane >> 4)) * 512;
      *reinterpret_cast<uint32_t*>(atom + 16 * (r % 32) + 4 * ((r % 128) / 32)) = word;
    }
  }
}

cudaError_t launch_quant_mxfp4(const uint16_t* X, int64_t R, int64_t K, uint8_t* codes, uint8_t* scales,
                               cudaStream_t st) {
  const int64_t items = (R + 127) / 128 * 128 * (K / 256);
  const int64_t blocks = ((items + kMxItems - 1) / kMxItems + 7) / 8;
  quant_mxfp4_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(X, R, K, codes, scales);
  return cudaGetLastError();
}

// NVFP4 per-tensor scale sg = amax(|X|) / (6 x 448), 1 when that is 0.  The
// amax is reduced into the output word as FP32 bits (non-negative floats
// order like their bit patterns), which a one-thread kernel then turns into sg.
__global__ void __launch_bounds__(256) amax_bits_kernel(const uint16_t* __restrict__ X, int64_t n8,
                                                        unsigned* __restrict__ out) {
  float amax = 0.0f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float v[8];
    bf16x8(reinterpret_cast<const uint4*>(X)[i], v);
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[k]));
  }
  amax = seg_max(amax, 32);
  if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(amax));
}

__global__ void nvfp4_scale_finish_kernel(float* sg) {
  const float amax = __uint_as_float(*reinterpret_cast<const unsigned*>(sg));
  const float s = __fdiv_rn(amax, 2688.0f);
  *sg = s == 0.0f ? 1.0f : s;
}

cudaError_t launch_nvfp4_tensor_scale(const uint16_t* X, int64_t n, float* sg, int num_sms, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(sg, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  const int64_t n8 = n / 8;
  int64_t blocks = (n8 + 255) / 256;
  if (blocks > 4LL * num_sms) blocks = 4LL * num_sms;
  if (blocks < 1) blocks = 1;
  amax_bits_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(X, n8, reinterpret_cast<unsigned*>(sg));
  nvfp4_scale_finish_kernel<<<1, 1, 0, st>>>(sg);
  return cudaGetLastError();
}

// E4M3 code -> its value (exact through FP16; the code in both bytes, so
// either half of the result holds it)
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(code * 0x0101u)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// NVFP4 ([LP] S10 names it; the vendor's two-level recipe): a warp per
// kMxItems consecutive (row r, 256 columns) items, lane l holds columns 8l .. 8l+7, a block of 16 columns
// is a pair of lanes.  Block scale sb = E4M3(amax_b / (6 sg)) (RNE, saturating),
// elements E2M1(v / (sb sg)); each step is one IEEE binary32 operation
// (__fmul_rn / __fdiv_rn); a block whose scale is 0 stores code 0.  The 256
// columns fill four scale atoms (64 columns each): the word of atom 4c + a
// (a = lane / 8) holds the scale bytes of lanes 8a, +2, +4, +6.
__global__ void __launch_bounds__(256) quant_nvfp4_kernel(const uint16_t* __restrict__ X, int64_t R, int64_t K,
                                                          const float* __restrict__ sgp, uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t nc = K / 256;
  const int64_t total = (R + 127) / 128 * 128 * nc;  // items: (row, 256 columns), padding rows included
  const int64_t item0 = ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * kMxItems;
  if (item0 >= total) return;  // whole warps only
  // item0 + u is row rr[u], chunk cc[u]: one division per warp, then a carry
  // (32-bit: rows < 2^31 and chunks < 2^23, as the call checks)
  int rr[kMxItems], cc[kMxItems];
  rr[0] = static_cast<int>(item0 / nc);
  cc[0] = static_cast<int>(item0 - static_cast<int64_t>(rr[0]) * nc);
#pragma unroll
  for (int u = 1; u < kMxItems; ++u) {
    const bool wrap = cc[u - 1] + 1 == nc;
    cc[u] = wrap ? 0 : cc[u - 1] + 1;
    rr[u] = wrap ? rr[u - 1] + 1 : rr[u - 1];
  }
  uint4 raw[kMxItems];
#pragma unroll
  for (int u = 0; u < kMxItems; ++u) {
    const int64_t item = item0 + u, r = rr[u], c = cc[u];
    raw[u] = (item < total && r < R) ? *reinterpret_cast<const uint4*>(X + r * K + c * 256 + 8 * lane)
                                     : make_uint4(0u, 0u, 0u, 0u);
  }
  const float sg = __ldg(sgp);
#pragma unroll
  for (int u = 0; u < kMxItems; ++u) {
    const int64_t item = item0 + u;
    if (item >= total) break;  // the same for the whole warp
    const int64_t r = rr[u], c = cc[u];
    uint32_t sc = 0;
    if (r < R) {
      float v[8];
      bf16x8(raw[u], v);
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
      amax = seg_max(amax, 2);
      sc = e4m3x2(__fdiv_rn(amax, __fmul_rn(6.0f, sg)), 0.0f) & 0xFFu;
      uint32_t qv = 0;
      if (sc != 0) {
        const float den = __fmul_rn(e4m3_value(sc), sg);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __fdiv_rn(v[i], den);
        qv = e2m1x8(v);
      }
      *reinterpret_cast<uint32_t*>(codes + r * (K / 2) + c * 128 + 4 * lane) = qv;
    }
    uint32_t word = sc << (8 * ((lane >> 1) & 3));
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    if ((lane & 7) == 0) {
      uint8_t* atom = scales + ((r / 128) * (K / 64) + 4 * c + (lane >> 3)) * 512;
      *reinterpret_cast<uint32_t*>(atom + 16 * (r % 32) + 4 * ((r % 128) / 32)) = word;
    }
  }
}

cudaError_t launch_quant_nvfp4(const uint16_t* X, int64_t R, int64_t K, const float* sg, uint8_t* codes,
                               uint8_t* scales, cudaStream_t st) {
  const int64_t items = (R + 127) / 128 * 128 * (K / 256);
  const int64_t blocks = ((items + kMxItems - 1) / kMxItems + 7) / 8;
  quant_nvfp4_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(X, R, K, sg, codes, scales);
  return cudaGetLastError();
}

}  // namespace qlin
