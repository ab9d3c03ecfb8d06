// W4A16 for small M (decode): split-K GEMV-style kernel whose inner product
// runs on the tensor cores through register-level mma.sync, so that the CUDA
// cores only unpack nibbles.
//
// [LP] S11 (packed INT4 -> unpack/dequantise -> multiply with BF16 activations
// -> accumulate) and S22 (FP32 accumulation).  Per group g of 128 columns the
// kernel uses
//     sum_k x_k s (q_k - z) = s ( sum_k x_k (128 + q_k) - (128 + z) sum_k x_k ),
// where 128 + q_k is exact in BF16.  The packed layout gives each lane of an
// mma.sync quad its own 32-bit word per record (four A-fragment pairs), so a
// pair comes out with one LOP3 after a right shift by a constant (a high
// multiply on the FMA pipe instead of the shift measured slower: it stalls
// dispatch); the MMA accumulates
// sum_k x_k (128 + q_k) in FP32 and the scale / zero-point are applied once
// per group and row in FP32 registers.
//
// One CTA = one 128-row tile x one K range.  Warp 4 streams, per stage of 256
// columns, the tile's packed codes (16 KB), scales and zero-points and the
// activation slice of every token into a ring of shared-memory stages with
// bulk copies (weights first, before waiting for the previous kernel on the
// stream).  Warps 0-3 each own 32 rows (two m16 blocks that share every B
// fragment) and every token (one or two n8 blocks).  Warp 5 forms the
// per-group activation sums sum_k x_k of each stage once for the whole CTA,
// on the tensor core (an m16 A operand of all ones), and leaves them in the
// stage for the folds.  The K ranges of one
// tile run as a thread-block cluster and add their partial sums through
// distributed shared memory, in rank order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <array>
#include <type_traits>
#include <mutex>
#include <unordered_map>

#include "qlin_internal.cuh"
#include "qlin_ptx.cuh"

namespace qlin {

constexpr int kMmaStageCols = 256;                 // K columns per stage (4 code tiles)
constexpr int kMmaCodeBytes = 4 * 4096;            // codes of one stage
constexpr int kMmaMetaOff = kMmaCodeBytes;         // group scales (128 FP16 each), then zeros (64 B each)
constexpr int kMmaXRow = kMmaStageCols * 2 + 16;   // 528 B per token row (conflict-free B fragments)
constexpr int kMmaRowBlocks = 2;                   // m16 row blocks per consumer warp
constexpr int kMmaConsumers = kTileN / (16 * kMmaRowBlocks);  // consumer warps, 32 rows each
constexpr int kMmaProducer = kMmaConsumers;        // bulk-copy warp
constexpr int kMmaSummer = kMmaConsumers + 1;      // activation-sum warp
constexpr int kMmaThreads = (kMmaConsumers + 2) * 32;
constexpr uint64_t kMmaWaitNs = 2000000000ull;
constexpr int kMmaMaxCluster = 16;                 // CTAs of one tile's split-K cluster (non-portable above 8)
constexpr int kMmaRedRows = 144;                   // >= splits x ceil(128 / splits) for splits <= 16

template <int NT, int G = 128>
struct MmaCfg {
  static constexpr int kTok = 8 * NT;
  static constexpr int kGps = kMmaStageCols / G;  // quantisation groups per stage
  static constexpr int kZeroOff = kMmaMetaOff + kGps * 256;
  static constexpr int kXOff = kMmaCodeBytes + (kGps * 320 + 1023) / 1024 * 1024;  // activation rows
  static constexpr int kSumOff = kXOff + kTok * kMmaXRow;  // FP32 activation sums [kGps groups][kTok tokens]
  static constexpr int kStage = ((kSumOff + kGps * kTok * 4) + 1023) / 1024 * 1024;
  // three CTAs fit per SM for M <= 8, two up to 32 (a ring of two stages at 32 tokens)
  static constexpr int kStages = NT == 4 ? 2 : 3;
  // split-K receive buffer: [source rank][row within the owner's slice][token
  // slot]; ranks x slice rows <= 140 for every split count up to 16
  static constexpr int kRedFloats = kTok * kMmaRedRows;
  static constexpr int kSmem = 1024 + kStages * kStage + 256 + kRedFloats * 4;
  static constexpr int kMinBlocks = NT == 1 ? 3 : 2;
  // independent MMA chains per group: one per 64-column tile up to 16
  // tokens; with more token blocks there is enough independent work per warp
  static constexpr int kChains = NT <= 2 ? 2 : 1;
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Same with a zero accumulator (starts a chain without clearing registers).
__device__ __forceinline__ void mma_bf16_16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// BF16x2 (128 + q) of the pair in the low nibbles of each half of v:
// (v & mask) | magic with mask = 0x000F000F and magic = 0x43004300 (a BF16
// with exponent 2^7 whose low mantissa bits take the nibble), as one logic op.
__device__ __forceinline__ uint32_t nib_pair_bf16(uint32_t v, uint32_t mask, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(mask), "r"(magic));
  return r;
}

// B fragments of two consecutive 16-column k-steps for tokens 8j .. 8j+7 of an
// activation block whose rows are `row_bytes` apart: lanes 8i .. 8i+7 address
// the rows at column offset 8i (x4 matrices = k-steps (0: cols 0-7, 8-15), (1: 16-23, 24-31)).
__device__ __forceinline__ void ldsm_b2(uint32_t addr, uint32_t (&b)[2][2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(b[0][0]), "=r"(b[0][1]), "=r"(b[1][0]), "=r"(b[1][1])
               : "r"(addr));
}

__device__ __forceinline__ float2 lds64f(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

// NT: n8 token blocks, M <= 8 * NT (NT = 1, 2, 4); EPI: bias / activation
// epilogue; G: quantisation group (32, 64, 128 columns), or 256 for per-channel
// scales (one group spanning K, folded once per 256-column stage: the fold is
// linear, so per-stage folds with the row's one scale and zero-point sum to
// the single fold over K)
template <int NT, bool EPI, int G>
__global__ void __launch_bounds__(kMmaThreads, MmaCfg<NT>::kMinBlocks) w4a16_mma_kernel(
    const uint16_t* __restrict__ X, const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
    const uint8_t* __restrict__ zeros, uint16_t* __restrict__ Y, int64_t M, int64_t N, int64_t K, int stages_per_split,
    int splits, int* err, Epi epi) {
  using C = MmaCfg<NT, G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + C::kStages * C::kStage);
  uint64_t* empty = full + C::kStages;
  uint64_t* summed = empty + C::kStages;  // activation sums of the stage are in place
  uint64_t* red_bar = summed + C::kStages;  // split-K: every rank's partial rows have arrived
  float* red = reinterpret_cast<float*>(ring + C::kStages * C::kStage + 256);
  __shared__ volatile int s_abort;
  // extraction constants, read back from shared memory so that the compiler
  // keeps them in registers: the nibble mask and the BF16 magic become the two
  // register operands of one LOP3
  __shared__ volatile uint32_t s_kc[2];

  const int split = blockIdx.x, nt = blockIdx.y;  // the K ranges of a tile form one cluster (rank = split)
  const int64_t KS = K / kMmaStageCols;
  const int s0 = split * stages_per_split;
  const int nst = static_cast<int>(imin64(KS, s0 + stages_per_split)) - s0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ngK = G == 256 ? 1 : K / G;  // groups per weight row
  const int64_t KB = K / kTileK;
  const int mrows = static_cast<int>(imin64(M, C::kTok));

  // split K: rank q of the tile's cluster owns rows [lo(q), lo(q + 1)), lo(q) = 128 q / splits
  // (at least eight rows for every split count up to 16)
  auto row_lo = [&](int q) { return q * kTileN / splits; };
  const int r_lo = row_lo(split), r_n = row_lo(split + 1) - r_lo;
  const int rstride = (kTileN + splits - 1) / splits;  // slice rows of the receive buffer
  // token groups a source sends per row: lane tq holds tokens 2tq, 2tq+1 (and
  // 8+2tq, 9+2tq); groups whose first token is >= M are all zero and not sent
  const int groups = NT == 1 ? (mrows + 1) / 2 : 4;

  const uint32_t tx = kMmaCodeBytes + C::kGps * 320 + mrows * kMmaStageCols * 2;
  auto issue_w = [&](int i) {  // weights of stage i (ring slot i % C::kStages)
    uint8_t* st = ring + (i % C::kStages) * C::kStage;
    uint64_t* bar = &full[i % C::kStages];
    const int64_t kb = static_cast<int64_t>(s0 + i) * 4;  // first 64-column block
    const int64_t g0 = G == 256 ? 0 : kb * 64 / G;  // first group
    mbar_arrive_expect_tx(bar, tx);
    bulk_load(st, codes + (static_cast<int64_t>(nt) * KB + kb) * 4096, kMmaCodeBytes, bar);
    bulk_load(st + kMmaMetaOff, scales + (static_cast<int64_t>(nt) * ngK + g0) * kTileN, C::kGps * 256, bar);
    bulk_load(st + C::kZeroOff, zeros + (static_cast<int64_t>(nt) * ngK + g0) * (kTileN / 2), C::kGps * 64, bar);
  };
  auto issue_x = [&](int i) {  // activation rows of stage i
    uint8_t* st = ring + (i % C::kStages) * C::kStage;
    const int64_t k0 = static_cast<int64_t>(s0 + i) * kMmaStageCols;
    for (int m = 0; m < mrows; ++m)
      bulk_load(st + C::kXOff + m * kMmaXRow, X + m * K + k0, kMmaStageCols * 2, &full[i % C::kStages]);
  };
  if (warp == kMmaProducer && lane == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kMmaConsumers);
      mbar_init(&summed[i], 4);
    }
    mbar_init(red_bar, 1);
    fence_mbar_init();
    // the owner's one arrival, with the bytes every rank will store into its slice
    if (splits > 1) mbar_arrive_expect_tx(red_bar, static_cast<uint32_t>(splits * r_n * groups * 2 * NT * 4));
    s_abort = 0;
    s_kc[0] = 0x000F000Fu;
    s_kc[1] = 0x43004300u;
    // weights never depend on the previous kernel on the stream: start them first
    for (int i = 0; i < nst && i < C::kStages; ++i) issue_w(i);
  }
  // token rows >= M are never copied: zero them once so B fragments need no bounds test
  for (int idx = threadIdx.x; idx < C::kStages * (C::kTok - mrows) * (kMmaXRow / 16); idx += kMmaThreads) {
    const int per = (C::kTok - mrows) * (kMmaXRow / 16);
    const int stg = idx / per, rem = idx % per;
    const int row = mrows + rem / (kMmaXRow / 16), c16 = rem % (kMmaXRow / 16);
    *reinterpret_cast<uint4*>(ring + stg * C::kStage + C::kXOff + row * kMmaXRow + c16 * 16) = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (splits > 1) cluster_arrive_relaxed();  // waited for before the first access to another CTA
  grid_dep_wait();
  grid_dep_launch();

  const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates
  // bias of this thread's output rows (direct path), loaded now and used at the end
  float bias_r[kMmaRowBlocks][2] = {};
  if constexpr (EPI) {
    if (splits == 1 && warp < kMmaConsumers) {
#pragma unroll
      for (int rb = 0; rb < kMmaRowBlocks; ++rb)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr)
          bias_r[rb][hr] =
              epi_bias(epi, static_cast<int64_t>(nt) * kTileN + warp * 16 * kMmaRowBlocks + 16 * rb + gq + hr * 8);
    }
  }
  float acc[kMmaRowBlocks][NT][4];
#pragma unroll
  for (int rb = 0; rb < kMmaRowBlocks; ++rb)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[rb][j][e] = 0.0f;

  if (warp == kMmaProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int i = 0; i < nst && i < C::kStages; ++i) issue_x(i);
      for (int i = C::kStages; i < nst; ++i) {
        if (!mbar_wait(&empty[i % C::kStages], ((i / C::kStages) & 1) ^ 1, kMmaWaitNs, &s_abort)) {
          set_error(err, QLIN_ERR_TIMEOUT);
          s_abort = 1;
          break;
        }
        issue_w(i);
        issue_x(i);
      }
    }
  } else if (warp == kMmaSummer) {
    // ------------------------------------------------------------ activation sums per group and token
    // M <= 8: C = ones(16 x 128) * X_g^T, every row of C holds sum_k x_k of the
    // n8 token block; lanes 0-3 (row 0) write tokens 2t, 2t + 1.
    // M > 8: C = X_g (16 tokens x 128) * ones(128 x 8) per block of 16 tokens,
    // one MMA per k-step; lanes 4g (column 0) write tokens g and g + 8.
    const uint32_t ones[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};  // BF16 1.0 pairs
    for (int i = 0; i < nst; ++i) {
      const int slot = i % C::kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (i / C::kStages) & 1, kMmaWaitNs, &s_abort))) {
        set_error(err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      const uint32_t st = smem_u32(ring + slot * C::kStage);
      float* sums = reinterpret_cast<float*>(ring + slot * C::kStage + C::kSumOff);  // [group][kTok tokens]
#pragma unroll
      for (int grp = 0; grp < C::kGps; ++grp) {
        float cs[2][4];  // two chains of G / 32 k-steps
        if constexpr (NT == 1) {
#pragma unroll
          for (int q = 0; q < G / 32; ++q) {
            uint32_t bb[2][2];
            ldsm_b2(st + C::kXOff + (lane & 7) * kMmaXRow + (grp * G + q * 32 + (lane >> 3) * 8) * 2, bb);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (q == 0)
                mma_bf16_16816_z(cs[h], ones, bb[h][0], bb[h][1]);
              else
                mma_bf16_16816(cs[h], ones, bb[h][0], bb[h][1]);
            }
          }
          if (lane < 4)
            *reinterpret_cast<float2*>(sums + grp * C::kTok + 2 * lane) =
                make_float2(cs[0][0] + cs[1][0], cs[0][1] + cs[1][1]);
        } else {
#pragma unroll
          for (int tb = 0; tb < NT / 2; ++tb) {  // 16 tokens per block
#pragma unroll
            for (int ks = 0; ks < G / 16; ++ks) {
              // A fragment of tokens 16tb .. 16tb+15 x columns 16ks..16ks+15: lanes
              // 0-15 address token rows (lane & 15) at column 16ks, lanes 16-31 at 16ks + 8
              uint32_t a[4];
              asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                           : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                           : "r"(st + C::kXOff + (tb * 16 + (lane & 15)) * kMmaXRow +
                                 (grp * G + ks * 16 + (lane >> 4) * 8) * 2));
              if (ks < 2)
                mma_bf16_16816_z(cs[ks & 1], a, ones[0], ones[1]);
              else
                mma_bf16_16816(cs[ks & 1], a, ones[0], ones[1]);
            }
            if (tq == 0) {
              sums[grp * C::kTok + tb * 16 + gq] = cs[0][0] + cs[1][0];
              sums[grp * C::kTok + tb * 16 + gq + 8] = cs[0][2] + cs[1][2];
            }
          }
        }
      }
      __syncwarp();
      if (lane < 4) mbar_arrive(&summed[slot]);
    }
  } else {
    // ------------------------------------------------------------ consumers: rows 32*warp .. 32*warp + 31
    // row block rb (m16) of this warp: rows 32 warp + 16 rb + (0..15); this
    // thread's rows in it are rr(rb) and rr(rb) + 8.  Both blocks share every B
    // fragment and activation sum.
    const int rbase = warp * 16 * kMmaRowBlocks + gq;
    auto rr = [&](int rb) { return rbase + 16 * rb; };
    const uint32_t kmask = s_kc[0], kmagic = s_kc[1];
    // pair in nibble positions i, i + 4 of w, as BF16x2 (128 + q): a constant
    // shift and one LOP3
    auto pair_at = [&](uint32_t w, int i) { return nib_pair_bf16(w >> (4 * i), kmask, kmagic); };
    // zero-point nibble of this thread's rows (all of the same parity): moved to
    // bits 16..19 of an FP32 whose exponent is 2^7, which reads as 128 + z exactly
    const uint32_t zsh = (rbase & 1) ? 12u : 16u;
    if (splits > 1) cluster_wait();  // overlaps the first stage's load
    for (int i = 0; i < nst; ++i) {
      const int slot = i % C::kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (i / C::kStages) & 1, kMmaWaitNs, &s_abort))) {
        set_error(err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      const uint32_t st = smem_u32(ring + slot * C::kStage);  // shared-space address of the stage
      const uint32_t sc = st + kMmaMetaOff;                   // FP16 scales [kGps][128]
      const uint32_t zp = st + C::kZeroOff;                   // zero nibbles [kGps][64]
      // word t (this lane's) of the records of each of this thread's rows in both
      // halves of a 64-column tile: w[rb][2h + e] = half h, row rr(rb) + 8e.  Each
      // tile's words are loaded one tile ahead to hide the shared-memory latency.
      uint32_t cw[kMmaRowBlocks][4];
      auto load_codes = [&](int kbl, uint32_t (&w)[kMmaRowBlocks][4]) {
        const uint32_t tile = st + kbl * 4096 + tq * 4;
#pragma unroll
        for (int rb = 0; rb < kMmaRowBlocks; ++rb) {
          w[rb][0] = lds32(tile + rr(rb) * 16);
          w[rb][1] = lds32(tile + (rr(rb) + 8) * 16);
          w[rb][2] = lds32(tile + 2048 + rr(rb) * 16);
          w[rb][3] = lds32(tile + 2048 + (rr(rb) + 8) * 16);
        }
      };
      load_codes(0, cw);
      bool sums_ok = true;
      // Groups: G = 128 spans two 64-column tiles (one MMA chain per tile up to
      // 16 tokens, summed at the fold), G = 64 one tile, G = 32 one half of a
      // tile (two k-steps).  The fold of group g:
      //   y += s (sum x (128 + q) - (128 + z) sum x); tokens 8j+2t, +1
      constexpr int kTpg = G >= 64 ? G / 64 : 1;      // tiles per outer step
      constexpr int kCh = G == 128 ? C::kChains : 1;  // MMA chains per group
      auto fold = [&](int g, const float (&cc)[kCh][kMmaRowBlocks][NT][4]) {
        if (g == 0)
          sums_ok = __all_sync(0xffffffffu, mbar_wait(&summed[slot], (i / C::kStages) & 1, kMmaWaitNs, &s_abort));
        float2 xv[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) xv[j] = lds64f(st + C::kSumOff + (g * C::kTok + j * 8 + 2 * tq) * 4);
#pragma unroll
        for (int rb = 0; rb < kMmaRowBlocks; ++rb)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int r = rr(rb) + hr * 8;
            const float s =
                __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(sc + (g * kTileN + r) * 2))));
            const uint32_t zb = lds8(zp + g * (kTileN / 2) + r / 2);
            const float cz = __uint_as_float(((zb << zsh) & 0x000F0000u) | 0x43000000u);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const float c0 = kCh == 2 ? cc[0][rb][j][hr * 2] + cc[kCh - 1][rb][j][hr * 2] : cc[0][rb][j][hr * 2];
              const float c1 =
                  kCh == 2 ? cc[0][rb][j][hr * 2 + 1] + cc[kCh - 1][rb][j][hr * 2 + 1] : cc[0][rb][j][hr * 2 + 1];
              acc[rb][j][hr * 2] = fmaf(s, fmaf(-cz, xv[j].x, c0), acc[rb][j][hr * 2]);
              acc[rb][j][hr * 2 + 1] = fmaf(s, fmaf(-cz, xv[j].y, c1), acc[rb][j][hr * 2 + 1]);
            }
          }
      };
#pragma unroll
      for (int ob = 0; ob < 4 / kTpg; ++ob) {
        float c[kCh][kMmaRowBlocks][NT][4];
#pragma unroll
        for (int kb2 = 0; kb2 < kTpg; ++kb2) {
          const int kbl = ob * kTpg + kb2;  // 64-column tile within the stage
          const int ch = kCh == 2 ? kb2 : 0;
          uint32_t cur[kMmaRowBlocks][4];
#pragma unroll
          for (int rb = 0; rb < kMmaRowBlocks; ++rb)
#pragma unroll
            for (int q = 0; q < 4; ++q) cur[rb][q] = cw[rb][q];
          if (kbl < 3) load_codes(kbl + 1, cw);
          // B fragments: one ldmatrix.x4 per token block covers two 16-column
          // k-steps; up to 16 tokens both halves of the tile are loaded up front
          constexpr int kBH = NT <= 2 ? 2 : 1;  // halves of B fragments held at once
          uint32_t b[kBH][NT][2][2];
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {  // k-step = columns 16a .. 16a+15 of half h
            const int h = ks >> 1, ia = 2 * (ks & 1);
            if (ks == 0 || (kBH == 1 && ks == 2)) {
#pragma unroll
              for (int hb = 0; hb < kBH; ++hb)
#pragma unroll
                for (int j = 0; j < NT; ++j)
                  ldsm_b2(st + C::kXOff + (j * 8 + (lane & 7)) * kMmaXRow +
                              (kbl * 64 + (h + hb) * 32 + (lane >> 3) * 8) * 2,
                          b[hb][j]);
            }
            // the chain starts from zero at the first k-step of its group (or tile)
            const bool start = G == 32 ? (ks & 1) == 0 : (ks == 0 && (kCh == 2 || kb2 == 0));
#pragma unroll
            for (int rb = 0; rb < kMmaRowBlocks; ++rb) {
              uint32_t a[4];
              a[0] = pair_at(cur[rb][2 * h], ia);          // row rr,   columns 2t, 2t+1
              a[1] = pair_at(cur[rb][2 * h + 1], ia);      // row rr+8, columns 2t, 2t+1
              a[2] = pair_at(cur[rb][2 * h], ia + 1);      // row rr,   columns 2t+8, 2t+9
              a[3] = pair_at(cur[rb][2 * h + 1], ia + 1);  // row rr+8, columns 2t+8, 2t+9
#pragma unroll
              for (int j = 0; j < NT; ++j) {
                const uint32_t(&bk)[2] = b[kBH == 2 ? h : 0][j][ks & 1];
                if (start)
                  mma_bf16_16816_z(c[ch][rb][j], a, bk[0], bk[1]);
                else
                  mma_bf16_16816(c[ch][rb][j], a, bk[0], bk[1]);
              }
            }
            if (G == 32 && (ks & 1)) fold(kbl * 2 + h, c);  // end of a 32-column group
          }
        }
        if (G >= 64) fold(ob, c);
      }
      if (!sums_ok) {
        set_error(err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
  }

  // ---------------------------------------------------------------- outputs
  // this thread's outputs: row 32 warp + 16 rb + gq + 8 hr, token 8 j + 2 tq + e
  if (splits == 1) {
    if (warp < kMmaConsumers) {
#pragma unroll
      for (int rb = 0; rb < kMmaRowBlocks; ++rb)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int64_t n = static_cast<int64_t>(nt) * kTileN + warp * 16 * kMmaRowBlocks + 16 * rb + gq + hr * 8;
          float o[2 * NT];  // tokens 8j + 2tq + e of row n
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) o[2 * j + e] = acc[rb][j][hr * 2 + e];
          if constexpr (EPI) epi_run(epi.act, o, bias_r[rb][hr]);
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
  // Split K: every CTA sends each row's token values to the row's owner with
  // one asynchronous remote store (8 or 16 bytes: the tokens this lane holds,
  // slot tq * 2NT + 2j + e for token 8j + 2tq + e) that completes its bytes on
  // the owner's red_bar, so no fence or barrier among the CTAs is needed.  Each
  // owner, once every rank's values have landed, adds the slots in rank order
  // (deterministic) from its own shared memory and writes Y.
  __syncwarp();
  if (warp >= kMmaConsumers) cluster_wait();  // the consumers waited at their start
  if (warp < kMmaConsumers && tq < groups) {
    const uint32_t red_u32 = smem_u32(red), bar_u32 = smem_u32(red_bar);
#pragma unroll
    for (int rb = 0; rb < kMmaRowBlocks; ++rb)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = warp * 16 * kMmaRowBlocks + 16 * rb + gq + hr * 8;
        const int q = (r * splits + splits - 1) / kTileN;  // owner: the last rank with lo(q) <= r
        const uint32_t dst = cluster_map(red_u32, static_cast<uint32_t>(q)) +
                             static_cast<uint32_t>(((split * rstride + r - row_lo(q)) * C::kTok + tq * 2 * NT) * 4);
        const uint32_t dbar = cluster_map(bar_u32, static_cast<uint32_t>(q));
        if constexpr (NT == 1) {
          st_async_v2(dst, acc[rb][0][hr * 2], acc[rb][0][hr * 2 + 1], dbar);
        } else {
#pragma unroll
          for (int j = 0; j < NT; j += 2)  // slots 2j .. 2j + 3: token blocks j and j + 1
            st_async_v4(dst + j * 8, acc[rb][j][hr * 2], acc[rb][j][hr * 2 + 1], acc[rb][j + 1][hr * 2],
                        acc[rb][j + 1][hr * 2 + 1], dbar);
        }
      }
  }
  if (!mbar_wait_cluster(red_bar, 0, kMmaWaitNs)) {
    set_error(err, QLIN_ERR_TIMEOUT);
    return;
  }
  for (int idx = threadIdx.x; idx < r_n * mrows; idx += kMmaThreads) {
    const int m = idx / r_n, rl = idx % r_n;
    const int slot = NT == 1 ? m : ((m & 7) >> 1) * 2 * NT + (m >> 3) * 2 + (m & 1);
    const float* src = red + rl * C::kTok + slot;
    float v = 0.0f;
    for (int p = 0; p < splits; ++p) v += src[p * rstride * C::kTok];
    const int64_t n = static_cast<int64_t>(nt) * kTileN + r_lo + rl;
    if constexpr (EPI) v = epi_apply(epi, v, n);
    Y[static_cast<int64_t>(m) * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

// Clusters of `cs` CTAs of w4a16_mma_kernel<NT, *, G> that fit on the GPU at
// once (cudaOccupancyMaxActiveClusters; wide clusters pack the GPCs less
// densely), for cs = 1 .. kMmaMaxCluster, queried once per device.
template <int NT, int G>
static int max_active_clusters(int cs) {
  static std::mutex mu;
  static std::unordered_map<int, std::array<int, kMmaMaxCluster + 1>> table;  // device -> count per size
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  auto it = table.find(dev);
  if (it == table.end()) {
    std::array<int, kMmaMaxCluster + 1> t{};
    if (set_smem_once(w4a16_mma_kernel<NT, false, G>, MmaCfg<NT, G>::kSmem, true) == cudaSuccess) {
      for (int c = 1; c <= kMmaMaxCluster; ++c) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(c), 1);
        cfg.blockDim = dim3(kMmaThreads);
        cfg.dynamicSmemBytes = MmaCfg<NT, G>::kSmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(c);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, w4a16_mma_kernel<NT, false, G>, &cfg) != cudaSuccess) n = 0;
        t[c] = n;
      }
    }
    (void)cudaGetLastError();
    it = table.emplace(dev, t).first;
  }
  return it->second[cs];
}

// Split K only for parallelism.  Time model per split count s (a cluster of s
// CTAs per tile): waves x (start-up + stages per CTA x the time one CTA takes
// for a stage), where a wave holds as many clusters as fit at once and the
// CTAs of a wave share the HBM bandwidth, or less when they are too few to
// keep enough bytes in flight (each has at most a ring of stages in flight for
// a loaded memory latency).  Fewer splits on a near tie.  The split-K sums
// never leave the GPC: no workspace.
template <int G>
static int active_clusters(int ntb, int cs) {
  return ntb == 1 ? max_active_clusters<1, G>(cs) : ntb == 2 ? max_active_clusters<2, G>(cs)
                                                               : max_active_clusters<4, G>(cs);
}

SplitPlan plan_w4a16_mma(int64_t M, int64_t N, int64_t K, int num_sms, int G) {
  (void)num_sms;  // the cluster occupancy table already counts the SMs
  if (G != 32 && G != 64 && G != 128) G = 256;  // per-channel scales (G == K): the 256-column instantiation
  SplitPlan p;
  const int64_t tiles = N / kTileN;
  const int64_t KS = K / kMmaStageCols;
  const int ntb = M <= 8 ? 1 : M <= 16 ? 2 : 4;  // n8 token blocks
  const double bw = 6.5e12, latency = 2.5e-6, startup = 3e-6;
  const int ring = ntb == 1 ? MmaCfg<1>::kStages : ntb == 2 ? MmaCfg<2>::kStages : MmaCfg<4>::kStages;
  const double stage_bytes = kMmaCodeBytes + 320.0 * (kMmaStageCols / G) + 2.0 * kMmaStageCols * static_cast<double>(M);
  const int64_t cap = KS < kMmaMaxCluster ? KS : kMmaMaxCluster;
  int64_t best_s = 1;
  double best_t = 1e30;
  for (int64_t c = 1; c <= cap; ++c) {
    const int64_t per = (KS + c - 1) / c;
    const int64_t s = (KS + per - 1) / per;  // splits actually formed
    if (s != c) continue;
    const int cs = static_cast<int>(s);
    const int64_t fit = G == 32 ? active_clusters<32>(ntb, cs) : G == 64 ? active_clusters<64>(ntb, cs)
                      : G == 256 ? active_clusters<256>(ntb, cs) : active_clusters<128>(ntb, cs);
    if (fit <= 0) continue;
    const int64_t waves = (tiles + fit - 1) / fit;
    const double conc = static_cast<double>((tiles < fit ? tiles : fit) * s);  // CTAs running together
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

bool mma_path_ok(int64_t M, int64_t K) { return M >= 1 && M <= 32 && K % kMmaStageCols == 0; }

template <int NT, bool EPI, int G>
static cudaError_t launch_mma(const uint16_t* X, const uint8_t* codes, const uint16_t* scales, const uint8_t* zeros,
                              uint16_t* Y, int64_t M, int64_t N, int64_t K, const SplitPlan& plan, int* err,
                              cudaStream_t st, const Epi& epi) {
  cudaError_t e = set_smem_once(w4a16_mma_kernel<NT, EPI, G>, MmaCfg<NT, G>::kSmem, true);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.splits), static_cast<unsigned>(N / kTileN));
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = MmaCfg<NT, G>::kSmem;
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
  return cudaLaunchKernelEx(&cfg, w4a16_mma_kernel<NT, EPI, G>, X, codes, scales, zeros, Y, M, N, K, plan.kb_per_split,
                            plan.splits, err, epi);
}

cudaError_t launch_w4a16_mma(const uint16_t* X, const uint8_t* codes, const uint16_t* scales, const uint8_t* zeros,
                             uint16_t* Y, int64_t M, int64_t N, int64_t K, int G, const SplitPlan& plan, void* ws,
                             int* err, cudaStream_t st, const Epi& epi) {
  (void)ws;  // the split-K reduction runs in distributed shared memory
  const bool fused = epi.bias != nullptr || epi.act != QLIN_ACT_NONE;
  auto go = [&](auto nt, auto ep, auto g) {
    return launch_mma<decltype(nt)::value, decltype(ep)::value, decltype(g)::value>(X, codes, scales, zeros, Y, M, N,
                                                                                      K, plan, err, st, epi);
  };
  auto by_group = [&](auto nt, auto ep) {
    if (G == 32) return go(nt, ep, std::integral_constant<int, 32>{});
    if (G == 64) return go(nt, ep, std::integral_constant<int, 64>{});
    if (G == 128) return go(nt, ep, std::integral_constant<int, 128>{});
    return go(nt, ep, std::integral_constant<int, 256>{});  // per-channel: G == K
  };
  auto by_epi = [&](auto nt) { return fused ? by_group(nt, std::true_type{}) : by_group(nt, std::false_type{}); };
  if (M <= 8) return by_epi(std::integral_constant<int, 1>{});
  if (M <= 16) return by_epi(std::integral_constant<int, 2>{});
  return by_epi(std::integral_constant<int, 4>{});
}

}  // namespace qlin
