// Tensor-core kernels for sm_103a: TMA -> shared memory -> tcgen05.mma with
// the accumulator in TMEM -> tcgen05.ld epilogue.
//
// Orientation ("swap AB"): the 128 weight rows of a tile are the MMA's M side
// and the tokens are its N side (16..256), so that a decode batch of a few
// tokens still fills the 128-row MMA and every weight is read once per token
// block.  D[n][m] = sum_k W[n][k] X[m][k] lands in TMEM lane n, column m.
// The one exception is FP8 block scaling with 128-token tiles, which runs
// token-major (tokens as M, 128 or 256 weight rows as N) so that its per-K-block
// promotion factor is one scalar per TMEM lane.
//
// W4A16 ([LP] S11, S23 "fast path"): the packed INT4 tile and its scales /
// zero-points are bulk-copied into shared memory; eight dequantisation warps
// turn them into BF16 s (q - z) written straight into the 128-byte-swizzled
// K-major layout the MMA reads; kind::f16 MMA (BF16 x BF16 -> FP32).
// W8A8 ([LP] S8, S9): E4M3 weight and activation tiles by TMA; kind::f8f6f4
// MMA; the epilogue applies sx[m] * sw.
//
// Persistent and warp-specialised: one CTA per SM walks a list of work units
// (output tile x K range).  Warp 0 streams every unit's tiles through one
// ring of shared-memory stages, so HBM traffic does not pause between units;
// warp 1 owns TMEM and issues the MMAs into one of two accumulators; the
// dequantisation warps (W4A16) fill a second ring with BF16 weight tiles; four
// epilogue warps (eight for block scaling from 32 tokens) drain the other
// accumulator meanwhile.  Every wait is bounded in time; on expiry the kernel
// records QLIN_ERR_TIMEOUT and leaves.
#include <cmath>
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "qlin_internal.cuh"
#include "qlin_ptx.cuh"

namespace qlin {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr int kSmemBudget = 225 * 1024;

// Block-scaled formats whose scales the MMA applies (template argument MX)
constexpr int kMxNone = 0;
constexpr int kMxF8 = 1;  // MXFP8: E4M3 elements, E8M0 scale per 32 (kind::mxf8f6f4, scale_vec::1X)
constexpr int kMxF4 = 2;  // MXFP4: E2M1 elements, E8M0 scale per 32 (kind::mxf4, scale_vec::2X)
constexpr int kNvF4 = 3;  // NVFP4: E2M1 elements, E4M3 scale per 16 (kind::mxf4nvf4, scale_vec::4X)

template <int BN, bool W4, int KPS, bool BS = false, int WN = 128, int MX = kMxNone, bool A8 = false>
struct TcCfg {
  static constexpr bool kF4 = MX == kMxF4 || MX == kNvF4;     // E2M1 operands, two per byte
  static constexpr int kBlkBytes = 128;                         // bytes of one row of a K block
  // K columns per block: 64 for W4A16 (one packed code tile), 128 for E4M3
  // operands, 256 for E2M1; W4A8 takes two code tiles (one quantisation
  // group) per block
  static constexpr int kCols = kF4 ? 256 : (W4 && !A8) ? 64 : 128;
  // TMA column step of a K block, in elements of the tensor map (BF16 for
  // W4A16 activations, bytes otherwise)
  static constexpr int kTmaX = (W4 && !A8) ? 64 : 128;
  static constexpr int kXBlk = BN * kBlkBytes;                  // token tile of one K block
  static constexpr int kWBlk = W4 ? (A8 ? 8192 : 4096) : WN * kBlkBytes;  // packed codes / E4M3 tile of one K block
  // group scales and zero-points of a stage: room for G = 32 (two groups per
  // 64-column block); G = 64 / 128 use the front of each region; W4A8: one
  // group (G = 128) per block
  static constexpr int kGroupsMax = W4 ? (A8 ? KPS : 2 * KPS) : 0;
  static constexpr int kScaleOff = KPS * kXBlk + KPS * kWBlk;   // scales, then zero-points (W4A16)
  static constexpr int kZeroOff = kScaleOff + kGroupsMax * 256;
  static constexpr int kMetaBytes = W4 ? ((kGroupsMax * 320 + 1023) / 1024) * 1024 : 0;
  // Block-scaled formats: the scale atoms of the stage's K block (kSfK
  // atoms of weight scales, then kSfK per 128 tokens), copied into TMEM by
  // the MMA thread.  An atom holds four scales of 128 rows: 128 columns of
  // MXFP8, 128 of MXFP4 (two per 256-column block), 64 of NVFP4 (four)
  static constexpr int kSfK = MX == kNvF4 ? 4 : MX == kMxF4 ? 2 : 1;
  static constexpr int kSfOff = KPS * kXBlk + KPS * kWBlk + kMetaBytes;
  static constexpr int kSfbAtoms = BN > 128 ? 2 : 1;                // token atoms of a tile
  static constexpr int kSfBytes = MX ? ((512 * kSfK * (1 + kSfbAtoms) + 1023) / 1024) * 1024 : 0;
  static constexpr int kStage = KPS * kXBlk + KPS * kWBlk + kMetaBytes + kSfBytes;
  static constexpr int kTxBase =
      KPS * kXBlk + KPS * kWBlk + (MX ? 512 * kSfK * (1 + kSfbAtoms) : 0);  // W4A16: plus 320 B per group
  // dequantised BF16 weight tiles: in TMEM (tcgen05.st, read by the MMA as
  // its A operand) when the accumulators leave room, else in shared memory
  static constexpr bool kATmem = W4 && BN <= 128;
  // A slots: W4A16 in TMEM hands the MMA two 64-column blocks per slot (64
  // TMEM columns), so that the issuing thread's fixed cost per hand-off (a
  // barrier wait, a fence, a commit) is paid once per 128 columns; W4A8 one
  // 128-column E4M3 block (32 columns); the shared-memory path one 64-column block
  static constexpr int kSlotBlocks = (kATmem && !A8) ? 2 : 1;
  static constexpr int kAStages = W4 ? (kATmem ? (A8 ? 8 : 4) : 4) : 0;
  static constexpr int kAStage = (W4 && !kATmem) ? 128 * kBlkBytes : 0;  // shared-memory bytes per slot
  static constexpr int kASlotCols = 32 * kSlotBlocks;           // TMEM columns per slot (64 BF16 per lane and block)
  // output staging: two boxes of 16 tokens x 128 rows of BF16 for the tensor stores
  // Block scaling with 128-token tiles runs token-major: the token tile is the
  // MMA's A operand (TMEM lane = token) and the weight tile of WN rows (one or
  // two 128-row scale blocks) its B operand, so the promotion factor
  // sx[kb][m] * sw[n / 128][kb] is one scalar per thread and 128 columns.
  static constexpr bool kTokM = BS && BN == 128;
  // Block-scaled formats with 256-token tiles have a single accumulator: the
  // epilogue drains it into registers (BF16 pairs) and hands it back before
  // writing, so that the next unit's MMAs overlap the stores
  static constexpr bool kEarly = MX && BN == 256;
  // epilogue warps: four (one per TMEM lane quadrant); with block scaling and
  // at least 32 tokens, or the early drain, eight, two per quadrant, each
  // taking half the columns
  static constexpr int kEpiWarps = ((BS && BN >= 32) || kEarly) ? 8 : 4;
  static constexpr int kEpiHalves = kEpiWarps / 4;
  static constexpr int kEpiBox = 16 * kTileN * 2;
  static constexpr int kEpiBoxes = kTokM ? 0 : 2 * kEpiHalves;  // token-major writes rows straight to Y
  static constexpr int kScaleVec = (BS && !kTokM) ? 2 * 128 * 4 : 0;  // sx * sw of one K block, two buffers
  static constexpr int kStagesRaw =
      (kSmemBudget - 2048 - kAStages * kAStage - kEpiBoxes * kEpiBox - kScaleVec) / kStage;
  static constexpr int kStages = kStagesRaw > 16 ? 16 : kStagesRaw;
  static constexpr int kAccCols = kTokM ? WN : BN;              // one accumulator
  // accumulators in TMEM: two (one unit while the epilogue drains the other);
  // block scaling and W4A8 keep up to four K-block partial products in flight
  // block-scaled formats with 256-token tiles keep one (the scale-factor ring takes the rest of TMEM)
  static constexpr int kAccBufs = BS ? (512 / kAccCols < 4 ? 512 / kAccCols : 4) : A8 ? 4 : (MX && BN == 256) ? 1 : 2;
  static constexpr int kAColBase = kAccBufs * BN;               // first TMEM column of the A slots
  // Block scale factors in TMEM: one slot per pipeline stage (the scale warp
  // fills slot s once stage s has landed, and the producer refills stage s
  // only after the MMAs that read slot s are done), four columns per atom (see
  // mma_mx8, mma_mxf4): kSfK atoms of weight scales and kSfK x kSfbAtoms of
  // token scales per slot
  static constexpr int kSfSlots = MX ? kStages : 0;
  static constexpr int kSfaCol = kAccBufs * BN;
  static constexpr int kSfbCol = kSfaCol + 4 * kSfK * kSfSlots;
  static constexpr int kTmemNeed =
      kAccBufs * BN + (kATmem ? kAStages * kASlotCols : 0) + 4 * kSfSlots * kSfK * (1 + kSfbAtoms);
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                 : kTmemNeed <= 256 ? 256 : 512;
  static constexpr int kDqWarps = W4 ? 8 : 0;
  // block-scaled formats: the warps that copy scales into TMEM; NVFP4 (12
  // atom copies per K block at 256 tokens) splits them over two, weight atoms
  // on the first, token atoms on the second
  static constexpr int kSfWarps = MX == kNvF4 ? 2 : MX ? 1 : 0;
  static constexpr int kEpiWarp0 = 2 + kDqWarps + kSfWarps;
  static constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
  // Register cap per thread.  Each of the SM's four sub-partitions holds 16 K
  // registers and takes every fourth warp, so the cap is set by the
  // sub-partition with the most warps: 14 warps (W4A16) -> 4 -> 128;
  // 10 warps -> 3 -> 168; 6 warps -> 2 -> 255 (232 kept).
  static constexpr int kMaxRegs = W4 ? 128 : kThreads > 256 ? 168 : 232;
  static constexpr int kSmemBytes = 1024 /*align slack*/ + kStages * kStage + kAStages * kAStage +
                                    kEpiBoxes * kEpiBox + kScaleVec + 1024 /*barriers*/;
  static_assert(kStages >= 2, "pipeline too shallow");
  static_assert(kXBlk % 1024 == 0 && kStage % 1024 == 0, "1024-byte alignment of swizzled tiles");
  static_assert(W4 || KPS == 1, "E4M3 stages hold one K block");
  static_assert(kTmemNeed <= 512, "TMEM budget");
  static_assert(!BS || (!W4 && BN <= 128), "block scaling: E4M3 operands, at most 128 tokens (running sums in registers)");
  static_assert(WN == 128 || (kTokM && WN == 256), "256-row weight tiles only token-major");
  static_assert(!MX || (!W4 && !BS && BN >= 32), "block-scaled formats: 8- or 4-bit float operands, at least 32 tokens per tile");
  // The FP4 MMAs (scale_vec::2X / 4X) take scale addresses a multiple of four
  // TMEM columns above the 32-column-aligned scale region; a 64-token tile
  // would start two columns into its token atom (32-token tiles run only as the
  // single token block of M <= 32, checked by the host)
  static_assert(!kF4 || BN != 64, "FP4: 32 (one token block), 128 or 256 tokens per tile");
  static_assert(!A8 || (W4 && !BS && !MX && BN <= 64), "W4A8: packed INT4 weights, at most 64 tokens per tile");
  static_assert(kSlotBlocks == 1 || KPS % 2 == 0, "two-block slots need an even number of blocks per stage");
};

struct TcArgs {
  const uint8_t* codes;
  const uint16_t* scales;
  const uint8_t* zeros;
  const float* sx;
  const float* sw;  // W8A8 block scaling: sx = [K/128][M], sw = [N/128][K/128]
  const uint8_t* sfa;  // block-scaled formats: scale atoms of the weights, [N/128][K atoms][512 B]
  const uint8_t* sfb;  // block-scaled formats: scale atoms of the tokens, [ceil(M/128)][K atoms][512 B]
                       // (NVFP4: sx / sw point at the two FP32 per-tensor scales)
  uint16_t* Y;
  float* partials;
  uint32_t* counters;
  int* err;
  int64_t M, N, K;
  int ntiles;        // N / 128
  int mblocks;       // token blocks
  int splits;        // K ranges per output tile
  int kb_per_split;  // K blocks per range (a multiple of the blocks per stage)
  int units;         // ntiles * mblocks * splits
  int mb_fast;       // unit order: token block fastest (weights streamed once) or weight tile fastest
  int x_keep;        // keep activation tiles in L2 (evict-last) when they are small
  int w_keep;        // keep weight tiles in L2 (evict-last): with the weight tile fastest, each one is
                     // read again by every later token block; otherwise they are streamed (evict-first)
  int G;             // W4A16 quantisation group (32, 64, 128, or K for per-channel scales)
  int gshift;        // log2 G; 31 for per-channel scales, so that every column maps to group 0
  Epi epi;           // output epilogue (bias, activation) of the *_fused calls
};

__device__ __forceinline__ uint16_t to_bf16(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

__device__ __forceinline__ void named_bar_epi() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }

// Eight columns of one 32-bit code word -> four BF16 pairs bf16(bf16(s) (q - z)):
// the caller rounds the FP16 group scale to BF16 once (s2), (q - z) is exact,
// and the product is rounded to BF16; component i is the pair in nibble
// positions i and i + 4.  Word t of a 32-column record holds pairs (columns
// 8i + 2t, +1) for i = 0..3.
__device__ __forceinline__ uint4 dequant8(uint32_t w, __nv_bfloat162 zoff, __nv_bfloat162 s2) {
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t v = ((w >> (4 * t)) & 0x000F000Fu) | 0x43004300u;  // BF16x2 (128 + q)
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v);
    b = __hmul2(__hsub2(b, zoff), s2);  // (q - z) is exact; the product with bf16(s) is rounded once
    o[t] = bf16x2_bits(b);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Work unit u -> (n tile, token block, K range).  The larger operand is
// streamed once and the smaller kept resident: when the activations are the
// smaller, tiles are taken in groups of kRasterN weight tiles x every token
// block, token block fastest, so that each weight tile is read from HBM once
// (its token blocks run at the same time); otherwise the weight tile varies
// fastest.  Weights that would fit in L2 are not assumed to stay there: the
// BF16 output streams through L2 as well (at 2048 tokens x 28672 rows, 117 MB).
constexpr int kRasterN = 16;
struct Unit {
  int nt, mb, split, kb0, nkb;
};
__device__ __forceinline__ Unit unit_of(const TcArgs& a, int u, int64_t KB) {
  Unit r;
  r.split = u % a.splits;
  const int tile = u / a.splits;
  if (a.mb_fast) {
    const int gsz = kRasterN * a.mblocks;
    const int g = tile / gsz, rem = tile % gsz;
    const int gn = a.ntiles - g * kRasterN < kRasterN ? a.ntiles - g * kRasterN : kRasterN;  // tiles in this group
    r.mb = rem % a.mblocks;
    r.nt = g * kRasterN + (rem / a.mblocks) % gn;
  } else {
    r.nt = tile % a.ntiles;
    r.mb = tile / a.ntiles;
  }
  r.kb0 = r.split * a.kb_per_split;
  const int64_t end = imin64(KB, static_cast<int64_t>(r.kb0) + a.kb_per_split);
  r.nkb = static_cast<int>(end - r.kb0);
  return r;
}

// EPI: the output epilogue (bias, activation) of the *_gemm_fused calls is compiled in;
// MX: block-scaled operands whose scales the MMA applies (kMxF8, kMxF4, kNvF4);
// A8: packed INT4 weights (W4 = true) dequantised to E4M3 times E4M3 tokens (W4A8)
template <int BN, bool W4, int KPS, bool BS, int WN, bool EPI, int MX = kMxNone, bool A8 = false>
__global__ void __maxnreg__((TcCfg<BN, W4, KPS, BS, WN, MX, A8>::kMaxRegs))
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_y, const __grid_constant__ TcArgs a) {
  using C = TcCfg<BN, W4, KPS, BS, WN, MX, A8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* aring = ring + C::kStages * C::kStage;
  uint8_t* epi_box = aring + C::kAStages * C::kAStage;  // [kEpiBoxes][16 tokens][128 rows] BF16
  float* scale_vec = reinterpret_cast<float*>(epi_box + C::kEpiBoxes * C::kEpiBox);  // [2][128] (block scaling)
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_box + C::kEpiBoxes * C::kEpiBox + C::kScaleVec);
  uint64_t* full = bars;                       // [kStages]  producer -> consumers (tx bytes)
  uint64_t* empty = full + C::kStages;         // [kStages]  consumers -> producer
  uint64_t* a_full = empty + C::kStages;       // [kAStages] dequant -> MMA
  uint64_t* a_empty = a_full + C::kAStages;    // [kAStages] MMA -> dequant
  uint64_t* acc_full = a_empty + C::kAStages;  // [kAccBufs] MMA -> epilogue
  uint64_t* acc_empty = acc_full + C::kAccBufs;  // [kAccBufs] epilogue -> MMA
  uint64_t* sf_full = acc_empty + C::kAccBufs;   // [kSfSlots] scale warp -> MMA (scales of stage s in TMEM)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_full + C::kSfSlots);
  __shared__ int s_last;
  __shared__ volatile int s_abort;  // set by the first role whose wait gave up

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t KB = a.K / C::kCols;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W4 ? 1 + C::kDqWarps : 1);
    }
    for (int i = 0; i < C::kAStages; ++i) {
      mbar_init(&a_full[i], C::kDqWarps / 2);  // one group of four warps fills a slot
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < C::kAccBufs; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], C::kEpiWarps);
    }
    for (int i = 0; i < C::kSfSlots; ++i) mbar_init(&sf_full[i], C::kSfWarps);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmap_x);
    if constexpr (!W4) prefetch_tensormap(&tmap_w);
    prefetch_tensormap(&tmap_y);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) grid_dep_launch();  // the next kernel may start its prologue

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_stream = a.w_keep ? policy_evict_last() : policy_evict_first();  // weight tiles
      const uint64_t pol_keep = a.x_keep ? policy_evict_last() : policy_evict_normal();
      const int64_t ng = W4 ? a.K / a.G : 0;  // groups per weight row (W4A16)
      // groups whose scales a stage loads: those of its KPS blocks (a G = 128
      // group spans two blocks, so a one-block stage loads the group it is in)
      const int gps = W4 ? (KPS * C::kCols >= a.G ? KPS * C::kCols / a.G : 1) : 0;
      const uint32_t tx_bytes = C::kTxBase + gps * 320;
      // weights never depend on the previous kernel: the first pass over the
      // ring is filled with weight tiles before waiting for that kernel; the
      // activation tiles follow once it has finished
      auto load_w = [&](int s, const Unit& un, int j) {
        uint8_t* st = ring + s * C::kStage;
        const int kb = un.kb0 + j * KPS;
        if constexpr (W4) {
          const int64_t g0 = (static_cast<int64_t>(kb) * C::kCols) >> a.gshift;
          const int64_t tpb = C::kCols / 64;  // packed code tiles per K block
          bulk_load_hint(st + KPS * C::kXBlk, a.codes + (static_cast<int64_t>(un.nt) * KB * tpb + kb * tpb) * 4096,
                         KPS * C::kWBlk, &full[s], pol_stream);
          bulk_load(st + C::kScaleOff, a.scales + (static_cast<int64_t>(un.nt) * ng + g0) * kTileN, gps * 256,
                    &full[s]);
          bulk_load(st + C::kZeroOff, a.zeros + (static_cast<int64_t>(un.nt) * ng + g0) * (kTileN / 2), gps * 64,
                    &full[s]);
        } else {
#pragma unroll
          for (int h = 0; h < WN / kTileN; ++h)  // one box of 128 rows per scale block
            tma_load_2d_hint(st + C::kXBlk + h * kTileN * C::kBlkBytes, &tmap_w, &full[s], kb * C::kTmaX,
                             un.nt * WN + h * kTileN, pol_stream);
          if constexpr (MX != kMxNone)  // the weight tile's scale atoms of this K block
            bulk_load(st + C::kSfOff, a.sfa + (static_cast<int64_t>(un.nt) * KB + kb) * (512 * C::kSfK),
                      512 * C::kSfK, &full[s]);
        }
      };
      auto load_x = [&](int s, const Unit& un, int j) {
        uint8_t* st = ring + s * C::kStage;
        const int kb = un.kb0 + j * KPS;
#pragma unroll
        for (int i = 0; i < KPS; ++i)
          tma_load_2d_hint(st + i * C::kXBlk, &tmap_x, &full[s], (kb + i) * C::kTmaX, un.mb * BN, pol_keep);
        if constexpr (MX != kMxNone) {  // the scale atoms of the 128 tokens holding this token block
          const int64_t natoms = (a.M + 127) / 128;  // atoms the caller's buffer holds
#pragma unroll
          for (int t = 0; t < C::kSfbAtoms; ++t) {
            // a 256-token tile past the last atom takes that atom again: its
            // tokens are beyond M (zero rows, outputs never written)
            const int64_t atom = imin64(static_cast<int64_t>(un.mb) * BN / 128 + t, natoms - 1);
            bulk_load(st + C::kSfOff + 512 * C::kSfK * (1 + t), a.sfb + (atom * KB + kb) * (512 * C::kSfK),
                      512 * C::kSfK, &full[s]);
          }
        }
      };
      int it = 0;
      // phase 1: weights of the first ring pass
      for (int u = blockIdx.x; u < a.units && it < C::kStages; u += gridDim.x) {
        const Unit un = unit_of(a, u, KB);
        for (int j = 0; j < un.nkb / KPS && it < C::kStages; ++j, ++it) {
          mbar_arrive_expect_tx(&full[it], tx_bytes);
          load_w(it, un, j);
        }
      }
      const int prefilled = it;
      grid_dep_wait();
      it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        const Unit un = unit_of(a, u, KB);
        for (int j = 0; j < un.nkb / KPS; ++j, ++it) {
          const int s = it % C::kStages;
          if (it >= prefilled) {
            if (!mbar_wait(&empty[s], ((it / C::kStages) & 1) ^ 1, kWaitLimitNs, &s_abort)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[s], tx_bytes);
            load_w(s, un, j);
          }
          load_x(s, un, j);
        }
      }
      if (!ok) {
        set_error(a.err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && BS) {
      // block scaling: every K block of 128 goes to its own partial product, in
      // one of kAccBufs TMEM buffers; the epilogue promotes it with the block scales
      constexpr uint32_t idesc = idesc_make(0, 0, 128, C::kTokM ? WN : BN);
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        const Unit un = unit_of(a, u, KB);
        for (int j = 0; j < un.nkb && ok; ++j, ++it) {
          const int pb = it % C::kAccBufs;
          if (!mbar_wait(&acc_empty[pb], ((it / C::kAccBufs) & 1) ^ 1, kWaitLimitNs, &s_abort)) {
            ok = false;
            break;
          }
          const int s = it % C::kStages;
          if (!mbar_wait(&full[s], (it / C::kStages) & 1, kWaitLimitNs, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tmem_d = tmem_base + pb * C::kAccCols;
          // weight-major: A = weight tile, B = token tile; token-major: swapped
          const uint32_t a_addr = smem_u32(ring + s * C::kStage + (C::kTokM ? 0 : C::kXBlk));
          const uint32_t b_addr = smem_u32(ring + s * C::kStage + (C::kTokM ? C::kXBlk : 0));
          const uint64_t ad0 = sdesc_sw128(a_addr), bd0 = sdesc_sw128(b_addr);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // 32 bytes of K per step: start address + 2 (16-byte units)
            mma_f8(tmem_d, ad0 + 2 * kk, bd0 + 2 * kk, idesc, kk != 0);
          mma_commit(&empty[s]);
          mma_commit(&acc_full[pb]);
        }
      }
      if (!ok) {
        set_error(a.err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
      }
    } else if (lane == 0 && MX != kMxNone) {
      // Block-scaled formats: per K block, once the scale warp has copied its
      // scale atoms into the stage's TMEM slot, four MMAs of 32 bytes of K.  MXFP8: k-step kk takes byte kk of each scale word;
      // MXFP4 (64 columns per step): atom kk / 2, bytes 2 (kk % 2) and +1;
      // NVFP4 (64 columns): atom kk, bytes 0..3
      int it = 0, ua = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x, ++ua) {
        const Unit un = unit_of(a, u, KB);
        const int acc = ua % C::kAccBufs;
        if (!mbar_wait(&acc_empty[acc], ((ua / C::kAccBufs) & 1) ^ 1, kWaitLimitNs, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + acc * C::kAccCols;
        const uint32_t tok_col = static_cast<uint32_t>((un.mb * BN) % 128) / 32;  // this block's tokens in the atom
        for (int j = 0; j < un.nkb && ok; ++j, ++it) {
          const int s = it % C::kStages;
          // the stage has landed and the scale warp's copies of its scales are done
          if (!mbar_wait(&sf_full[s], (it / C::kStages) & 1, kWaitLimitNs, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t t_sfa = tmem_base + C::kSfaCol + s * 4 * C::kSfK;
          const uint32_t t_sfb = tmem_base + C::kSfbCol + s * 4 * C::kSfK * C::kSfbAtoms;
          const uint32_t st_u32 = smem_u32(ring + s * C::kStage);
          const uint64_t ad0 = sdesc_sw128(st_u32 + C::kXBlk), bd0 = sdesc_sw128(st_u32);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = ad0 + 2 * kk, bd = bd0 + 2 * kk;  // 32 bytes of K per step
            const uint32_t accum = (j | kk) != 0;
            if constexpr (MX == kMxF8) {
              mma_mx8(tmem_d, ad, bd, idesc_mx(BN, kk, kk), t_sfa, t_sfb + tok_col, accum);
            } else if constexpr (MX == kMxF4) {
              const uint32_t c = kk >> 1, id = 2 * (kk & 1);
              mma_mxf4(tmem_d, ad, bd, idesc_f4(BN, id, id, 1), t_sfa + 4 * c, t_sfb + 4 * c * C::kSfbAtoms + tok_col,
                       accum);
            } else {
              mma_nvf4(tmem_d, ad, bd, idesc_f4(BN, 0, 0, 0), t_sfa + 4 * kk,
                       t_sfb + 4 * kk * C::kSfbAtoms + tok_col, accum);
            }
          }
          mma_commit(&empty[s]);
        }
        mma_commit(&acc_full[acc]);
      }
      if (!ok) {
        set_error(a.err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
      }
    } else if (lane == 0 && A8) {
      // W4A8: every K block (one quantisation group) goes to its own partial
      // product in one of kAccBufs TMEM buffers, A = the block's E4M3 (q - z)
      // written into a TMEM slot by the dequantisation warps; the epilogue
      // applies the group scale
      constexpr uint32_t idesc = idesc_make(0, 0, 128, BN);
      int it = 0, ait = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        const Unit un = unit_of(a, u, KB);
        for (int j = 0; j < un.nkb / KPS && ok; ++j, ++it) {
          const int s = it % C::kStages;
          if (!mbar_wait(&full[s], (it / C::kStages) & 1, kWaitLimitNs, &s_abort)) {
            ok = false;
            break;
          }
#pragma unroll 1
          for (int i = 0; i < KPS; ++i, ++ait) {
            const int ai = ait % C::kAStages, pb = ait % C::kAccBufs;
            if (!mbar_wait(&a_full[ai], (ait / C::kAStages) & 1, kWaitLimitNs, &s_abort) ||
                !mbar_wait(&acc_empty[pb], ((ait / C::kAccBufs) & 1) ^ 1, kWaitLimitNs, &s_abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = tmem_base + C::kAColBase + ai * C::kASlotCols;
            const uint64_t bd0 = sdesc_sw128(smem_u32(ring + s * C::kStage + i * C::kXBlk));
            const uint32_t tmem_d = tmem_base + pb * C::kAccCols;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // 32 bytes of K per MMA = 8 TMEM columns of A
              mma_f8_tmem_a(tmem_d, a_addr + kk * 8, bd0 + 2 * kk, idesc, kk != 0);
            mma_commit(&a_empty[ai]);
            mma_commit(&acc_full[pb]);
          }
          mma_commit(&empty[s]);
        }
      }
      if (!ok) {
        set_error(a.err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
      }
    } else if (lane == 0 && C::kSlotBlocks == 2) {
      // W4A16 with A in TMEM: per slot (two 64-column blocks) one barrier wait,
      // eight MMAs with the B descriptors stepped by 32 bytes, one commit
      constexpr uint32_t idesc = idesc_make(1, 1, 128, BN);
      int it = 0, pit = 0, ua = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x, ++ua) {
        const Unit un = unit_of(a, u, KB);
        const int acc = ua % C::kAccBufs;
        if (!mbar_wait(&acc_empty[acc], ((ua / C::kAccBufs) & 1) ^ 1, kWaitLimitNs, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + acc * C::kAccCols;
        for (int j = 0; j < un.nkb / KPS && ok; ++j, ++it) {
          // No wait on full[s]: the dequantisation group that filled a slot of
          // this stage waited on full[s] before arriving on a_full, so the
          // a_full wait below already orders these MMAs after the stage's copies
          const int s = it % C::kStages;
          const uint32_t st_u32 = smem_u32(ring + s * C::kStage);
#pragma unroll
          for (int ip = 0; ip < KPS / 2; ++ip, ++pit) {
            const int ai = pit % C::kAStages;
            if (!mbar_wait(&a_full[ai], (pit / C::kAStages) & 1, kWaitLimitNs, &s_abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_slot = tmem_base + C::kAColBase + ai * C::kASlotCols;
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
              const uint64_t bd = sdesc_sw128(st_u32 + (2 * ip + blk) * C::kXBlk);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)  // 16 BF16 of K per MMA: 8 TMEM columns of A, 32 bytes of B
                mma_f16_tmem_a(tmem_d, a_slot + blk * 32 + kk * 8, bd + 2 * kk, idesc, (j | ip | blk | kk) != 0);
            }
            mma_commit(&a_empty[ai]);
          }
          mma_commit(&empty[s]);
        }
        mma_commit(&acc_full[acc]);  // arrives when this unit's MMAs are done
      }
      if (!ok) {
        set_error(a.err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
      }
    } else if (lane == 0) {
      constexpr uint32_t idesc = W4 ? idesc_make(1, 1, 128, BN) : idesc_make(0, 0, 128, BN);
      int it = 0, ait = 0, ua = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x, ++ua) {
        const Unit un = unit_of(a, u, KB);
        const int acc = ua % C::kAccBufs;
        if (!mbar_wait(&acc_empty[acc], ((ua / C::kAccBufs) & 1) ^ 1, kWaitLimitNs, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + acc * C::kAccCols;
        for (int j = 0; j < un.nkb / KPS && ok; ++j, ++it) {
          const int s = it % C::kStages;
          // W4A16: the a_full wait below orders the MMAs after the stage's
          // copies (its dequantisation group waited on full[s] first)
          if (!W4 && !mbar_wait(&full[s], (it / C::kStages) & 1, kWaitLimitNs, &s_abort)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int i = 0; i < KPS; ++i, ++ait) {
            uint32_t a_addr;
            const int ai = W4 ? ait % C::kAStages : 0;
            if constexpr (W4) {
              if (!mbar_wait(&a_full[ai], (ait / C::kAStages) & 1, kWaitLimitNs, &s_abort)) {
                ok = false;
                break;
              }
              a_addr = C::kATmem ? tmem_base + C::kAColBase + ai * C::kASlotCols : smem_u32(aring + ai * C::kAStage);
            } else {
              a_addr = smem_u32(ring + s * C::kStage + KPS * C::kXBlk);
            }
            tc_fence_after();
            // descriptors of the first k-step; a step of 32 bytes of K adds 2 to
            // the start address (16-byte units, bits 0..13; shared addresses < 256 KB)
            const uint64_t bd0 = sdesc_sw128(smem_u32(ring + s * C::kStage + i * C::kXBlk));
            const uint64_t ad0 = C::kATmem ? 0 : sdesc_sw128(a_addr);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {  // 32 bytes of K per MMA
              const uint64_t bd = bd0 + 2 * kk;
              const uint32_t accum = (j | i | kk) != 0;
              if constexpr (C::kATmem)
                mma_f16_tmem_a(tmem_d, a_addr + kk * 8, bd, idesc, accum);  // 16 BF16 of K = 8 columns
              else if constexpr (W4)
                mma_f16(tmem_d, ad0 + 2 * kk, bd, idesc, accum);
              else
                mma_f8(tmem_d, ad0 + 2 * kk, bd, idesc, accum);
            }
            if constexpr (W4) mma_commit(&a_empty[ai]);
          }
          mma_commit(&empty[s]);
        }
        mma_commit(&acc_full[acc]);  // arrives when this unit's MMAs are done
      }
      if (!ok) {
        set_error(a.err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
      }
    }
  } else if (warp < C::kEpiWarp0) {
    if constexpr (MX != kMxNone) {
      // ------------------------------------------------------------ scale warps (block-scaled formats)
      // Per K block: wait for the stage, copy its scale atoms from shared
      // memory into the stage's TMEM slot (tcgen05.cp), and commit the copies
      // to sf_full[s] (one arrival per scale warp).  Slot s is free again when
      // the producer refills stage s: that happens only after the MMAs that
      // read the slot are done.
      if (lane == 0) {
        int it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
          const Unit un = unit_of(a, u, KB);
          for (int j = 0; j < un.nkb; ++j, ++it) {
            const int s = it % C::kStages;
            if (!mbar_wait(&full[s], (it / C::kStages) & 1, kWaitLimitNs, &s_abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t t_sfa = tmem_base + C::kSfaCol + s * 4 * C::kSfK;
            const uint32_t t_sfb = tmem_base + C::kSfbCol + s * 4 * C::kSfK * C::kSfbAtoms;
            const uint32_t st_u32 = smem_u32(ring + s * C::kStage);
            const int sfw = warp - 2 - C::kDqWarps;  // which scale warp (0 .. kSfWarps - 1)
#pragma unroll
            for (int c = 0; c < C::kSfK; ++c) {
              if (C::kSfWarps == 1 || sfw == 0) tc_cp_atom(t_sfa + 4 * c, sdesc_atom(st_u32 + C::kSfOff + 512 * c));
              if (C::kSfWarps == 1 || sfw == 1) {
#pragma unroll
                for (int t = 0; t < C::kSfbAtoms; ++t)  // K atom c, tokens 128 t ..: columns 4 (c kSfbAtoms + t) ..
                  tc_cp_atom(t_sfb + 4 * (c * C::kSfbAtoms + t),
                             sdesc_atom(st_u32 + C::kSfOff + 512 * C::kSfK * (1 + t) + 512 * c));
              }
            }
            mma_commit(&sf_full[s]);  // arrives when this warp's copies are done
          }
        }
        if (!ok) {
          set_error(a.err, QLIN_ERR_TIMEOUT);
          s_abort = 1;
        }
      }
    }
    // ---------------------------------------------------------------- dequantisation (W4A8)
    if constexpr (W4 && A8) {
      // The two groups of four warps take the K blocks (128 columns = one
      // quantisation group) in turn; the warp of TMEM lane quadrant q turns rows
      // 32q..32q+31 into E4M3 (q - z): integers in [-15, 15], exact in E4M3.
      // A nibble pair becomes FP16x2 (1024 + q) with one LOP3, (q - z) with one
      // HSUB2 and an E4M3 pair with one CVT; the 128 columns go to the slot in
      // natural order, four per TMEM column.
      const int quad = warp & 3;
      const int r = quad * 32 + lane;
      const int grp = (warp - 2) >> 2;
      int it = 0, ait = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        const Unit un = unit_of(a, u, KB);
        for (int j = 0; j < un.nkb / KPS && ok; ++j, ++it) {
          const int s = it % C::kStages;
          if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (it / C::kStages) & 1, kWaitLimitNs, &s_abort))) {
            ok = false;
            break;
          }
          const uint32_t sts = smem_u32(ring + s * C::kStage);
#pragma unroll 1
          for (int i = 0; i < KPS; ++i, ++ait) {
            const bool mine = (ait & 1) == grp;
            const int ai = ait % C::kAStages;
            uint4 c[4];  // records of row r: code tile 0 halves 0, 1, then code tile 1 halves 0, 1
            uint32_t zoff = 0;
            if (mine) {
              if (!__all_sync(0xffffffffu,
                              mbar_wait(&a_empty[ai], ((ait / C::kAStages) & 1) ^ 1, kWaitLimitNs, &s_abort))) {
                ok = false;
                break;
              }
#pragma unroll
              for (int rec = 0; rec < 4; ++rec) c[rec] = lds128(sts + KPS * C::kXBlk + i * 8192 + rec * 2048 + r * 16);
              const uint32_t zb = lds8(sts + C::kZeroOff + i * 64 + r / 2);
              zoff = (0x6400u + ((r & 1) ? (zb >> 4) : (zb & 15u))) * 0x10001u;  // FP16x2 (1024 + z)
            }
            if (i == KPS - 1) {
              __syncwarp();
              if (lane == 0) mbar_arrive(&empty[s]);  // this warp has read all of the stage it needs
            }
            if (!mine) continue;
            tc_fence_after();
#pragma unroll
            for (int rec = 0; rec < 4; ++rec) {
              const uint32_t w[4] = {c[rec].x, c[rec].y, c[rec].z, c[rec].w};
              uint32_t e[4][4];  // e[t][g8]: E4M3 of columns 8 g8 + 2t (low byte) and 8 g8 + 2t + 1
#pragma unroll
              for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8)
                  e[t][g8] = e4m3x2_of_f16x2(hsub2_bits(((w[t] >> (4 * g8)) & 0x000F000Fu) | 0x64006400u, zoff));
              uint32_t v[8];  // TMEM column 2 g8 + j of the record: columns 8 g8 + 4 j .. + 3
#pragma unroll
              for (int g8 = 0; g8 < 4; ++g8)
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) v[2 * g8 + jj] = e[2 * jj][g8] | (e[2 * jj + 1][g8] << 16);
              tmem_st8(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + C::kAColBase + ai * C::kASlotCols +
                           rec * 8,
                       v);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[ai]);
          }
        }
      }
      if (!ok) {
        set_error(a.err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
      }
    } else if constexpr (W4) {
      // ------------------------------------------------------------ dequantisation (W4A16)
      // Two groups of four warps take the 64-column blocks in turn (group g the
      // blocks with ait % 2 == g), so that two blocks are dequantised at once;
      // within a group, the warp of TMEM lane quadrant q does rows 32q..32q+31,
      // all 64 columns.
      const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
      const int r = quad * 32 + lane;            // weight row of the tile
      const int grp = (warp - 2) >> 2;
      int it = 0, ait = 0;
      bool ok = true;
      // the whole loop per group size, so that the group arithmetic is constant
      auto dq_loop = [&](auto gconst) {
        constexpr int gshift = decltype(gconst)::value;  // log2 G
        for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
          const Unit un = unit_of(a, u, KB);
          for (int j = 0; j < un.nkb / KPS && ok; ++j, ++it) {
            const int s = it % C::kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (it / C::kStages) & 1, kWaitLimitNs, &s_abort))) {
              ok = false;  // leave as a whole warp
              break;
            }
            const uint8_t* st = ring + s * C::kStage;
            const int kb = un.kb0 + j * KPS;
  #pragma unroll
            for (int i = 0; i < KPS; ++i, ++ait) {
              const bool mine = (ait & 1) == grp;
              const int ai = ait % C::kAStages;
              uint4 c[2];
              float scale[2] = {0.0f, 0.0f}, zq[2] = {0.0f, 0.0f};  // per 32-column half (they differ for G = 32)
              if (mine) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&a_empty[ai], ((ait / C::kAStages) & 1) ^ 1, kWaitLimitNs, &s_abort))) {
                  ok = false;
                  break;
                }
                const uint32_t sts = smem_u32(st);
                c[0] = lds128(sts + KPS * C::kXBlk + i * 4096 + r * 16);         // columns 0..31
                c[1] = lds128(sts + KPS * C::kXBlk + i * 4096 + 2048 + r * 16);  // columns 32..63
  #pragma unroll
                for (int h = 0; h < 2; ++h) {  // group of this half within the stage (one group for G >= 64)
                  if (h == 1 && gshift > 5) {  // G >= 64: both halves in one group
                    scale[1] = scale[0];
                    zq[1] = zq[0];
                    break;
                  }
                  const int gi = (((kb + i) * 64 + h * 32) >> gshift) - ((kb * 64) >> gshift);
                  scale[h] = __half2float(
                      __ushort_as_half(static_cast<unsigned short>(lds16(sts + C::kScaleOff + gi * 256 + r * 2))));
                  const uint32_t zb = lds8(sts + C::kZeroOff + gi * 64 + r / 2);
                  zq[h] = static_cast<float>((r & 1) ? (zb >> 4) : (zb & 15u));
                }
              }
              if (i == KPS - 1) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);  // this warp has read all of the stage it needs
              }
              if (!mine) continue;
              {
                uint8_t* arow = aring + ai * C::kAStage + r * 128;
  #pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const __nv_bfloat162 zoff = __float2bfloat162_rn(128.0f + zq[h]);
                  const __nv_bfloat162 s2 = __float2bfloat162_rn(scale[h]);
                  const uint32_t words[4] = {c[h].x, c[h].y, c[h].z, c[h].w};
                  uint4 d[4];
  #pragma unroll
                  for (int t = 0; t < 4; ++t) d[t] = dequant8(words[t], zoff, s2);
                  // 16-byte chunk cc = 4h + i holds columns 8cc..8cc+7: position i of words 0..3
                  *reinterpret_cast<uint4*>(arow + (((h * 4 + 0) ^ (r & 7)) << 4)) = make_uint4(d[0].x, d[1].x, d[2].x, d[3].x);
                  *reinterpret_cast<uint4*>(arow + (((h * 4 + 1) ^ (r & 7)) << 4)) = make_uint4(d[0].y, d[1].y, d[2].y, d[3].y);
                  *reinterpret_cast<uint4*>(arow + (((h * 4 + 2) ^ (r & 7)) << 4)) = make_uint4(d[0].z, d[1].z, d[2].z, d[3].z);
                  *reinterpret_cast<uint4*>(arow + (((h * 4 + 3) ^ (r & 7)) << 4)) = make_uint4(d[0].w, d[1].w, d[2].w, d[3].w);
                }
                fence_proxy_async_smem();
              }
              __syncwarp();
              if (lane == 0) mbar_arrive(&a_full[ai]);
            }
          }
        }
      };
      // A in TMEM: a group takes two consecutive blocks (one slot) in turn;
      // lane r of the slot holds row r, 32 columns x two BF16 per block
      auto dq_pairs = [&](auto gconst) {
        constexpr int gshift = decltype(gconst)::value;  // log2 G (31: per-channel)
        int pit = 0;
        for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
          const Unit un = unit_of(a, u, KB);
          for (int j = 0; j < un.nkb / KPS && ok; ++j, ++it) {
            const int s = it % C::kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (it / C::kStages) & 1, kWaitLimitNs, &s_abort))) {
              ok = false;
              break;
            }
            const uint32_t sts = smem_u32(ring + s * C::kStage);
            const int kb = un.kb0 + j * KPS;
#pragma unroll
            for (int ip = 0; ip < KPS / 2; ++ip, ++pit) {
              const bool mine = (pit & 1) == grp;
              const int ai = pit % C::kAStages;
              uint4 c[2][2];
              float scale[2][2] = {}, zq[2][2] = {};  // [block][32-column half]
              if (mine) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&a_empty[ai], ((pit / C::kAStages) & 1) ^ 1, kWaitLimitNs, &s_abort))) {
                  ok = false;
                  break;
                }
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                  const int i = 2 * ip + blk;
                  c[blk][0] = lds128(sts + KPS * C::kXBlk + i * 4096 + r * 16);         // columns 0..31
                  c[blk][1] = lds128(sts + KPS * C::kXBlk + i * 4096 + 2048 + r * 16);  // columns 32..63
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    if (h == 1 && gshift > 5) {  // G >= 64: both halves in one group
                      scale[blk][1] = scale[blk][0];
                      zq[blk][1] = zq[blk][0];
                      break;
                    }
                    const int gi = (((kb + i) * 64 + h * 32) >> gshift) - ((kb * 64) >> gshift);
                    scale[blk][h] = __half2float(
                        __ushort_as_half(static_cast<unsigned short>(lds16(sts + C::kScaleOff + gi * 256 + r * 2))));
                    const uint32_t zb = lds8(sts + C::kZeroOff + gi * 64 + r / 2);
                    zq[blk][h] = static_cast<float>((r & 1) ? (zb >> 4) : (zb & 15u));
                  }
                }
              }
              if (ip == KPS / 2 - 1) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);  // this warp has read all of the stage it needs
              }
              if (!mine) continue;
              tc_fence_after();
#pragma unroll
              for (int blk = 0; blk < 2; ++blk)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const __nv_bfloat162 zoff = __float2bfloat162_rn(128.0f + zq[blk][h]);
                  const __nv_bfloat162 s2 = __float2bfloat162_rn(scale[blk][h]);
                  const uint32_t words[4] = {c[blk][h].x, c[blk][h].y, c[blk][h].z, c[blk][h].w};
                  uint32_t v[16];  // v[p] = columns 2p, 2p+1 of the half; pair p = 4i + t is word t, position i
#pragma unroll
                  for (int t = 0; t < 4; ++t) {
                    const uint4 d = dequant8(words[t], zoff, s2);
                    v[t] = d.x;
                    v[4 + t] = d.y;
                    v[8 + t] = d.z;
                    v[12 + t] = d.w;
                  }
                  tmem_st16(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + C::kAColBase + ai * C::kASlotCols +
                                blk * 32 + h * 16,
                            v);
                }
              tmem_st_wait();
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&a_full[ai]);
            }
          }
        }
      };
      if constexpr (C::kATmem) {
        if (a.G == 32) dq_pairs(std::integral_constant<int, 5>{});
        else if (a.G == 64) dq_pairs(std::integral_constant<int, 6>{});
        else if (a.G == 128) dq_pairs(std::integral_constant<int, 7>{});
        else dq_pairs(std::integral_constant<int, 31>{});  // per-channel (G == K): the group index is always 0
      } else {
        if (a.G == 32) dq_loop(std::integral_constant<int, 5>{});
        else if (a.G == 64) dq_loop(std::integral_constant<int, 6>{});
        else if (a.G == 128) dq_loop(std::integral_constant<int, 7>{});
        else dq_loop(std::integral_constant<int, 31>{});  // per-channel (G == K): the group index is always 0
      }
      if (!ok) {
        set_error(a.err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    grid_dep_wait();  // outputs and the workspace may still be in use by the previous kernel
    const int t = threadIdx.x - C::kEpiWarp0 * 32;  // 0 .. kEpiWarps * 32 - 1
    const int quad = warp & 3;                       // TMEM lane quadrant of this warp
    const float s_w = (W4 || BS || MX) ? 1.0f : *a.sw;
    const float s_nv = MX == kNvF4 ? __ldg(a.sx) * __ldg(a.sw) : 1.0f;  // NVFP4: the two per-tensor scales
    int ua = 0;
    uint32_t epi_n = 0;  // staging boxes used so far
    int kbi = 0;         // K blocks promoted so far (block scaling)
    for (int u = blockIdx.x; u < a.units; u += gridDim.x, ++ua) {
      if constexpr (A8) {
        // ---- W4A8: every K block's partial product is promoted with the group
        // scale of this thread's weight row (TMEM lane quad * 32 + lane),
        // r[c] += P[c] * s[n][g], in K-block order; then y = r * sx[m]
        const Unit un = unit_of(a, u, KB);
        const int row = quad * 32 + lane;
        const int64_t n = static_cast<int64_t>(un.nt) * kTileN + row;
        const int64_t mbase = static_cast<int64_t>(un.mb) * BN;
        const bool direct = a.splits == 1;
        const float bias_n = EPI ? epi_bias(a.epi, n) : 0.0f;
        const uint16_t* sp = a.scales + static_cast<int64_t>(un.nt) * KB * kTileN + row;  // [group][128 rows]
        float sn = un.nkb > 0 ? __half2float(__ushort_as_half(__ldg(sp + static_cast<int64_t>(un.kb0) * kTileN))) : 0.0f;
        float rr[BN];
#pragma unroll
        for (int c = 0; c < BN; ++c) rr[c] = 0.0f;
        bool have = true;
        for (int j = 0; j < un.nkb; ++j, ++kbi) {
          const int pb = kbi % C::kAccBufs;
          const float f = sn;
          if (j + 1 < un.nkb)  // the next group's scale while this one is promoted
            sn = __half2float(__ushort_as_half(__ldg(sp + static_cast<int64_t>(un.kb0 + j + 1) * kTileN)));
          if (have && !__all_sync(0xffffffffu, mbar_wait(&acc_full[pb], (kbi / C::kAccBufs) & 1, kWaitLimitNs,
                                                           &s_abort))) {
            have = false;
            set_error(a.err, QLIN_ERR_TIMEOUT);
            s_abort = 1;
          }
          if (!have) continue;
          tc_fence_after();
          const uint32_t tmem_d = tmem_base + pb * C::kAccCols + (static_cast<uint32_t>(quad * 32) << 16);
          constexpr int kChunk = 16;  // columns per TMEM load: the running sums already hold up to 64 registers
#pragma unroll
          for (int c0 = 0; c0 < BN; c0 += kChunk) {
            uint32_t v[kChunk / 16][16];
#pragma unroll
            for (int q = 0; q < kChunk / 16; ++q) tmem_ld16(tmem_d + c0 + q * 16, v[q]);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < kChunk / 16; ++q) reg_fence16(v[q]);
            if (c0 + kChunk == BN) {  // all of the buffer is in registers: it may take the next K block
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_empty[pb]);
            }
#pragma unroll
            for (int c = 0; c < kChunk; ++c) rr[c0 + c] = fmaf(__uint_as_float(v[c >> 4][c & 15]), f, rr[c0 + c]);
          }
        }
        // the token scales are applied where the values are written, 16 tokens at a time
        if (direct) {
#pragma unroll
          for (int c0 = 0; c0 < BN; c0 += 16) {
            if (mbase + c0 < a.M) {  // the same for the four warps: they skip the barriers together
              uint16_t* box = reinterpret_cast<uint16_t*>(epi_box + (epi_n & 1) * C::kEpiBox);
              if (t == 0) bulk_wait_read<1>();
              named_bar_epi();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int64_t m = mbase + c0 + i;
                float v = m < a.M ? rr[c0 + i] * __ldg(a.sx + m) : 0.0f;
                if constexpr (EPI) v = epi_act(a.epi.act, v, bias_n);
                box[i * kTileN + row] = m < a.M ? to_bf16(v) : uint16_t(0);
              }
              fence_proxy_async_smem();
              named_bar_epi();
              if (t == 0) tma_store_2d(&tmap_y, box, un.nt * kTileN, static_cast<int>(mbase + c0));
              ++epi_n;
            }
          }
        } else {
          if (have) {
#pragma unroll
            for (int c = 0; c < BN; ++c) {
              const int64_t m = mbase + c;
              if (m < a.M) __stcg(a.partials + (static_cast<int64_t>(un.split) * a.M + m) * a.N + n, rr[c] * __ldg(a.sx + m));
            }
          }
          // last-arriver reduction of the K ranges, in split order (deterministic)
          __threadfence();
          named_bar_epi();
          const int64_t tile = static_cast<int64_t>(un.mb) * a.ntiles + un.nt;
          if (t == 0) s_last = !s_abort && (atomicAdd(a.counters + tile, 1u) == static_cast<uint32_t>(a.splits - 1));
          named_bar_epi();
          if (s_last) {
            __threadfence();
#pragma unroll 1
            for (int c = 0; c < BN; ++c) {
              const int64_t m = mbase + c;
              if (m >= a.M) break;
              float acc_v = 0.0f;
              for (int sp2 = 0; sp2 < a.splits; ++sp2) {  // read and clear: the workspace is left zero-filled
                float* p = a.partials + (static_cast<int64_t>(sp2) * a.M + m) * a.N + n;
                acc_v += __ldcg(p);
                __stcg(p, 0.0f);
              }
              if constexpr (EPI) acc_v = epi_act(a.epi.act, acc_v, bias_n);
              a.Y[m * a.N + n] = to_bf16(acc_v);
            }
            if (t == 0) a.counters[tile] = 0u;
          }
          named_bar_epi();
        }
        continue;
      } else if constexpr (C::kTokM) {
        // ---- block scaling, token-major: thread = token m (TMEM lane quad * 32 +
        // lane), columns [cbase, cbase + 64) of the weight tile; every K block's
        // partial product is promoted as r[c] += P[c] * (sx[kb][m] * sw[nt][kb])
        constexpr int kCw = WN / C::kEpiHalves;
        constexpr int kChunk = kCw > 64 ? 16 : kCw;  // TMEM columns loaded per wait
        constexpr int kAll = C::kEpiWarps * 32;
        const int te = threadIdx.x - C::kEpiWarp0 * 32;
        const int cbase = (te >> 7) * kCw;
        const Unit un = unit_of(a, u, KB);
        const int64_t m = static_cast<int64_t>(un.mb) * BN + quad * 32 + lane;
        const int64_t n0 = static_cast<int64_t>(un.nt) * WN + cbase;
        const bool mok = m < a.M;
        const bool direct = a.splits == 1;
        // the next K block's scales are loaded while the current one is promoted
        const float* swp = a.sw + (n0 / kTileN) * KB;  // this thread's columns lie in one scale block
        float sxn = 0.0f, swn = 0.0f;
        if (un.nkb > 0) {
          swn = __ldg(swp + un.kb0);
          if (mok) sxn = __ldg(a.sx + un.kb0 * a.M + m);
        }
        float r[kCw];
#pragma unroll
        for (int c = 0; c < kCw; ++c) r[c] = 0.0f;
        bool have = true;
        for (int j = 0; j < un.nkb; ++j, ++kbi) {
          const int pb = kbi % C::kAccBufs;
          const float f = sxn * swn;
          if (j + 1 < un.nkb) {
            const int64_t kb1 = un.kb0 + j + 1;
            swn = __ldg(swp + kb1);
            if (mok) sxn = __ldg(a.sx + kb1 * a.M + m);
          }
          if (have && !__all_sync(0xffffffffu, mbar_wait(&acc_full[pb], (kbi / C::kAccBufs) & 1, kWaitLimitNs,
                                                           &s_abort))) {
            have = false;
            set_error(a.err, QLIN_ERR_TIMEOUT);
            s_abort = 1;
          }
          if (!have) continue;
          tc_fence_after();
          const uint32_t tmem_d =
              tmem_base + pb * C::kAccCols + cbase + (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll
          for (int c0 = 0; c0 < kCw; c0 += kChunk) {
            uint32_t v[kChunk / 16][16];
#pragma unroll
            for (int q = 0; q < kChunk / 16; ++q) tmem_ld16(tmem_d + c0 + q * 16, v[q]);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < kChunk / 16; ++q) reg_fence16(v[q]);  // no use of v is hoisted above the wait
            if (c0 + kChunk == kCw) {  // all in registers: the buffer may take the next K block
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_empty[pb]);
            }
#pragma unroll
            for (int c = 0; c < kChunk; ++c) r[c0 + c] = fmaf(__uint_as_float(v[c >> 4][c & 15]), f, r[c0 + c]);
          }
        }
        if (direct) {
          if (have && mok) {
            uint4* yrow = reinterpret_cast<uint4*>(a.Y + m * a.N + n0);
#pragma unroll
            for (int c = 0; c < kCw; c += 8) {
              if constexpr (EPI) {  // bias of columns n0 + c .. (one weight row each)
#pragma unroll
                for (int i = 0; i < 8; ++i) r[c + i] = epi_cols(a.epi, r[c + i], n0 + c + i);
              }
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                w[i] = static_cast<uint32_t>(to_bf16(r[c + 2 * i])) | (static_cast<uint32_t>(to_bf16(r[c + 2 * i + 1])) << 16);
              yrow[c / 8] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        } else {
          if (have && mok) {
            float4* prow = reinterpret_cast<float4*>(a.partials + (static_cast<int64_t>(un.split) * a.M + m) * a.N + n0);
#pragma unroll
            for (int c = 0; c < kCw; c += 4) __stcg(prow + c / 4, make_float4(r[c], r[c + 1], r[c + 2], r[c + 3]));
          }
          // last-arriver reduction of the K ranges, in split order (deterministic)
          __threadfence();
          named_bar(1, kAll);
          const int64_t tile = static_cast<int64_t>(un.mb) * a.ntiles + un.nt;
          if (te == 0) s_last = !s_abort && (atomicAdd(a.counters + tile, 1u) == static_cast<uint32_t>(a.splits - 1));
          named_bar(1, kAll);
          if (s_last) {
            __threadfence();
            if (mok) {
              for (int c = 0; c < kCw; c += 4) {
                float4 acc_v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                for (int sp = 0; sp < a.splits; ++sp) {  // read and clear: the workspace is left zero-filled
                  float4* pp = reinterpret_cast<float4*>(a.partials + (static_cast<int64_t>(sp) * a.M + m) * a.N + n0 + c);
                  const float4 x = __ldcg(pp);
                  acc_v.x += x.x;
                  acc_v.y += x.y;
                  acc_v.z += x.z;
                  acc_v.w += x.w;
                  __stcg(pp, make_float4(0.0f, 0.0f, 0.0f, 0.0f));
                }
                if constexpr (EPI) {
                  acc_v.x = epi_cols(a.epi, acc_v.x, n0 + c);
                  acc_v.y = epi_cols(a.epi, acc_v.y, n0 + c + 1);
                  acc_v.z = epi_cols(a.epi, acc_v.z, n0 + c + 2);
                  acc_v.w = epi_cols(a.epi, acc_v.w, n0 + c + 3);
                }
                const uint32_t lo = static_cast<uint32_t>(to_bf16(acc_v.x)) | (static_cast<uint32_t>(to_bf16(acc_v.y)) << 16);
                const uint32_t hi = static_cast<uint32_t>(to_bf16(acc_v.z)) | (static_cast<uint32_t>(to_bf16(acc_v.w)) << 16);
                *reinterpret_cast<uint2*>(a.Y + m * a.N + n0 + c) = make_uint2(lo, hi);
              }
            }
            if (te == 0) a.counters[tile] = 0u;
          }
          named_bar(1, kAll);
        }
        continue;
      } else if constexpr (BS) {
        // ---- block scaling: promote every K block's partial product into FP32
        // running sums, r[c] += P[c] * sx[kb][m_c] * sw[nt][kb], in K-block order.
        // Epilogue warp e owns TMEM lanes quad * 32.. (its rows of the tile) and
        // token columns [cbase, cbase + kCw) of the token block.
        constexpr int kCw = BN / C::kEpiHalves;
        constexpr int kAll = C::kEpiWarps * 32;
        const int te = threadIdx.x - C::kEpiWarp0 * 32;  // 0 .. kAll - 1
        const int half = te >> 7, th = te & 127;
        const int cbase = half * kCw;
        const Unit un = unit_of(a, u, KB);
        const int64_t n = static_cast<int64_t>(un.nt) * kTileN + quad * 32 + lane;
        const int64_t mbase = static_cast<int64_t>(un.mb) * BN;
        const bool direct = a.splits == 1;
        const float bias_n = EPI ? epi_bias(a.epi, n) : 0.0f;
        // thread te < BN stages the factor of token mbase + te; the next K
        // block's factor is loaded while the current one is promoted
        const int64_t mt = mbase + te;
        const bool stager = te < BN && mt < a.M && un.nkb > 0;
        const float* swp = a.sw + static_cast<int64_t>(un.nt) * KB;
        // raw scales, multiplied only where they are stored: the product does
        // not wait for the loads right after they are issued
        float sxn = 0.0f, swn = 0.0f;
        if (stager) {
          sxn = __ldg(a.sx + un.kb0 * a.M + mt);
          swn = __ldg(swp + un.kb0);
        }
        float r[kCw];
#pragma unroll
        for (int c = 0; c < kCw; ++c) r[c] = 0.0f;
        bool have = true;
        for (int j = 0; j < un.nkb; ++j, ++kbi) {
          const int pb = kbi % C::kAccBufs;
          float* fv = scale_vec + (kbi & 1) * 128;
          if (te < BN) fv[te] = sxn * swn;
          if (stager && j + 1 < un.nkb) {
            const int64_t kb1 = un.kb0 + j + 1;
            sxn = __ldg(a.sx + kb1 * a.M + mt);
            swn = __ldg(swp + kb1);
          }
          if (have && !__all_sync(0xffffffffu, mbar_wait(&acc_full[pb], (kbi / C::kAccBufs) & 1, kWaitLimitNs,
                                                           &s_abort))) {
            have = false;
            set_error(a.err, QLIN_ERR_TIMEOUT);
            s_abort = 1;
          }
          // every epilogue warp takes part, also one whose wait gave up
          named_bar(1, kAll);
          if (!have) continue;
          tc_fence_after();
          const uint32_t tmem_d =
              tmem_base + pb * C::kAccCols + cbase + (static_cast<uint32_t>(quad * 32) << 16);
          uint32_t v[kCw / 16][16];
#pragma unroll
          for (int q = 0; q < kCw / 16; ++q) tmem_ld16(tmem_d + q * 16, v[q]);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < kCw / 16; ++q) reg_fence16(v[q]);  // no use of v is hoisted above the wait
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[pb]);  // in registers: the buffer may take the next K block
          const float4* f4 = reinterpret_cast<const float4*>(fv + cbase);
#pragma unroll
          for (int q = 0; q < kCw / 4; ++q) {
            const float4 x = f4[q];
            r[4 * q] = fmaf(__uint_as_float(v[q >> 2][(4 * q) & 15]), x.x, r[4 * q]);
            r[4 * q + 1] = fmaf(__uint_as_float(v[q >> 2][(4 * q + 1) & 15]), x.y, r[4 * q + 1]);
            r[4 * q + 2] = fmaf(__uint_as_float(v[q >> 2][(4 * q + 2) & 15]), x.z, r[4 * q + 2]);
            r[4 * q + 3] = fmaf(__uint_as_float(v[q >> 2][(4 * q + 3) & 15]), x.w, r[4 * q + 3]);
          }
        }
#pragma unroll
        for (int c0 = 0; c0 < kCw; c0 += 16) {
          const int64_t m0 = mbase + cbase + c0;
          if (direct) {
            if (m0 < a.M) {  // the same for the 128 threads of this half: they skip the barriers together
              uint16_t* box = reinterpret_cast<uint16_t*>(epi_box + (half * 2 + (epi_n & 1)) * C::kEpiBox);
              if (th == 0) bulk_wait_read<1>();
              named_bar(2 + half, 128);
#pragma unroll
              for (int i = 0; i < 16; ++i)
                box[i * kTileN + quad * 32 + lane] = to_bf16(EPI ? epi_sparse(a.epi.act, r[c0 + i], bias_n) : r[c0 + i]);
              fence_proxy_async_smem();
              named_bar(2 + half, 128);
              if (th == 0) tma_store_2d(&tmap_y, box, un.nt * kTileN, static_cast<int>(m0));
              ++epi_n;
            }
          } else if (have) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int64_t m = m0 + i;
              if (m < a.M) __stcg(a.partials + (static_cast<int64_t>(un.split) * a.M + m) * a.N + n, r[c0 + i]);
            }
          }
        }
        if (!direct) {
          // last-arriver reduction of the K ranges, in split order (deterministic)
          __threadfence();
          named_bar(1, kAll);
          const int64_t tile = static_cast<int64_t>(un.mb) * a.ntiles + un.nt;
          if (te == 0) s_last = !s_abort && (atomicAdd(a.counters + tile, 1u) == static_cast<uint32_t>(a.splits - 1));
          named_bar(1, kAll);
          if (s_last) {
            __threadfence();
#pragma unroll 1
            for (int c0 = cbase; c0 < cbase + kCw; c0 += 16) {
              if (mbase + c0 >= a.M) break;
              float acc_v[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) acc_v[i] = 0.0f;
              // 16 tokens x several splits of independent loads in flight per thread
#pragma unroll 4
              for (int sp = 0; sp < a.splits; ++sp) {
                float* p = a.partials + (static_cast<int64_t>(sp) * a.M + mbase + c0) * a.N + n;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  if (mbase + c0 + i < a.M) {  // read and clear: the workspace is left zero-filled
                    acc_v[i] += __ldcg(p + static_cast<int64_t>(i) * a.N);
                    __stcg(p + static_cast<int64_t>(i) * a.N, 0.0f);
                  }
              }
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int64_t m = mbase + c0 + i;
                if (m < a.M) a.Y[m * a.N + n] = to_bf16(EPI ? epi_sparse(a.epi.act, acc_v[i], bias_n) : acc_v[i]);
              }
            }
            if (te == 0) a.counters[tile] = 0u;
          }
          named_bar(1, kAll);
        }
        continue;
      } else if constexpr (C::kEarly) {
        // ---- single 256-token accumulator (block-scaled formats, never split
        // along K: see the planners): warp (quadrant, half) owns TMEM lanes
        // quad * 32.. and tokens [128 half, 128 half + 128); it reads all 128
        // columns as BF16 pairs (64 registers), hands the accumulator back,
        // then writes them through the staging boxes
        const Unit un = unit_of(a, u, KB);
        const int half = t >> 7, th = t & 127;
        const int cbase = half * 128;
        const int64_t mbase = static_cast<int64_t>(un.mb) * BN;
        // bias of this thread's row (TMEM lane quad * 32 + lane), loaded while the MMAs run
        const float bias_n = EPI ? epi_bias(a.epi, static_cast<int64_t>(un.nt) * kTileN + quad * 32 + lane) : 0.0f;
        const bool have =
            __all_sync(0xffffffffu, mbar_wait(&acc_full[0], ua & 1, kWaitLimitNs, &s_abort));
        if (!have) {
          set_error(a.err, QLIN_ERR_TIMEOUT);
          s_abort = 1;
        }
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + cbase + (static_cast<uint32_t>(quad * 32) << 16);
        uint32_t pk[64];  // BF16 pairs: tokens cbase + 2i (low half), + 1
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t v[2][16];
          if (have) {
            tmem_ld16(tmem_d + c0, v[0]);
            tmem_ld16(tmem_d + c0 + 16, v[1]);
            tmem_ld_wait();
            reg_fence16(v[0]);
            reg_fence16(v[1]);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0 = have ? __uint_as_float(v[i >> 3][(2 * i) & 15]) * s_nv : 0.0f;
            float x1 = have ? __uint_as_float(v[i >> 3][(2 * i + 1) & 15]) * s_nv : 0.0f;
            if constexpr (EPI) {
              x0 = epi_act(a.epi.act, x0, bias_n);
              x1 = epi_act(a.epi.act, x1, bias_n);
            }
            pk[c0 / 2 + i] = bf16x2_bits(__floats2bfloat162_rn(x0, x1));  // x0 in the low half
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[0]);  // the next unit's MMAs may start
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 16) {
          const int64_t m0 = mbase + cbase + c0;
          if (m0 < a.M) {  // the same for the 128 threads of this half: they skip the barriers together
            uint16_t* box = reinterpret_cast<uint16_t*>(epi_box + (half * 2 + (epi_n & 1)) * C::kEpiBox);
            if (th == 0) bulk_wait_read<1>();
            named_bar(2 + half, 128);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t w = pk[(c0 + i) >> 1];
              box[i * kTileN + quad * 32 + lane] =
                  m0 + i < a.M ? static_cast<uint16_t>((i & 1) ? (w >> 16) : (w & 0xFFFFu)) : uint16_t(0);
            }
            fence_proxy_async_smem();
            named_bar(2 + half, 128);
            if (th == 0) tma_store_2d(&tmap_y, box, un.nt * kTileN, static_cast<int>(m0));
            ++epi_n;
          }
        }
        continue;
      }
      const Unit un = unit_of(a, u, KB);
      const int acc = ua % C::kAccBufs;
      const int64_t n = static_cast<int64_t>(un.nt) * kTileN + quad * 32 + lane;
      const float bias_n = EPI ? epi_bias(a.epi, n) : 0.0f;  // loaded while the MMAs run
      // A warp whose wait gave up skips this unit's data but keeps taking part
      // in the named barriers below, so that they always see all 128 threads.
      const bool have =
          __all_sync(0xffffffffu, mbar_wait(&acc_full[acc], (ua / C::kAccBufs) & 1, kWaitLimitNs, &s_abort));
      if (!have) {
        set_error(a.err, QLIN_ERR_TIMEOUT);
        s_abort = 1;
      }
      tc_fence_after();
      const int64_t mbase = static_cast<int64_t>(un.mb) * BN;
      const uint32_t tmem_d = tmem_base + acc * C::kAccCols + (static_cast<uint32_t>(quad * 32) << 16);
      const bool direct = a.splits == 1;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t v[16];
        if (have) {
          tmem_ld16(tmem_d + c0, v);
          tmem_ld_wait();
        }
        if (have && c0 + 16 >= BN) {  // the whole accumulator has been read: hand it back to the MMA
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[acc]);
        }
        if (direct) {
          // 16 tokens x 128 rows as BF16 into a staging box, then one tensor store
          // (rows past M are clipped by the tensor map); the two boxes alternate
          // over the stores issued.  Whether this block of tokens exists is the
          // same for all 128 threads, so they skip the barriers together.
          if (mbase + c0 < a.M) {
            uint16_t* box = reinterpret_cast<uint16_t*>(epi_box + (epi_n & 1) * C::kEpiBox);
            if (t == 0) bulk_wait_read<1>();  // the store before last, from this box, has read it
            named_bar_epi();
            float o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int64_t m = mbase + c0 + i;
              const float x = have ? __uint_as_float(v[i]) : 0.0f;
              o[i] = W4 ? x : MX ? (MX == kNvF4 ? x * s_nv : x) : (m < a.M ? (x * __ldg(a.sx + m)) * s_w : 0.0f);
            }
            if constexpr (EPI) epi_run(a.epi.act, o, bias_n);
#pragma unroll
            for (int i = 0; i < 16; ++i)  // this thread's row of the tile: TMEM lane quad * 32 + lane
              box[i * kTileN + quad * 32 + lane] = mbase + c0 + i < a.M ? to_bf16(o[i]) : uint16_t(0);
            fence_proxy_async_smem();
            named_bar_epi();
            if (t == 0) tma_store_2d(&tmap_y, box, un.nt * kTileN, static_cast<int>(mbase + c0));
            ++epi_n;
          }
        } else if (have) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int64_t m = mbase + c0 + i;
            if (m < a.M)
              __stcg(a.partials + (static_cast<int64_t>(un.split) * a.M + m) * a.N + n, __uint_as_float(v[i]));
          }
        }
      }
      if (!direct) {
        // last-arriver reduction of the K ranges, in split order (deterministic)
        __threadfence();
        named_bar_epi();
        const int64_t tile = static_cast<int64_t>(un.mb) * a.ntiles + un.nt;
        if (t == 0) s_last = !s_abort && (atomicAdd(a.counters + tile, 1u) == static_cast<uint32_t>(a.splits - 1));
        named_bar_epi();
        if (s_last) {
          __threadfence();
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 16) {
            if (mbase + c0 >= a.M) break;
            float acc_v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc_v[i] = 0.0f;
            // 16 tokens x several splits of independent loads in flight per thread
#pragma unroll 4
            for (int s = 0; s < a.splits; ++s) {
              float* p = a.partials + (static_cast<int64_t>(s) * a.M + mbase + c0) * a.N + n;
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (mbase + c0 + i < a.M) {  // read and clear: the workspace is left zero-filled
                  acc_v[i] += __ldcg(p + static_cast<int64_t>(i) * a.N);
                  __stcg(p + static_cast<int64_t>(i) * a.N, 0.0f);
                }
            }
            if constexpr (!W4 && !MX) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int64_t m = mbase + c0 + i;
                acc_v[i] = m < a.M ? (acc_v[i] * __ldg(a.sx + m)) * s_w : 0.0f;
              }
            } else if constexpr (MX == kNvF4) {
#pragma unroll
              for (int i = 0; i < 16; ++i) acc_v[i] *= s_nv;
            }
            if constexpr (EPI) epi_run(a.epi.act, acc_v, bias_n);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int64_t m = mbase + c0 + i;
              if (m < a.M) a.Y[m * a.N + n] = to_bf16(acc_v[i]);
            }
          }
          if (t == 0) a.counters[tile] = 0u;
        }
        named_bar_epi();  // s_last is read by all before the next unit rewrites it
      }
    }
    if ((t & 127) == 0) bulk_wait_all();  // every tensor store has written its box (one issuer per half)
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, C::kTmemCols);
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

// Cost of a unit on one SM in cycles at 2.07 GHz, measured on GB300 per token
// tile: cycles per K block (64 columns W4A16, 128 E4M3), a start-up and drain
// cost paid once per CTA, and the split-K fix-up of a unit (partial sums
// written, the last arriver's reduction), which grows with the tile and, by
// half again per extra split, with the split count.  W4A16 (16 .. 256 tokens)
// from one unit per SM at three depths of K, a linear fit; E4M3 (64 .. 256)
// with the split count forced.
struct TcCost {
  double kb, once, fix;
};
static TcCost tc_cost(bool w4, int bn) {
  const int i = bn >= 256 ? 4 : bn >= 128 ? 3 : bn >= 64 ? 2 : bn >= 32 ? 1 : 0;
  static const double kb8[5] = {590, 590, 590, 594, 657}, once8[5] = {10.5e3, 10.5e3, 10.5e3, 15e3, 24.5e3};
  static const double kb4[5] = {539, 541, 597, 616, 927}, once4[5] = {13.1e3, 13e3, 15.1e3, 17.4e3, 24e3};
  static const double fix[5] = {12e3, 16e3, 23e3, 40e3, 70e3};
  return TcCost{w4 ? kb4[i] : kb8[i], w4 ? once4[i] : once8[i], fix[i]};
}

// Token tile and split count for M > 32 (tiles of 64 tokens or more), chosen
// together to minimise max(memory time, rounds of units x unit cost + once).
// Ties keep the wider tile (fewer re-reads of the weights).
static void plan_tc_joint(TcPlan& p, int64_t M, int64_t N, int64_t K, int num_sms, int cols, bool w4, int max_bn,
                          int min_bn) {
  const int64_t KB = K / cols;
  const double wbytes = static_cast<double>(N) * static_cast<double>(K) * (w4 ? 0.51953125 : 1.0);
  const double xbytes = static_cast<double>(M) * static_cast<double>(K) * (w4 ? 2.0 : 1.0);
  const double ybytes = 2.0 * static_cast<double>(M) * static_cast<double>(N);
  double best = 1e30;
  int top = pick_bn(M) < max_bn ? pick_bn(M) : max_bn;
  if (top < min_bn) top = min_bn;
  const int low = std::max(w4 ? 16 : 64, min_bn);  // W4A16 plans every token tile this way
  for (int bn = top; bn >= low; bn /= 2) {
    const TcCost cost = tc_cost(w4, bn);
    // A in TMEM (BN <= 128): slots of two blocks; narrow tiles four blocks per
    // stage, so that a stage still carries enough bytes
    const int kps = (w4 && bn <= 32 && KB % 4 == 0) ? 4 : (w4 && bn <= 128) ? 2 : 1;
    const int64_t KS = KB / kps;
    const int64_t mblocks = (M + bn - 1) / bn;
    const int64_t tiles = (N / kTileN) * mblocks;
    const int64_t min_stages = (4 + kps - 1) / kps;
    int64_t max_s = KS / min_stages;
    if (max_s < 1) max_s = 1;
    if (max_s > 8) max_s = 8;
    const double t_mem = (wbytes * static_cast<double>(mblocks > 4 ? 4 : mblocks) + xbytes + ybytes) / 6.5e12;
    for (int c = 1; c <= max_s; ++c) {
      const int64_t per = (KS + c - 1) / c;
      if ((KS + per - 1) / per != c) continue;  // that many splits would not form
      const double rounds = std::ceil(static_cast<double>(tiles * c) / num_sms);
      const double fix = c > 1 ? cost.fix * (1.0 + 0.5 * (c - 2)) : 0.0;
      const double cyc = rounds * (static_cast<double>(per * kps) * cost.kb + fix) + cost.once;
      const double t = std::max(cyc / 2.07e9, t_mem);
      if (t < best) {
        best = t;
        p.bn = bn;
        p.kps = kps;
        p.mblocks = mblocks;
        p.split.splits = c;
        p.split.kb_per_split = static_cast<int>(per) * kps;
        p.split.tiles = tiles;
      }
    }
  }
  p.split.ws_bytes = p.split.splits > 1 ? counters_bytes(p.split.tiles) +
                                              sizeof(float) * static_cast<size_t>(p.split.splits) * M * N
                                        : 0;
}

static TcPlan plan_tc(int64_t M, int64_t N, int64_t K, int num_sms, int cols, bool w4, int max_bn = 256,
                      int tile_n = kTileN, bool joint = true, int min_bn = 0) {
  TcPlan p;
  p.bn = pick_bn(M) < max_bn ? pick_bn(M) : max_bn;
  p.wn = tile_n;
  if (joint && (p.bn >= 64 || w4) && tile_n == kTileN) {
    plan_tc_joint(p, M, N, K, num_sms, cols, w4, max_bn, min_bn);
    return p;
  }
  p.mblocks = (M + p.bn - 1) / p.bn;
  const int64_t tiles = (N / tile_n) * p.mblocks;
  const int64_t KB = K / cols;
  // K blocks per pipeline stage: small token tiles carry little activation
  // data, so W4A16 stages bundle several 4 KB code blocks to keep enough bytes
  // in flight per SM
  p.kps = 1;
  if (w4 && p.bn <= 32 && KB % 4 == 0) p.kps = 4;
  else if (w4 && p.bn <= 128) p.kps = 2;  // A in TMEM: slots of two blocks (K % 128 == 0 makes KB even)
  const int64_t KS = KB / p.kps;  // stages along K
  // Split K by a small cost model: the time of a split count c is the larger
  // of the memory time (all bytes at the HBM rate, or one unit's bytes at a
  // single SM's streaming rate, times the rounds of units per SM) and the MMA
  // time (rounds x one unit's FLOPs at one SM's rate), plus a fixed cost for
  // the partial-sum fix-up when c > 1.  Partial sums are FP32, written and read
  // back once.  At least 4 blocks of K per unit; fewer splits on a tie.
  const double wbytes = static_cast<double>(N) * static_cast<double>(K) * (w4 ? 0.51953125 : 1.0);
  const double xbytes = static_cast<double>(M) * static_cast<double>(K) * (w4 ? 2.0 : 1.0);
  const double ybytes = 2.0 * static_cast<double>(M) * static_cast<double>(N);
  const double flops = 2.0 * static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K);
  const double hbm = 6.5e12, sm_stream = 80e9;
  const double sm_mma = (w4 ? 1.9e15 : 3.9e15) * 0.7 / num_sms;
  const int64_t min_stages = (4 + p.kps - 1) / p.kps;
  int64_t max_s = KS / min_stages;
  if (max_s < 1) max_s = 1;
  if (max_s > 32) max_s = 32;
  if (p.bn >= 128 && max_s > 2) max_s = 2;  // wide token tiles: the fix-up of many partials costs more than it gains
  if (tiles >= num_sms) max_s = 1;          // enough tiles for every SM: splitting only adds partial-sum traffic
  int s = 1;
  double best = 1e30;
  for (int c = 1; c <= max_s; ++c) {
    const double units = static_cast<double>(tiles) * c;
    const double rounds = std::ceil(units / num_sms);
    const double partial = c > 1 ? 8.0 * c * static_cast<double>(M) * static_cast<double>(N) : 0.0;
    const double bytes = wbytes * static_cast<double>(p.mblocks > 4 ? 1 : p.mblocks) + xbytes + ybytes + partial;
    const double t_mem = std::max(bytes / hbm, rounds * (bytes / units) / sm_stream);
    const double t_mma = rounds * (flops / units) / sm_mma;
    const double t = std::max(t_mem, t_mma) + (c > 1 ? 2e-6 : 0.0);
    if (t < best * 0.97) {
      best = t;
      s = c;
    }
  }
  const int per = static_cast<int>((KS + s - 1) / s);  // stages per split
  s = static_cast<int>((KS + per - 1) / per);
  p.split.splits = s;
  p.split.kb_per_split = per * p.kps;
  p.split.tiles = tiles;
  p.split.ws_bytes = s > 1 ? counters_bytes(tiles) + sizeof(float) * static_cast<size_t>(s) * M * N : 0;
  return p;
}

TcPlan plan_w4a16_tc(int64_t M, int64_t N, int64_t K, int num_sms) { return plan_tc(M, N, K, num_sms, 64, true); }
TcPlan plan_w8a8_tc(int64_t M, int64_t N, int64_t K, int num_sms) { return plan_tc(M, N, K, num_sms, 128, false); }
// W4A8: K blocks of 128 columns (one quantisation group, two code tiles) and
// at most 64 tokens per tile (the promotion keeps a row's running sums in
// registers); the E4M3 tile plan with those limits.
TcPlan plan_w4a8_tc(int64_t M, int64_t N, int64_t K, int num_sms) { return plan_tc(M, N, K, num_sms, 128, false, 64); }

// MXFP8 runs on the E4M3 tile plan with at least 32 tokens per tile: a token
// tile then starts on a 32-token boundary of its scale atom (the MMA reads a
// tile's token scales from whole TMEM columns of 32 lanes).  256-token tiles
// keep one accumulator: two would leave no TMEM for the scale-factor ring.
TcPlan plan_mxfp8_tc(int64_t M, int64_t N, int64_t K, int num_sms) {
  TcPlan p = plan_tc(M, N, K, num_sms, 128, false, 256);
  if (p.bn == 256 && p.split.splits > 1) p = plan_tc(M, N, K, num_sms, 128, false, 128);  // 256: never split
  if (p.bn < 32) p.bn = 32;  // the same single token block for M <= 16
  return p;
}
// FP4 (MXFP4, NVFP4): a K block of 256 E2M1 columns is 128 bytes per row,
// the bytes and K blocks of an E4M3 problem of K / 2 columns; the MXFP8 plan
// of that problem, without 64-token tiles (see TcCfg): one 32-token block up
// to 32 tokens, 128- or 256-token tiles beyond.
TcPlan plan_fp4_tc(int64_t M, int64_t N, int64_t K, int num_sms) {
  if (M <= 32) return plan_mxfp8_tc(M, N, K / 2, num_sms);
  TcPlan p = plan_tc(M, N, K / 2, num_sms, 128, false, 256, kTileN, true, 128);
  if (p.bn == 256 && p.split.splits > 1) p = plan_tc(M, N, K / 2, num_sms, 128, false, 128, kTileN, true, 128);
  return p;
}
// Block scaling keeps the running sums of a 128-token tile in registers.  With
// 128-token tiles the weight tile is 256 rows (two scale blocks) when N allows
// and there are still enough tiles for every SM: a wider MMA moves fewer
// shared-memory bytes per FLOP.
TcPlan plan_w8a8_block_tc(int64_t M, int64_t N, int64_t K, int num_sms) {
  const int bn = pick_bn(M) < 128 ? pick_bn(M) : 128;
  const int64_t mblocks = (M + bn - 1) / bn;
  const int wn = (bn == 128 && N % 256 == 0 && (N / 256) * mblocks >= num_sms) ? 256 : 128;
  return plan_tc(M, N, K, num_sms, 128, false, 128, wn, false);
}

template <int BN, bool W4, int KPS, bool BS = false, int WN = 128, bool EPI = false, int MX = kMxNone, bool A8 = false>
static cudaError_t launch_tc(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty, TcArgs args,
                             const TcPlan& plan, void* ws, int num_sms, cudaStream_t st) {
  using C = TcCfg<BN, W4, KPS, BS, WN, MX, A8>;
  if (C::kEarly && plan.split.splits != 1) return cudaErrorInvalidValue;  // its epilogue writes Y directly
  cudaError_t e = set_smem_once(tc_gemm_kernel<BN, W4, KPS, BS, WN, EPI, MX, A8>, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  args.counters = static_cast<uint32_t*>(ws);
  args.partials = ws ? reinterpret_cast<float*>(static_cast<char*>(ws) + counters_bytes(plan.split.tiles)) : nullptr;
  args.ntiles = static_cast<int>(args.N / WN);
  args.mblocks = static_cast<int>(plan.mblocks);
  args.splits = plan.split.splits;
  args.kb_per_split = plan.split.kb_per_split;
  args.units = static_cast<int>(plan.split.tiles * plan.split.splits);
  {
    const double l2_half = 63.0 * 1024 * 1024;  // half of the 126 MB L2
    const double wb = static_cast<double>(args.N) * static_cast<double>(args.K) * (W4 ? 0.51953125 : C::kF4 ? 0.5 : 1.0);
    const double xb = static_cast<double>(args.M) * static_cast<double>(args.K) * ((W4 && !A8) ? 2.0 : C::kF4 ? 0.5 : 1.0);
    args.mb_fast = xb < wb ? 1 : 0;
    args.x_keep = xb <= l2_half / 2 ? 1 : 0;
    args.w_keep = !args.mb_fast && args.mblocks > 1 && wb <= l2_half ? 1 : 0;
  }
  const int grid = args.units < num_sms ? args.units : num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap with the previous kernel's tail
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<BN, W4, KPS, BS, WN, EPI, MX, A8>, tx, tw, ty, args);
}

template <bool W4, bool EPI>
static cudaError_t launch_tc_bn(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty, const TcArgs& a,
                                const TcPlan& plan, void* ws, int num_sms, cudaStream_t st) {
  if constexpr (W4) {
    if (plan.bn == 16) return plan.kps == 4 ? launch_tc<16, true, 4, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st)
                                            : launch_tc<16, true, 2, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
    if (plan.bn == 32) return plan.kps == 4 ? launch_tc<32, true, 4, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st)
                                            : launch_tc<32, true, 2, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
    if (plan.bn == 64) return launch_tc<64, true, 2, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
    if (plan.bn == 128) return launch_tc<128, true, 2, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
    return launch_tc<256, true, 1, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
  } else {
    switch (plan.bn) {
      case 16: return launch_tc<16, false, 1, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
      case 32: return launch_tc<32, false, 1, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
      case 64: return launch_tc<64, false, 1, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
      case 128: return launch_tc<128, false, 1, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
      default: return launch_tc<256, false, 1, false, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
    }
  }
}

cudaError_t launch_w4a16_tc(const uint16_t* X, const uint8_t* codes, const uint16_t* scales, const uint8_t* zeros,
                            uint16_t* Y, int64_t M, int64_t N, int64_t K, int G, const TcPlan& plan, void* ws,
                            int* err, int num_sms, cudaStream_t st, const Epi& epi) {
  CUtensorMap tx, ty;
  if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, K * 2, 64, plan.bn))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Y, N, M, N * 2, kTileN, 16, false))
    return cudaErrorInvalidValue;
  TcArgs a{};
  a.codes = codes;
  a.scales = scales;
  a.zeros = zeros;
  a.G = G;
  a.gshift = G == 32 ? 5 : G == 64 ? 6 : G == 128 ? 7 : 31;
  a.Y = Y;
  a.err = err;
  a.M = M;
  a.N = N;
  a.K = K;
  a.epi = epi;
  return (epi.bias || epi.act) ? launch_tc_bn<true, true>(tx, tx, ty, a, plan, ws, num_sms, st)
                                : launch_tc_bn<true, false>(tx, tx, ty, a, plan, ws, num_sms, st);
}

cudaError_t launch_w8a8_tc(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, uint16_t* Y,
                           int64_t M, int64_t N, int64_t K, const TcPlan& plan, void* ws, int* err, int num_sms,
                           cudaStream_t st, const Epi& epi) {
  CUtensorMap tx, tw, ty;
  if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Xq, K, M, K, 128, plan.bn)) return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wq, K, N, K, 128, 128)) return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Y, N, M, N * 2, kTileN, 16, false))
    return cudaErrorInvalidValue;
  TcArgs a{};
  a.sx = sx;
  a.sw = sw;
  a.Y = Y;
  a.err = err;
  a.M = M;
  a.N = N;
  a.K = K;
  a.epi = epi;
  return (epi.bias || epi.act) ? launch_tc_bn<false, true>(tx, tw, ty, a, plan, ws, num_sms, st)
                                : launch_tc_bn<false, false>(tx, tw, ty, a, plan, ws, num_sms, st);
}

template <bool EPI>
static cudaError_t launch_w4a8_bn(const CUtensorMap& tx, const CUtensorMap& ty, const TcArgs& a, const TcPlan& plan,
                                  void* ws, int num_sms, cudaStream_t st) {
  switch (plan.bn) {
    case 16: return launch_tc<16, true, 1, false, 128, EPI, false, true>(tx, tx, ty, a, plan, ws, num_sms, st);
    case 32: return launch_tc<32, true, 1, false, 128, EPI, false, true>(tx, tx, ty, a, plan, ws, num_sms, st);
    default: return launch_tc<64, true, 1, false, 128, EPI, false, true>(tx, tx, ty, a, plan, ws, num_sms, st);
  }
}

cudaError_t launch_w4a8_tc(const uint8_t* Xq, const float* sx, const uint8_t* codes, const uint16_t* scales,
                           const uint8_t* zeros, uint16_t* Y, int64_t M, int64_t N, int64_t K, const TcPlan& plan,
                           void* ws, int* err, int num_sms, cudaStream_t st, const Epi& epi) {
  CUtensorMap tx, ty;
  if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Xq, K, M, K, 128, plan.bn)) return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Y, N, M, N * 2, kTileN, 16, false))
    return cudaErrorInvalidValue;
  TcArgs a{};
  a.codes = codes;
  a.scales = scales;
  a.zeros = zeros;
  a.G = kGroup;
  a.gshift = 7;
  a.sx = sx;
  a.Y = Y;
  a.err = err;
  a.M = M;
  a.N = N;
  a.K = K;
  a.epi = epi;
  return (epi.bias || epi.act) ? launch_w4a8_bn<true>(tx, ty, a, plan, ws, num_sms, st)
                                : launch_w4a8_bn<false>(tx, ty, a, plan, ws, num_sms, st);
}

template <bool EPI>
static cudaError_t launch_mxfp8_bn(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty, const TcArgs& a,
                                   const TcPlan& plan, void* ws, int num_sms, cudaStream_t st) {
  switch (plan.bn) {
    case 32: return launch_tc<32, false, 1, false, 128, EPI, kMxF8>(tx, tw, ty, a, plan, ws, num_sms, st);
    case 64: return launch_tc<64, false, 1, false, 128, EPI, kMxF8>(tx, tw, ty, a, plan, ws, num_sms, st);
    case 128: return launch_tc<128, false, 1, false, 128, EPI, kMxF8>(tx, tw, ty, a, plan, ws, num_sms, st);
    default: return launch_tc<256, false, 1, false, 128, EPI, kMxF8>(tx, tw, ty, a, plan, ws, num_sms, st);
  }
}

cudaError_t launch_mxfp8_tc(const uint8_t* Xq, const uint8_t* xs, const uint8_t* Wq, const uint8_t* ws_sf,
                            uint16_t* Y, int64_t M, int64_t N, int64_t K, const TcPlan& plan, void* ws, int* err,
                            int num_sms, cudaStream_t st, const Epi& epi) {
  CUtensorMap tx, tw, ty;
  if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Xq, K, M, K, 128, plan.bn)) return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wq, K, N, K, 128, 128)) return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Y, N, M, N * 2, kTileN, 16, false))
    return cudaErrorInvalidValue;
  TcArgs a{};
  a.sfa = ws_sf;
  a.sfb = xs;
  a.Y = Y;
  a.err = err;
  a.M = M;
  a.N = N;
  a.K = K;
  a.epi = epi;
  return (epi.bias || epi.act) ? launch_mxfp8_bn<true>(tx, tw, ty, a, plan, ws, num_sms, st)
                                : launch_mxfp8_bn<false>(tx, tw, ty, a, plan, ws, num_sms, st);
}

template <int MX, bool EPI>
static cudaError_t launch_fp4_bn(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty, const TcArgs& a,
                                 const TcPlan& plan, void* ws, int num_sms, cudaStream_t st) {
  switch (plan.bn) {
    case 32:  // only as the single token block: its scales start at column 0 of the token atom
      if (plan.mblocks != 1) return cudaErrorInvalidValue;
      return launch_tc<32, false, 1, false, 128, EPI, MX>(tx, tw, ty, a, plan, ws, num_sms, st);
    case 128: return launch_tc<128, false, 1, false, 128, EPI, MX>(tx, tw, ty, a, plan, ws, num_sms, st);
    case 256: return launch_tc<256, false, 1, false, 128, EPI, MX>(tx, tw, ty, a, plan, ws, num_sms, st);
    default: return cudaErrorInvalidValue;
  }
}

// MXFP4 (sgx == sgw == nullptr) and NVFP4: packed E2M1 operands, K / 2 bytes per row
cudaError_t launch_fp4_tc(const uint8_t* Xq, const uint8_t* xs, const float* sgx, const uint8_t* Wq,
                          const uint8_t* ws_sf, const float* sgw, uint16_t* Y, int64_t M, int64_t N, int64_t K,
                          bool nv, const TcPlan& plan, void* ws, int* err, int num_sms, cudaStream_t st,
                          const Epi& epi) {
  CUtensorMap tx, tw, ty;
  if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Xq, K / 2, M, K / 2, 128, plan.bn))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wq, K / 2, N, K / 2, 128, 128))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Y, N, M, N * 2, kTileN, 16, false))
    return cudaErrorInvalidValue;
  TcArgs a{};
  a.sfa = ws_sf;
  a.sfb = xs;
  a.sx = sgx;
  a.sw = sgw;
  a.Y = Y;
  a.err = err;
  a.M = M;
  a.N = N;
  a.K = K;
  a.epi = epi;
  if (epi.bias || epi.act)
    return nv ? launch_fp4_bn<kNvF4, true>(tx, tw, ty, a, plan, ws, num_sms, st)
              : launch_fp4_bn<kMxF4, true>(tx, tw, ty, a, plan, ws, num_sms, st);
  return nv ? launch_fp4_bn<kNvF4, false>(tx, tw, ty, a, plan, ws, num_sms, st)
            : launch_fp4_bn<kMxF4, false>(tx, tw, ty, a, plan, ws, num_sms, st);
}

template <bool EPI>
static cudaError_t launch_block_bn(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty, const TcArgs& a,
                                   const TcPlan& plan, void* ws, int num_sms, cudaStream_t st) {
  switch (plan.bn) {
    case 16: return launch_tc<16, false, 1, true, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
    case 32: return launch_tc<32, false, 1, true, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
    case 64: return launch_tc<64, false, 1, true, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
    default:
      return plan.wn == 256 ? launch_tc<128, false, 1, true, 256, EPI>(tx, tw, ty, a, plan, ws, num_sms, st)
                            : launch_tc<128, false, 1, true, 128, EPI>(tx, tw, ty, a, plan, ws, num_sms, st);
  }
}

cudaError_t launch_w8a8_block_tc(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, uint16_t* Y,
                                 int64_t M, int64_t N, int64_t K, const TcPlan& plan, void* ws, int* err, int num_sms,
                                 cudaStream_t st, const Epi& epi) {
  CUtensorMap tx, tw, ty;
  if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Xq, K, M, K, 128, plan.bn)) return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wq, K, N, K, 128, 128)) return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Y, N, M, N * 2, kTileN, 16, false))
    return cudaErrorInvalidValue;
  TcArgs a{};
  a.sx = sx;
  a.sw = sw;
  a.Y = Y;
  a.err = err;
  a.M = M;
  a.N = N;
  a.K = K;
  a.epi = epi;
  return (epi.bias || epi.act) ? launch_block_bn<true>(tx, tw, ty, a, plan, ws, num_sms, st)
                                : launch_block_bn<false>(tx, tw, ty, a, plan, ws, num_sms, st);
}

}  // namespace qlin
