// Routed-expert GEMMs with MXFP4 weights on the block-scaled tensor-core MMA
// (tcgen05.mma.cta_group::2.kind::mxf4): the experts' E2M1 bytes go from HBM to shared memory by
// TMA exactly as stored and are multiplied as stored, their E8M0 scales applied by the MMA
// itself, so no instruction of the kernel touches a weight value (page "What K3 actually is",
// srikanthmalla.com: MXFP4 expert weights, and the dequantizing path's lost 4-bit arithmetic
// rate that this kernel keeps; page "Lesson 6 - LatentMoE", kimi-k3-course.pages.dev, eq. 11 for
// the routed experts' gate/up and down projections).
//
// The token rows arrive as three-term MXFP4 records (mx.cuh), so every product is E2M1 x E2M1:
//
//   D[f][j] = sum_t sum_c W_e[f][c] * 2^sw[f][c/32] * Q_t[row0 + j][c] * 2^sx_t[row0 + j][c/32]
//
// Swapped operands as in the bf16 grouped kernel: the expert's weights are the M = 256 side (128
// rows in each CTA of the pair), its token rows the N side (at most 192 per tile, each expert's
// rows cut into ceil(rows / 192) tiles of equal width rounded up to 16).  Per 256-element k-block
// each CTA stages 16 KB of weights and 3 x 12 KB of token terms; the even CTA issues 3 terms x 4
// MMAs of K = 64.  Decode tiles (16 token rows) put the three terms side by side in N instead:
// one MMA of N = 48 per K = 64 (a CTA-pair MMA of N <= 64 costs the same issue time whatever N
// is, about 49 cycles, so three N = 16 MMAs per 4 KB of weights would bound the weight stream
// near half of HBM bandwidth); the epilogue adds the three terms' accumulator columns.
//
// Scale factors live in TMEM (two slots of 64 columns beside the two 192-column accumulators).
// The producer brings each pair of k-blocks' scale bytes into a ring of their own by TMA (the
// weight rows' scales, and all 192 token rows' scales of the three terms, since both CTAs' MMA
// halves read every token row); a group of four scale warps (one per TMEM lane quadrant) copies
// them from shared memory into TMEM with tcgen05.st in the layout the MMA reads: weight row m at
// lane m, column + m/32 (four columns per 128 scale blocks); token row n at lane n % 32 of every
// quadrant, column + n/32.  A slot is rewritten once the MMAs that read it have completed (a
// commit multicast to both CTAs).
//
// Epilogues: gate/up tiles (128 features: rows 0..15 of each 32-row quarter are gate rows, 16..31
// the matching up rows) compute SiLU(gate) * up, stage 64 tokens x 64 features in shared memory
// and quantise them into three-term MXFP4 records (one 32-feature block per thread), the down
// projection's input; down tiles (256 output features) scale each token column by its routing
// weight and write fp16 rows.  Every wait is bounded; after an abort the even CTA waits for its
// loads and MMAs in flight before the pair lets go of shared memory and TMEM.
#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lmoe {
namespace {

using namespace tc;
constexpr int kWRows = 128;                              // weight rows per CTA (M = 256 per pair)
constexpr int KB = 256;                                  // K elements per stage (128 packed bytes)
constexpr uint32_t kWBytes = kWRows * 128;               // 16 KB
constexpr int kThreads = 320;                            // producer, MMA, 4 epilogue, 4 scale warps
constexpr int kEpiStride = 72;                           // floats per staged token: blocks at 0 and 36

// Layout of the kernel for token tiles of NT columns: 192 (prefill; the dispatch's 192-row tile
// list) or 16 (decode; its 16-row unit list).  Decode tiles carry a few token rows against whole
// weight tiles, so their stages are small and the ring is deep (eight k-blocks of weights in
// flight per CTA instead of three): the kernel then streams weights as fast as HBM delivers them.
//
// F8: the token rows are MXFP8 records (one E4M3 term) and the MMA is kind::mxf8f6f4 (E2M1 x
// E4M3, K = 32 per instruction, 8 per k-block).  That kind reads 4-bit elements from shared
// memory one per byte: the weights land by TMA as CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B (16
// packed elements of global memory padded to 16 bytes), two 128-element boxes per k-block, and
// the transaction count of such a load is its packed (global) size.  Each token row's k-block is
// two 128-byte chunks.
template <int NT, bool F8 = false>
struct MxCfg {
  static constexpr int kN = NT;                                      // token columns per tile (MMA N)
  static constexpr int kTerms = F8 ? 1 : kMxTerms;                   // activation terms per record
  static constexpr int kXRows = NT / 2;                              // token rows per CTA
  static constexpr uint32_t kXTermBytes = kXRows * 128;              // one term's (F8: one chunk's) rows of a k-block
  static constexpr uint32_t kWSmem = F8 ? 2 * kWBytes : kWBytes;     // weight bytes of a k-block in shared memory
  static constexpr uint32_t kStageBytes = kWSmem + (F8 ? 2 : kMxTerms) * kXTermBytes;
  static constexpr int kStages = NT >= 64 ? 3 : (F8 ? 5 : 8);
  // scale ring: per stage the scale bytes of kSfKb k-blocks of this CTA's weight rows, and of all
  // NT token rows of each term (both CTAs' MMA halves read every token row)
  // scale ring: kSfKb k-blocks per stage (8 scale bytes of every row each): four for decode's
  // MXFP4 units, whose producer issue rate bounds them, two where shared memory is scarce
  static constexpr int kSfKb = (NT < 32 && !F8) ? 4 : 2;
  static constexpr uint32_t kSfRowBytes = 8 * kSfKb;                  // bytes of a row per stage
  static constexpr uint32_t kWsBytes = kWRows * kSfRowBytes;          // this CTA's weight rows
  static constexpr uint32_t kXsTermBytes = NT * kSfRowBytes;
  static constexpr uint32_t kSfStageBytes = kWsBytes + kTerms * kXsTermBytes;
  static constexpr int kSfStages = NT >= 64 ? 3 : 4;
  // token boxes sized to the tile: 8, 32 or 96 rows of each term per CTA (tiles of N <= 16, <= 64,
  // <= 192 tokens) and 16, 64 or 192 rows of their scales
  static constexpr int kNumBoxes = NT >= 64 ? 3 : 1;
  // TMEM: two accumulators (at least 32 columns apart: the epilogue reads 32 at a time), then the
  // scale slots: weight scales in 8 columns (4 per 4-block chunk, one per lane quadrant), token
  // scales of term t and chunk h at 8 + t * 16 + h * 8 (row n at + n / 32; decode: the 48 MMA
  // rows of chunk h at 8 + 16 h, row n at + n / 32).  Every scale-factor
  // address the MMA is given is a multiple of 4 columns (weights) or 8 (tokens) from a 64-column
  // slot start: the MMA reads its scale operands at such aligned addresses only.
  // decode: N = 3 * 16 token-term columns, CTA c providing rows 24 c + 8 q + j' (term q of token
  // 8 c + j'), the three terms of a k-block being contiguous 8-row swizzle atoms in its stage
  static constexpr bool kTermsInN = !F8 && NT < 32;
  static constexpr int kMmaN = kTermsInN ? kMxTerms * NT : NT;
  static constexpr uint32_t kAccCols = kTermsInN ? 64 : (NT >= 32 ? NT : 32);
  static constexpr uint32_t kChunkCols = 8;
  static constexpr uint32_t kSfCols = 64;
  static constexpr int kSfSlots = NT >= 32 ? 2 : 4;
  static constexpr uint32_t kSfBase = 2 * kAccCols;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kEpiTokens = NT >= 64 ? 64 : 32;              // tokens per GLU epilogue chunk
  static constexpr uint32_t kEpiBytes = kEpiTokens * kEpiStride * 4; // >= the down epilogue's 8 KB
  static constexpr size_t kSmem =
      (size_t)kStages * kStageBytes + (size_t)kSfStages * kSfStageBytes + kEpiBytes + 1024 + 512;
  static_assert(kSfBase + kSfSlots * kSfCols <= kTmemCols, "TMEM budget");
  static_assert(kSfBase % 64 == 0 && kSfCols % 64 == 0, "scale slots start on 64-column boundaries");
  static_assert(8 + kMxTerms * 2 * kChunkCols <= kSfCols, "scale slot");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert(kEpiBytes >= 4 * 32 * 32 * 2, "down epilogue staging");
  static_assert(!kTermsInN || (NT == 16 && kXTermBytes == 1024 && kMmaN <= 64), "decode: terms as 8-row atoms");
  static_assert(kStageBytes % 1024 == 0 && kXTermBytes % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
};
static_assert(MxCfg<192>::kN == kTileMx, "the dispatch cuts expert rows into tiles of this kernel's width");
static_assert(MxCfg<16>::kN == kTileS, "decode units are the dispatch's 16-row units");
static_assert(MxCfg<192, true>::kN == kTileMx && MxCfg<16, true>::kN == kTileS, "MXFP8 tiles: the same lists");
__host__ __device__ constexpr int x_box_rows(int NT, int b) {
  return NT < 64 ? NT / 2 : (b == 0 ? 8 : b == 1 ? 32 : NT / 2);
}
__host__ __device__ constexpr int box_for(int n) { return n <= 16 ? 0 : n <= 64 ? 1 : 2; }

struct MxParams {
  int num_kb;             // 256-element k-blocks (even: K % 512 == 0)
  int K;                  // reduction width
  int num_wt;             // weight tiles per expert
  int glu_h;              // > 0: gate/up weights [2h][K], 128 features per tile; 0: 256 rows per tile
  const int4* tiles;      // NT = 192: tiles {expert, first tile of expert, rows of expert, first row};
                          // NT = 16: units {expert, first row, rows (<= 16), 0}
  const int32_t* num_tiles;
  void* C;                // GLU: records of the activations [rows][ldc bytes]; down: fp16 [rows][ldc]
  int64_t ldc;
  int out_k;              // GLU: h (the width the records hold)
  const float* row_scale; // down: routing weight per row
  uint32_t* status;
  uint64_t timeout_ns;
  int inject;             // test hook: pair 0 skips its first stage (loads and signal)
};

struct MxTile {
  int expert, wt;
  int row0, nrows, n;
};

__device__ __forceinline__ int4 mx_entry(const MxParams& p, int t) { return p.tiles[t / p.num_wt]; }

template <int NT>
__device__ __forceinline__ MxTile decode_mx(const MxParams& p, int t, int4 tl) {
  MxTile ti;
  ti.expert = tl.x;
  if (NT == 16) {  // a unit of at most 16 rows, against weight tile t % num_wt
    ti.wt = t - (t / p.num_wt) * p.num_wt;
    ti.row0 = tl.y;
    ti.nrows = tl.z;
    ti.n = 16;
    return ti;
  }
  const int rows = tl.z;
  const int ntiles = (rows + NT - 1) / NT;
  const int local = t - tl.y * p.num_wt;
  ti.wt = local / ntiles;
  const int j = local - ti.wt * ntiles;
  // equal widths (multiples of 16, at most NT): width * (ntiles - 1) < rows, so no tile is empty
  const int width = ((rows + ntiles - 1) / ntiles + 15) & ~15;
  ti.row0 = tl.w + j * width;
  ti.nrows = min(width, rows - j * width);
  ti.n = (ti.nrows + 15) & ~15;
  return ti;
}

// 32 token columns of an accumulator row, r[i] = token c0 + i.  With the terms in N (16-token
// tiles) token j's three terms sit in columns 24 (j / 8) + 8 q + j % 8 and are added here (fp32,
// term order); tokens 16..31 read as 0.
template <bool kTermsInN>
__device__ __forceinline__ void load_acc(uint32_t taddr, uint32_t (&r)[32]) {
  if (!kTermsInN) {
    ptx::tmem_ld_32x32b_x32(taddr, r);
    ptx::tmem_ld_wait();
    return;
  }
  uint32_t a[32], b[32];
  ptx::tmem_ld_32x32b_x32(taddr, a);
  ptx::tmem_ld_32x32b_x32(taddr + 32, b);
  ptx::tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    r[j] = __float_as_uint(__uint_as_float(a[j]) + __uint_as_float(a[8 + j]) + __uint_as_float(a[16 + j]));
    r[8 + j] = __float_as_uint(__uint_as_float(a[24 + j]) + __uint_as_float(b[j]) + __uint_as_float(b[8 + j]));
  }
#pragma unroll
  for (int j = 16; j < 32; ++j) r[j] = 0u;
}

// Epilogue-warp barrier (the 4 epilogue warps only).
__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <bool GLU, int NT, bool F8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_mx_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmWs,
                 const __grid_constant__ CUtensorMap tmX0, const __grid_constant__ CUtensorMap tmX1,
                 const __grid_constant__ CUtensorMap tmX2, const __grid_constant__ CUtensorMap tmXs0,
                 const __grid_constant__ CUtensorMap tmXs1, const __grid_constant__ CUtensorMap tmXs2,
                 const MxParams p) {
  using C = MxCfg<NT, F8>;
  constexpr int kStages = C::kStages, kSfStages = C::kSfStages, kSfSlots = C::kSfSlots;
  constexpr uint32_t kStageBytes = C::kStageBytes, kXTermBytes = C::kXTermBytes, kSfStageBytes = C::kSfStageBytes;
  constexpr uint32_t kXsTermBytes = C::kXsTermBytes, kEpiBytes = C::kEpiBytes, kSfBase = C::kSfBase;
  constexpr uint32_t kWsBytes = C::kWsBytes, kSfRowBytes = C::kSfRowBytes;
  constexpr int kSfKb = C::kSfKb;
  constexpr uint32_t kSfCols = C::kSfCols, kAccCols = C::kAccCols, kChunkCols = C::kChunkCols;
  constexpr uint32_t kTmemCols = C::kTmemCols;
  constexpr int kEpiTokens = C::kEpiTokens;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // same offset in both CTAs
  uint8_t* sf_ring = smem + kStages * kStageBytes;
  float* epi = reinterpret_cast<float*>(sf_ring + kSfStages * kSfStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(epi) + kEpiBytes);
  uint64_t* empty = full + kStages;
  uint64_t* sfr_full = empty + kStages;        // scale ring: bytes landed (this CTA)
  uint64_t* sfr_empty = sfr_full + kSfStages;  // scale ring: copied to TMEM by the 4 scale warps
  uint64_t* sf_full = sfr_empty + kSfStages;   // TMEM scale slot written (even CTA, 8 warps)
  uint64_t* sf_empty = sf_full + kSfSlots;     // TMEM scale slot read by its MMAs (both CTAs)
  uint64_t* tmem_full = sf_empty + kSfSlots;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain_bar = tmem_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* epi_ok = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0: issues the MMAs; 1: partner
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  ptx::ArmedStages armed, armed_sf;  // producer: operand stages (even CTA) and scale stages armed

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kSfStages; ++s) {
      ptx::mbar_init(&sfr_full[s], 1);
      ptx::mbar_init(&sfr_empty[s], 4);
    }
    for (int s = 0; s < kSfSlots; ++s) {
      ptx::mbar_init(&sf_full[s], 8);  // 4 scale warps in each CTA of the pair
      ptx::mbar_init(&sf_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tmem_full[a], 1);
      ptx::mbar_init(&tmem_empty[a], 8);  // 4 epilogue warps in each CTA of the pair
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmWs);
    ptx::prefetch_tmap(&tmX0);
    ptx::prefetch_tmap(&tmX1);
    ptx::prefetch_tmap(&tmX2);
    ptx::prefetch_tmap(&tmXs0);
    ptx::prefetch_tmap(&tmXs1);
    ptx::prefetch_tmap(&tmXs2);
  }
  if (warp == 1) ptx::tmem_alloc_pair(tmem_holder, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before any signal crosses the pair
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int total = *p.num_tiles * p.num_wt;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    int stage = 0, sstage = 0;
    uint32_t phase = 0, sphase = 0;
    bool first = true;
    int4 entry = pair < total ? mx_entry(p, pair) : make_int4(0, 0, 0, 0);
    for (int t = pair; t < total; t += npairs) {
      const MxTile ti = decode_mx<NT>(p, t, entry);
      if (t + npairs < total) entry = mx_entry(p, t + npairs);
      const int xrow0 = ti.row0 + (int)rank * (ti.n >> 1);  // this CTA's N/2 token rows
      const int wrow_glu = (ti.wt * 128 + (int)rank * 64) / 16;                // GLU: first 16-row group
      const int wrow = ti.wt * 2 * kWRows + (int)rank * kWRows;                // down: first weight row
      const int bsel = C::kNumBoxes == 1 ? 0 : box_for(ti.n);
      const CUtensorMap* tmX = bsel == 0 ? &tmX0 : bsel == 1 ? &tmX1 : &tmX2;
      const CUtensorMap* tmXs = bsel == 0 ? &tmXs0 : bsel == 1 ? &tmXs1 : &tmXs2;
      // bytes a stage's loads deliver: weights (F8: counted packed), token rows of each term or chunk
      const uint32_t stage_tx = kWBytes + (F8 ? 2u : (uint32_t)kMxTerms) * (uint32_t)x_box_rows(NT, bsel) * 128u;
      const uint32_t sf_tx = kWsBytes + (uint32_t)C::kTerms * (uint32_t)(2 * x_box_rows(NT, bsel)) * kSfRowBytes;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (kb % kSfKb == 0) {
          // scale bytes of k-blocks kb .. kb+kSfKb-1 (8 bytes each of every row) into this CTA's
          // scale ring (past the last k-block: the boxes' fill)
          if (!ptx::mbar_wait_bounded(&sfr_empty[sstage], sphase ^ 1u, abort_flag, p.status, p.timeout_ns,
                                      kWaitProducer))
            goto done;
          uint8_t* ss = sf_ring + sstage * kSfStageBytes;
          ptx::mbar_arrive_expect_tx(&sfr_full[sstage], sf_tx);
          armed_sf.arm(sstage, sphase);
          const int xb = 8 * kb;  // byte of k-block kb in a scale row (16-byte aligned: kb even)
          if (GLU)
            ptx::tma_load_5d(ss, &tmWs, &sfr_full[sstage], xb, 0, 0, wrow_glu, ti.expert);
          else
            ptx::tma_load_3d(ss, &tmWs, &sfr_full[sstage], xb, wrow, ti.expert);
          if (C::kTermsInN)  // decode: the three terms' scale bytes in one box {16 B, NT rows, 3 terms}
            ptx::tma_load_3d(ss + kWsBytes, tmXs, &sfr_full[sstage], xb, ti.row0, 0);
          else
#pragma unroll
            for (int q = 0; q < C::kTerms; ++q)
              ptx::tma_load_2d(ss + kWsBytes + q * kXsTermBytes, tmXs, &sfr_full[sstage], q * (p.K / 32) + xb,
                               ti.row0);
          if (++sstage == kSfStages) {
            sstage = 0;
            sphase ^= 1u;
          }
        }
        // the stage's last reader has finished: the MMA's commit arrives in both CTAs of the pair
        if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns, kWaitProducer))
          goto done;
        uint8_t* sW = smem + stage * kStageBytes;
        uint8_t* sX = sW + C::kWSmem;  // F8: the weight chunks take 2 x kWBytes
        const uint32_t bar = ptx::mapa_shared(&full[stage], 0);  // the even CTA's full[stage]
        const bool skip = p.inject && first && pair == 0;  // test hook, the same in both CTAs
        first = false;
        if (!skip) {
          if (rank == 0) {
            ptx::mbar_arrive_expect_tx(&full[stage], 2 * stage_tx);
            armed.arm(stage, phase);
          }
          if (F8) {  // two 128-element weight chunks (padded to a byte each), two 128-byte token chunks
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              if (GLU)
                ptx::tma_load_5d_pair(sW + c * kWBytes, &tmW, bar, kb * 256 + c * 128, 0, 0, wrow_glu, ti.expert);
              else
                ptx::tma_load_3d_pair(sW + c * kWBytes, &tmW, bar, kb * 256 + c * 128, wrow, ti.expert);
              ptx::tma_load_2d_pair(sX + c * kXTermBytes, tmX, bar, kb * 256 + c * 128, xrow0);
            }
          } else {
            if (GLU)  // 4 x (16 gate rows, 16 up rows) of features wt*128 + rank*64 ..
              ptx::tma_load_5d_pair(sW, &tmW, bar, kb * 128, 0, 0, wrow_glu, ti.expert);
            else
              ptx::tma_load_3d_pair(sW, &tmW, bar, kb * 128, wrow, ti.expert);
            if (C::kTermsInN)  // decode: the three terms' 8 rows in one box {128 B, 8 rows, 3 terms}, term-major
              ptx::tma_load_3d_pair(sX, tmX, bar, kb * 128, xrow0, 0);
            else
#pragma unroll
              for (int q = 0; q < kMxTerms; ++q)  // term q: 96 rows x 128 bytes at byte q * K/2 + kb * 128 of each record
                ptx::tma_load_2d_pair(sX + q * kXTermBytes, tmX, bar, q * (p.K / 2) + kb * 128, xrow0);
          }
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    int s = 0, g = 0;
    uint32_t ph = 0;
    int it = 0;
    int4 entry = pair < total ? mx_entry(p, pair) : make_int4(0, 0, 0, 0);
    for (int t = pair; t < total; t += npairs, ++it) {
      const MxTile ti = decode_mx<NT>(p, t, entry);
      if (t + npairs < total) entry = mx_entry(p, t + npairs);
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!ptx::mbar_wait_bounded(&tmem_empty[acc], (use & 1u) ^ 1u, abort_flag, p.status, p.timeout_ns,
                                  kWaitAccFree))
        goto done;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)acc * kAccCols;
      for (int kb = 0; kb < p.num_kb; ++kb, ++g) {
        const int slot = g % kSfSlots;
        if (!ptx::mbar_wait_bounded(&full[s], ph, abort_flag, p.status, p.timeout_ns, kWaitFull)) goto done;
        if (!ptx::mbar_wait_bounded(&sf_full[slot], (uint32_t)(g / kSfSlots) & 1u, abort_flag, p.status,
                                    p.timeout_ns, kWaitConverted))
          goto done;
        ptx::tc_fence_after();
        const uint32_t w_addr = ptx::smem_addr(smem + s * kStageBytes);
        const uint32_t x_addr = w_addr + C::kWSmem;
        const uint32_t sf = tmem_base + kSfBase + (uint32_t)slot * kSfCols;
        if (F8) {  // 8 MMAs of K = 32: chunk c = kk / 4, scale byte kk % 4 of the chunk's columns
#pragma unroll
          for (int kk = 0; kk < KB / 32; ++kk) {
            const uint32_t c = (uint32_t)(kk >> 2), sub = (uint32_t)(kk & 3);
            ptx::mma_mxf8f6f4_pair(d_tmem, ptx::sw128_kmajor_desc(w_addr + c * kWBytes + sub * 32),
                                   ptx::sw128_kmajor_desc(x_addr + c * kXTermBytes + sub * 32),
                                   ptx::idesc_mxf8f6f4_e2m1_e4m3(2 * kWRows, ti.n, sub, sub), sf + 4u * c,
                                   sf + 8u + kChunkCols * c, (kb | kk) != 0 ? 1u : 0u);
          }
        } else {
#pragma unroll
        for (int kk = 0; kk < KB / 64; ++kk) {
          const uint32_t sf_id = 2u * (uint32_t)(kk & 1);
          const uint64_t a_desc = ptx::sw128_kmajor_desc(w_addr + kk * 32);
          if (C::kTermsInN) {  // the three terms' 24 rows of each CTA as one operand: N = 48
            ptx::mma_mxf4_pair(d_tmem, a_desc, ptx::sw128_kmajor_desc(x_addr + kk * 32),
                               ptx::idesc_mxf4(2 * kWRows, C::kMmaN, sf_id, sf_id), sf + 4u * (uint32_t)(kk >> 1),
                               sf + 8u + 2u * kChunkCols * (uint32_t)(kk >> 1), (kb | kk) != 0 ? 1u : 0u);
          } else {
            const uint32_t idesc = ptx::idesc_mxf4(2 * kWRows, ti.n, sf_id, sf_id);
#pragma unroll
            for (int q = 0; q < kMxTerms; ++q)
              ptx::mma_mxf4_pair(d_tmem, a_desc, ptx::sw128_kmajor_desc(x_addr + q * kXTermBytes + kk * 32), idesc,
                                 sf + 4u * (uint32_t)(kk >> 1),
                                 sf + 8u + 2u * kChunkCols * (uint32_t)q + kChunkCols * (uint32_t)(kk >> 1),
                                 (kb | kk | q) != 0 ? 1u : 0u);
          }
        }
        }
        ptx::mma_commit_pair_both(&empty[s]);  // both CTAs' copies of the stage are free
        ptx::mma_commit_pair_both(&sf_empty[slot]);
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      ptx::mma_commit_pair(&tmem_full[acc]);
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------------ scale warps (both CTAs)
    const int q = warp & 3;  // TMEM lane quadrant this warp writes
    const uint32_t lane_base = tmem_base + ((uint32_t)(32 * q) << 16) + kSfBase;
    int g = 0, ss = 0;
    uint32_t sph = 0;
    for (int t = pair; t < total; t += npairs) {
      for (int kb = 0; kb < p.num_kb; ++kb, ++g) {
        const int slot = g % kSfSlots;
        int ok = 1;
        if (lane == 0) {
          if (kb % kSfKb == 0)
            ok = ptx::mbar_wait_bounded(&sfr_full[ss], sph, abort_flag, p.status, p.timeout_ns, kWaitFull);
          ok = ok && ptx::mbar_wait_bounded(&sf_empty[slot], ((uint32_t)(g / kSfSlots) & 1u) ^ 1u, abort_flag,
                                            p.status, p.timeout_ns, kWaitAccFree);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) goto sf_done;
        {
          const uint8_t* st = sf_ring + ss * kSfStageBytes + 8 * (kb % kSfKb);  // this k-block's 8 bytes of a row
          const uint2 wv = *reinterpret_cast<const uint2*>(st + (32 * q + lane) * kSfRowBytes);
          ptx::tc_fence_after();
          const uint32_t col = lane_base + (uint32_t)slot * kSfCols;
          ptx::tmem_st_32x32b_x1(col + (uint32_t)q, wv.x);       // weight scale blocks 0..3 of the k-block
          ptx::tmem_st_32x32b_x1(col + 4u + (uint32_t)q, wv.y);  // blocks 4..7
          if (NT >= 32) {
            uint32_t lo[C::kTerms][8], hi[C::kTerms][8];
#pragma unroll
            for (int tt = 0; tt < C::kTerms; ++tt)
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                uint2 v = make_uint2(0u, 0u);
                if (c < NT / 32)
                  v = *reinterpret_cast<const uint2*>(st + kWsBytes + tt * kXsTermBytes + (32 * c + lane) * kSfRowBytes);
                lo[tt][c] = v.x;
                hi[tt][c] = v.y;
              }
#pragma unroll
            for (int tt = 0; tt < C::kTerms; ++tt) {
              ptx::tmem_st_32x32b_x8(col + 8u + 2u * kChunkCols * tt, lo[tt]);
              ptx::tmem_st_32x32b_x8(col + 8u + 2u * kChunkCols * tt + kChunkCols, hi[tt]);
            }
          } else if (F8) {  // one term: token rows 0 .. NT-1 in lanes 0 .. NT-1, chunk h at 8 + 8 h
            uint2 v = make_uint2(0u, 0u);
            if (lane < NT) v = *reinterpret_cast<const uint2*>(st + kWsBytes + lane * kSfRowBytes);
            ptx::tmem_st_32x32b_x1(col + 8u, v.x);
            ptx::tmem_st_32x32b_x1(col + 8u + kChunkCols, v.y);
          } else {  // MMA rows n = 24 c + 8 q + j' (term q, token 8 c + j'): row n at lane n % 32,
                    // column + n / 32 of chunk h's pair of columns at 8 + 2 h kChunkCols
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int n = 32 * half + lane;
              uint2 v = make_uint2(0u, 0u);
              if (n < C::kMmaN) {
                const int c = n / 24, tt = (n % 24) >> 3, j = 8 * c + (n & 7);
                v = *reinterpret_cast<const uint2*>(st + kWsBytes + tt * kXsTermBytes + j * kSfRowBytes);
              }
              ptx::tmem_st_32x32b_x1(col + 8u + (uint32_t)half, v.x);
              ptx::tmem_st_32x32b_x1(col + 8u + 2u * kChunkCols + (uint32_t)half, v.y);
            }
          }
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (rank == 0)
              ptx::mbar_arrive(&sf_full[slot]);
            else
              ptx::mbar_arrive_remote(&sf_full[slot], 0);
            if (kb % kSfKb == kSfKb - 1 || kb == p.num_kb - 1)
              ptx::mbar_arrive(&sfr_empty[ss]);  // every k-block of the stage copied
          }
        }
        if (kb % kSfKb == kSfKb - 1 || kb == p.num_kb - 1) {
          if (++ss == kSfStages) {
            ss = 0;
            sph ^= 1u;
          }
        }
      }
    }
  sf_done:;
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int etid = threadIdx.x - 64;  // 0..127
    int it = 0;
    int4 entry = pair < total ? mx_entry(p, pair) : make_int4(0, 0, 0, 0);
    for (int t = pair; t < total; t += npairs, ++it) {
      const MxTile ti = decode_mx<NT>(p, t, entry);
      if (t + npairs < total) entry = mx_entry(p, t + npairs);
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      // down x p: the item's row scales, lane l holding token 32 c + l
      constexpr int kChunks = (NT + 31) / 32;
      float sc_reg[kChunks];
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const int jl = c * 32 + lane;
        sc_reg[c] = !GLU && jl < ti.nrows ? p.row_scale[ti.row0 + jl] : 0.0f;
      }
      // one warp waits; the decision is shared so that the four warps leave (or stay) together
      if (warp == 2 && lane == 0) {
        const int ok =
            ptx::mbar_wait_bounded(&tmem_full[acc], use & 1u, abort_flag, p.status, p.timeout_ns, kWaitAccFull);
        if (ok && rank == 0) ptx::mbar_arrive_remote(&tmem_full[acc], 1);
        *epi_ok = ok;
      }
      epi_barrier();
      const int ok = *epi_ok;
      epi_barrier();  // every warp has read the flag before the next item rewrites it
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * kAccCols;
      if (GLU) {
        // this CTA's 64 features fb .. fb+63: warp q holds 16 of them.  64 tokens at a time are
        // staged as fp32 [token][2 blocks of 32 features] (block b at float 36 b of a 72-float
        // row), then thread (token j, block b) quantises its 32 values into the record of row j
        const int fb = ti.wt * 128 + (int)rank * 64;
        uint8_t* out = static_cast<uint8_t*>(p.C);
        const int64_t half_k = p.out_k / 2, sc0 = mx3_scale_offset(p.out_k), kscale = p.out_k / 32;
        const int foff = 36 * (q >> 1) + 16 * (q & 1);  // this warp's 16 features in a staged row
        for (int c0 = 0; c0 < ti.n; c0 += kEpiTokens) {
#pragma unroll
          for (int h2 = 0; h2 < kEpiTokens / 32; ++h2) {
            if (c0 + 32 * h2 >= ti.n) break;  // uniform
            uint32_t r[32];
            load_acc<C::kTermsInN>(t_row + c0 + 32 * h2, r);
            // token pair (2i, 2i+1): lanes < 16 finish token 2i, lanes >= 16 token 2i+1
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
              const float send = __uint_as_float(lane < 16 ? r[2 * i2 + 1] : r[2 * i2]);
              const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
              const float gt = lane < 16 ? __uint_as_float(r[2 * i2]) : recv;
              const float up = lane < 16 ? recv : __uint_as_float(r[2 * i2 + 1]);
              epi[(32 * h2 + 2 * i2 + (lane >> 4)) * kEpiStride + foff + (lane & 15)] = silu(gt) * up;
            }
          }
          epi_barrier();
          {
            const int j = etid >> 1, b = etid & 1;
            if (c0 + j < ti.nrows) {
              float v[32];
              const float4* src = reinterpret_cast<const float4*>(epi + j * kEpiStride + 36 * b);
#pragma unroll
              for (int e4 = 0; e4 < 8; ++e4) {
                const float4 f = src[e4];
                v[4 * e4] = f.x;
                v[4 * e4 + 1] = f.y;
                v[4 * e4 + 2] = f.z;
                v[4 * e4 + 3] = f.w;
              }
              uint8_t* rec = out + (int64_t)(ti.row0 + c0 + j) * p.ldc;
              const int f = fb + 32 * b;
              if (F8) {  // MXFP8 record: E4M3 codes at byte f, the scale after the K codes
                uint32_t codes[8], scb8;
                mx::quantize_block8(v, codes, scb8);
                *reinterpret_cast<uint4*>(rec + f) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
                *reinterpret_cast<uint4*>(rec + f + 16) = make_uint4(codes[4], codes[5], codes[6], codes[7]);
                rec[mx8_scale_offset(p.out_k) + f / 32] = (uint8_t)scb8;
              } else {
                uint32_t packed[kMxTerms][4], scb[kMxTerms];
                mx::quantize_block(v, packed, scb);
#pragma unroll
                for (int tt = 0; tt < kMxTerms; ++tt) {
                  *reinterpret_cast<uint4*>(rec + tt * half_k + f / 2) =
                      make_uint4(packed[tt][0], packed[tt][1], packed[tt][2], packed[tt][3]);
                  rec[sc0 + tt * kscale + f / 32] = (uint8_t)scb[tt];
                }
              }
            }
          }
          epi_barrier();  // the staging tile is rewritten by the next chunk
        }
      } else {
        // 32 output features per warp; each 32-token chunk goes through shared memory as
        // [token][feature] fp16 and leaves in 16-byte stores
        const int f0 = ti.wt * 2 * kWRows + (int)rank * kWRows + 32 * q;
        __half* out = static_cast<__half*>(p.C);
        uint16_t* st = reinterpret_cast<uint16_t*>(epi) + q * (32 * 32);
        for (int c0 = 0; c0 < ti.n; c0 += 32) {
          uint32_t r[32];
          load_acc<C::kTermsInN>(t_row + c0, r);
          const int c = c0 >> 5;
          float scv = 0.f;
#pragma unroll
          for (int cc = 0; cc < kChunks; ++cc)
            if (cc == c) scv = sc_reg[cc];
#pragma unroll
          for (int i2 = 0; i2 < 32; ++i2) {
            const float sc = __shfl_sync(0xffffffffu, scv, i2);
            st[i2 * 32 + lane] = __half_as_ushort(__float2half_rn(__uint_as_float(r[i2]) * sc));
          }
          __syncwarp();
#pragma unroll
          for (int v = lane; v < 32 * 4; v += 32) {
            const int j = v >> 2, part = v & 3;
            if (c0 + j < ti.nrows)
              *reinterpret_cast<uint4*>(out + (int64_t)(ti.row0 + c0 + j) * p.ldc + f0 + 8 * part) =
                  *reinterpret_cast<const uint4*>(st + j * 32 + 8 * part);
          }
          __syncwarp();
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          ptx::mbar_arrive(&tmem_empty[acc]);
        else
          ptx::mbar_arrive_remote(&tmem_empty[acc], 0);
      }
    }
  }
done:
  ptx::tc_fence_before();
  __syncthreads();  // every role has left its loop; the abort flag no longer changes
  if (*abort_flag) {  // let the loads and MMAs in flight finish before the pair lets go of them
    if (warp == 0 && lane == 0) {
      ptx::drain_armed(sfr_full, armed_sf, p.timeout_ns);  // this CTA's scale loads
      if (rank == 0) ptx::drain_armed(full, armed, p.timeout_ns);  // both halves' operand loads
    }
    if (rank == 0 && warp == 1 && lane == 0) ptx::drain_mma_pair(drain_bar, p.timeout_ns);
    __syncthreads();
  }
  ptx::cluster_sync();  // the partner no longer reads this CTA's shared memory or signals it
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <bool GLU, int NT, bool F8>
cudaError_t launch_mx_inst(const CUtensorMap (&maps)[8], const MxParams& p, long long items, cudaStream_t s) {
  auto kern = tc_mx_kernel<GLU, NT, F8>;
  constexpr size_t kSmem = MxCfg<NT, F8>::kSmem;
  static PerDeviceValue max_pairs_of;
  std::atomic<int>* slot = max_pairs_of.current();
  if (!slot) return cudaErrorInvalidDevice;
  int max_pairs = slot->load(std::memory_order_acquire);
  if (max_pairs == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_pairs = n;
    slot->store(n, std::memory_order_release);
  }
  const int pairs = (int)(items < max_pairs ? items : max_pairs);
  kern<<<2 * pairs, kThreads, kSmem, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], p);
  return cudaGetLastError();
}

bool encode_u8(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
               const cuuint32_t* box, bool swizzle128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !ptr) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_tc_mx(const TcMx& g, const int4* tiles, const int32_t* num_tiles, int max_tiles, int unit_rows,
                         uint32_t* status, uint64_t timeout_ns, cudaStream_t s, int inject) {
  const bool glu = g.glu_h > 0;
  if (!g.w.ptr || !g.w_scale || !g.x || !g.C || !tiles || !num_tiles) return cudaErrorInvalidValue;
  if (unit_rows != MxCfg<192>::kN && unit_rows != MxCfg<16>::kN) return cudaErrorInvalidValue;
  const bool decode = unit_rows == MxCfg<16>::kN;
  if (g.K % 512 || g.rows < 1) return cudaErrorInvalidValue;
  if (glu ? (g.glu_h % 128 || g.out_features != g.glu_h || g.out_features % 512 || g.w.rows != 2 * g.glu_h)
          : (g.out_features % (2 * kWRows) || g.w.rows != g.out_features || !g.row_scale || g.ldc % 8))
    return cudaErrorInvalidValue;
  const bool f8 = g.f8;
  const int64_t x_rec = f8 ? mx8_row_bytes(g.K) : mx3_row_bytes(g.K), kscale = g.K / 32, E = g.w.depth;
  const int terms = f8 ? 1 : kMxTerms;
  CUtensorMap maps[8];  // weights, weight scales, token terms (3 box heights), token scales (3)
  bool ok = glu ? make_map_glu_interleaved(&maps[0], g.w, g.glu_h, kWRows / 32, true, f8)
                : make_map_fp4(&maps[0], g.w, kWRows, 128, true, f8);
  // decode (MXFP4 records): the three terms are a dimension of the maps, so that one load brings
  // a k-block of all three (their 8-row atoms term-major, as separate loads would place them);
  // the producer's issue rate, not HBM, had bounded the decode units at six loads per k-block
  const bool terms_dim = decode && !f8;
  const cuuint32_t sf_row = terms_dim ? MxCfg<16, false>::kSfRowBytes : 16;  // scale bytes of a row per stage
  for (int b = 0; b < 3; ++b) {  // the decode layout uses its one box size in all three slots
    const int rows_b = x_box_rows(unit_rows, b);
    if (terms_dim) {
      // token bytes {K/2, rows, 3 terms} (row stride: a record, term stride K/2): boxes {128, 8, 3}
      const cuuint64_t dims3[3] = {(cuuint64_t)(g.K / 2), (cuuint64_t)g.rows, (cuuint64_t)kMxTerms};
      const cuuint64_t strides3[2] = {(cuuint64_t)x_rec, (cuuint64_t)(g.K / 2)};
      const cuuint32_t box3[3] = {128, (cuuint32_t)rows_b, (cuuint32_t)kMxTerms};
      ok = ok && encode_u8(&maps[2 + b], g.x, 3, dims3, strides3, box3, true);
      // scale bytes {K/32, rows, 3 terms}: boxes {16, 16, 3}
      const cuuint64_t sdims3[3] = {(cuuint64_t)kscale, (cuuint64_t)g.rows, (cuuint64_t)kMxTerms};
      const cuuint64_t sstrides3[2] = {(cuuint64_t)x_rec, (cuuint64_t)kscale};
      const cuuint32_t sbox3[3] = {sf_row, (cuuint32_t)(2 * rows_b), (cuuint32_t)kMxTerms};
      ok = ok && encode_u8(&maps[5 + b], static_cast<const uint8_t*>(g.x) + mx3_scale_offset(g.K), 3, sdims3,
                           sstrides3, sbox3, false);
      continue;
    }
    // the token bytes of the records as a 2-D byte array {3 K/2 (MXFP8: K), rows}: boxes of 128 bytes
    const cuuint64_t dims[2] = {(cuuint64_t)(f8 ? g.K : kMxTerms * g.K / 2), (cuuint64_t)g.rows};
    const cuuint64_t strides[1] = {(cuuint64_t)x_rec};
    const cuuint32_t box[2] = {128, (cuuint32_t)rows_b};
    ok = ok && encode_u8(&maps[2 + b], g.x, 2, dims, strides, box, true);
    // the records' scale bytes {3 K/32, rows}: boxes of 16 bytes x (2 x the term box) rows
    const cuuint64_t sdims[2] = {(cuuint64_t)(terms * kscale), (cuuint64_t)g.rows};
    const cuuint32_t sbox[2] = {16, (cuuint32_t)(2 * rows_b)};
    ok = ok && encode_u8(&maps[5 + b],
                         static_cast<const uint8_t*>(g.x) + (f8 ? mx8_scale_offset(g.K) : mx3_scale_offset(g.K)), 2,
                         sdims, strides, sbox, false);
  }
  if (glu) {  // weight scales [E][2h][K/32] as {K/32, 16, 2, h/16, E}: the rows in the weights' order
    const int64_t h = g.glu_h;
    const cuuint64_t dims[5] = {(cuuint64_t)kscale, 16, 2, (cuuint64_t)(h / 16), (cuuint64_t)E};
    const cuuint64_t strides[4] = {(cuuint64_t)kscale, (cuuint64_t)(h * kscale), (cuuint64_t)(16 * kscale),
                                   (cuuint64_t)(2 * h * kscale)};
    const cuuint32_t box[5] = {sf_row, 16, 2, (cuuint32_t)(kWRows / 32), 1};
    ok = ok && encode_u8(&maps[1], g.w_scale, 5, dims, strides, box, false);
  } else {    // weight scales [E][rows][K/32]
    const cuuint64_t dims[3] = {(cuuint64_t)kscale, (cuuint64_t)g.w.rows, (cuuint64_t)E};
    const cuuint64_t strides[2] = {(cuuint64_t)kscale, (cuuint64_t)(g.w.rows * kscale)};
    const cuuint32_t box[3] = {sf_row, (cuuint32_t)kWRows, 1};
    ok = ok && encode_u8(&maps[1], g.w_scale, 3, dims, strides, box, false);
  }
  if (!ok) return cudaErrorInvalidValue;
  MxParams p = {};
  p.num_kb = g.K / KB;
  p.K = g.K;
  p.num_wt = glu ? g.glu_h / 128 : g.out_features / (2 * kWRows);
  p.glu_h = glu ? g.glu_h : 0;
  p.tiles = tiles;
  p.num_tiles = num_tiles;
  p.C = g.C;
  p.ldc = glu ? (f8 ? mx8_row_bytes(g.out_features) : mx3_row_bytes(g.out_features)) : g.ldc;
  p.out_k = g.out_features;
  p.row_scale = g.row_scale;
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.inject = inject;
  const long long items = (long long)max_tiles * p.num_wt;
  if (items == 0) return cudaSuccess;
  if (f8) {
    if (decode)
      return glu ? launch_mx_inst<true, 16, true>(maps, p, items, s) : launch_mx_inst<false, 16, true>(maps, p, items, s);
    return glu ? launch_mx_inst<true, 192, true>(maps, p, items, s) : launch_mx_inst<false, 192, true>(maps, p, items, s);
  }
  if (decode)
    return glu ? launch_mx_inst<true, 16, false>(maps, p, items, s) : launch_mx_inst<false, 16, false>(maps, p, items, s);
  return glu ? launch_mx_inst<true, 192, false>(maps, p, items, s) : launch_mx_inst<false, 192, false>(maps, p, items, s);
}

}  // namespace lmoe
