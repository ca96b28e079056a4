// Grouped expert GEMM for experts that receive few rows (decode-sized batches): the roles of
// the operands are swapped, so that the expert's weights fill the 128-row M side of the
// tcgen05 MMA and the expert's token rows are the N side (a multiple of 16), instead of a
// 128-row token tile that is almost empty (page "What K3 actually is", srikanthmalla.com,
// first section: decode is bound by reading the active expert weights).
//
//   D[f][j] = sum_c W_e[f][c] * X[row_j][c]     (f: 128 weight rows, j: the unit's token rows)
//
// Gate/up tiles hold 64 features: in every 32-row quarter of the M side, rows 0..15 are gate
// rows and rows 16..31 the matching up rows, so one warp holds both halves of each GLU pair
// and combines them with a lane shuffle.  Down tiles hold 128 output features and scale each
// token column by its routing weight p.
//
// MXFP4 weights stream as 256-element super-blocks (128 contiguous bytes per weight row, 16 KB
// per stage, stored with the 128-byte swizzle) and are converted to fp16 in 64-element
// sub-blocks by 8 converter warps (hardware E2M1 pair conversion times the E8M0 block scale),
// each handed to the MMA as soon as it is ready.  bf16 weights go to the MMA straight from TMA,
// 64 elements per stage.  A unit is one entry of the dispatch's 16-row tile list (an expert's
// rows in groups of at most 16), so decode batches run N = 16 MMAs.  Every wait is bounded.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lmoe {
namespace {

using namespace tc;

constexpr int kWRows = 128;  // weight rows per tile (MMA M)
constexpr int kBox = 16;     // rows per TMA box (weights and tokens)
constexpr int kBase = 192;   // producer, MMA, 4 epilogue warps

template <bool FP4W>
struct SwapCfg {
  static constexpr int kSub = FP4W ? 4 : 1;                 // 64-element sub-blocks per TMA stage
  static constexpr int kMaxN = kTileS;                      // token rows per unit (16-row tile list)
  static constexpr int kS1 = FP4W ? 4 : 10;
  static constexpr int kS2 = FP4W ? 8 : 1;
  static constexpr uint32_t kAConvBytes = kWRows * BK * 2;  // 16 KB 16-bit A sub-tile
  static constexpr uint32_t kWStageBytes = FP4W ? kWRows * BK * kSub / 2 : kAConvBytes;  // 16 KB
  static constexpr uint32_t kXSubBytes = kMaxN * BK * 2;    // token sub-tile (2 KB)
  static constexpr uint32_t kStage1Bytes = kWStageBytes + kSub * kXSubBytes;  // 24 KB or 18 KB
  static constexpr uint32_t kRing1 = kS1 * kStage1Bytes;
  static constexpr uint32_t kRing2 = FP4W ? kS2 * kAConvBytes : 0;
  static constexpr uint32_t kTmemCols = 32;                 // two accumulators of kMaxN columns
  static constexpr int kConvWarps = FP4W ? 8 : 0;
  static constexpr int kThreads = kBase + 32 * kConvWarps;
  static constexpr size_t kSmem = (size_t)kRing1 + kRing2 + 1024 + 512;
};

struct SwapParams {
  int num_kb;  // 64-element k-blocks
  int num_wt;  // weight tiles per expert
  int glu_h;   // > 0: gate/up weights [2h][K] (64 features per tile); 0: plain rows (128 per tile)
  int w_rows;  // weight rows per expert
  const int4* tiles_s;  // {expert, first row, rows}
  const int32_t* num_tiles_s;
  int skip_rows_upto;   // units with at most this many rows belong to another kernel
  void* C;
  int64_t ldc;
  const float* row_scale;
  const uint8_t* w_scale;
  uint32_t* status;
  uint64_t timeout_ns;
  int inject;  // test hook: CTA 0 skips its first stage (loads and signal) so a bounded wait runs out
};

struct SwapTile {
  int expert, row0, nrows, nb, wt;
};

__device__ __forceinline__ SwapTile decode_swap(const SwapParams& p, int u) {
  SwapTile t;
  const int q = u / p.num_wt;
  t.wt = u - q * p.num_wt;
  const int4 tl = p.tiles_s[q];
  t.expert = tl.x;
  t.row0 = tl.y;
  t.nrows = tl.z;
  t.nb = 1;
  return t;
}

// Weight row (within the expert) held by M-side row r of tile wt.
__device__ __forceinline__ int weight_row(const SwapParams& p, int wt, int r) {
  if (p.glu_h > 0) {
    const int qq = r >> 5, w = r & 31;
    const int j = wt * 64 + 16 * qq + (w & 15);
    return w < 16 ? j : p.glu_h + j;
  }
  return wt * kWRows + r;
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

template <bool GLU, bool OUT_F16, bool AB_F16, bool FP4W>
__global__ void __launch_bounds__(SwapCfg<FP4W>::kThreads, 1)
    tc_swap_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const SwapParams p) {
  using C = SwapCfg<FP4W>;
  constexpr int S1 = C::kS1, S2 = C::kS2, SUB = C::kSub, MAXN = C::kMaxN;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* ring2 = smem + C::kRing1;
  uint64_t* full1 = reinterpret_cast<uint64_t*>(ring2 + C::kRing2);
  uint64_t* empty1 = full1 + S1;
  uint64_t* full2 = empty1 + S1;
  uint64_t* empty2 = full2 + S2;
  uint64_t* tmem_full = empty2 + S2;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain_bar = tmem_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ptx::ArmedStages armed;  // producer: ring stages with loads issued (teardown after an abort)
  if (threadIdx.x == 0) {
    for (int s = 0; s < S1; ++s) {
      ptx::mbar_init(&full1[s], 1);
      ptx::mbar_init(&empty1[s], 1);
    }
    for (int s = 0; s < S2; ++s) {
      ptx::mbar_init(&full2[s], C::kConvWarps > 0 ? C::kConvWarps : 1);
      ptx::mbar_init(&empty2[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tmem_full[a], 1);
      ptx::mbar_init(&tmem_empty[a], 4);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
  }
  if (warp == 1) ptx::tmem_alloc(tmem_holder, C::kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = *p.num_tiles_s * p.num_wt;
  const int num_st = p.num_kb / SUB;  // TMA stages per unit

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    bool first = true;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const SwapTile ti = decode_swap(p, u);
      if (ti.nrows <= p.skip_rows_upto) continue;
      const uint32_t tx = C::kWStageBytes + (uint32_t)SUB * C::kXSubBytes;
      for (int st = 0; st < num_st; ++st) {
        if (!ptx::mbar_wait_bounded(&empty1[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns, kWaitProducer)) goto done;
        const bool skip = p.inject && first && blockIdx.x == 0;  // test hook: drop one stage
        first = false;
        if (!skip) {
          uint8_t* sW = smem + stage * C::kStage1Bytes;
          uint8_t* sX = sW + C::kWStageBytes;
          ptx::mbar_arrive_expect_tx(&full1[stage], tx);
          armed.arm(stage, phase);
          const int kx = FP4W ? st * (BK * SUB / 2) : st * BK;  // bytes (packed) or elements
          // weights: one box of 128 rows (gate/up: 4 x (16 gate rows, 16 up rows) of features wt*64..)
          if (GLU)
            ptx::tma_load_5d(sW, &tmW, &full1[stage], kx, 0, 0, ti.wt * 4, ti.expert);
          else
            ptx::tma_load_3d(sW, &tmW, &full1[stage], kx, ti.wt * kWRows, ti.expert);
          // tokens: the unit's 16 rows for the stage's SUB 64-column blocks, one box
          ptx::tma_load_3d(sX, &tmX, &full1[stage], 0, ti.row0, st * SUB);
        }
        if (++stage == S1) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc0 = AB_F16 ? ptx::idesc_f16_f32(kWRows, 0) : ptx::idesc_bf16_f32(kWRows, 0);
    int s1 = 0, s2 = 0;
    uint32_t ph1 = 0, ph2 = 0;
    int it = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const SwapTile ti = decode_swap(p, u);
      if (ti.nrows <= p.skip_rows_upto) continue;
      const uint32_t idesc = idesc0 | ((uint32_t)((ti.nb * kBox) >> 3) << 17);  // N = 16 * nb
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      ++it;
      if (!ptx::mbar_wait_bounded(&tmem_empty[acc], (use & 1u) ^ 1u, abort_flag, p.status, p.timeout_ns, kWaitAccFree))
        goto done;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * MAXN);
      for (int st = 0; st < num_st; ++st) {
        if (!ptx::mbar_wait_bounded(&full1[s1], ph1, abort_flag, p.status, p.timeout_ns, kWaitFull)) goto done;
        const uint32_t st_addr = ptx::smem_addr(smem + s1 * C::kStage1Bytes);
#pragma unroll
        for (int sb = 0; sb < SUB; ++sb) {
          if (FP4W && !ptx::mbar_wait_bounded(&full2[s2], ph2, abort_flag, p.status, p.timeout_ns, kWaitConverted)) goto done;
          ptx::tc_fence_after();
          const uint32_t a_addr = FP4W ? ptx::smem_addr(ring2 + s2 * C::kAConvBytes) : st_addr;
          const uint32_t b_addr = st_addr + C::kWStageBytes + sb * C::kXSubBytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            ptx::mma_f16(d_tmem, ptx::sw128_kmajor_desc(a_addr + kk * 32),
                         ptx::sw128_kmajor_desc(b_addr + kk * 32), idesc, (st | sb | kk) != 0 ? 1u : 0u);
          if (FP4W) {
            ptx::mma_commit(&empty2[s2]);
            if (++s2 == S2) {
              s2 = 0;
              ph2 ^= 1u;
            }
          }
        }
        ptx::mma_commit(&empty1[s1]);
        if (++s1 == S1) {
          s1 = 0;
          ph1 ^= 1u;
        }
      }
      ptx::mma_commit(&tmem_full[acc]);
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------------ epilogue (transposed)
    const int q = warp & 3;
    int it = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const SwapTile ti = decode_swap(p, u);
      if (ti.nrows <= p.skip_rows_upto) continue;
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      ++it;
      int ok = 1;
      if (lane == 0) ok = ptx::mbar_wait_bounded(&tmem_full[acc], use & 1u, abort_flag, p.status, p.timeout_ns, kWaitAccFull);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * MAXN);
      uint16_t* out = static_cast<uint16_t*>(p.C);
      const int col = GLU ? ti.wt * 64 + 16 * q + (lane & 15) : ti.wt * kWRows + 32 * q + lane;
      for (int ch = 0; ch < ti.nb; ++ch) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(t_row + ch * kBox, r);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kBox; ++i) {
          const int j = ch * kBox + i;
          if (j < ti.nrows) {  // uniform across the warp
            const int row = ti.row0 + j;
            const float v = __uint_as_float(r[i]);
            float o;
            bool write;
            if (GLU) {
              const float up = __shfl_down_sync(0xffffffffu, v, 16);
              o = silu(v) * up;
              write = lane < 16;
            } else {
              o = v * p.row_scale[row];
              write = true;
            }
            if (write) {
              const uint32_t bits = OUT_F16 ? (uint32_t)__half_as_ushort(__float2half_rn(o))
                                            : (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(o));
              out[(int64_t)row * p.ldc + col] = (uint16_t)bits;
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tmem_empty[acc]);
    }
  } else if (FP4W && warp >= 6) {
    // ------------------------------------------------------------------ E2M1 -> fp16 converters
    const int cid = threadIdx.x - kBase;  // 0..255
    const int r = cid >> 1, half = cid & 1;
    const int kscale = p.num_kb * 2;     // E8M0 bytes per weight row
    int s1 = 0, s2 = 0;
    uint32_t ph1 = 0, ph2 = 0;
    bool bad = false;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const SwapTile ti = decode_swap(p, u);
      if (ti.nrows <= p.skip_rows_upto) continue;
      const int wrow = weight_row(p, ti.wt, r);
      const uint4* srow =
          reinterpret_cast<const uint4*>(p.w_scale + ((int64_t)ti.expert * p.w_rows + wrow) * kscale);
      uint4 sc16 = make_uint4(0, 0, 0, 0);
      for (int st = 0; st < num_st; ++st) {
        if ((st & 1) == 0) sc16 = __ldg(srow + (st >> 1));  // scales of 2 stages (512 elements)
        // each 64-element sub-block is handed to the MMA as soon as it is converted
        int ok = 1;
        if (lane == 0) ok = ptx::mbar_wait_bounded(&full1[s1], ph1, abort_flag, p.status, p.timeout_ns);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) goto conv_done;
#pragma unroll
        for (int sb = 0; sb < SUB; ++sb) {
          ok = 1;
          if (lane == 0) ok = ptx::mbar_wait_bounded(&empty2[s2], ph2 ^ 1u, abort_flag, p.status, p.timeout_ns);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) goto conv_done;
          {
            // raw rows are 128 bytes with the 128-byte swizzle: chunk j of row r sits at j ^ (r % 8)
            const int chunk = 2 * sb + half;
            const uint4 qv =
                *reinterpret_cast<const uint4*>(smem + s1 * C::kStage1Bytes + r * 128 + ((chunk ^ (r & 7)) << 4));
            const int byte = 8 * (st & 1) + chunk;  // scale index within the 16-byte vector
            const int wsel = byte >> 2;
            const uint32_t sw = wsel == 0 ? sc16.x : wsel == 1 ? sc16.y : wsel == 2 ? sc16.z : sc16.w;
            uint32_t o[16];
            e2m1x32_to_f16(qv, e8m0_to_f16x2((sw >> ((byte & 3) * 8)) & 0xFFu, &bad), o);
            uint8_t* dst = ring2 + s2 * C::kAConvBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(dst + (((4 * half + c) ^ (r & 7)) << 4)) =
                  make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&full2[s2]);
          if (++s2 == S2) {
            s2 = 0;
            ph2 ^= 1u;
          }
        }
        if (++s1 == S1) {
          s1 = 0;
          ph1 ^= 1u;
        }
      }
    }
  conv_done:
    if (bad) report(p.status, kStatusDeviceCheck);
  }
done:
  ptx::tc_fence_before();
  __syncthreads();  // every role has left its loop; the abort flag no longer changes
  if (*abort_flag) {  // let the loads and MMAs in flight finish before the CTA lets go of them
    if (warp == 0 && lane == 0) ptx::drain_armed(full1, armed, p.timeout_ns);
    if (warp == 1 && lane == 0) ptx::drain_mma(drain_bar, p.timeout_ns);
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <bool GLU, bool OUT_F16, bool AB_F16, bool FP4W>
cudaError_t launch_swap_inst(const CUtensorMap& w, const CUtensorMap& x, const SwapParams& p, int grid,
                             cudaStream_t s) {
  using C = SwapCfg<FP4W>;
  auto kern = tc_swap_kernel<GLU, OUT_F16, AB_F16, FP4W>;
  static PerDeviceValue attr_set;
  std::atomic<int>* set = attr_set.current();
  if (!set) return cudaErrorInvalidDevice;
  if (set->load(std::memory_order_acquire) == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    set->store(1, std::memory_order_release);
  }
  kern<<<grid, C::kThreads, C::kSmem, s>>>(w, x, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_swap(const TcSwap& g, uint32_t* status, uint64_t timeout_ns, int num_sms, cudaStream_t s,
                           int inject) {
  const bool glu = g.epi == kEpiGluBF16 || g.epi == kEpiGluF16;
  const bool out_f16 = g.epi == kEpiGluF16 || g.epi == kEpiScaleF16;
  const bool fp4 = g.w_scale != nullptr;
  if (g.K % BK || (fp4 && g.K % 512)) return cudaErrorInvalidValue;
  if (glu ? (g.glu_h % 64 || g.out_features != g.glu_h) : g.out_features % kWRows) return cudaErrorInvalidValue;
  if (fp4 && !g.ab_f16) return cudaErrorInvalidValue;
  CUtensorMap mw, mx;
  const bool wmap = glu ? make_map_glu_interleaved(&mw, g.w, g.glu_h, kWRows / 32, fp4)
                        : (fp4 ? make_map_fp4(&mw, g.w, kWRows, BK * SwapCfg<true>::kSub / 2, /*swizzle128=*/true)
                               : make_map(&mw, g.w, kWRows));
  if (!wmap) return cudaErrorInvalidValue;
  if (!make_map_kslabs(&mx, g.act, kBox, fp4 ? SwapCfg<true>::kSub : SwapCfg<false>::kSub)) return cudaErrorInvalidValue;
  SwapParams p = {};
  p.num_kb = g.K / BK;
  p.num_wt = glu ? g.glu_h / 64 : g.out_features / kWRows;
  p.glu_h = glu ? g.glu_h : 0;
  p.w_rows = (int)g.w.rows;
  p.tiles_s = g.tiles_s;
  p.num_tiles_s = g.num_tiles_s;
  p.skip_rows_upto = g.skip_rows_upto;
  p.C = g.C;
  p.ldc = g.ldc;
  p.row_scale = g.row_scale;
  p.w_scale = g.w_scale;
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.inject = inject;
  const long long units = (long long)g.max_tiles_s * p.num_wt;
  if (units == 0) return cudaSuccess;
  const int grid = (int)(units < num_sms ? units : num_sms);
  if (fp4) {
    return glu ? launch_swap_inst<true, true, true, true>(mw, mx, p, grid, s)
               : launch_swap_inst<false, true, true, true>(mw, mx, p, grid, s);
  }
  if (g.ab_f16 || out_f16) return cudaErrorInvalidValue;
  return glu ? launch_swap_inst<true, false, false, false>(mw, mx, p, grid, s)
             : launch_swap_inst<false, false, false, false>(mw, mx, p, grid, s);
}

}  // namespace lmoe
