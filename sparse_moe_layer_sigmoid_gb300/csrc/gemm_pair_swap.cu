// Grouped expert GEMM on CTA pairs with swapped operands, for experts that receive many rows
// (prefill): the expert's weights are the M = 256 side of tcgen05.mma.cta_group::2 (128 weight
// rows in each CTA of the pair) and the expert's token rows are the N side.  Each expert's rows
// are cut into ceil(rows / 256) token tiles of equal width rounded up to 16, so an expert is
// padded by at most 15 rows per tile, where 256-row (or 128-row) M tiles of tokens pad it by up
// to 255 (127) rows (page "Lesson 6 - LatentMoE", kimi-k3-course.pages.dev, eq. 11: the routed
// experts' gate/up and down projections; section "Deriving the headline number" for their
// shapes).
//
//   D[f][j] = sum_c W_e[f][c] * X[row0 + j][c]     f: 256 weight rows, j < N token rows
//
// MMA operand split: A (weights) rows 0..127 come from the even CTA, 128..255 from the odd one;
// B (tokens) rows 0..N/2-1 from the even CTA and N/2..N-1 from the odd one; each CTA's TMEM
// receives its 128 weight rows x N token columns.
//
// Gate/up tiles hold 128 features (64 per CTA): in every 32-row quarter of a CTA's weights,
// rows 0..15 are gate rows and rows 16..31 the matching up rows, so one warp holds both halves
// of each GLU pair and combines them with a lane shuffle.  Down tiles hold 256 output features
// and scale each token column by its routing weight p.  The epilogue writes the transposed tile
// (token rows of the output) directly.
//
// Pipeline and cross-CTA protocol as in the CTA-pair GEMM: both CTAs' loads signal the even
// CTA's full[s]; the even CTA's MMA frees stages on its own empty[s] and its producer forwards
// each release to the odd CTA; accumulator-ready is forwarded by one even epilogue warp; all 8
// epilogue warps release accumulators on the even CTA.  Every wait is bounded.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lmoe {
namespace {

using namespace tc;
constexpr int kWRows = 128;                             // weight rows per CTA (M = 256 per pair)
constexpr int kMaxN = 256;                              // token columns per tile (MMA N)
constexpr uint32_t kWBytes = kWRows * BK * 2;           // 16 KB
constexpr uint32_t kXBytes = (kMaxN / 2) * BK * 2;      // 16 KB: 128 token rows per CTA, one box
constexpr uint32_t kStageBytes = kWBytes + kXBytes;     // 32 KB
constexpr int kStages = 6;
constexpr int kThreads = 192;                           // producer, MMA, 4 epilogue warps
constexpr uint32_t kTmemCols = 2 * kMaxN;               // two fp32 accumulators
constexpr uint32_t kStageOut = 32 * 32 * 2;             // per epilogue warp: 32 tokens x 32 bf16
constexpr size_t kSmem = (size_t)kStages * kStageBytes + 4 * kStageOut + 1024 + 512;

struct PSwapParams {
  int num_kb;        // 64-element k-blocks
  int num_wt;        // weight tiles per expert
  int glu_h;         // > 0: gate/up weights [2h][K], 128 features per tile; 0: 256 rows per tile
  const int4* tiles; // token tiles of 256 rows: {expert, first tile of expert, tiles of expert, first row}
  const int32_t* num_tiles;
  void* C;
  int64_t ldc;
  const float* row_scale;
  uint32_t* status;
  uint64_t timeout_ns;
  int inject;  // test hook: pair 0 skips its first stage (loads and signal) so a bounded wait runs out
};

struct PSwapTile {
  int expert, wt;
  int row0, nrows;  // the tile's token rows
  int n;            // MMA N: nrows rounded up to 16
};

// Work item t: expert-major, then weight tile, then token tile (consecutive items share the
// weight tile, so an expert's weights are read from HBM once and re-read from L2).  The table
// entry of item t is loaded one item ahead (pswap_entry) and decoded when the item starts, so
// no role waits on a global load between items.
__device__ __forceinline__ int4 pswap_entry(const PSwapParams& p, int t) { return p.tiles[t / p.num_wt]; }

__device__ __forceinline__ PSwapTile decode_pswap(const PSwapParams& p, int t, int4 tl) {
  const int rows = tl.z;
  const int ntiles = (rows + kMaxN - 1) / kMaxN;
  const int local = t - tl.y * p.num_wt;
  PSwapTile ti;
  ti.expert = tl.x;
  ti.wt = local / ntiles;
  const int j = local - ti.wt * ntiles;
  // ntiles = ceil(rows / 256) tiles of equal width (multiple of 16, at most 256): every tile has
  // at least one row because width * (ntiles - 1) <= 256 * (ntiles - 1) < rows
  const int width = ((rows + ntiles - 1) / ntiles + 15) & ~15;
  ti.row0 = tl.w + j * width;
  ti.nrows = min(width, rows - j * width);
  ti.n = (ti.nrows + 15) & ~15;
  return ti;
}

template <bool GLU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_pair_swap_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                        const PSwapParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // same offset in both CTAs
  uint8_t* out_stage = smem + kStages * kStageBytes;  // epilogue transposes, one per warp
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stage + 4 * kStageOut);
  uint64_t* empty = full + kStages;
  uint64_t* tmem_full = empty + kStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain_bar = tmem_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0: issues the MMAs; 1: partner
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  ptx::ArmedStages armed;  // even producer: stages armed (both halves' loads land on its full[s])

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tmem_full[a], 1);
      ptx::mbar_init(&tmem_empty[a], 8);  // 4 epilogue warps in each CTA of the pair
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
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
    int stage = 0, iter = 0;
    uint32_t phase = 0;
    bool first = true;
    int4 entry = pair < total ? pswap_entry(p, pair) : make_int4(0, 0, 0, 0);
    for (int t = pair; t < total; t += npairs) {
      const PSwapTile ti = decode_pswap(p, t, entry);
      if (t + npairs < total) entry = pswap_entry(p, t + npairs);
      // this CTA's token rows: N/2 from row0 + rank * N/2 (one 128-row box; rows past N/2 unused)
      const int xrow0 = ti.row0 + (int)rank * (ti.n >> 1);
      for (int kb = 0; kb < p.num_kb; ++kb, ++iter) {
        if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns, kWaitProducer))
          goto done;
        // the MMA read both CTAs' copy of this stage: pass the release on to the partner
        if (rank == 0 && iter >= kStages) ptx::mbar_arrive_remote(&empty[stage], 1);
        uint8_t* sW = smem + stage * kStageBytes;
        uint8_t* sX = sW + kWBytes;
        const uint32_t bar = ptx::mapa_shared(&full[stage], 0);  // the even CTA's full[stage]
        const bool skip = p.inject && first && pair == 0;  // test hook, the same in both CTAs
        first = false;
        if (!skip) {
          if (rank == 0) {
            ptx::mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes);
            armed.arm(stage, phase);
          }
          if (GLU) {  // 4 x (16 gate rows, 16 up rows) of features wt*128 + rank*64 ..
            ptx::tma_load_5d_pair(sW, &tmW, bar, kb * BK, 0, 0, (ti.wt * 128 + (int)rank * 64) / 16, ti.expert);
          } else {
            ptx::tma_load_3d_pair(sW, &tmW, bar, kb * BK, ti.wt * 2 * kWRows + (int)rank * kWRows, ti.expert);
          }
          ptx::tma_load_3d_pair(sX, &tmX, bar, kb * BK, xrow0, 0);
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc0 = ptx::idesc_bf16_f32(2 * kWRows, 0);
    int s = 0;
    uint32_t ph = 0;
    int it = 0;
    int4 entry = pair < total ? pswap_entry(p, pair) : make_int4(0, 0, 0, 0);
    for (int t = pair; t < total; t += npairs, ++it) {
      const PSwapTile ti = decode_pswap(p, t, entry);
      if (t + npairs < total) entry = pswap_entry(p, t + npairs);
      const uint32_t idesc = idesc0 | ((uint32_t)(ti.n >> 3) << 17);
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!ptx::mbar_wait_bounded(&tmem_empty[acc], (use & 1u) ^ 1u, abort_flag, p.status, p.timeout_ns,
                                  kWaitAccFree))
        goto done;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kMaxN);
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!ptx::mbar_wait_bounded(&full[s], ph, abort_flag, p.status, p.timeout_ns, kWaitFull)) goto done;
        ptx::tc_fence_after();
        const uint32_t w_addr = ptx::smem_addr(smem + s * kStageBytes);
        const uint32_t x_addr = w_addr + kWBytes;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          ptx::mma_f16_pair(d_tmem, ptx::sw128_kmajor_desc(w_addr + kk * 32), ptx::sw128_kmajor_desc(x_addr + kk * 32),
                            idesc, (kb | kk) != 0 ? 1u : 0u);
        ptx::mma_commit_pair(&empty[s]);
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      ptx::mma_commit_pair(&tmem_full[acc]);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue (both CTAs, transposed)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint16_t* out = static_cast<uint16_t*>(p.C);
    int it = 0;
    int4 entry = pair < total ? pswap_entry(p, pair) : make_int4(0, 0, 0, 0);
    for (int t = pair; t < total; t += npairs, ++it) {
      const PSwapTile ti = decode_pswap(p, t, entry);
      if (t + npairs < total) entry = pswap_entry(p, t + npairs);
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      // down x p: the item's row scales, lane l holding token 32 c + l, loaded while the
      // accumulator is still being computed
      float sc_reg[kMaxN / 32];
#pragma unroll
      for (int c = 0; c < kMaxN / 32; ++c) {
        const int jl = c * 32 + lane;
        sc_reg[c] = !GLU && jl < ti.nrows ? p.row_scale[ti.row0 + jl] : 0.0f;
      }
      int ok = 1;
      if (lane == 0) {
        ok = ptx::mbar_wait_bounded(&tmem_full[acc], use & 1u, abort_flag, p.status, p.timeout_ns, kWaitAccFull);
        if (ok && rank == 0 && warp == 2) ptx::mbar_arrive_remote(&tmem_full[acc], 1);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kMaxN);
      // This warp's output features: GLU 16 (lanes l and l+16 hold gate and up of feature l),
      // down 32.  Each 32-token chunk goes through shared memory as [token][feature] bf16 and
      // leaves in 16-byte stores.
      constexpr int FW = GLU ? 16 : 32;
      const int f0 = GLU ? ti.wt * 128 + (int)rank * 64 + 16 * q : ti.wt * 2 * kWRows + (int)rank * kWRows + 32 * q;
      uint16_t* st = reinterpret_cast<uint16_t*>(out_stage + q * kStageOut);
#pragma unroll
      for (int c = 0; c < kMaxN / 32; ++c) {
        const int c0 = c * 32;
        if (c0 >= ti.n) break;
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(t_row + c0, r);
        ptx::tmem_ld_wait();
        if (GLU) {
          // token pair (2i, 2i+1): lanes < 16 finish token 2i, lanes >= 16 token 2i+1
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float send = __uint_as_float(lane < 16 ? r[2 * i + 1] : r[2 * i]);
            const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
            const float g = lane < 16 ? __uint_as_float(r[2 * i]) : recv;
            const float u = lane < 16 ? recv : __uint_as_float(r[2 * i + 1]);
            st[(2 * i + (lane >> 4)) * FW + (lane & 15)] = __bfloat16_as_ushort(__float2bfloat16_rn(silu(g) * u));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float sc = __shfl_sync(0xffffffffu, sc_reg[c], i);
            st[i * FW + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[i]) * sc));
          }
        }
        __syncwarp();
        // 32 tokens x FW features = 32 * FW / 8 vectors of 16 bytes
#pragma unroll
        for (int v = lane; v < 32 * FW / 8; v += 32) {
          const int j = v / (FW / 8), part = v % (FW / 8);
          if (c0 + j < ti.nrows)
            *reinterpret_cast<uint4*>(out + (int64_t)(ti.row0 + c0 + j) * p.ldc + f0 + 8 * part) =
                *reinterpret_cast<const uint4*>(st + j * FW + 8 * part);
        }
        __syncwarp();
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
  if (*abort_flag) {  // the even CTA lets both halves' loads and its MMAs finish
    if (rank == 0 && warp == 0 && lane == 0) ptx::drain_armed(full, armed, p.timeout_ns);
    if (rank == 0 && warp == 1 && lane == 0) ptx::drain_mma_pair(drain_bar, p.timeout_ns);
    __syncthreads();
  }
  ptx::cluster_sync();  // the partner no longer reads this CTA's shared memory or signals it
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <bool GLU>
cudaError_t launch_pswap_inst(const CUtensorMap& w, const CUtensorMap& x, const PSwapParams& p, long long items,
                              cudaStream_t s) {
  auto kern = tc_pair_swap_kernel<GLU>;
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
  kern<<<2 * pairs, kThreads, kSmem, s>>>(w, x, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_pair_swap(const TcSwap& g, const int4* tiles_p, const int32_t* num_tiles_p, int max_tiles_p,
                                uint32_t* status, uint64_t timeout_ns, cudaStream_t s, int inject) {
  const bool glu = g.epi == kEpiGluBF16;
  if (g.epi != kEpiGluBF16 && g.epi != kEpiScaleBF16) return cudaErrorInvalidValue;
  if (g.w_scale || g.ab_f16 || g.K % BK || g.ldc % 8) return cudaErrorInvalidValue;
  if (glu ? (g.glu_h % 128 || g.out_features != g.glu_h) : g.out_features % (2 * kWRows))
    return cudaErrorInvalidValue;
  if (!tiles_p || !num_tiles_p) return cudaErrorInvalidValue;
  CUtensorMap mw, mx;
  if (!(glu ? make_map_glu_interleaved(&mw, g.w, g.glu_h, kWRows / 32) : make_map(&mw, g.w, kWRows)) ||
      !make_map(&mx, g.act, kMaxN / 2))
    return cudaErrorInvalidValue;
  PSwapParams p = {};
  p.num_kb = g.K / BK;
  p.num_wt = glu ? g.glu_h / 128 : g.out_features / (2 * kWRows);
  p.glu_h = glu ? g.glu_h : 0;
  p.tiles = tiles_p;
  p.num_tiles = num_tiles_p;
  p.C = g.C;
  p.ldc = g.ldc;
  p.row_scale = g.row_scale;
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.inject = inject;
  const long long items = (long long)max_tiles_p * p.num_wt;
  if (items == 0) return cudaSuccess;
  return glu ? launch_pswap_inst<true>(mw, mx, p, items, s) : launch_pswap_inst<false>(mw, mx, p, items, s);
}

}  // namespace lmoe
