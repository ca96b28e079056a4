// Paired-CTA persistent GEMM on the 5th-generation tensor cores for the dense 16-bit
// contractions with many rows: W_down, the shared experts' gate/up and the final GEMM of the
// layer (page "Lesson 6 - LatentMoE", kimi-k3-course.pages.dev, eq. 11).
//
//   C[r][n] = epilogue( sum_c A[r][c] * B[n][c] ),  A, B bf16 K-major, fp32 accumulation.
//
// Two CTAs of a cluster (a CTA pair on two SMs) share one 256 x 256 output tile: the even CTA
// issues tcgen05.mma.cta_group::2 with M = 256, which reads A rows 0..127 and B rows 0..127 from
// its own shared memory and A rows 128..255 and B rows 128..255 from its partner's, and writes
// each CTA's 128 rows of D into that CTA's TMEM.  Each CTA therefore stages 32 KB per 64-wide
// k-block (its A rows and half of B) instead of the 48 KB a single-CTA 128 x 256 tile needs: a
// third less L2->SM traffic per FLOP and a deeper ring (6 stages) in the same shared memory.
//
// Protocol (all waits bounded; on timeout the status word is flagged and the CTA unwinds):
//   * both CTAs' TMA loads signal the even CTA's full[s] (cp.async.bulk.tensor .cta_group::2);
//     the even CTA's producer posts the expected bytes of both halves;
//   * the even CTA's MMA commits stage release to its own empty[s]; its producer, on seeing the
//     release, forwards one arrival to the odd CTA's empty[s] before refilling;
//   * the MMA commits accumulator-ready to the even CTA's tmem_full[a]; one even epilogue warp
//     forwards it to the odd CTA; all 8 epilogue warps of the pair release the accumulator on
//     the even CTA's tmem_empty[a].
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lmoe {
namespace {

using namespace tc;
constexpr int kRows = 128;                          // A rows and B rows each CTA stages
constexpr int BN = 256;                             // output columns of a pair tile (before GLU)
constexpr uint32_t kHalfBytes = kRows * BK * 2;     // 16 KB: one 128-row x 64-col bf16 box
constexpr uint32_t kStageBytes = 2 * kHalfBytes;    // this CTA's A rows + its half of B
constexpr int kStages = 6;
constexpr int kThreads = 192;                       // producer, MMA, 4 epilogue warps
constexpr uint32_t kTmemCols = 2 * BN;              // two fp32 accumulators
constexpr size_t kSmem = (size_t)kStages * kStageBytes + 1024 + 512;

struct PairParams {
  int M, N;
  int num_kb, kb0, kb0_per_group;
  int a_kb_period;  // A's K coordinate repeats every a_kb_period k-blocks (K-concatenated B terms)
  int glu_h;
  int num_m_tiles, num_n_tiles;  // 256-row tiles, 256-column (GLU: 128-output) tiles
  void* C;
  int64_t ldc;
  const float* row_scale;
  uint32_t* status;
  uint64_t timeout_ns;
  int inject;  // test hook: pair 0 skips its first stage (loads and signal) so a bounded wait runs out
};

struct PairTile {
  int row0, row_end, n0, group;  // row0: first of the tile's 256 rows
};

template <int BN_OUT>
__device__ __forceinline__ PairTile decode_pair_tile(const PairParams& p, int t) {
  PairTile ti;
  const int m = t % p.num_m_tiles, n = t / p.num_m_tiles;
  ti.row0 = m * kTileP;
  ti.row_end = min(ti.row0 + kTileP, p.M);
  ti.n0 = n * BN_OUT;
  ti.group = 0;
  return ti;
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const PairParams p) {
  constexpr bool GLU = EPI == kEpiGluBF16;
  constexpr int BN_OUT = GLU ? BN / 2 : BN;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // same offset in both CTAs
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
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
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB0);
    ptx::prefetch_tmap(&tmB1);
  }
  if (warp == 1) ptx::tmem_alloc_pair(tmem_holder, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before any signal crosses the pair
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int total = p.num_m_tiles * p.num_n_tiles;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    int stage = 0, iter = 0;
    uint32_t phase = 0;
    // Boxes of k-block kb: A rows row0 + rank*128 at K block ka; this CTA's half of B (the even
    // CTA takes B rows n0..n0+127 or, for GLU, the gate rows; the odd CTA the next 128 rows or
    // the matching up rows).  Non-GLU B is K-concatenated: groups of kb0_per_group k-blocks of
    // B0 (group offset goff, block kin within it), then B1 from kb0 on.  The K positions advance
    // by counting, with no division per k-block: the producer's issue latency is on the
    // pipeline's critical path.
    constexpr bool PERIODIC = EPI == kEpiF32;  // the router's terms: A's K wraps every a_kb_period
    bool first = true;
    for (int t = pair; t < total; t += npairs) {
      const PairTile ti = decode_pair_tile<BN_OUT>(p, t);
      const int ay = ti.row0 + (int)rank * kRows;
      const int by = GLU ? (int)rank * p.glu_h + ti.n0 % p.glu_h : ti.n0 + (int)rank * kRows;
      const int bz_glu = ti.group + ti.n0 / p.glu_h;
      int ka = 0, goff = 0, kin = 0;
      bool second = p.kb0 == 0;
      for (int kb = 0; kb < p.num_kb; ++kb, ++iter) {
        if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns, kWaitProducer))
          goto done;
        // the MMA read both CTAs' copy of this stage: pass the release on to the partner
        if (rank == 0 && iter >= kStages) ptx::mbar_arrive_remote(&empty[stage], 1);
        uint8_t* sA = smem + stage * kStageBytes;
        const uint32_t bar = ptx::mapa_shared(&full[stage], 0);  // the even CTA's full[stage]
        const bool skip = p.inject && first && pair == 0;  // test hook, the same in both CTAs
        first = false;
        if (!skip) {
          if (rank == 0) {
            ptx::mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes);
            armed.arm(stage, phase);
          }
          ptx::tma_load_3d_pair(sA, &tmA, bar, ka * BK, ay, 0);
          if (GLU)
            ptx::tma_load_3d_pair(sA + kHalfBytes, &tmB0, bar, kb * BK, by, bz_glu);
          else
            ptx::tma_load_3d_pair(sA + kHalfBytes, second ? &tmB1 : &tmB0, bar, kin * BK, by,
                                  second ? 0 : ti.group + goff);
        }
        if (PERIODIC) {
          if (++ka == p.a_kb_period) ka = 0;
        } else {
          ++ka;
        }
        if (!GLU) {
          if (!second && kb + 1 == p.kb0) {
            second = true;
            kin = 0;
          } else if (!second && ++kin == p.kb0_per_group) {
            kin = 0;
            ++goff;
          } else if (second) {
            ++kin;
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
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(2 * kRows, BN);
    int s = 0;
    uint32_t ph = 0;
    int it = 0;
    for (int t = pair; t < total; t += npairs, ++it) {
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!ptx::mbar_wait_bounded(&tmem_empty[acc], (use & 1u) ^ 1u, abort_flag, p.status, p.timeout_ns,
                                        kWaitAccFree))
        goto done;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!ptx::mbar_wait_bounded(&full[s], ph, abort_flag, p.status, p.timeout_ns, kWaitFull)) goto done;
        ptx::tc_fence_after();
        const uint32_t a_addr = ptx::smem_addr(smem + s * kStageBytes);
        const uint32_t b_addr = a_addr + kHalfBytes;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          ptx::mma_f16_pair(d_tmem, ptx::sw128_kmajor_desc(a_addr + kk * 32), ptx::sw128_kmajor_desc(b_addr + kk * 32),
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
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int it = 0;
    for (int t = pair; t < total; t += npairs, ++it) {
      const PairTile ti = decode_pair_tile<BN_OUT>(p, t);
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      int ok = 1;
      if (lane == 0) {
        ok = ptx::mbar_wait_bounded(&tmem_full[acc], use & 1u, abort_flag, p.status, p.timeout_ns,
                                          kWaitAccFull);
        if (ok && rank == 0 && warp == 2) ptx::mbar_arrive_remote(&tmem_full[acc], 1);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      const int row = ti.row0 + (int)rank * kRows + q * 32 + lane;
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      store_accumulator<BN, EPI>(t_row, row, row < ti.row_end, ti.n0, p.N, p.C, p.ldc, p.row_scale);
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

template <int EPI>
cudaError_t launch_inst(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const PairParams& p,
                        long long pair_tiles, cudaStream_t s) {
  auto kern = tc_pair_kernel<EPI>;
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
  const int pairs = (int)(pair_tiles < max_pairs ? pair_tiles : max_pairs);
  kern<<<2 * pairs, kThreads, kSmem, s>>>(a, b0, b1, p);
  return cudaGetLastError();
}

}  // namespace

bool tc_pair_supported(const TcGemm& g) {
  const bool glu = g.epi == kEpiGluBF16;
  if (g.tiles || g.b_scale || g.ab_f16) return false;
  if (g.epi != kEpiBF16 && g.epi != kEpiGluBF16 && g.epi != kEpiF32) return false;
  const int a_period = g.a_k_period ? g.a_k_period : g.K;
  if (g.K % BK || g.k0_len % BK || g.k0_per_group % BK || a_period % BK || g.K % a_period) return false;
  if (a_period != g.K && g.epi != kEpiF32) return false;  // a periodic A only with the fp32 epilogue
  if (glu) return g.N % (BN / 2) == 0 && g.glu_h % kRows == 0;
  return g.N % (g.epi == kEpiF32 ? 4 : 32) == 0;
}

cudaError_t launch_tc_pair(const TcGemm& g, uint32_t* status, uint64_t timeout_ns, cudaStream_t s, int inject) {
  if (!tc_pair_supported(g)) return cudaErrorInvalidValue;
  const bool glu = g.epi == kEpiGluBF16;
  const int bn_out = glu ? BN / 2 : BN;
  CUtensorMap ma, mb0, mb1;
  if (!make_map(&ma, g.A) || !make_map(&mb0, g.B0)) return cudaErrorInvalidValue;
  if (g.B1.ptr) {
    if (!make_map(&mb1, g.B1)) return cudaErrorInvalidValue;
  } else {
    mb1 = mb0;
  }
  PairParams p = {};
  p.M = g.M;
  p.N = g.N;
  p.num_kb = g.K / BK;
  p.kb0 = g.k0_len / BK;
  p.kb0_per_group = g.k0_per_group / BK;
  p.a_kb_period = (g.a_k_period ? g.a_k_period : g.K) / BK;
  p.glu_h = glu ? g.glu_h : 1;
  p.num_m_tiles = (g.M + kTileP - 1) / kTileP;
  p.num_n_tiles = (g.N + bn_out - 1) / bn_out;
  p.C = g.C;
  p.ldc = g.ldc;
  p.row_scale = g.row_scale;
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.inject = inject;
  const long long tiles = (long long)p.num_m_tiles * p.num_n_tiles;
  if (tiles == 0) return cudaSuccess;
  switch (g.epi) {
    case kEpiGluBF16: return launch_inst<kEpiGluBF16>(ma, mb0, mb1, p, tiles, s);
    case kEpiF32: return launch_inst<kEpiF32>(ma, mb0, mb1, p, tiles, s);
    default: return launch_inst<kEpiBF16>(ma, mb0, mb1, p, tiles, s);
  }
}

}  // namespace lmoe
