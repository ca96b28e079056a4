// Persistent GEMM on the 5th-generation tensor cores (tcgen05 + TMEM, operands staged by TMA)
// for every dense contraction of the layer: the router logits, W_down, the routed experts'
// gate/up and down projections (grouped by expert), the shared experts' gate/up, and the final
// GEMM that concatenates the shared experts' down projections with W_up along K (page "Lesson 6
// - LatentMoE", kimi-k3-course.pages.dev, eq. 11; section "Deriving the headline number" for
// the gate/up/down structure of an expert).
//
//   C[r][n] = epilogue( sum_c A[r][c] * B[n][c] ),  A, B K-major 16-bit, fp32 accumulation.
//
// CTA roles: warp 0 issues TMA loads (one thread), warp 1 owns TMEM and issues the MMAs (one
// thread), warps 2..5 drain the accumulator (tcgen05.ld) and run the epilogue.  Tiles are
// 128 x 256 x 64 with a multi-stage shared-memory ring and two TMEM accumulators, so the
// epilogue of one tile overlaps the main loop of the next.
//
// MXFP4 weights (B as E2M1 pairs + one E8M0 scale per 32 elements along K): TMA stages the
// packed bytes, and 16 converter warps turn each 256 x 64 block into fp16 with the hardware
// pair conversion (cvt.rn.f16x2.e2m1x2) times the block scale, writing the 128-byte-swizzled
// K-major layout the MMA reads; the MMA then runs kind::f16 with fp16 activations.  Values are
// exact: an E2M1 value times a power of two fits fp16 for scale exponents in [-24, 13].
//
// Every wait is bounded: on timeout the CTA flags the device status word and unwinds through
// the normal teardown (no trap, no hang).
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lmoe {
namespace {

using namespace tc;
constexpr int BM = 128;
constexpr int kBoxRows = 128;
constexpr uint32_t kBoxBytes = kBoxRows * BK * 2;  // 16 KB: one 128-row x 64-col 16-bit box
constexpr int kBaseThreads = 192;                   // producer, MMA, 4 epilogue warps

template <int BN, bool FP4B>
struct Cfg {
  static constexpr int kS1 = FP4B ? 5 : 4;                       // TMA ring stages
  static constexpr int kS2 = FP4B ? 3 : 0;                       // converted-B ring stages
  static constexpr uint32_t kABytes = BM * BK * 2;               // 16 KB
  static constexpr uint32_t kBBytes = BN * BK * 2;               // 32 KB (16-bit B tile)
  static constexpr uint32_t kBRawBytes = BN * BK / 2;            // 8 KB (packed E2M1)
  static constexpr uint32_t kStage1Bytes = kABytes + (FP4B ? kBRawBytes : kBBytes);
  static constexpr uint32_t kRing1 = kS1 * kStage1Bytes;
  static constexpr uint32_t kRing2 = kS2 * kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;                  // two fp32 accumulators
  static constexpr int kConvWarps = FP4B ? BN / 16 : 0;          // 2 * BN threads: one per (B row, K half)
  static constexpr int kRowsPerThread = FP4B ? 2 * BN / (32 * kConvWarps) : 0;
  static constexpr int kThreads = kBaseThreads + 32 * kConvWarps;
  static constexpr size_t kSmem = (size_t)kRing1 + kRing2 + 1024 + 512;
};

struct TcParams {
  int M, N;
  int num_kb, kb0, kb0_per_group;
  int a_kb_period;  // A's K coordinate repeats every a_kb_period k-blocks (K-concatenated B terms)
  int glu_h;
  int num_m_tiles, num_n_tiles;
  const int4* tiles;
  const int32_t* num_tiles;
  void* C;
  int64_t ldc;
  const float* row_scale;
  const uint8_t* b_scale;  // MXFP4 B: E8M0 [group][rows][K/32]
  int b_rows;              // MXFP4 B: rows per group
  uint32_t* status;
  uint64_t timeout_ns;
  int inject;
  // split-K (dense, few output tiles): k_splits ranges of kb_per_split k-blocks, raw fp32 accumulator
  // tiles to partial[split][row][n_tile * BN + c] (ldp columns, split_stride floats per split)
  int k_splits, kb_per_split;
  float* partial;
  int64_t ldp, split_stride;
};

struct Tile {
  int row0, row_end, n0, group;
  int kb_lo, kb_hi, split;
};

// Grouped mode: the tile-table entry of work item t, loaded one item ahead of its use so that no
// role waits on a global load between items ({expert, first m-tile, rows, first row}).
template <bool GROUPED>
__device__ __forceinline__ int4 tile_entry(const TcParams& p, int t) {
  return GROUPED ? p.tiles[t / p.num_n_tiles] : make_int4(0, 0, 0, 0);
}

template <int BN_OUT, bool GROUPED>
__device__ __forceinline__ Tile decode_tile(const TcParams& p, int t, int4 tl) {
  Tile ti;
  if (GROUPED) {
    const int mt = (tl.z + BM - 1) / BM;  // m-tiles of the expert
    const int local = t - tl.y * p.num_n_tiles;
    const int n = local / mt, m = local - n * mt;
    ti.row0 = tl.w + m * BM;
    ti.row_end = min(ti.row0 + BM, tl.w + tl.z);
    ti.n0 = n * BN_OUT;
    ti.group = tl.x;
    ti.kb_lo = 0;
    ti.kb_hi = p.num_kb;
    ti.split = 0;
  } else {
    const int mn = p.num_m_tiles * p.num_n_tiles;
    const int sp = t / mn, r = t - sp * mn;
    const int m = r % p.num_m_tiles, n = r / p.num_m_tiles;
    ti.row0 = m * BM;
    ti.row_end = min(ti.row0 + BM, p.M);
    ti.n0 = n * BN_OUT;
    ti.group = 0;
    ti.split = sp;
    ti.kb_lo = sp * p.kb_per_split;
    ti.kb_hi = min(p.num_kb, ti.kb_lo + p.kb_per_split);
  }
  return ti;
}

template <int BN, int EPI, bool GROUPED, bool AB_F16, bool FP4B, bool SPLIT = false>
__global__ void __launch_bounds__(Cfg<BN, FP4B>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const TcParams p) {
  using C = Cfg<BN, FP4B>;
  constexpr bool GLU = EPI == kEpiGluBF16 || EPI == kEpiGluF16;
  constexpr int BN_OUT = GLU ? BN / 2 : BN;
  constexpr int S1 = C::kS1, S2 = C::kS2 > 0 ? C::kS2 : 1;

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
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB0);
    ptx::prefetch_tmap(&tmB1);
  }
  if (warp == 1) ptx::tmem_alloc(tmem_holder, C::kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int total = (GROUPED ? *p.num_tiles : p.num_m_tiles * p.k_splits) * p.num_n_tiles;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    bool first = true;
    int4 entry = (int)blockIdx.x < total ? tile_entry<GROUPED>(p, blockIdx.x) : make_int4(0, 0, 0, 0);
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile ti = decode_tile<BN_OUT, GROUPED>(p, t, entry);
      if (t + (int)gridDim.x < total) entry = tile_entry<GROUPED>(p, t + gridDim.x);
      // K positions of k-block kb, advanced by counting (no division per k-block: the producer's
      // issue latency is on the pipeline's critical path): A's block ka wraps every a_kb_period;
      // non-GLU B is K-concatenated, groups of kb0_per_group blocks of B0 (offset goff, block kin
      // within it), then B1 from kb0 on.
      int ka = ti.kb_lo % p.a_kb_period;
      bool second = ti.kb_lo >= p.kb0;
      int goff = second ? 0 : ti.kb_lo / p.kb0_per_group;
      int kin = second ? ti.kb_lo - p.kb0 : ti.kb_lo - goff * p.kb0_per_group;
      const int grp = GLU ? ti.group + ti.n0 / p.glu_h : 0, j0 = GLU ? ti.n0 % p.glu_h : 0;
      for (int kb = ti.kb_lo; kb < ti.kb_hi; ++kb) {
        if (!ptx::mbar_wait_bounded(&empty1[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns, kWaitProducer)) goto done;
        const bool skip = p.inject && first && blockIdx.x == 0;  // test hook: drop one stage signal
        first = false;
        if (!skip) {
          uint8_t* sA = smem + stage * C::kStage1Bytes;
          uint8_t* sB = sA + C::kABytes;
          constexpr uint32_t kBoxB = FP4B ? kBoxRows * BK / 2 : kBoxBytes;  // bytes of one B box
          const int kx = FP4B ? kb * (BK / 2) : kb * BK;                     // B inner coordinate
          ptx::mbar_arrive_expect_tx(&full1[stage], C::kStage1Bytes);
          armed.arm(stage, phase);
          ptx::tma_load_3d(sA, &tmA, &full1[stage], ka * BK, ti.row0, 0);
          if (GLU) {
            ptx::tma_load_3d(sB, &tmB0, &full1[stage], kx, j0, grp);
            ptx::tma_load_3d(sB + kBoxB, &tmB0, &full1[stage], kx, p.glu_h + j0, grp);
          } else if (!second) {
            const int kin_el = kin * (FP4B ? BK / 2 : BK);
#pragma unroll
            for (int h = 0; h < BN / kBoxRows; ++h)
              ptx::tma_load_3d(sB + h * kBoxB, &tmB0, &full1[stage], kin_el, ti.n0 + h * kBoxRows, ti.group + goff);
          } else {
#pragma unroll
            for (int h = 0; h < BN / kBoxRows; ++h)
              ptx::tma_load_3d(sB + h * kBoxB, &tmB1, &full1[stage], kin * BK, ti.n0 + h * kBoxRows, 0);
          }
        }
        if (++ka == p.a_kb_period) ka = 0;
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
        if (++stage == S1) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = AB_F16 ? ptx::idesc_f16_f32(BM, BN) : ptx::idesc_bf16_f32(BM, BN);
    int s1 = 0, s2 = 0;
    uint32_t ph1 = 0, ph2 = 0;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      int kb_lo = 0, kb_hi = p.num_kb;
      if (!GROUPED) {
        const Tile ti = decode_tile<BN_OUT, GROUPED>(p, t, make_int4(0, 0, 0, 0));
        kb_lo = ti.kb_lo;
        kb_hi = ti.kb_hi;
      }
      if (!ptx::mbar_wait_bounded(&tmem_empty[acc], (use & 1u) ^ 1u, abort_flag, p.status, p.timeout_ns, kWaitAccFree))
        goto done;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (FP4B && !ptx::mbar_wait_bounded(&full2[s2], ph2, abort_flag, p.status, p.timeout_ns, kWaitConverted)) goto done;
        if (!ptx::mbar_wait_bounded(&full1[s1], ph1, abort_flag, p.status, p.timeout_ns, kWaitFull)) goto done;
        ptx::tc_fence_after();
        const uint32_t a_addr = ptx::smem_addr(smem + s1 * C::kStage1Bytes);
        const uint32_t b_addr = FP4B ? ptx::smem_addr(ring2 + s2 * C::kBBytes) : a_addr + C::kABytes;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          ptx::mma_f16(d_tmem, ptx::sw128_kmajor_desc(a_addr + kk * 32), ptx::sw128_kmajor_desc(b_addr + kk * 32),
                       idesc, (kb != kb_lo || kk != 0) ? 1u : 0u);
        ptx::mma_commit(&empty1[s1]);
        if (++s1 == S1) {
          s1 = 0;
          ph1 ^= 1u;
        }
        if (FP4B) {
          ptx::mma_commit(&empty2[s2]);
          if (++s2 == S2) {
            s2 = 0;
            ph2 ^= 1u;
          }
        }
      }
      ptx::mma_commit(&tmem_full[acc]);
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int it = 0;
    int4 entry = (int)blockIdx.x < total ? tile_entry<GROUPED>(p, blockIdx.x) : make_int4(0, 0, 0, 0);
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const Tile ti = decode_tile<BN_OUT, GROUPED>(p, t, entry);
      if (t + (int)gridDim.x < total) entry = tile_entry<GROUPED>(p, t + gridDim.x);
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      int ok = 1;
      if (lane == 0) ok = ptx::mbar_wait_bounded(&tmem_full[acc], use & 1u, abort_flag, p.status, p.timeout_ns, kWaitAccFull);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      const int row = ti.row0 + q * 32 + lane;
      const bool live = row < ti.row_end;
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (SPLIT)  // raw accumulator columns of n tile n0 / BN_OUT, reduced later in split order
        store_accumulator<BN, kEpiF32>(t_row, row, live, (ti.n0 / BN_OUT) * BN, (int)p.ldp,
                                       p.partial + (int64_t)ti.split * p.split_stride, p.ldp, nullptr);
      else
        store_accumulator<BN, EPI>(t_row, row, live, ti.n0, p.N, p.C, p.ldc, p.row_scale);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tmem_empty[acc]);
    }
  } else if (FP4B && warp >= 6) {
    // ------------------------------------------------------------------ E2M1 -> fp16 converters
    // Thread i converts one 32-element scale block (half i%2 of the k-block) of B rows i/2,
    // i/2 + 32 * kConvWarps / 2, ... (kRowsPerThread rows); consecutive threads read consecutive
    // 16-byte chunks.  Each k-block is handed to the MMA as soon as it is converted.
    constexpr int G = 1;
    constexpr int RPT = C::kRowsPerThread > 0 ? C::kRowsPerThread : 1;  // (instantiated only with FP4B)
    const int cid = threadIdx.x - kBaseThreads;  // 0 .. 32 * kConvWarps - 1
    const int half = cid & 1;
    int rows[RPT];
#pragma unroll
    for (int h = 0; h < RPT; ++h) rows[h] = (cid >> 1) + h * (16 * C::kConvWarps);
    const int kscale = p.num_kb * 2;  // E8M0 bytes per B row (K / 32)
    int s1 = 0, s2 = 0;
    uint32_t ph1 = 0, ph2 = 0;
    bool bad = false;
    int4 entry = (int)blockIdx.x < total ? tile_entry<GROUPED>(p, blockIdx.x) : make_int4(0, 0, 0, 0);
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile ti = decode_tile<BN_OUT, GROUPED>(p, t, entry);
      if (t + (int)gridDim.x < total) entry = tile_entry<GROUPED>(p, t + gridDim.x);
      const uint4* srow[RPT];
#pragma unroll
      for (int h = 0; h < RPT; ++h) {
        const int r = rows[h];
        int brow, bgrp;
        if (GLU) {
          bgrp = ti.group + ti.n0 / p.glu_h;
          const int j0 = ti.n0 % p.glu_h;
          brow = r < kBoxRows ? j0 + r : p.glu_h + j0 + (r - kBoxRows);
        } else {
          bgrp = ti.group;
          brow = ti.n0 + r;
        }
        srow[h] = reinterpret_cast<const uint4*>(p.b_scale + ((int64_t)bgrp * p.b_rows + brow) * kscale);
      }
      uint4 sc16[RPT];
      for (int kb0 = 0; kb0 < p.num_kb; kb0 += G) {  // num_kb % 8 == 0
        if ((kb0 & 7) == 0) {
#pragma unroll
          for (int h = 0; h < RPT; ++h) sc16[h] = __ldg(srow[h] + (kb0 >> 3));  // scales of 8 k-blocks
        }
        int gs1[G], gs2[G];
        uint32_t gp1[G], gp2[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          gs1[g] = s1;
          gp1[g] = ph1;
          gs2[g] = s2;
          gp2[g] = ph2;
          if (++s1 == S1) {
            s1 = 0;
            ph1 ^= 1u;
          }
          if (++s2 == S2) {
            s2 = 0;
            ph2 ^= 1u;
          }
        }
        int ok = 1;
        if (lane == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g)
            ok = ok && ptx::mbar_wait_bounded(&full1[gs1[g]], gp1[g], abort_flag, p.status, p.timeout_ns) &&
                 ptx::mbar_wait_bounded(&empty2[gs2[g]], gp2[g] ^ 1u, abort_flag, p.status, p.timeout_ns);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) goto conv_done;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int kb = kb0 + g;
          const int byte = (kb & 7) * 2 + half;  // scale index within the 16-byte vector
          const int wsel = byte >> 2;
#pragma unroll
          for (int h = 0; h < RPT; ++h) {
            const int r = rows[h];
            const uint4 qv =
                *reinterpret_cast<const uint4*>(smem + gs1[g] * C::kStage1Bytes + C::kABytes + r * (BK / 2) + half * 16);
            const uint32_t sw = wsel == 0 ? sc16[h].x : wsel == 1 ? sc16[h].y : wsel == 2 ? sc16[h].z : sc16[h].w;
            uint32_t o[16];
            e2m1x32_to_f16(qv, e8m0_to_f16x2((sw >> ((byte & 3) * 8)) & 0xFFu, &bad), o);
            uint8_t* dst = ring2 + gs2[g] * C::kBBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(dst + (((4 * half + c) ^ (r & 7)) << 4)) =
                  make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
          }
        }
        fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor cores
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) ptx::mbar_arrive(&full2[gs2[g]]);
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

template <int BN, int EPI, bool GROUPED, bool AB_F16, bool FP4B, bool SPLIT = false>
cudaError_t launch_inst(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const TcParams& p,
                        int grid, cudaStream_t s) {
  using C = Cfg<BN, FP4B>;
  auto kern = tc_gemm_kernel<BN, EPI, GROUPED, AB_F16, FP4B, SPLIT>;
  static PerDeviceValue attr_set;
  std::atomic<int>* set = attr_set.current();
  if (!set) return cudaErrorInvalidDevice;
  if (set->load(std::memory_order_acquire) == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    set->store(1, std::memory_order_release);
  }
  kern<<<grid, C::kThreads, C::kSmem, s>>>(a, b0, b1, p);
  return cudaGetLastError();
}

// Split-K reduction: out[row][f] = epilogue( sum over splits, in split order, of the partial
// accumulators ).  GLU outputs f read gate column (f / 128) * 256 + f % 128 and the up column 128
// to the right; the other epilogues read column f.  Four outputs per thread.
template <int EPI>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part, int splits,
                                                            int64_t split_stride, int64_t ldp, int M, int N,
                                                            void* __restrict__ C, int64_t ldc) {
  constexpr bool GLU = EPI == kEpiGluBF16 || EPI == kEpiGluF16;
  const int n4 = N / 4;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)M * n4) return;
  const int row = (int)(i / n4), f0 = (int)(i - (int64_t)row * n4) * 4;
  // the four outputs f0..f0+3 are adjacent partial columns (f0 % 4 == 0; GLU blocks of 128): one
  // 16-byte load per split (and one for the up half), eight splits in flight, added in split order
  const int64_t col = GLU ? (int64_t)(f0 / 128) * 256 + f0 % 128 : f0;
  const float* src = part + (int64_t)row * ldp + col;
  float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
  for (int sp0 = 0; sp0 < splits; sp0 += 8) {
    float4 a[8], b[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      a[q] = sp0 + q < splits ? *reinterpret_cast<const float4*>(src + (sp0 + q) * split_stride)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
      b[q] = GLU && sp0 + q < splits ? *reinterpret_cast<const float4*>(src + (sp0 + q) * split_stride + 128)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (sp0 + q < splits) {
        g[0] += a[q].x; g[1] += a[q].y; g[2] += a[q].z; g[3] += a[q].w;
        if (GLU) {
          u[0] += b[q].x; u[1] += b[q].y; u[2] += b[q].z; u[3] += b[q].w;
        }
      }
  }
  float v[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] = GLU ? silu(g[e]) * u[e] : g[e];
  if (EPI == kEpiF32) {
    *reinterpret_cast<float4*>(static_cast<float*>(C) + (int64_t)row * ldc + f0) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
    constexpr bool F16 = EPI == kEpiF16 || EPI == kEpiGluF16;
    const uint32_t a = F16 ? pack_f16x2(v[0], v[1]) : pack_bf16x2(v[0], v[1]);
    const uint32_t b = F16 ? pack_f16x2(v[2], v[3]) : pack_bf16x2(v[2], v[3]);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(C) + (int64_t)row * ldc + f0) = make_uint2(a, b);
  }
}

template <int EPI>
cudaError_t launch_split(const CUtensorMap& ma, const CUtensorMap& mb0, const CUtensorMap& mb1, const TcParams& p,
                         int grid, cudaStream_t s) {
  cudaError_t e = launch_inst<256, EPI, false, false, false, true>(ma, mb0, mb1, p, grid, s);
  if (e != cudaSuccess) return e;
  const int64_t n = (int64_t)p.M * (p.N / 4);
  splitk_reduce_kernel<EPI><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p.partial, p.k_splits, p.split_stride, p.ldp,
                                                                       p.M, p.N, p.C, p.ldc);
  return cudaGetLastError();
}

}  // namespace

size_t tc_splitk_partial_bytes(int num_sms) { return (size_t)num_sms * 256 * BM * sizeof(float); }

cudaError_t launch_tc_gemm(const TcGemm& g, uint32_t* status, uint64_t timeout_ns, int inject_fault, int num_sms,
                           cudaStream_t s) {
  const bool glu = g.epi == kEpiGluBF16 || g.epi == kEpiGluF16;
  const bool grouped = g.tiles != nullptr;
  const bool fp4 = g.b_scale != nullptr;
  const int bn = 256;
  const int bn_out = glu ? bn / 2 : bn;
  if (g.K % BK || g.k0_len % BK || g.k0_per_group % BK) return cudaErrorInvalidValue;
  if (glu ? g.N % bn_out : g.N % (g.epi == kEpiF32 ? 4 : 32)) return cudaErrorInvalidValue;
  const int a_period = g.a_k_period ? g.a_k_period : g.K;
  if (a_period % BK || g.K % a_period) return cudaErrorInvalidValue;
  if (fp4 && (!g.ab_f16 || g.B1.ptr || g.K % 512 || g.k0_len != g.K || g.k0_per_group != g.K))
    return cudaErrorInvalidValue;
  if (glu && g.glu_h % kBoxRows) return cudaErrorInvalidValue;
  CUtensorMap ma, mb0, mb1;
  if (!make_map(&ma, g.A)) return cudaErrorInvalidValue;
  if (!(fp4 ? make_map_fp4(&mb0, g.B0) : make_map(&mb0, g.B0))) return cudaErrorInvalidValue;
  if (g.B1.ptr) {
    if (!make_map(&mb1, g.B1)) return cudaErrorInvalidValue;
  } else {
    mb1 = mb0;
  }
  TcParams p = {};
  p.M = g.M;
  p.N = g.N;
  p.num_kb = g.K / BK;
  p.kb0 = g.k0_len / BK;
  p.kb0_per_group = g.k0_per_group / BK;
  p.a_kb_period = a_period / BK;
  p.glu_h = glu ? g.glu_h : 1;
  p.num_m_tiles = (g.M + BM - 1) / BM;
  p.num_n_tiles = (g.N + bn_out - 1) / bn_out;
  p.tiles = g.tiles;
  p.num_tiles = g.num_tiles;
  p.C = g.C;
  p.ldc = g.ldc;
  p.row_scale = g.row_scale;
  p.b_scale = g.b_scale;
  p.b_rows = (int)g.B0.rows;
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.inject = inject_fault;
  p.k_splits = 1;
  p.kb_per_split = p.num_kb;
  const long long tiles = grouped ? (long long)g.max_tiles * p.num_n_tiles : (long long)p.num_m_tiles * p.num_n_tiles;
  if (tiles == 0) return cudaSuccess;
  const int grid = (int)(tiles < num_sms ? tiles : num_sms);
  // At most half as many output tiles as SMs: split K so that tiles x splits fills the GPU.  The
  // split count depends on the tile count and K, so for one M tile (up to 128 rows) on N and K
  // only: every batch of up to 128 rows sums in the same order.
  int splits = 1;
  if (!grouped && !fp4 && !g.ab_f16 && g.partial && tiles * 2 <= num_sms && g.N % 4 == 0 &&
      (g.epi == kEpiBF16 || g.epi == kEpiF16 || g.epi == kEpiGluBF16 || g.epi == kEpiF32)) {
    splits = num_sms / (int)tiles;
    if (splits > p.num_kb / 4) splits = p.num_kb / 4;  // at least 4 k-blocks per split
    if (splits < 1) splits = 1;
  }
  const bool defer = g.defer && g.epi == kEpiF32;
  if (defer) g.defer->splits = 0;
  if (g.launch_count) *g.launch_count += splits > 1 && !defer ? 2 : 1;
  if (fp4) {
    if (!grouped) return cudaErrorInvalidValue;
    switch (g.epi) {
      case kEpiGluF16: return launch_inst<256, kEpiGluF16, true, true, true>(ma, mb0, mb1, p, grid, s);
      case kEpiScaleF16: return launch_inst<256, kEpiScaleF16, true, true, true>(ma, mb0, mb1, p, grid, s);
    }
    return cudaErrorInvalidValue;
  }
  if (g.ab_f16) return cudaErrorInvalidValue;  // fp16 operands only come with converted MXFP4 weights
  if (splits > 1) {
    p.kb_per_split = (p.num_kb + splits - 1) / splits;
    p.k_splits = (p.num_kb + p.kb_per_split - 1) / p.kb_per_split;
    p.partial = g.partial;
    p.ldp = (int64_t)p.num_n_tiles * 256;
    p.split_stride = (int64_t)p.num_m_tiles * BM * p.ldp;
    if ((size_t)p.k_splits * p.split_stride * sizeof(float) > g.partial_bytes) return cudaErrorInvalidValue;
    const long long work = tiles * p.k_splits;
    const int grid_s = (int)(work < num_sms ? work : num_sms);
    if (defer) {  // the consumer adds the partial sums
      *g.defer = SplitPartials{p.partial, p.k_splits, p.split_stride, p.ldp};
      return launch_inst<256, kEpiF32, false, false, false, true>(ma, mb0, mb1, p, grid_s, s);
    }
    switch (g.epi) {
      case kEpiBF16: return launch_split<kEpiBF16>(ma, mb0, mb1, p, grid_s, s);
      case kEpiF16: return launch_split<kEpiF16>(ma, mb0, mb1, p, grid_s, s);
      case kEpiGluBF16: return launch_split<kEpiGluBF16>(ma, mb0, mb1, p, grid_s, s);
      case kEpiF32: return launch_split<kEpiF32>(ma, mb0, mb1, p, grid_s, s);
    }
    return cudaErrorInvalidValue;
  }
  switch (g.epi) {
    case kEpiBF16:
      return grouped ? launch_inst<256, kEpiBF16, true, false, false>(ma, mb0, mb1, p, grid, s)
                     : launch_inst<256, kEpiBF16, false, false, false>(ma, mb0, mb1, p, grid, s);
    case kEpiF16:
      return grouped ? cudaErrorInvalidValue : launch_inst<256, kEpiF16, false, false, false>(ma, mb0, mb1, p, grid, s);
    case kEpiGluBF16:
      return grouped ? launch_inst<256, kEpiGluBF16, true, false, false>(ma, mb0, mb1, p, grid, s)
                     : launch_inst<256, kEpiGluBF16, false, false, false>(ma, mb0, mb1, p, grid, s);
    case kEpiScaleBF16:
      return grouped ? launch_inst<256, kEpiScaleBF16, true, false, false>(ma, mb0, mb1, p, grid, s)
                     : cudaErrorInvalidValue;
    case kEpiF32:
      return launch_inst<256, kEpiF32, false, false, false>(ma, mb0, mb1, p, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lmoe
