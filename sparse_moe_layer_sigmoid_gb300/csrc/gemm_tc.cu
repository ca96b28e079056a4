// Persistent bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM, operands staged by
// TMA) for every dense contraction of the layer: W_down, the routed experts' gate/up and down
// projections (grouped by expert), the shared experts' gate/up, and the final GEMM that
// concatenates the shared experts' down projections with W_up along K (page "Lesson 6 -
// LatentMoE", kimi-k3-course.pages.dev, eq. 11; section "Deriving the headline number" for
// the gate/up/down structure of an expert).
//
//   C[r][n] = epilogue( sum_c A[r][c] * B[n][c] ),  A, B bf16 K-major, fp32 accumulation.
//
// CTA = 6 warps: warp 0 issues TMA loads (one thread), warp 1 owns TMEM and issues the MMAs
// (one thread), warps 2..5 drain the accumulator (tcgen05.ld) and run the epilogue.  Tiles are
// 128 x BN x 64 (BN = 256 or 128) with a 4..6-stage shared-memory ring and two TMEM
// accumulators, so the epilogue of one tile overlaps the main loop of the next.  Every wait is
// bounded: on timeout the CTA flags the device status word and unwinds (no trap, no hang).
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace lmoe {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int kThreads = 192;
constexpr int kBoxRows = 128;
constexpr uint32_t kBoxBytes = kBoxRows * BK * 2;  // 16 KB: one 128-row x 64-col bf16 box

template <int BN>
struct Cfg {
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr uint32_t kABytes = BM * BK * 2;
  static constexpr uint32_t kBBytes = BN * BK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;  // two fp32 accumulators of BN columns
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + 1024 + 256;
};

struct TcParams {
  int M, N;
  int num_kb, kb0, kb0_per_group;
  int a_kb_period;  // A's K coordinate repeats every a_kb_period k-blocks (K-concatenated B terms)
  int glu_h;
  int num_m_tiles, num_n_tiles;
  const int4* tiles;
  const int32_t* num_tiles;
  const int32_t* offsets;
  void* C;
  int64_t ldc;
  const float* row_scale;
  uint32_t* status;
  uint64_t timeout_ns;
  int inject;
};

struct Tile {
  int row0, row_end, n0, group;
};

template <int BN_OUT, bool GROUPED>
__device__ __forceinline__ Tile decode_tile(const TcParams& p, int t) {
  Tile ti;
  if (GROUPED) {
    const int q = t / p.num_n_tiles;
    const int4 tl = p.tiles[q];
    const int local = t - tl.y * p.num_n_tiles;
    const int n = local / tl.z, m = local - n * tl.z;
    ti.row0 = p.offsets[tl.x] + m * BM;
    ti.row_end = min(ti.row0 + BM, p.offsets[tl.x + 1]);
    ti.n0 = n * BN_OUT;
    ti.group = tl.x;
  } else {
    const int m = t % p.num_m_tiles, n = t / p.num_m_tiles;
    ti.row0 = m * BM;
    ti.row_end = min(ti.row0 + BM, p.M);
    ti.n0 = n * BN_OUT;
    ti.group = 0;
  }
  return ti;
}

template <int BN, int EPI, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const TcParams p) {
  using C = Cfg<BN>;
  constexpr bool GLU = EPI == kEpiGluBF16;
  constexpr int BN_OUT = GLU ? BN / 2 : BN;
  constexpr int S = C::kStages;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * C::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* tmem_full = empty + S;
  uint64_t* tmem_empty = tmem_full + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tmem_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tmem_full[a], 1);
      ptx::mbar_init(&tmem_empty[a], 4);
    }
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

  const int total = (GROUPED ? *p.num_tiles : p.num_m_tiles) * p.num_n_tiles;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    bool first = true;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile ti = decode_tile<BN_OUT, GROUPED>(p, t);
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns)) goto done;
        const bool skip = p.inject && first && blockIdx.x == 0;  // test hook: drop one stage signal
        first = false;
        if (!skip) {
          uint8_t* sA = smem + stage * C::kStageBytes;
          uint8_t* sB = sA + C::kABytes;
          ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          ptx::tma_load_3d(sA, &tmA, &full[stage], (kb % p.a_kb_period) * BK, ti.row0, 0);
          if (GLU) {
            const int grp = ti.group + ti.n0 / p.glu_h, j0 = ti.n0 % p.glu_h;
            ptx::tma_load_3d(sB, &tmB0, &full[stage], kb * BK, j0, grp);
            ptx::tma_load_3d(sB + kBoxBytes, &tmB0, &full[stage], kb * BK, p.glu_h + j0, grp);
          } else if (kb < p.kb0) {
            const int goff = kb / p.kb0_per_group, kin = (kb - goff * p.kb0_per_group) * BK;
#pragma unroll
            for (int h = 0; h < BN / kBoxRows; ++h)
              ptx::tma_load_3d(sB + h * kBoxBytes, &tmB0, &full[stage], kin, ti.n0 + h * kBoxRows,
                               ti.group + goff);
          } else {
            const int kin = (kb - p.kb0) * BK;
#pragma unroll
            for (int h = 0; h < BN / kBoxRows; ++h)
              ptx::tma_load_3d(sB + h * kBoxBytes, &tmB1, &full[stage], kin, ti.n0 + h * kBoxRows, 0);
          }
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!ptx::mbar_wait_bounded(&tmem_empty[acc], (use & 1u) ^ 1u, abort_flag, p.status, p.timeout_ns))
        goto done;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!ptx::mbar_wait_bounded(&full[stage], phase, abort_flag, p.status, p.timeout_ns)) goto done;
        ptx::tc_fence_after();
        const uint32_t a_addr = ptx::smem_addr(smem + stage * C::kStageBytes);
        const uint32_t b_addr = a_addr + C::kABytes;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          ptx::mma_f16(d_tmem, ptx::sw128_kmajor_desc(a_addr + kk * 32), ptx::sw128_kmajor_desc(b_addr + kk * 32),
                       idesc, (kb | kk) != 0 ? 1u : 0u);
        ptx::mma_commit(&empty[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      ptx::mma_commit(&tmem_full[acc]);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const Tile ti = decode_tile<BN_OUT, GROUPED>(p, t);
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      int ok = 1;
      if (lane == 0) ok = ptx::mbar_wait_bounded(&tmem_full[acc], use & 1u, abort_flag, p.status, p.timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      const int row = ti.row0 + q * 32 + lane;
      const bool live = row < ti.row_end;
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (GLU) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.ldc + ti.n0;
#pragma unroll 1
        for (int c = 0; c < BN_OUT; c += 32) {
          uint32_t g[32], u[32];
          ptx::tmem_ld_32x32b_x32(t_row + c, g);
          ptx::tmem_ld_32x32b_x32(t_row + BN_OUT + c, u);
          ptx::tmem_ld_wait();
          if (live) {
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
              const float a1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
              packed[i] = pack_bf16x2(a0, a1);
            }
            uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
          }
        }
      } else {
        const float sc = (EPI == kEpiScaleBF16 && live) ? p.row_scale[row] : 1.0f;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          if (ti.n0 + c >= p.N) break;  // ragged last column tile (fp32: N % 4 == 0, else N % 32 == 0)
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(t_row + c, r);
          ptx::tmem_ld_wait();
          if (live) {
            if (EPI == kEpiF32) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(p.C) + (int64_t)row * p.ldc + ti.n0 + c);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (ti.n0 + c + 4 * i < p.N) dst[i] = make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
            } else {
              uint32_t packed[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                packed[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * sc, __uint_as_float(r[2 * i + 1]) * sc);
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.ldc +
                                                    ti.n0 + c);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tmem_empty[acc]);
    }
  }
done:
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const TcOperand& op) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !op.ptr) return false;
  const int64_t depth_stride = op.depth > 1 ? op.depth_stride : op.rows * op.row_stride;
  cuuint64_t dims[3] = {(cuuint64_t)op.cols, (cuuint64_t)op.rows, (cuuint64_t)op.depth};
  cuuint64_t strides[2] = {(cuuint64_t)op.row_stride * 2, (cuuint64_t)depth_stride * 2};
  cuuint32_t box[3] = {BK, kBoxRows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(op.ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int EPI, bool GROUPED>
cudaError_t launch_inst(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const TcParams& p,
                        int grid, cudaStream_t s) {
  auto kern = tc_gemm_kernel<BN, EPI, GROUPED>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<BN>::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<grid, kThreads, Cfg<BN>::kSmem, s>>>(a, b0, b1, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_gemm(const TcGemm& g, uint32_t* status, uint64_t timeout_ns, int inject_fault, int num_sms,
                           cudaStream_t s) {
  const bool glu = g.epi == kEpiGluBF16;
  const bool grouped = g.tiles != nullptr;
  const int bn = 256;
  const int bn_out = glu ? bn / 2 : bn;
  if (g.K % BK || g.k0_len % BK || g.k0_per_group % BK) return cudaErrorInvalidValue;
  if (glu ? g.N % bn_out : g.N % (g.epi == kEpiF32 ? 4 : 32)) return cudaErrorInvalidValue;
  const int a_period = g.a_k_period ? g.a_k_period : g.K;
  if (a_period % BK || g.K % a_period) return cudaErrorInvalidValue;
  if (glu && g.glu_h % kBoxRows) return cudaErrorInvalidValue;
  CUtensorMap ma, mb0, mb1;
  if (!make_map(&ma, g.A) || !make_map(&mb0, g.B0)) return cudaErrorInvalidValue;
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
  p.offsets = g.offsets;
  p.C = g.C;
  p.ldc = g.ldc;
  p.row_scale = g.row_scale;
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.inject = inject_fault;
  const long long tiles = grouped ? (long long)g.max_tiles * p.num_n_tiles : (long long)p.num_m_tiles * p.num_n_tiles;
  if (tiles == 0) return cudaSuccess;
  const int grid = (int)(tiles < num_sms ? tiles : num_sms);
  switch (g.epi) {
    case kEpiBF16:
      return grouped ? launch_inst<256, kEpiBF16, true>(ma, mb0, mb1, p, grid, s)
                     : launch_inst<256, kEpiBF16, false>(ma, mb0, mb1, p, grid, s);
    case kEpiGluBF16:
      return grouped ? launch_inst<256, kEpiGluBF16, true>(ma, mb0, mb1, p, grid, s)
                     : launch_inst<256, kEpiGluBF16, false>(ma, mb0, mb1, p, grid, s);
    case kEpiScaleBF16:
      return grouped ? launch_inst<256, kEpiScaleBF16, true>(ma, mb0, mb1, p, grid, s)
                     : launch_inst<256, kEpiScaleBF16, false>(ma, mb0, mb1, p, grid, s);
    case kEpiF32:
      return launch_inst<256, kEpiF32, false>(ma, mb0, mb1, p, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lmoe
