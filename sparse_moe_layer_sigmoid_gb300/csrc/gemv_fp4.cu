// Routed experts with MXFP4 weights for expert batches of at most 4 token rows (decode), on
// the CUDA cores.  Such a batch is a matrix-vector product bound by reading the expert's weight
// bytes (page "What K3 actually is", srikanthmalla.com, first section: decode streams the
// active experts' weights; page "Lesson 6 - LatentMoE", kimi-k3-course.pages.dev, eq. 11 for the
// expert GLU and down projections).
//
//   gate/up: a[row][f] = SiLU(G_e[f] . x_row) * (U_e[f] . x_row)
//   down:    o[row][f] = p_row * (D_e[f] . a_row)
//
// Work item: (16-row unit of the dispatch's unit list with at most 4 rows, 32 weight rows:
// gate/up 16 features' gate and up rows, down 32 features).  One producer thread streams each
// item's whole weight rows and their E8M0 scale rows into a shared-memory ring with TMA (one box
// per 16 or 32 rows, each row read front to back), so a few hundred KB per SM are in flight
// without registers; 8 compute warps take 4 rows each, lane l the 32-element K blocks l, l+32,
// ..., reading 16-byte words of the staged rows.  Each CTA works through a contiguous range of
// items and stages a unit's token rows in shared memory once, each row scaled by a power of two
// 2^-s_t so that |x| <= 1.  Per K block, the unscaled E2M1 values (|q| <= 6, exact in fp16)
// times the scaled activations are summed in fp16 (16 products per half of an f16x2:
// |partial| <= 96, no overflow), widened to fp32 and accumulated times the block's E8M0 scale
// 2^(e-127) (exact in fp32); a warp butterfly reduces over lanes and the result is multiplied
// back by 2^s_t.  Units with more rows run on the tensor-core decode kernel.  Every wait is
// bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lmoe {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kThreads = 32 * (kComputeWarps + 1);  // + one producer warp
constexpr int kItemRows = 32;                       // weight rows per item
constexpr int kRowsPerWarp = kItemRows / kComputeWarps;
constexpr int kMaxChunks = 128;                     // 32-element K blocks: K <= 4096
constexpr int kJ = kMaxChunks / 32;
constexpr uint32_t kActBytes = 4 * kJ * 4 * 32 * 16;  // 32 KB: 4 token rows of up to 4096 fp16
constexpr int kMaxStages = 4;
constexpr uint32_t kSmemLimit = 227 * 1024;

struct GemvParams {
  int K;                  // reduction width (multiple of 512, at most 4096)
  int glu_h;              // > 0: gate rows f, up rows glu_h + f; 0: plain rows
  int feats_per_item;     // GLU 16, plain 32
  int num_fb;             // items per unit
  int w_rows;             // weight rows per expert
  int stages;             // ring depth
  uint32_t row_bytes;     // K / 2
  uint32_t srow_bytes;    // K / 32
  uint32_t stage_bytes;   // kItemRows * (row_bytes + srow_bytes)
  const __half* act;      // [rows][K] fp16
  const int4* tiles_s;    // {expert, first row, rows}
  const int32_t* num_tiles_s;
  __half* out;            // fp16 outputs
  int64_t ldc;
  const float* row_scale; // plain: routing weight per row
  uint32_t* status;
  uint64_t timeout_ns;
  int inject;             // test hook: CTA 0 skips its first stage (loads and signal)
};

// Activations in shared memory: token t, 16-byte quarter i of K block c = 32 j + l at
// [t][j][i][l], so lane l's loads of one quarter are consecutive 16-byte words.
__device__ __forceinline__ int act_index(int t, int j, int i, int l) { return ((t * kJ + j) * 4 + i) * 32 + l; }

__device__ __forceinline__ void e2m1x32_unscaled(const uint4& q, uint32_t (&o)[16]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o[4 * i]), "=r"(o[4 * i + 1]), "=r"(o[4 * i + 2]), "=r"(o[4 * i + 3])
        : "r"(w[i]));
  }
}

// Item it of a CTA's range: unit q (tiles_s entry) and feature block fb.
struct GemvItem {
  int q, fb;
};
__device__ __forceinline__ GemvItem gemv_item(const GemvParams& p, int it) {
  GemvItem g;
  g.q = it / p.num_fb;
  g.fb = it - g.q * p.num_fb;
  return g;
}

// Partial dot product of one 32-element K block: E2M1 weights wq (with E8M0 scale byte sc) against
// the NT staged token blocks xa, added to acc[t] (fp16 pair sums within the block, fp32 across).
// scmax tracks the largest scale byte seen (checked once per row group by the caller).
template <int NT>
__device__ __forceinline__ void block_dot(const uint4& wq, uint32_t sc, const uint32_t (&xa)[NT][16], float (&acc)[NT],
                                          uint32_t& scmax) {
  uint32_t q[16];
  e2m1x32_unscaled(wq, q);
  scmax = max(scmax, sc);
  const float scale = __uint_as_float(sc == 0u ? 0x00400000u : (sc << 23));  // 2^(e - 127)
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    __half2 s2 = __float2half2_rn(0.f);
#pragma unroll
    for (int k = 0; k < 16; ++k)
      s2 = __hfma2(*reinterpret_cast<const __half2*>(&q[k]), *reinterpret_cast<const __half2*>(&xa[t][k]), s2);
    const float2 f = __half22float2(s2);
    acc[t] = fmaf(f.x + f.y, scale, acc[t]);
  }
}

template <int NT>
__device__ __forceinline__ void load_act(const uint4* __restrict__ act_s, int t0, int j, int l, uint32_t (&xa)[NT][16]) {
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = act_s[act_index(t0 + t, j, i, l)];
      xa[t][4 * i] = v.x;
      xa[t][4 * i + 1] = v.y;
      xa[t][4 * i + 2] = v.z;
      xa[t][4 * i + 3] = v.w;
    }
}

// Dot products of the warp's staged weight rows (indices srow into the stage) with staged token
// rows t0 .. t0 + NT - 1.  Lane l takes the K blocks l, l + 32, ...; when K holds a half round of
// 16 blocks at the end (K = 3584: 112 blocks), the two half-warps split the rows there instead
// of leaving half the lanes idle: lanes 0-15 take rows 0 and 1, lanes 16-31 rows 2 and 3.
template <int NT>
__device__ __forceinline__ void warp_rows(const GemvParams& p, const uint8_t* __restrict__ wst,
                                          const uint8_t* __restrict__ sst, const uint4* __restrict__ act_s, int t0,
                                          const int (&srow)[kRowsPerWarp], int lane, float (&acc)[kRowsPerWarp][NT],
                                          bool& bad) {
  static_assert(kRowsPerWarp == 4, "the half-round split pairs rows 0-1 with 2-3");
  const int nchunks = p.K / 32;  // a multiple of 16 (K % 512 == 0)
  const int nfull = nchunks >> 5;
  uint32_t scmax = 0;
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
#pragma unroll 1
  for (int j = 0; j < nfull; ++j) {
    const int c = 32 * j + lane;
    uint32_t xa[NT][16];
    load_act<NT>(act_s, t0, j, lane, xa);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const uint4 wq = *reinterpret_cast<const uint4*>(wst + srow[r] * p.row_bytes + 16 * c);
      const uint32_t sc = (uint32_t)sst[srow[r] * p.srow_bytes + c];
      block_dot<NT>(wq, sc, xa, acc[r], scmax);
    }
  }
  if (nchunks & 31) {
    const int hl = lane & 15;
    const bool upper = lane >= 16;
    const int c = 32 * nfull + hl;
    uint32_t xa[NT][16];
    load_act<NT>(act_s, t0, nfull, hl, xa);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = upper ? srow[rr + 2] : srow[rr];
      const uint4 wq = *reinterpret_cast<const uint4*>(wst + row * p.row_bytes + 16 * c);
      const uint32_t sc = (uint32_t)sst[row * p.srow_bytes + c];
      float part[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) part[t] = upper ? acc[rr + 2][t] : acc[rr][t];
      block_dot<NT>(wq, sc, xa, part, scmax);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        acc[rr][t] = upper ? acc[rr][t] : part[t];
        acc[rr + 2][t] = upper ? part[t] : acc[rr + 2][t];
      }
    }
  }
  // scale bytes past 2^13 (and the NaN code 255) would leave fp16's range: a device check
  bad |= scmax > 127u + 13u;
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r][t] += __shfl_xor_sync(0xffffffffu, acc[r][t], off);
}

// One warp's share of an item: GLU features f0 + 2w, f0 + 2w + 1 (staged rows 2w, 2w + 1 are
// their gate rows, 16 + 2w, 16 + 2w + 1 their up rows); plain features f0 + 4w .. f0 + 4w + 3.
// Four token rows run as two passes of two (the weights are re-read from shared memory), which
// keeps the register count of the 4-row case at that of the 2-row case.
template <bool GLU, int NT>
__device__ __forceinline__ void item_rows(const GemvParams& p, const uint8_t* wst, const uint8_t* sst,
                                          const uint4* act_s, const float* tok_mul, int row0, int nrows, int fb,
                                          int warp, int lane, bool& bad) {
  int srow[kRowsPerWarp];
  int f0;
  if (GLU) {
    f0 = fb * p.feats_per_item + 2 * warp;
    srow[0] = 2 * warp;           // gate f0
    srow[1] = 16 + 2 * warp;      // up f0
    srow[2] = 2 * warp + 1;       // gate f0 + 1
    srow[3] = 16 + 2 * warp + 1;  // up f0 + 1
  } else {
    f0 = fb * p.feats_per_item + kRowsPerWarp * warp;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) srow[r] = kRowsPerWarp * warp + r;
  }
  constexpr int TP = NT > 2 ? 2 : NT;  // token rows per pass
#pragma unroll
  for (int t0 = 0; t0 < NT; t0 += TP) {
    float acc[kRowsPerWarp][TP];
    warp_rows<TP>(p, wst, sst, act_s, t0, srow, lane, acc, bad);
    // every lane holds every sum; lane (row or feature, token) of this pass writes one output
    const int r = lane >> 1, tt = lane & 1, t = t0 + tt;
    if (tt < TP && t < nrows) {
      if (GLU) {
        if (r < 2) {
          float g = 0.f, u = 0.f;
#pragma unroll
          for (int ff = 0; ff < 2; ++ff)
#pragma unroll
            for (int k = 0; k < TP; ++k)
              if (ff == r && k == tt) {
                g = acc[2 * ff][k];
                u = acc[2 * ff + 1][k];
              }
          g *= tok_mul[t];
          u *= tok_mul[t];
          p.out[(int64_t)(row0 + t) * p.ldc + f0 + r] = __float2half_rn(silu(g) * u);
        }
      } else if (r < kRowsPerWarp) {
        float v = 0.f;
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
          for (int k = 0; k < TP; ++k)
            if (rr == r && k == tt) v = acc[rr][k];
        p.out[(int64_t)(row0 + t) * p.ldc + f0 + r] = __float2half_rn(v * tok_mul[t] * p.row_scale[row0 + t]);
      }
    }
  }
}

// Barrier of the compute warps only (the producer warp runs ahead on its own).
__device__ __forceinline__ void compute_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(kComputeWarps * 32) : "memory");
}

template <bool GLU>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_fp4_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                    const GemvParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 127u) & ~127u) - raw);
  uint4* act_s = reinterpret_cast<uint4*>(smem);
  uint8_t* ring = smem + kActBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)p.stages * p.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  uint32_t* amax_bits = reinterpret_cast<uint32_t*>(empty + kMaxStages);
  float* tok_mul = reinterpret_cast<float*>(amax_bits + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tok_mul + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = *p.num_tiles_s * p.num_fb;
  const int per_cta = (total + gridDim.x - 1) / gridDim.x;
  const int it_begin = blockIdx.x * per_cta;
  const int it_end = min(total, it_begin + per_cta);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], kComputeWarps);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmS);
  }
  __syncthreads();

  if (warp == kComputeWarps) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool first = true;
      ptx::ArmedStages armed;
      for (int it = it_begin; it < it_end; ++it) {
        const GemvItem g = gemv_item(p, it);
        const int4 tl = p.tiles_s[g.q];
        if (tl.z > kGemvMaxRows) continue;  // the tensor-core kernel takes this unit
        if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns, kWaitProducer))
          break;
        const bool skip = p.inject && first && blockIdx.x == 0;  // test hook: drop one stage
        first = false;
        if (!skip) {
          uint8_t* wst = ring + (size_t)stage * p.stage_bytes;
          uint8_t* sst = wst + kItemRows * p.row_bytes;
          ptx::mbar_arrive_expect_tx(&full[stage], p.stage_bytes);
          armed.arm(stage, phase);
          const int base = tl.x * p.w_rows;  // first weight row of the expert
          const int f0 = g.fb * p.feats_per_item;
          if (GLU) {  // 16 gate rows, then the 16 matching up rows
            ptx::tma_load_3d(wst, &tmW, &full[stage], 0, 0, base + f0);
            ptx::tma_load_3d(wst + 16 * p.row_bytes, &tmW, &full[stage], 0, 0, base + p.glu_h + f0);
            ptx::tma_load_2d(sst, &tmS, &full[stage], 0, base + f0);
            ptx::tma_load_2d(sst + 16 * p.srow_bytes, &tmS, &full[stage], 0, base + p.glu_h + f0);
          } else {
            ptx::tma_load_3d(wst, &tmW, &full[stage], 0, 0, base + f0);
            ptx::tma_load_2d(sst, &tmS, &full[stage], 0, base + f0);
          }
        }
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // the CTA stays resident until its loads have landed (after an abort some were not
      // consumed; in a normal run every armed stage has already completed)
      ptx::drain_armed(full, armed, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------------ compute warps
    const int ctid = threadIdx.x;  // 0 .. 32 * kComputeWarps - 1
    const int vec_per_row = p.K / 8;
    bool bad = false;
    int staged = -1;
    int stage = 0;
    uint32_t phase = 0;
    for (int it = it_begin; it < it_end; ++it) {
      const GemvItem g = gemv_item(p, it);
      const int4 tl = p.tiles_s[g.q];
      const int nrows = tl.z;
      if (nrows > kGemvMaxRows) continue;
      if (g.q != staged) {
        // stage the unit's rows scaled by 2^-s_t, where 2^s_t > max |x_t|
        compute_barrier();
        if (ctid < 4) amax_bits[ctid] = 0u;
        compute_barrier();
        for (int t = 0; t < nrows; ++t) {
          const uint4* src = reinterpret_cast<const uint4*>(p.act + (int64_t)(tl.y + t) * p.K);
          float m = 0.f;
          for (int v = ctid; v < vec_per_row; v += kComputeWarps * 32) {
            const uint4 x = __ldg(src + v);
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&xs[k]));
              m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
          if (lane == 0) atomicMax(&amax_bits[t], __float_as_uint(m));
        }
        compute_barrier();
        if (ctid < 4) {
          const float m = __uint_as_float(amax_bits[ctid]);
          // power of two above m (1 for m == 0); x * 2^-s keeps x's fp16 bits for |x| >= 2^-10
          const int e = m > 0.f ? max(ilogbf(m) + 1, -14) : 0;
          tok_mul[ctid] = ldexpf(1.f, e);
        }
        compute_barrier();
        for (int t = 0; t < nrows; ++t) {
          const uint4* src = reinterpret_cast<const uint4*>(p.act + (int64_t)(tl.y + t) * p.K);
          const __half2 inv = __float2half2_rn(1.f / tok_mul[t]);  // power of two: exact
          for (int v = ctid; v < vec_per_row; v += kComputeWarps * 32) {
            uint4 x = __ldg(src + v);
            uint32_t* xs = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              __half2 h = __hmul2(*reinterpret_cast<__half2*>(&xs[k]), inv);
              xs[k] = *reinterpret_cast<uint32_t*>(&h);
            }
            const int c = v >> 2, i = v & 3;
            act_s[act_index(t, c >> 5, i, c & 31)] = x;
          }
        }
        compute_barrier();
        staged = g.q;
      }
      int ok = 1;
      if (lane == 0) ok = ptx::mbar_wait_bounded(&full[stage], phase, abort_flag, p.status, p.timeout_ns, kWaitFull);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const uint8_t* wst = ring + (size_t)stage * p.stage_bytes;
      const uint8_t* sst = wst + kItemRows * p.row_bytes;
      if (nrows == 1)
        item_rows<GLU, 1>(p, wst, sst, act_s, tok_mul, tl.y, nrows, g.fb, warp, lane, bad);
      else if (nrows == 2)
        item_rows<GLU, 2>(p, wst, sst, act_s, tok_mul, tl.y, nrows, g.fb, warp, lane, bad);
      else
        item_rows<GLU, 4>(p, wst, sst, act_s, tok_mul, tl.y, nrows, g.fb, warp, lane, bad);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[stage]);
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (bad) report(p.status, kStatusDeviceCheck);
  }
}

// Packed E2M1 weights [rows_total][K/2] viewed as {256 bytes, K/512, rows_total}: a box of
// {256, K/512, box_rows} brings box_rows whole rows, each contiguous in shared memory.
bool make_map_weight_rows(CUtensorMap* m, const void* ptr, int64_t rows_total, int64_t row_bytes, int box_rows) {
  tc::EncodeTiledFn enc = tc::encode_fn();
  if (!enc || !ptr || row_bytes % 256 || row_bytes / 256 > 256) return false;
  cuuint64_t dims[3] = {256, (cuuint64_t)(row_bytes / 256), (cuuint64_t)rows_total};
  cuuint64_t strides[2] = {256, (cuuint64_t)row_bytes};
  cuuint32_t box[3] = {256, (cuuint32_t)(row_bytes / 256), (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E8M0 scales [rows_total][K/32] as a 2-D map with boxes of box_rows whole scale rows.
bool make_map_scale_rows(CUtensorMap* m, const void* ptr, int64_t rows_total, int64_t srow_bytes, int box_rows) {
  tc::EncodeTiledFn enc = tc::encode_fn();
  if (!enc || !ptr || srow_bytes % 16 || srow_bytes > 256) return false;
  cuuint64_t dims[2] = {(cuuint64_t)srow_bytes, (cuuint64_t)rows_total};
  cuuint64_t strides[1] = {(cuuint64_t)srow_bytes};
  cuuint32_t box[2] = {(cuuint32_t)srow_bytes, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemv_fp4(const TcSwap& g, uint32_t* status, uint64_t timeout_ns, int num_sms, cudaStream_t s,
                            int inject) {
  const bool glu = g.epi == kEpiGluF16;
  if (!g.w_scale || (g.epi != kEpiGluF16 && g.epi != kEpiScaleF16)) return cudaErrorInvalidValue;
  if (g.K % 512 || g.K > kMaxChunks * 32 || g.ldc <= 0) return cudaErrorInvalidValue;
  const int feats = glu ? kItemRows / 2 : kItemRows;
  if (g.out_features % feats || (glu && g.glu_h != g.out_features)) return cudaErrorInvalidValue;
  GemvParams p = {};
  p.K = g.K;
  p.glu_h = glu ? g.glu_h : 0;
  p.feats_per_item = feats;
  p.num_fb = g.out_features / feats;
  p.w_rows = (int)g.w.rows;
  p.row_bytes = (uint32_t)(g.K / 2);
  p.srow_bytes = (uint32_t)(g.K / 32);
  p.stage_bytes = kItemRows * (p.row_bytes + p.srow_bytes);
  const uint32_t avail = kSmemLimit - kActBytes - 256 - 128;
  p.stages = (int)(avail / p.stage_bytes);
  if (p.stages > kMaxStages) p.stages = kMaxStages;
  if (p.stages < 2) return cudaErrorInvalidValue;
  p.act = static_cast<const __half*>(g.act.ptr);
  p.tiles_s = g.tiles_s;
  p.num_tiles_s = g.num_tiles_s;
  p.out = static_cast<__half*>(g.C);
  p.ldc = g.ldc;
  p.row_scale = g.row_scale;
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.inject = inject;
  const int64_t rows_total = g.w.depth * g.w.rows;
  CUtensorMap mw, ms;
  if (!make_map_weight_rows(&mw, g.w.ptr, rows_total, p.row_bytes, glu ? kItemRows / 2 : kItemRows) ||
      !make_map_scale_rows(&ms, g.w_scale, rows_total, p.srow_bytes, glu ? kItemRows / 2 : kItemRows))
    return cudaErrorInvalidValue;
  const long long items = (long long)g.max_tiles_s * p.num_fb;
  if (items == 0) return cudaSuccess;
  const int grid = (int)(items < num_sms ? items : num_sms);
  const size_t smem = kActBytes + (size_t)p.stages * p.stage_bytes + 256 + 128;
  auto kern = glu ? gemv_fp4_kernel<true> : gemv_fp4_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, s>>>(mw, ms, p);
  return cudaGetLastError();
}

}  // namespace lmoe
