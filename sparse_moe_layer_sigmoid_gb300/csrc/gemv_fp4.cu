// Routed experts with MXFP4 weights for expert batches of at most 4 token rows (decode), on
// the CUDA cores.  Such a batch is a matrix-vector product bound by reading the expert's weight
// bytes (page "What K3 actually is", srikanthmalla.com, first section: decode streams the
// active experts' weights; page "Lesson 6 - LatentMoE", kimi-k3-course.pages.dev, eq. 11 for the
// expert GLU and down projections), so the weights stream straight from HBM with coalesced
// 16-byte loads and are used once per token row.
//
//   gate/up: a[row][f] = SiLU(G_e[f] . x_row) * (U_e[f] . x_row)
//   down:    o[row][f] = p_row * (D_e[f] . a_row)
//
// Work item: (16-row unit of the dispatch's unit list with at most 4 rows, block of features);
// each CTA takes a contiguous range of items, so it stages a unit's token rows in shared memory
// once for many items, each row scaled by a power of two 2^-s_t with |x| <= 1 after scaling.
// Each warp takes 4 weight rows (gate/up: 2 features, their gate and up rows), lane l the
// 32-element K blocks l, l+32, l+64, l+96.  Per block, the unscaled
// E2M1 values (|q| <= 6, exact in fp16) times the scaled activations are summed in fp16 (16
// products per half of an f16x2: |partial| <= 96, no overflow), the partial is widened to fp32
// and accumulated times the block's E8M0 scale 2^(e-127) (exact in fp32).  A warp butterfly
// reduces over lanes; the result is multiplied back by 2^s_t.  Units with more rows run on the
// tensor-core decode kernel.
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace lmoe {
namespace {

constexpr int kThreads = 256;      // 8 warps
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = 4;    // weight rows per warp per item
constexpr int kMaxChunks = 128;    // 32-element K blocks: K <= 4096
constexpr int kJ = kMaxChunks / 32;

struct GemvParams {
  int K;                  // reduction width (multiple of 32, at most 4096)
  int glu_h;              // > 0: gate rows f, up rows glu_h + f; 0: plain rows
  int feats_per_item;     // features per item: GLU 2 per warp, plain 4 per warp
  int num_fb;             // feature blocks per unit
  int w_rows;             // weight rows per expert
  const uint8_t* w;       // [E][w_rows][K/2]
  const uint8_t* ws;      // [E][w_rows][K/32]
  const __half* act;      // [rows][K] fp16
  const int4* tiles_s;    // {expert, first row, rows}
  const int32_t* num_tiles_s;
  __half* out;            // fp16 outputs
  int64_t ldc;
  const float* row_scale; // plain: routing weight per row
  uint32_t* status;
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

// One warp: dot products of R weight rows with NT staged token rows.
template <int NT, int R>
__device__ __forceinline__ void warp_rows(const GemvParams& p, const uint4* __restrict__ act_s, int expert,
                                          const int* wrow, int lane, float (&acc)[R][NT], bool& bad) {
  const int nchunks = p.K / 32;
  const int nj = (nchunks + 31) / 32;
  const size_t row_bytes = (size_t)p.K / 2;
  const uint8_t* wrow_ptr[R];
  const uint8_t* srow_ptr[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const size_t rbase = (size_t)expert * p.w_rows + wrow[r];
    wrow_ptr[r] = p.w + rbase * row_bytes;
    srow_ptr[r] = p.ws + rbase * nchunks;
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
  }
  // weights of K block j + 1 are in flight while block j is used
  uint4 wq[R], wn[R];
  uint32_t sc[R], sn[R];
  {
    const bool live0 = lane < nchunks;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      wq[r] = live0 ? __ldg(reinterpret_cast<const uint4*>(wrow_ptr[r]) + lane) : make_uint4(0, 0, 0, 0);
      sc[r] = live0 ? (uint32_t)__ldg(srow_ptr[r] + lane) : 127u;
    }
  }
#pragma unroll 1
  for (int j = 0; j < nj; ++j) {
    const int c = 32 * j + lane;
    const bool live = c < nchunks;
    const int cn = c + 32;
    const bool live_n = j + 1 < nj && cn < nchunks;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      wn[r] = live_n ? __ldg(reinterpret_cast<const uint4*>(wrow_ptr[r]) + cn) : make_uint4(0, 0, 0, 0);
      sn[r] = live_n ? (uint32_t)__ldg(srow_ptr[r] + cn) : 127u;
    }
    uint32_t xa[NT][16];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // blocks past the end of K were never staged: zero, not stale bits (0 * inf = NaN)
        const uint4 v = live ? act_s[act_index(t, j, i, lane)] : make_uint4(0, 0, 0, 0);
        xa[t][4 * i] = v.x;
        xa[t][4 * i + 1] = v.y;
        xa[t][4 * i + 2] = v.z;
        xa[t][4 * i + 3] = v.w;
      }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      uint32_t q[16];
      e2m1x32_unscaled(wq[r], q);
      bad |= sc[r] == 255u || sc[r] > 127u + 13u;
      const float scale = __uint_as_float(sc[r] == 0u ? 0x00400000u : (sc[r] << 23));  // 2^(e - 127)
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        __half2 s2 = __float2half2_rn(0.f);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          s2 = __hfma2(*reinterpret_cast<const __half2*>(&q[k]), *reinterpret_cast<const __half2*>(&xa[t][k]), s2);
        const float2 f = __half22float2(s2);
        acc[r][t] = fmaf(f.x + f.y, scale, acc[r][t]);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      wq[r] = wn[r];
      sc[r] = sn[r];
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r][t] += __shfl_xor_sync(0xffffffffu, acc[r][t], off);
}

template <bool GLU, int NT>
__device__ __forceinline__ void item_rows(const GemvParams& p, const uint4* act_s, const float* tok_mul, int expert,
                                          int row0, int nrows, int fb, int warp, int lane, bool& bad) {
  int wrow[kRowsPerWarp];
  int f0;
  if (GLU) {
    f0 = fb * p.feats_per_item + warp * (kRowsPerWarp / 2);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) wrow[r] = (r & 1) ? p.glu_h + f0 + (r >> 1) : f0 + (r >> 1);
  } else {
    f0 = fb * p.feats_per_item + warp * kRowsPerWarp;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) wrow[r] = f0 + r;
  }
  // four token rows: two passes of two weight rows each (register budget of two CTAs per SM)
  constexpr int RP = NT == 4 ? 2 : kRowsPerWarp;
  float acc[kRowsPerWarp][NT];
#pragma unroll
  for (int h = 0; h < kRowsPerWarp; h += RP) {
    float part[RP][NT];
    warp_rows<NT, RP>(p, act_s, expert, wrow + h, lane, part, bad);
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[h + r][t] = part[r][t];
  }
  // every lane holds every sum; lane (r, t) writes one output
  if (GLU) {
    const int fr = lane >> 2, t = lane & 3;  // feature of the warp, token
    if (lane < 4 * (kRowsPerWarp / 2) && t < nrows && t < NT) {
      float g = 0.f, u = 0.f;
#pragma unroll
      for (int r = 0; r < kRowsPerWarp / 2; ++r)
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
          if (r == fr && tt == t) {
            g = acc[2 * r][tt];
            u = acc[2 * r + 1][tt];
          }
      g *= tok_mul[t];
      u *= tok_mul[t];
      p.out[(int64_t)(row0 + t) * p.ldc + f0 + fr] = __float2half_rn(silu(g) * u);
    }
  } else {
    const int r = lane >> 2, t = lane & 3;
    if (r < kRowsPerWarp && t < nrows && t < NT) {
      float v = 0.f;
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
          if (rr == r && tt == t) v = acc[rr][tt];
      p.out[(int64_t)(row0 + t) * p.ldc + f0 + r] = __float2half_rn(v * tok_mul[t] * p.row_scale[row0 + t]);
    }
  }
}

template <bool GLU>
__global__ void __launch_bounds__(kThreads, 2) gemv_fp4_kernel(const GemvParams p) {
  __shared__ uint4 act_s[4 * kJ * 4 * 32];  // 32 KB
  __shared__ uint32_t amax_bits[4];
  __shared__ float tok_mul[4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = *p.num_tiles_s * p.num_fb;
  const int per_cta = (total + gridDim.x - 1) / gridDim.x;
  const int it_end = min(total, (int)(blockIdx.x + 1) * per_cta);
  const int vec_per_row = p.K / 8;  // 16-byte vectors of fp16 per token row
  bool bad = false;
  int staged = -1;
  for (int it = blockIdx.x * per_cta; it < it_end; ++it) {
    const int q = it / p.num_fb, fb = it - q * p.num_fb;
    const int4 tl = p.tiles_s[q];
    const int nrows = tl.z;
    if (nrows > kGemvMaxRows) continue;  // the tensor-core kernel takes this unit
    if (q != staged) {
      // stage the unit's rows scaled by 2^-s_t, where 2^s_t >= max |x_t|
      __syncthreads();
      if (threadIdx.x < 4) amax_bits[threadIdx.x] = 0u;
      __syncthreads();
      for (int t = 0; t < nrows; ++t) {
        const uint4* src = reinterpret_cast<const uint4*>(p.act + (int64_t)(tl.y + t) * p.K);
        float m = 0.f;
        for (int v = threadIdx.x; v < vec_per_row; v += kThreads) {
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
      __syncthreads();
      if (threadIdx.x < 4) {
        const float m = __uint_as_float(amax_bits[threadIdx.x]);
        // power of two >= m (1 for m == 0 or tiny m); fp16 x * 2^-s stays exact above 2^-24
        const int e = m > 0.f ? max(ilogbf(m) + 1, -14) : 0;
        tok_mul[threadIdx.x] = ldexpf(1.f, e);
      }
      __syncthreads();
      for (int t = 0; t < nrows; ++t) {
        const uint4* src = reinterpret_cast<const uint4*>(p.act + (int64_t)(tl.y + t) * p.K);
        const __half2 inv = __float2half2_rn(1.f / tok_mul[t]);  // power of two: exact
        for (int v = threadIdx.x; v < vec_per_row; v += kThreads) {
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
      // rows past nrows are never read (NT covers them only when nrows == NT)
      __syncthreads();
      staged = q;
    }
    if (nrows == 1)
      item_rows<GLU, 1>(p, act_s, tok_mul, tl.x, tl.y, nrows, fb, warp, lane, bad);
    else if (nrows == 2)
      item_rows<GLU, 2>(p, act_s, tok_mul, tl.x, tl.y, nrows, fb, warp, lane, bad);
    else
      item_rows<GLU, 4>(p, act_s, tok_mul, tl.x, tl.y, nrows, fb, warp, lane, bad);
  }
  if (bad) report(p.status, kStatusDeviceCheck);
}

}  // namespace

cudaError_t launch_gemv_fp4(const TcSwap& g, uint32_t* status, int num_sms, cudaStream_t s) {
  const bool glu = g.epi == kEpiGluF16;
  if (!g.w_scale || (g.epi != kEpiGluF16 && g.epi != kEpiScaleF16)) return cudaErrorInvalidValue;
  if (g.K % 32 || g.K > kMaxChunks * 32 || g.ldc <= 0) return cudaErrorInvalidValue;
  const int feats = glu ? kWarps * kRowsPerWarp / 2 : kWarps * kRowsPerWarp;
  if (g.out_features % feats || (glu && g.glu_h != g.out_features)) return cudaErrorInvalidValue;
  GemvParams p = {};
  p.K = g.K;
  p.glu_h = glu ? g.glu_h : 0;
  p.feats_per_item = feats;
  p.num_fb = g.out_features / feats;
  p.w_rows = (int)g.w.rows;
  p.w = static_cast<const uint8_t*>(g.w.ptr);
  p.ws = g.w_scale;
  p.act = static_cast<const __half*>(g.act.ptr);
  p.tiles_s = g.tiles_s;
  p.num_tiles_s = g.num_tiles_s;
  p.out = static_cast<__half*>(g.C);
  p.ldc = g.ldc;
  p.row_scale = g.row_scale;
  p.status = status;
  const long long items = (long long)g.max_tiles_s * p.num_fb;
  if (items == 0) return cudaSuccess;
  const long long cap = 2LL * num_sms;  // two CTAs per SM (register-limited)
  const int grid = (int)(items < cap ? items : cap);
  if (glu)
    gemv_fp4_kernel<true><<<grid, kThreads, 0, s>>>(p);
  else
    gemv_fp4_kernel<false><<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace lmoe
