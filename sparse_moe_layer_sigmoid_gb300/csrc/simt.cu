// fp32 CUDA-core GEMM used for the router logits (fp32 accumulation, fixed K order) and for
// every contraction of fp32 layers.  C[r][n] = epilogue( sum_c A[r][c] * B[n][c] ).
//
// Modes: dense or grouped (rows come from the dispatch tile list and B from the tile's
// expert); B as up to six K segments (the final GEMM concatenates the shared-expert down
// projections and W_up along K); GLU (output j = SiLU(gate_j) * up_j with gate/up rows
// j and j + glu_h); optional per-row scale (the routed down projection's p).
#include "common.cuh"
#include "internal.h"

namespace lmoe {
namespace {

constexpr int BM = 128, BN = 64, BK = 16, NT = 256;
constexpr int TM = 8, TN = 4;  // per-thread micro tile (16 x 16 threads)

template <typename T>
__device__ __forceinline__ float ld_as_f32(const void* base, int64_t i) {
  return to_f32(static_cast<const T*>(base)[i]);
}

template <typename TA, typename TB, bool GLU>
__global__ void __launch_bounds__(NT) simt_gemm_kernel(SimtGemm g) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ float Bu[GLU ? BK : 1][BN + 4];

  int row0, row_end, group = 0;
  if (g.tiles) {
    if ((int)blockIdx.x >= *g.num_tiles) return;
    const int4 tl = g.tiles[blockIdx.x];
    group = tl.x;
    row0 = g.offsets[tl.x] + (blockIdx.x - tl.y) * kTileM;
    row_end = min(row0 + kTileM, g.offsets[tl.x + 1]);
  } else {
    row0 = blockIdx.x * BM;
    row_end = min(row0 + BM, g.M);
  }
  const int n0 = blockIdx.y * BN;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;

  float acc[TM][TN], accu[GLU ? TM : 1][GLU ? TN : 1];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
  if (GLU) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) accu[GLU ? i : 0][GLU ? j : 0] = 0.f;
  }

  int seg = 0, seg_k0 = 0;
  for (int kt = 0; kt < g.K; kt += BK) {
    while (seg + 1 < g.nseg && kt >= seg_k0 + g.seg[seg].k_len) {
      seg_k0 += g.seg[seg].k_len;
      ++seg;
    }
    const SimtSegment sg = g.seg[seg];
    const int kl = kt - seg_k0;
    const int goff = kl / sg.k_per_group, kin = kl % sg.k_per_group;
    // A tile: 128 rows x 16 k
#pragma unroll
    for (int i = 0; i < (BM * BK) / NT; ++i) {
      const int e = tid + i * NT, r = e / BK, c = e % BK;
      const int row = row0 + r;
      As[c][r] = (row < row_end) ? ld_as_f32<TA>(g.A, (int64_t)row * g.lda + kt + c) : 0.f;
    }
    // B tile: 64 output columns x 16 k
#pragma unroll
    for (int i = 0; i < (BN * BK) / NT; ++i) {
      const int e = tid + i * NT, n = e / BK, c = e % BK;
      const int col = n0 + n;
      float bv = 0.f, uv = 0.f;
      if (col < g.N) {
        int grp = group + goff, brow = col;
        if (GLU) {
          grp += col / g.glu_h;
          brow = col % g.glu_h;
        }
        const int64_t base = (int64_t)grp * sg.group_stride + kin + c;
        bv = ld_as_f32<TB>(sg.ptr, base + (int64_t)brow * sg.ld);
        if (GLU) uv = ld_as_f32<TB>(sg.ptr, base + (int64_t)(brow + g.glu_h) * sg.ld);
      }
      Bs[c][n] = bv;
      if (GLU) Bu[GLU ? c : 0][n] = uv;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < BK; ++c) {
      float a[TM], b[TN], u[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) a[i] = As[c][ty * TM + i];
#pragma unroll
      for (int j = 0; j < TN; ++j) {
        b[j] = Bs[c][tx * TN + j];
        if (GLU) u[j] = Bu[GLU ? c : 0][tx * TN + j];
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if (GLU) accu[GLU ? i : 0][GLU ? j : 0] = fmaf(a[i], u[j], accu[GLU ? i : 0][GLU ? j : 0]);
        }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int row = row0 + ty * TM + i;
    if (row >= row_end) continue;
    const float sc = g.row_scale ? g.row_scale[row] : 1.0f;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int col = n0 + tx * TN + j;
      if (col >= g.N) continue;
      float v = acc[i][j];
      if (GLU) v = silu(v) * accu[GLU ? i : 0][GLU ? j : 0];
      v *= sc;
      if (g.c_dtype == kF32) static_cast<float*>(g.C)[(int64_t)row * g.ldc + col] = v;
      else static_cast<__nv_bfloat16*>(g.C)[(int64_t)row * g.ldc + col] = __float2bfloat16_rn(v);
    }
  }
}

template <typename TA, typename TB>
cudaError_t launch_typed(const SimtGemm& g, cudaStream_t s) {
  const int mblocks = g.tiles ? g.max_tiles : (g.M + BM - 1) / BM;
  dim3 grid(mblocks, (g.N + BN - 1) / BN);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  if (g.glu_h > 0) simt_gemm_kernel<TA, TB, true><<<grid, NT, 0, s>>>(g);
  else simt_gemm_kernel<TA, TB, false><<<grid, NT, 0, s>>>(g);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t s) {
  if (g.K % BK != 0) return cudaErrorInvalidValue;
  for (int i = 0; i < g.nseg; ++i)
    if (g.seg[i].k_len % BK != 0 || g.seg[i].k_per_group % BK != 0) return cudaErrorInvalidValue;
  if (g.a_dtype == kF32 && g.b_dtype == kF32) return launch_typed<float, float>(g, s);
  if (g.a_dtype == kBF16 && g.b_dtype == kF32) return launch_typed<__nv_bfloat16, float>(g, s);
  if (g.a_dtype == kF32 && g.b_dtype == kBF16) return launch_typed<float, __nv_bfloat16>(g, s);
  return launch_typed<__nv_bfloat16, __nv_bfloat16>(g, s);
}

}  // namespace lmoe
