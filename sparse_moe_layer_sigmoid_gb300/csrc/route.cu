// Router, top-k selection and expert dispatch (page "Lesson 6 - LatentMoE",
// kimi-k3-course.pages.dev, section "show me the actual equation", eq. 13; and
// "Kimi K3 architectural innovations", manishklach.github.io, section "A router decision is
// also a scheduling decision": selections become expert batches).
//
// Everything here is integer or per-token fp32 work on CUDA cores; the router GEMM itself is
// the fp32 CUDA-core GEMM of simt.cu.  All results are deterministic: no reduction depends on
// thread scheduling (counts use atomicOr on bit masks, which commute exactly).
#include "common.cuh"
#include "internal.h"

namespace lmoe {
namespace {

__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp per token.  Keys are packed as (orderable(s + b) << 32) | (~expert) so that the
// 64-bit maximum is the largest key and, among equal keys, the lowest expert index.
template <int NPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits,
                                                   const float* __restrict__ bias, int T, int E, int k,
                                                   int32_t* __restrict__ idx, float* __restrict__ p) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* row = logits + (size_t)warp * E;
  uint64_t key[NPL];
  float sv[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0;
    sv[i] = 0.f;
    if (e < E) {
      const float s = 1.0f / (1.0f + expf(-row[e]));
      const float kf = bias ? s + bias[e] : s;
      key[i] = ((uint64_t)orderable(kf) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e);
      sv[i] = s;
    }
  }
  float sum = 0.f;
  int my_e = 0;
  float my_s = 0.f;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off);
      best = o > best ? o : best;
    }
    const int e_win = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFu));
    const int owner = e_win & 31, slot = e_win >> 5;
    float s_here = 0.f;
    if (lane == owner) {
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (i == slot) {
          s_here = sv[i];
          key[i] = 0;
        }
    }
    const float s_win = __shfl_sync(0xffffffffu, s_here, owner);
    sum += s_win;  // rank order
    if (lane == j) {
      my_e = e_win;
      my_s = s_win;
    }
  }
  if (lane < k) {
    idx[(size_t)warp * k + lane] = my_e;
    p[(size_t)warp * k + lane] = my_s / sum;
  }
}

constexpr int kMaskWords = kDispatchChunk / 32;

// Per-chunk bit mask of the tokens that selected each expert.  Returns false (and reports)
// for an index outside [0,E) or an expert listed twice for one token.
__device__ __forceinline__ void build_masks(const int32_t* __restrict__ idx, int T, int E, int k, uint32_t* mask,
                                            uint32_t* status) {
  for (int i = threadIdx.x; i < E * kMaskWords; i += blockDim.x) mask[i] = 0;
  __syncthreads();
  const int t = blockIdx.x * kDispatchChunk + threadIdx.x;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)t * k + j];
      if (e < 0 || e >= E) {
        report(status, kStatusDeviceCheck);
        continue;
      }
      const uint32_t bit = 1u << (threadIdx.x & 31);
      const uint32_t old = atomicOr(&mask[e * kMaskWords + (threadIdx.x >> 5)], bit);
      if (old & bit) report(status, kStatusDeviceCheck);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kDispatchChunk) dispatch_count_kernel(const int32_t* __restrict__ idx, int T,
                                                                        int E, int k,
                                                                        int32_t* __restrict__ chunk_counts,
                                                                        uint32_t* status) {
  extern __shared__ uint32_t mask[];
  build_masks(idx, T, E, k, mask, status);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w) c += __popc(mask[e * kMaskWords + w]);
    chunk_counts[(size_t)blockIdx.x * E + e] = c;
  }
}

__global__ void __launch_bounds__(1024) dispatch_scan_kernel(const int32_t* __restrict__ chunk_counts,
                                                             int nchunks, int E, int32_t* __restrict__ chunk_base,
                                                             int32_t* __restrict__ offsets, int4* __restrict__ tiles,
                                                             int32_t* __restrict__ num_tiles) {
  __shared__ int s_cnt[1024];
  __shared__ int s_tiles[1024];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E)
    for (int c = 0; c < nchunks; ++c) total += chunk_counts[(size_t)c * E + e];
  const int nt = (total + kTileM - 1) / kTileM;
  s_cnt[e] = total;
  s_tiles[e] = nt;
  __syncthreads();
  // Hillis-Steele inclusive scans over 1024 entries (fixed order, integer: exact).
  for (int off = 1; off < 1024; off <<= 1) {
    const int a = e >= off ? s_cnt[e - off] : 0;
    const int b = e >= off ? s_tiles[e - off] : 0;
    __syncthreads();
    s_cnt[e] += a;
    s_tiles[e] += b;
    __syncthreads();
  }
  const int row0 = s_cnt[e] - total;
  const int tile0 = s_tiles[e] - nt;
  if (e < E) {
    offsets[e] = row0;
    int run = row0;
    for (int c = 0; c < nchunks; ++c) {
      chunk_base[(size_t)c * E + e] = run;
      run += chunk_counts[(size_t)c * E + e];
    }
    for (int j = 0; j < nt; ++j) tiles[tile0 + j] = make_int4(e, tile0, nt, 0);
  }
  if (e == E - 1) {
    offsets[E] = s_cnt[e];
    *num_tiles = s_tiles[e];
  }
}

__global__ void __launch_bounds__(kDispatchChunk) dispatch_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ p, int T, int E, int k,
    const int32_t* __restrict__ chunk_base, int32_t* __restrict__ tok_of_row, int32_t* __restrict__ row_of,
    float* __restrict__ p_row) {
  extern __shared__ uint32_t mask[];
  build_masks(idx, T, E, k, mask, nullptr);
  const int t = blockIdx.x * kDispatchChunk + threadIdx.x;
  if (t >= T) return;
  const int w = threadIdx.x >> 5;
  const uint32_t below = (1u << (threadIdx.x & 31)) - 1u;
  for (int j = 0; j < k; ++j) {
    const int e = idx[(size_t)t * k + j];
    if (e < 0 || e >= E) {
      if (row_of) row_of[(size_t)t * k + j] = -1;
      continue;
    }
    const uint32_t* m = mask + e * kMaskWords;
    int rank = __popc(m[w] & below);
    for (int q = 0; q < w; ++q) rank += __popc(m[q]);
    const int row = chunk_base[(size_t)blockIdx.x * E + e] + rank;
    if (row_of) row_of[(size_t)t * k + j] = row;
    if (tok_of_row) tok_of_row[row] = t;
    if (p_row) p_row[row] = p ? p[(size_t)t * k + j] : 1.0f;
  }
}

// One warp per token: read the token's row once, write it to each of its k rows.
__global__ void __launch_bounds__(256) scatter_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                           const int32_t* __restrict__ row_of, int T, int k,
                                                           int nvec) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int rows[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) rows[j] = (j < k) ? row_of[(size_t)t * k + j] : -1;
  const uint4* s = src + (size_t)t * nvec;
  for (int v = lane; v < nvec; v += 32) {
    const uint4 val = s[v];
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < k && rows[j] >= 0) dst[(size_t)rows[j] * nvec + v] = val;
  }
}

}  // namespace

cudaError_t launch_router_logits(const void* x, int x_dtype, const void* w_router, int w_dtype, float* logits,
                                 int T, int E, int d, cudaStream_t s) {
  SimtGemm g = {};
  g.A = x;
  g.lda = d;
  g.a_dtype = x_dtype;
  g.b_dtype = w_dtype;
  g.nseg = 1;
  g.seg[0] = SimtSegment{w_router, d, 0, d, d};
  g.M = T;
  g.N = E;
  g.K = d;
  g.C = logits;
  g.ldc = E;
  g.c_dtype = kF32;
  return launch_simt_gemm(g, s);
}

cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* idx, float* p,
                        cudaStream_t s) {
  const int warps_per_block = 8;
  dim3 grid((T + warps_per_block - 1) / warps_per_block), block(32 * warps_per_block);
  const int npl = (E + 31) / 32;
  if (npl <= 1) topk_kernel<1><<<grid, block, 0, s>>>(logits, bias, T, E, k, idx, p);
  else if (npl <= 2) topk_kernel<2><<<grid, block, 0, s>>>(logits, bias, T, E, k, idx, p);
  else if (npl <= 4) topk_kernel<4><<<grid, block, 0, s>>>(logits, bias, T, E, k, idx, p);
  else if (npl <= 8) topk_kernel<8><<<grid, block, 0, s>>>(logits, bias, T, E, k, idx, p);
  else if (npl <= 16) topk_kernel<16><<<grid, block, 0, s>>>(logits, bias, T, E, k, idx, p);
  else if (npl <= 28) topk_kernel<28><<<grid, block, 0, s>>>(logits, bias, T, E, k, idx, p);
  else topk_kernel<32><<<grid, block, 0, s>>>(logits, bias, T, E, k, idx, p);
  return cudaGetLastError();
}

cudaError_t launch_dispatch(const int32_t* idx, const float* p, int T, int E, int k, const DispatchBuffers& b,
                            uint32_t* status, int* launches, cudaStream_t s) {
  const int nchunks = (T + kDispatchChunk - 1) / kDispatchChunk;
  const size_t smem = (size_t)E * kMaskWords * sizeof(uint32_t);
  dispatch_count_kernel<<<nchunks, kDispatchChunk, smem, s>>>(idx, T, E, k, b.chunk_counts, status);
  dispatch_scan_kernel<<<1, 1024, 0, s>>>(b.chunk_counts, nchunks, E, b.chunk_base, b.offsets, b.tiles,
                                          b.num_tiles);
  dispatch_scatter_kernel<<<nchunks, kDispatchChunk, smem, s>>>(idx, p, T, E, k, b.chunk_base, b.tok_of_row,
                                                                b.row_of, b.p_row);
  if (launches) *launches += 3;
  return cudaGetLastError();
}

cudaError_t launch_scatter_rows(const void* src, void* dst, const int32_t* row_of, int T, int k, int width,
                                int elem_bytes, cudaStream_t s) {
  const int nvec = width * elem_bytes / 16;
  const int warps = 8;
  scatter_rows_kernel<<<(T + warps - 1) / warps, 32 * warps, 0, s>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), row_of, T, k, nvec);
  return cudaGetLastError();
}

}  // namespace lmoe
