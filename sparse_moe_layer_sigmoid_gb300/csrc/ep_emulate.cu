// Expert-parallel dispatch and combine, emulated on one GPU (page "What K3 actually is",
// srikanthmalla.com, opening section: a routed token crosses the expert-parallel all-to-all at
// the experts' input width, k x 7168 values at full width and half that at the latent width;
// page "Lesson 6 - LatentMoE", kimi-k3-course.pages.dev, table "What scales with what").
//
// R virtual ranks: rank r owns tokens [r T/R, (r+1) T/R) and experts [r E/R, (r+1) E/R).  Every
// selected (token t, expert e) pair is one row of W values (W = l for LatentMoE's latent rows
// z = W_down x, W = d for a conventional MoE that dispatches x itself).  One pass:
//   plan      per (expert, source rank) row counts from the dispatch's expert-sorted rows, and
//             the offsets of every (source, destination) cell in both buffers;
//   pack      each source rank's rows into its send region, ordered (destination, expert, token);
//   exchange  send[src][dst] -> recv[dst][src] for all R x R cells (the all-to-all; on one GPU a
//             copy through HBM, on a real system the NVLink transfer);
//   return    the expert outputs (identity experts: the received rows) back, recv -> send order;
//   combine   each token's k rows in rank order, p-weighted (the layer's combine kernel).
// Row (t, j) of the dispatch (expert e, row i of the expert-sorted order) sits at send position
//   send_base[src][dst] + P[e][src] + (i - offsets[e] - Q[e][src]),
// with Q[e][r] the rows of expert e from ranks below r (an expert's rows are token-ascending, so
// a rank's rows of one expert are contiguous) and P[e][r] the rows of rank r for experts of the
// same destination below e.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace lmoe {
namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int lower_bound_i32(const int32_t* a, int n, int32_t v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < v)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

// One CTA.  plan layout: Q [E][R], P [E][R], cells [R][R] (src-major), send_base [R][R]
// (src-major), recv_base [R][R] (dst-major).
__global__ void __launch_bounds__(kPlanThreads) ep_plan_kernel(const int32_t* __restrict__ offsets,
                                                               const int32_t* __restrict__ tok_of_row, int T, int E,
                                                               int R, int32_t* __restrict__ plan) {
  int32_t* Q = plan;
  int32_t* P = Q + E * R;
  int32_t* cells = P + E * R;
  int32_t* send_base = cells + R * R;
  int32_t* recv_base = send_base + R * R;
  const int tr = T / R, er = E / R;
  // Q[e][r] = rows of expert e whose token is below rank r's first token; Q[e][R] would be the count
  for (int c = threadIdx.x; c < E * R; c += blockDim.x) {
    const int e = c / R, r = c - e * R;
    const int o0 = offsets[e];
    Q[c] = lower_bound_i32(tok_of_row + o0, offsets[e + 1] - o0, r * tr);
  }
  __syncthreads();
  // P[e][r] over the experts of e's destination in increasing order; cells[r][dst] the total
  for (int c = threadIdx.x; c < R * R; c += blockDim.x) {
    const int dst = c / R, r = c - dst * R;
    int run = 0;
    for (int e = dst * er; e < (dst + 1) * er; ++e) {
      P[e * R + r] = run;
      const int hi = r + 1 < R ? Q[e * R + r + 1] : offsets[e + 1] - offsets[e];
      run += hi - Q[e * R + r];
    }
    cells[r * R + dst] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int c = 0; c < R * R; ++c) {  // (src, dst) order
      send_base[c] = acc;
      acc += cells[c];
    }
    acc = 0;
    for (int dst = 0; dst < R; ++dst)  // (dst, src) order
      for (int src = 0; src < R; ++src) {
        recv_base[dst * R + src] = acc;
        acc += cells[src * R + dst];
      }
  }
}

// Copy one row of `bytes` (multiple of 16) with the warp, 16-byte vectors.
__device__ __forceinline__ void copy_row(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int bytes,
                                         int lane) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  const int n = bytes >> 4;
#pragma unroll 4
  for (int v = lane; v < n; v += 32) d[v] = __ldg(s + v);
}

// One warp per (t, j): the token's row into its send position; ep_row_of[t][j] = that position.
__global__ void ep_pack_kernel(const uint8_t* __restrict__ src, int64_t src_ld, int row_bytes,
                               const int32_t* __restrict__ idx, const int32_t* __restrict__ row_of,
                               const int32_t* __restrict__ offsets, const int32_t* __restrict__ plan, int T, int E,
                               int R, int k, uint8_t* __restrict__ send, int32_t* __restrict__ ep_row_of) {
  const int32_t* Q = plan;
  const int32_t* P = Q + E * R;
  const int32_t* send_base = P + E * R + R * R;
  const int tr = T / R, er = E / R;
  const int lane = threadIdx.x & 31;
  const int64_t pairs = (int64_t)T * k;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; w < pairs;
       w += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int t = (int)(w / k);
    const int e = idx[w], i = row_of[w];
    const int r = t / tr, dst = e / er;
    const int pos = send_base[r * R + dst] + P[e * R + r] + (i - offsets[e] - Q[e * R + r]);
    if (lane == 0) ep_row_of[w] = pos;
    copy_row(src + (int64_t)t * src_ld, send + (int64_t)pos * row_bytes, row_bytes, lane);
  }
}

// The all-to-all, one warp per destination row.  forward: recv (dst, src) order <- send (src,
// dst) order; backward: the reverse.
__global__ void ep_exchange_kernel(const uint8_t* __restrict__ from, uint8_t* __restrict__ to, int row_bytes,
                                   int64_t rows, const int32_t* __restrict__ plan, int E, int R, int forward) {
  const int32_t* cells = plan + 2 * E * R;
  const int32_t* send_base = cells + R * R;
  const int32_t* recv_base = send_base + R * R;
  const int32_t* to_base = forward ? recv_base : send_base;  // cell starts in the destination order
  const int lane = threadIdx.x & 31;
  for (int64_t q = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; q < rows;
       q += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    // the cell holding destination row q: the last start <= q among the R x R starts (ascending)
    int lo = 0, hi = R * R - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (to_base[mid] <= q)
        lo = mid;
      else
        hi = mid - 1;
    }
    // (an empty cell starts where the next one does; the search passes over it)
    const int a = lo / R, b = lo - a * R;  // forward: (dst, src); backward: (src, dst)
    const int64_t from_row = forward ? (int64_t)send_base[b * R + a] + (q - recv_base[lo])
                                     : (int64_t)recv_base[b * R + a] + (q - send_base[lo]);
    copy_row(from + from_row * row_bytes, to + q * row_bytes, row_bytes, lane);
  }
}

}  // namespace

size_t ep_plan_ints(int E, int R) { return (size_t)2 * E * R + (size_t)3 * R * R; }

cudaError_t launch_ep_plan(const int32_t* offsets, const int32_t* tok_of_row, int T, int E, int R, int32_t* plan,
                           cudaStream_t s) {
  ep_plan_kernel<<<1, kPlanThreads, 0, s>>>(offsets, tok_of_row, T, E, R, plan);
  return cudaGetLastError();
}

cudaError_t launch_ep_pack(const void* src, int64_t src_ld_bytes, int row_bytes, const int32_t* idx,
                           const int32_t* row_of, const int32_t* offsets, const int32_t* plan, int T, int E, int R,
                           int k, void* send, int32_t* ep_row_of, int num_sms, cudaStream_t s) {
  const int64_t pairs = (int64_t)T * k;
  if (pairs == 0) return cudaSuccess;
  const int64_t blocks = (pairs + 7) / 8;  // 8 warps per CTA
  const int grid = (int)(blocks < 16LL * num_sms ? blocks : 16LL * num_sms);
  ep_pack_kernel<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(src), src_ld_bytes, row_bytes, idx, row_of,
                                      offsets, plan, T, E, R, k, static_cast<uint8_t*>(send), ep_row_of);
  return cudaGetLastError();
}

cudaError_t launch_ep_exchange(const void* from, void* to, int row_bytes, int64_t rows, const int32_t* plan, int E,
                               int R, int forward, int num_sms, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;
  const int grid = (int)(blocks < 16LL * num_sms ? blocks : 16LL * num_sms);
  ep_exchange_kernel<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(from), static_cast<uint8_t*>(to), row_bytes,
                                          rows, plan, E, R, forward);
  return cudaGetLastError();
}

}  // namespace lmoe
