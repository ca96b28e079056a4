// Deterministic combine + RMSNorm (page "Lesson 6 - LatentMoE", kimi-k3-course.pages.dev:
// eq. 11 "u = sum over the selected experts of p_i E_i(W_down x)", and section "What extreme
// sparsity breaks": RMSNorm between aggregation and W_up).
//
// One CTA of 512 threads per token, whatever the batch size (the reduction tree below depends on
// the CTA's width only, so a token's output does not depend on the batch).  The k expert rows of
// the token are summed in rank order j = 0..k-1 in fp32 registers (the same order on every run),
// U rows' loads in flight at a time (all 16 of a short batch's token at once, where latency rules;
// fewer for long batches, where occupancy does), then sum(u^2) is reduced in a fixed tree and
// n = u * g / sqrt(mean(u^2) + eps) is written.  HBM-bound: it reads k rows per token once.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace lmoe {
namespace {

constexpr int kThreads = 512;
constexpr int kShortBatch = 256;  // batches up to this many tokens load all of a token's rows at once

template <typename T>
struct Vec {  // 16-byte vector of T
  static constexpr int N = 16 / sizeof(T);
};

__device__ __forceinline__ void unpack(const uint4& v, float (&f)[8], __nv_bfloat16) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[8], __half) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[8], float) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ uint4 pack(const float (&f)[8], __nv_bfloat16) {
  uint4 v;
  v.x = pack_bf16x2(f[0], f[1]);
  v.y = pack_bf16x2(f[2], f[3]);
  v.z = pack_bf16x2(f[4], f[5]);
  v.w = pack_bf16x2(f[6], f[7]);
  return v;
}
__device__ __forceinline__ uint4 pack(const float (&f)[8], float) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}

template <typename T, typename TO, int VPT, int U>
__global__ void __launch_bounds__(kThreads) combine_kernel(const T* __restrict__ o, const int32_t* __restrict__ row_of,
                                                           const float* __restrict__ p,
                                                           const float* __restrict__ gain, float eps, int k,
                                                           int width, TO* __restrict__ out, int64_t ld_out) {
  static_assert(Vec<T>::N == Vec<TO>::N, "input and output vectors must hold the same element count");
  constexpr int EPV = Vec<T>::N;
  const int t = blockIdx.x;
  const int nvec = width / EPV;
  float acc[VPT][8];
#pragma unroll
  for (int i = 0; i < VPT; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;

  // the token's k row indices and weights first (one round of loads), then U expert rows at a
  // time: their loads are all issued before any is summed, and the sums still run in rank order
  // j = 0..k-1 (U does not change the arithmetic).
  __shared__ int s_r[32];
  __shared__ float s_w[32];
  if (threadIdx.x < k) {
    s_r[threadIdx.x] = row_of[(size_t)t * k + threadIdx.x];
    s_w[threadIdx.x] = p ? p[(size_t)t * k + threadIdx.x] : 1.0f;
  }
  __syncthreads();
  for (int j0 = 0; j0 < k; j0 += U) {
    int r[U];
    float w[U];
    uint4 raw[U][VPT];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + u;
      r[u] = j < k ? s_r[j] : -1;
      w[u] = j < k ? s_w[j] : 1.0f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (r[u] < 0) continue;
      const uint4* src = reinterpret_cast<const uint4*>(o + (size_t)r[u] * width);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = threadIdx.x + i * kThreads;
        if (v < nvec) raw[u][i] = __ldg(src + v);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (r[u] < 0) continue;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = threadIdx.x + i * kThreads;
        if (v < nvec) {
          float f[8];
          unpack(raw[u][i], f, T());
#pragma unroll
          for (int e = 0; e < EPV; ++e) acc[i][e] = p ? fmaf(w[u], f[e], acc[i][e]) : acc[i][e] + f[e];
        }
      }
    }
  }

  float scale = 1.0f;
  if (gain) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int e = 0; e < EPV; ++e) ss = fmaf(acc[i][e], acc[i][e], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    __shared__ float warp_ss[kThreads / 32];
    if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) tot += warp_ss[w];
    scale = 1.0f / sqrtf(tot / (float)width + eps);
  }

  uint4* dst = reinterpret_cast<uint4*>(out + (size_t)t * ld_out);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * kThreads;
    if (v < nvec) {
      float f[8];
#pragma unroll
      for (int e = 0; e < EPV; ++e) f[e] = gain ? acc[i][e] * __ldg(gain + v * EPV + e) * scale : acc[i][e];
      dst[v] = pack(f, TO());
    }
  }
}

template <typename T, typename TO, int VPT>
void launch_vpt(const T* op, const int32_t* row_of, const float* p, const float* gain, float eps, int T_, int k,
                int width, TO* dp, int64_t ld_out, cudaStream_t s) {
  constexpr int U_LONG = VPT == 1 ? 8 : 2;
  if (T_ <= kShortBatch)
    combine_kernel<T, TO, VPT, 16 / VPT><<<T_, kThreads, 0, s>>>(op, row_of, p, gain, eps, k, width, dp, ld_out);
  else
    combine_kernel<T, TO, VPT, U_LONG><<<T_, kThreads, 0, s>>>(op, row_of, p, gain, eps, k, width, dp, ld_out);
}

template <typename T, typename TO>
cudaError_t launch_typed(const void* o, const int32_t* row_of, const float* p, const float* gain, float eps, int T_,
                         int k, int width, void* out, int64_t ld_out, cudaStream_t s) {
  const int nvec = width / Vec<T>::N;
  const T* op = static_cast<const T*>(o);
  TO* dp = static_cast<TO*>(out);
  if (nvec <= kThreads)
    launch_vpt<T, TO, 1>(op, row_of, p, gain, eps, T_, k, width, dp, ld_out, s);
  else if (nvec <= 2 * kThreads)
    launch_vpt<T, TO, 2>(op, row_of, p, gain, eps, T_, k, width, dp, ld_out, s);
  else if (nvec <= 4 * kThreads)
    launch_vpt<T, TO, 4>(op, row_of, p, gain, eps, T_, k, width, dp, ld_out, s);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const void* o, int in_dtype, int out_dtype, const int32_t* row_of, const float* p,
                           const float* gain, float eps, int T, int k, int width, void* out, int64_t ld_out,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (in_dtype == kF32 && out_dtype == kF32)
    return launch_typed<float, float>(o, row_of, p, gain, eps, T, k, width, out, ld_out, s);
  if (in_dtype == kBF16 && out_dtype == kBF16)
    return launch_typed<__nv_bfloat16, __nv_bfloat16>(o, row_of, p, gain, eps, T, k, width, out, ld_out, s);
  if (in_dtype == kF16 && out_dtype == kBF16)
    return launch_typed<__half, __nv_bfloat16>(o, row_of, p, gain, eps, T, k, width, out, ld_out, s);
  return cudaErrorInvalidValue;
}

}  // namespace lmoe
