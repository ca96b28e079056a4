// Rows of z = W_down x into expert-contiguous order as three-term MXFP4 records, or MXFP8
// records (mx.cuh), the input formats of the block-scaled routed-expert GEMMs (page "Lesson 6 - LatentMoE",
// kimi-k3-course.pages.dev, eq. 11: each selected expert reads W_down x; the rows are grouped by
// expert the way "Kimi K3 architectural innovations", manishklach.github.io, section "A router
// decision is also a scheduling decision", converts selections into expert batches).
//
// Each token's row is quantised once and copied to its k destination rows.  W warps per CTA (one
// for long batches, where the CTA's tokens pipeline; four when every token has a CTA of its own):
// thread 0 loads the next token's row (cp.async.bulk) while the CTA quantises the current one
// (thread i takes the 32-element blocks i, i + 32 W, ...), and thread j writes the record to the
// token's j-th destination row with a bulk store (row_of == nullptr: row t to row t).  Two row
// buffers and two record buffers.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "latentmoe.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace lmoe {
namespace {

__device__ __forceinline__ void load32(const __half* p, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = reinterpret_cast<const uint4*>(p)[q];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      v[8 * q + 2 * i] = f.x;
      v[8 * q + 2 * i + 1] = f.y;
    }
  }
}
__device__ __forceinline__ void load32(const __nv_bfloat16* p, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = reinterpret_cast<const uint4*>(p)[q];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      v[8 * q + 2 * i] = f.x;
      v[8 * q + 2 * i + 1] = f.y;
    }
  }
}

template <int W>
__device__ __forceinline__ void cta_sync() {
  if (W == 1)
    __syncwarp();
  else
    __syncthreads();
}

template <typename TIn, bool F8, int W>
__global__ void __launch_bounds__(32 * W) scatter_mx3_kernel(const TIn* __restrict__ src, uint8_t* __restrict__ dst,
                                                             const int32_t* __restrict__ row_of, int T, int k, int K,
                                                             uint32_t* status, uint64_t timeout_ns) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[2];
  __shared__ int abort_flag;
  const int lane = threadIdx.x;  // the thread's index in the CTA
  const uint32_t in_bytes = (uint32_t)K * sizeof(TIn);
  const uint32_t rec_bytes = (uint32_t)(F8 ? mx8_row_bytes(K) : mx3_row_bytes(K));
  const uint32_t in_stride = (in_bytes + 127u) & ~127u, rec_stride = (rec_bytes + 127u) & ~127u;
  unsigned char* in_buf = smem;                   // [2][in_stride]
  unsigned char* rec_buf = smem + 2 * in_stride;  // [2][rec_stride]
  const int first = blockIdx.x, stride = gridDim.x;
  const int n = first < T ? (T - first + stride - 1) / stride : 0;  // tokens first, first + stride, ...
  if (lane == 0) {
    ptx::mbar_init(&full[0], 1);
    ptx::mbar_init(&full[1], 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  cta_sync<W>();
  auto load = [&](int i) {
    uint64_t* bar = &full[i & 1];
    ptx::mbar_arrive_expect_tx(bar, in_bytes);
    ptx::bulk_load(in_buf + (size_t)(i & 1) * in_stride, src + (size_t)(first + i * stride) * K, in_bytes, bar);
  };
  int issued = 0;
  if (lane == 0 && n > 0) {
    load(0);
    issued = 1;
  }
  int i = 0;
  const int nblocks = K / 32;
  const uint32_t half_k = (uint32_t)K / 2, sc_off = (uint32_t)mx3_scale_offset(K);
  for (; i < n; ++i) {
    // the other row buffer was last read while token i-1 was quantised (finished): refill it
    if (lane == 0 && i + 1 < n) {
      load(i + 1);
      issued = i + 2;
    }
    const int t = first + i * stride;
    const int r = row_of ? (lane < k ? row_of[(size_t)t * k + lane] : -1) : (lane == 0 ? t : -1);
    const bool ok = ptx::mbar_wait_bounded(&full[i & 1], (uint32_t)(i >> 1) & 1u, &abort_flag, status, timeout_ns);
    if (W == 1 ? !__all_sync(0xffffffffu, ok) : !__syncthreads_and(ok)) break;
    // record buffer i&1 was last stored from by token i-2: at most one group (token i-1) may
    // still be reading shared memory
    ptx::bulk_wait_read<1>();
    cta_sync<W>();
    const TIn* row = reinterpret_cast<const TIn*>(in_buf + (size_t)(i & 1) * in_stride);
    unsigned char* rec = rec_buf + (size_t)(i & 1) * rec_stride;
    for (int b = lane; b < nblocks; b += 32 * W) {
      float v[32];
      load32(row + 32 * b, v);
      if (F8) {
        uint32_t codes[8], sc;
        mx::quantize_block8(v, codes, sc);
        *reinterpret_cast<uint4*>(rec + 32 * b) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
        *reinterpret_cast<uint4*>(rec + 32 * b + 16) = make_uint4(codes[4], codes[5], codes[6], codes[7]);
        rec[K + b] = (unsigned char)sc;
      } else {
        uint32_t packed[kMxTerms][4], sc[kMxTerms];
        mx::quantize_block(v, packed, sc);
#pragma unroll
        for (int q = 0; q < kMxTerms; ++q) {
          *reinterpret_cast<uint4*>(rec + q * half_k + 16 * b) =
              make_uint4(packed[q][0], packed[q][1], packed[q][2], packed[q][3]);
          rec[sc_off + q * (K / 32) + b] = (unsigned char)sc[q];
        }
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> bulk-copy reads
    cta_sync<W>();
    if (r >= 0) ptx::bulk_store(dst + (size_t)r * rec_bytes, rec, rec_bytes);
    ptx::bulk_commit();
  }
  if (lane == 0)  // after a wait gave up: let the loads still in flight land before the CTA exits
    for (int j = i; j < issued; ++j) {
      const uint32_t bar = ptx::smem_addr(&full[j & 1]);
      const uint64_t t0 = globaltimer_ns();
      while (!ptx::mbar_try_wait(bar, (uint32_t)(j >> 1) & 1u) && globaltimer_ns() - t0 < timeout_ns) {
      }
    }
  ptx::bulk_wait_all();
}

}  // namespace

size_t scatter_mx3_smem_bytes(int K, int in_elem_bytes, bool f8) {
  const size_t in_stride = ((size_t)K * in_elem_bytes + 127) & ~(size_t)127;
  const size_t rec_stride = ((size_t)(f8 ? mx8_row_bytes(K) : mx3_row_bytes(K)) + 127) & ~(size_t)127;
  return 2 * in_stride + 2 * rec_stride;
}

template <typename TIn, bool F8>
cudaError_t launch_scatter_typed(const void* src, void* dst, const int32_t* row_of, int T, int k, int K, uint32_t* status,
                                 uint64_t timeout_ns, size_t smem, int grid, cudaStream_t s) {
  // a CTA per token: four warps share each token's blocks; otherwise one warp pipelines its tokens
  const bool wide = grid >= T;
  auto kern = wide ? scatter_mx3_kernel<TIn, F8, 4> : scatter_mx3_kernel<TIn, F8, 1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, wide ? 128 : 32, smem, s>>>(static_cast<const TIn*>(src), static_cast<uint8_t*>(dst), row_of, T, k, K,
                                           status, timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_scatter_mx3(const void* src, int src_dtype, void* dst, const int32_t* row_of, int T, int k, int K,
                               uint32_t* status, uint64_t timeout_ns, int num_sms, cudaStream_t s, bool f8) {
  if (T <= 0) return cudaSuccess;
  if (k < 1 || k > 32 || K % 512 || (src_dtype != kF16 && src_dtype != kBF16) ||
      (reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u))
    return cudaErrorInvalidValue;
  const size_t smem = scatter_mx3_smem_bytes(K, 2, f8);
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  const int per_sm = (int)((200 * 1024) / (smem + 1024)) < 8 ? (int)((200 * 1024) / (smem + 1024)) : 8;
  const int grid = T < per_sm * num_sms ? T : per_sm * num_sms;
  if (src_dtype == kF16)
    return f8 ? launch_scatter_typed<__half, true>(src, dst, row_of, T, k, K, status, timeout_ns, smem, grid, s)
              : launch_scatter_typed<__half, false>(src, dst, row_of, T, k, K, status, timeout_ns, smem, grid, s);
  return f8 ? launch_scatter_typed<__nv_bfloat16, true>(src, dst, row_of, T, k, K, status, timeout_ns, smem, grid, s)
            : launch_scatter_typed<__nv_bfloat16, false>(src, dst, row_of, T, k, K, status, timeout_ns, smem, grid, s);
}

}  // namespace lmoe

namespace {
lmoe_status quantize_rows(const void* src, int32_t src_dtype, int64_t rows, int32_t K, void* dst, void* stream,
                          bool f8) {
  if (rows < 0 || rows > INT32_MAX || K <= 0 || K % 512 || (rows > 0 && (!src || !dst)))
    return LMOE_ERR_INVALID_ARG;
  if (src_dtype != LMOE_BF16 && src_dtype != LMOE_F16) return LMOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u)) return LMOE_ERR_INVALID_ARG;
  if (rows == 0) return LMOE_OK;
  int dev = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LMOE_ERR_CUDA;
  const cudaError_t e =
      lmoe::launch_scatter_mx3(src, src_dtype == LMOE_BF16 ? lmoe::kBF16 : lmoe::kF16, dst, nullptr, (int)rows, 1, K,
                               nullptr, 4000000000ull, num_sms, static_cast<cudaStream_t>(stream), f8);
  return e == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}
}  // namespace

// Test hooks (declared in latentmoe.h): the three-term MXFP4 / the MXFP8 records of rows x K values.
extern "C" lmoe_status latentmoe_mx3_quantize(const void* src, int32_t src_dtype, int64_t rows, int32_t K, void* dst,
                                              void* stream) {
  return quantize_rows(src, src_dtype, rows, K, dst, stream, false);
}
extern "C" lmoe_status latentmoe_mx8_quantize(const void* src, int32_t src_dtype, int64_t rows, int32_t K, void* dst,
                                              void* stream) {
  return quantize_rows(src, src_dtype, rows, K, dst, stream, true);
}
