// Tensor-core rate microbenchmark: back-to-back tcgen05.mma of one kind on every SM, for the
// roofline denominators of the expert GEMMs.  The block-scaled FP4 rate has no library
// measurement to read; this one runs the exact instruction shape the expert kernels issue
// (cta_group::2, M = 256, N = 256: kind::f16 with K = 16, or kind::mxf4 with K = 64 and E8M0
// scales), so rate(mxf4) / rate(f16) is the ratio of the two peaks on this GPU.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "latentmoe.h"
#include "ptx.cuh"

namespace lmoe {
namespace {

constexpr int kThreads = 128;
constexpr uint32_t kOperandBytes = 48 * 1024;  // A 128 rows + B 128 rows per CTA, 128-byte rows (+ spare)
constexpr size_t kSmem = kOperandBytes + 1024;

template <bool MXF4>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mma_rate_kernel(int iters, uint64_t timeout_ns, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ uint32_t tmem_holder;
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = ptx::cluster_ctarank();
  // operand values do not change the rate: E2M1 / fp16 bit patterns of small numbers
  for (uint32_t i = threadIdx.x; i < kOperandBytes / 4; i += kThreads) reinterpret_cast<uint32_t*>(smem)[i] = 0x22222222u;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&done_bar, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) ptx::tmem_alloc_pair(&tmem_holder, 512);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_holder;
  if (MXF4) {  // scales 2^0 in the scale columns 256..511 of every lane
    uint32_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0x7F7F7F7Fu;
    for (uint32_t c = 256; c < 512; c += 8) ptx::tmem_st_32x32b_x8(tmem + ((uint32_t)(32 * warp) << 16) + c, v);
    ptx::tmem_st_wait();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (threadIdx.x == 0 && rank == 0) {
    const uint32_t a = ptx::smem_addr(smem), b = a + 16384;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (MXF4)
          ptx::mma_mxf4_pair(tmem, ptx::sw128_kmajor_desc(a + 32 * kk), ptx::sw128_kmajor_desc(b + 32 * kk),
                             ptx::idesc_mxf4(256, 256, 0, 0), tmem + 256, tmem + 320, 1u);
        else
          ptx::mma_f16_pair(tmem, ptx::sw128_kmajor_desc(a + 32 * kk), ptx::sw128_kmajor_desc(b + 32 * kk),
                            ptx::idesc_bf16_f32(256, 256), 1u);
      }
    }
    ptx::mma_commit_pair(&done_bar);
    const uint32_t bar = ptx::smem_addr(&done_bar);
    const uint64_t t0 = globaltimer_ns();
    bool ok = true;
    while (!ptx::mbar_try_wait(bar, 0))
      if (globaltimer_ns() - t0 > timeout_ns) {
        ok = false;
        break;
      }
    if (!ok) {
      report(status, kStatusTimeout);
      ptx::drain_mma_pair(&done_bar, timeout_ns);  // a second commit: every MMA issued has completed
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace
}  // namespace lmoe

extern "C" lmoe_status latentmoe_mma_peak(int32_t kind, double* tflops, void* stream) {
  using namespace lmoe;
  if (!tflops || (kind != 0 && kind != 1)) return LMOE_ERR_INVALID_ARG;
  *tflops = 0.0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LMOE_ERR_CUDA;
  auto kern = kind ? mma_rate_kernel<true> : mma_rate_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) != cudaSuccess)
    return LMOE_ERR_CUDA;
  const int pairs = num_sms / 2;
  const int iters = kind ? 3000 : 1000;  // about 0.5-1 ms per launch
  uint32_t* status = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  lmoe_status st = LMOE_OK;
  float best = 0.f;
  if (cudaMallocAsync(reinterpret_cast<void**>(&status), sizeof(uint32_t), s) != cudaSuccess ||
      cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess || cudaEventCreate(&e0) != cudaSuccess ||
      cudaEventCreate(&e1) != cudaSuccess) {
    st = LMOE_ERR_CUDA;
  } else {
    for (int rep = 0; rep < 4 && st == LMOE_OK; ++rep) {  // the first launch warms up
      float ms = 0.f;
      if (cudaEventRecord(e0, s) != cudaSuccess) st = LMOE_ERR_CUDA;
      kern<<<2 * pairs, kThreads, kSmem, s>>>(iters, 2000000000ull, status);
      if (cudaGetLastError() != cudaSuccess || cudaEventRecord(e1, s) != cudaSuccess ||
          cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
        st = LMOE_ERR_CUDA;
      else if (rep > 0 && (best == 0.f || ms < best))
        best = ms;
    }
    uint32_t word = 0;
    if (st == LMOE_OK && cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
      st = LMOE_ERR_CUDA;
    if (st == LMOE_OK && word) st = LMOE_ERR_TIMEOUT;
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (status) cudaFreeAsync(status, s);
  cudaStreamSynchronize(s);
  if (st != LMOE_OK) return st;
  const double k = kind ? 64.0 : 16.0;
  const double flops = (double)pairs * iters * 4 * 2.0 * 256 * 256 * k;
  *tflops = flops / (best * 1e-3) / 1e12;
  return LMOE_OK;
}
