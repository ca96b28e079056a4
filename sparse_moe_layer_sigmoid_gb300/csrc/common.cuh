// Shared device/host helpers for the LatentMoE kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace lmoe {

// Bits of the device status word.  Kernels OR these in; the host maps them to
// LMOE_ERR_TIMEOUT / LMOE_ERR_DEVICE_CHECK.
enum : uint32_t { kStatusTimeout = 1u, kStatusDeviceCheck = 2u };
// Diagnostic bits naming the wait that ran out (bits 8..15 of the status word).
enum : uint32_t {
  kWaitProducer = 1u << 8,    // producer: stage free
  kWaitAccFree = 1u << 9,     // MMA: accumulator drained
  kWaitFull = 1u << 10,       // MMA: operands landed
  kWaitConverted = 1u << 11,  // MMA: converted operands ready
  kWaitAccFull = 1u << 12,    // epilogue: accumulator complete
  kWaitMmaDone = 1u << 13     // producer: own MMA finished with a stage (paired CTAs)
};
// Diagnostic bit beside kStatusDeviceCheck: a router logit recomputed exactly differed from the
// GEMM's by more than half the margin the top-k selection relies on.
constexpr uint32_t kStatusRouterMargin = 1u << 16;

enum DType : int { kF32 = 0, kBF16 = 1, kMXFP4 = 2, kF16 = 3 /* internal: fp16 activations */ };

// Rows of one grouped-GEMM M tile; the dispatch step builds its tile list in these units.
constexpr int kTileM = 128;
// Rows of one unit of the swapped-operand (decode) expert GEMM: a second, finer tile list.
constexpr int kTileS = 16;
// Rows of the M tile a pair of clustered CTAs shares (each CTA computes 128 of them).
constexpr int kTileP = 256;
// Token rows of one tile of the block-scaled (MXFP4) expert GEMM.
constexpr int kTileMx = 192;
// Tokens per dispatch chunk (one CTA, one bit per token in the per-expert masks).
constexpr int kDispatchChunk = 256;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu(float v) { return v / (1.0f + expf(-v)); }

__device__ __forceinline__ void report(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

}  // namespace lmoe
