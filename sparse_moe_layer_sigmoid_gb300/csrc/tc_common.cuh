// Helpers shared by the tcgen05 GEMM kernels: tensor-map encoding (TMA descriptors) and the
// in-shared-memory E2M1 -> fp16 conversion of MXFP4 weights.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace lmoe {
namespace tc {

constexpr int BK = 64;          // K elements per pipeline stage (128 bytes of 16-bit data)

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// fp16 bits (duplicated into both halves) of 2^(s-127) for an E8M0 byte s; sets *bad when the
// decoded block could leave the exact fp16 range (6 * scale above 65504) or s is NaN.
__device__ __forceinline__ uint32_t e8m0_to_f16x2(uint32_t s, bool* bad) {
  const int e = (int)s - 127;
  uint32_t h;
  if (s == 255u || e > 13) {
    *bad = true;
    h = 0;
  } else if (e >= -14) {
    h = (uint32_t)(e + 15) << 10;
  } else if (e >= -24) {
    h = 1u << (e + 24);  // subnormal
  } else {
    h = 0;
  }
  return h | (h << 16);
}

// 32 E2M1 values (16 bytes, element 2i in the low nibble of byte i) times a scale -> 16 f16x2.
__device__ __forceinline__ void e2m1x32_to_f16(const uint4& q, uint32_t scale2, uint32_t (&o)[16]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  const __half2 sc = *reinterpret_cast<const __half2*>(&scale2);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t r0, r1, r2, r3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(w[i]));
    const uint32_t rr[4] = {r0, r1, r2, r3};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&rr[j]), sc);
      o[4 * i + j] = *reinterpret_cast<uint32_t*>(&v);
    }
  }
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}


typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
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

// 16-bit operand [depth][rows][cols]: boxes of 64 cols x box_rows rows, 128-byte swizzle.
inline bool make_map(CUtensorMap* m, const TcOperand& op, int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !op.ptr) return false;
  const int64_t depth_stride = op.depth > 1 ? op.depth_stride : op.rows * op.row_stride;
  cuuint64_t dims[3] = {(cuuint64_t)op.cols, (cuuint64_t)op.rows, (cuuint64_t)op.depth};
  cuuint64_t strides[2] = {(cuuint64_t)op.row_stride * 2, (cuuint64_t)depth_stride * 2};
  cuuint32_t box[3] = {BK, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(op.ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed E2M1 operand [depth][rows][cols/2 bytes] (element strides in `op`): boxes of
// box_bytes bytes (2 elements per byte) x box_rows rows, no swizzle, or the 128-byte swizzle
// (box_bytes == 128) when the reader takes column slices of the rows.
inline bool make_map_fp4(CUtensorMap* m, const TcOperand& op, int box_rows = 128, int box_bytes = BK / 2,
                         bool swizzle128 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !op.ptr) return false;
  const int64_t rb = op.row_stride / 2;  // bytes per row
  const int64_t depth_stride = op.depth > 1 ? op.depth_stride / 2 : op.rows * rb;
  cuuint64_t dims[3] = {(cuuint64_t)(op.cols / 2), (cuuint64_t)op.rows, (cuuint64_t)op.depth};
  cuuint64_t strides[2] = {(cuuint64_t)rb, (cuuint64_t)depth_stride};
  cuuint32_t box[3] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(op.ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace tc
}  // namespace lmoe
