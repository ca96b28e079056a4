// Helpers shared by the tcgen05 GEMM kernels: tensor-map encoding (TMA descriptors), the
// in-shared-memory E2M1 -> fp16 conversion of MXFP4 weights, and the accumulator epilogue.
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

// Epilogue of one warp over a 128 x BN fp32 accumulator: `t_row` addresses the warp's 32 TMEM
// lanes (one output row each, row `row` of C, stored only when `live`).  GLU epilogues read gate
// columns [0, BN/2) and up columns [BN/2, BN) and store BN/2 outputs SiLU(gate) * up; the
// others store columns n0 .. n0+BN-1 (clipped at N) of acc, times row_scale[row] for kEpiScale*.
template <int BN, int EPI>
__device__ __forceinline__ void store_accumulator(uint32_t t_row, int row, bool live, int n0, int N, void* C,
                                                  int64_t ldc, const float* row_scale) {
  constexpr bool GLU = EPI == kEpiGluBF16 || EPI == kEpiGluF16;
  constexpr bool SCALE = EPI == kEpiScaleBF16 || EPI == kEpiScaleF16;
  constexpr bool OUT_F16 = EPI == kEpiF16 || EPI == kEpiGluF16 || EPI == kEpiScaleF16;
  constexpr int BN_OUT = GLU ? BN / 2 : BN;
  if (GLU) {
    uint16_t* out = static_cast<uint16_t*>(C) + (int64_t)row * ldc + n0;
#pragma unroll 1
    for (int c = 0; c < BN_OUT; c += 32) {
      uint32_t g[32], u[32];
      ptx::tmem_ld_32x32b_x32(t_row + c, g);
      ptx::tmem_ld_32x32b_x32(t_row + BN_OUT + c, u);
      ptx::tmem_ld_wait();
      if (live) {
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
          const float a1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
          packed[i] = OUT_F16 ? pack_f16x2(a0, a1) : pack_bf16x2(a0, a1);
        }
        uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
      }
    }
  } else {
    const float sc = (SCALE && live) ? row_scale[row] : 1.0f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      if (n0 + c >= N) break;  // ragged last column tile (fp32: N % 4 == 0, else N % 32 == 0)
      uint32_t r[32];
      ptx::tmem_ld_32x32b_x32(t_row + c, r);
      ptx::tmem_ld_wait();
      if (live) {
        if (EPI == kEpiF32) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(C) + (int64_t)row * ldc + n0 + c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (n0 + c + 4 * i < N) dst[i] = make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
        } else {
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float v0 = __uint_as_float(r[2 * i]) * sc, v1 = __uint_as_float(r[2 * i + 1]) * sc;
            packed[i] = OUT_F16 ? pack_f16x2(v0, v1) : pack_bf16x2(v0, v1);
          }
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(C) + (int64_t)row * ldc + n0 + c);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
      }
    }
  }
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

// Gate/up weights [depth][2h][cols] (gate rows 0..h-1, up rows h..2h-1) viewed as 5-D
// {cols, 16, 2, h/16, depth} with a box of {64 elements, 16, 2, groups, 1}: one load brings
// `groups` x (16 gate rows, then the matching 16 up rows), 128-byte swizzled rows in that order.
// `fp4`: the operand holds packed E2M1 bytes (cols/2 bytes per row, 128-byte box rows = 256
// elements); otherwise bf16.  `padded4` (with fp4): 4-bit elements that land one per byte
// (CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B: 16 packed elements padded to 16 bytes), 128-element
// boxes, for MMA kinds that read 4-bit operands from byte containers.
inline bool make_map_glu_interleaved(CUtensorMap* m, const TcOperand& op, int glu_h, int groups, bool fp4 = false,
                                     bool padded4 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !op.ptr || glu_h % 16 || op.rows != 2 * (int64_t)glu_h) return false;
  const int64_t rs = fp4 ? op.row_stride / 2 : op.row_stride * 2;  // bytes per row
  const int64_t depth_stride = op.depth > 1 ? (fp4 ? op.depth_stride / 2 : op.depth_stride * 2) : op.rows * rs;
  const bool pad = fp4 && padded4;
  cuuint64_t dims[5] = {(cuuint64_t)(fp4 && !pad ? op.cols / 2 : op.cols), 16, 2, (cuuint64_t)(glu_h / 16),
                        (cuuint64_t)op.depth};
  cuuint64_t strides[4] = {(cuuint64_t)rs, (cuuint64_t)(glu_h * rs), (cuuint64_t)(16 * rs), (cuuint64_t)depth_stride};
  cuuint32_t box[5] = {fp4 ? 128u : (cuuint32_t)BK, 16, 2, (cuuint32_t)groups, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(m, pad ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B
                    : (fp4 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16),
             5, const_cast<void*>(op.ptr),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 16-bit operand [rows][cols] viewed as 3-D {64, rows, cols/64}: a box of {64, box_rows, slabs}
// lands as `slabs` consecutive 64-column blocks of box_rows 128-byte swizzled rows each.
inline bool make_map_kslabs(CUtensorMap* m, const TcOperand& op, int box_rows, int slabs) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !op.ptr || op.cols % BK || op.depth != 1) return false;
  cuuint64_t dims[3] = {(cuuint64_t)BK, (cuuint64_t)op.rows, (cuuint64_t)(op.cols / BK)};
  cuuint64_t strides[2] = {(cuuint64_t)op.row_stride * 2, (cuuint64_t)BK * 2};
  cuuint32_t box[3] = {BK, (cuuint32_t)box_rows, (cuuint32_t)slabs};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(op.ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed E2M1 operand [depth][rows][cols/2 bytes] (element strides in `op`): boxes of
// box_bytes bytes (2 elements per byte) x box_rows rows, no swizzle, or the 128-byte swizzle
// (box_bytes == 128) when the reader takes column slices of the rows.
// `padded4`: 4-bit elements landing one per byte (see make_map_glu_interleaved), boxes of
// box_bytes elements.
inline bool make_map_fp4(CUtensorMap* m, const TcOperand& op, int box_rows = 128, int box_bytes = BK / 2,
                         bool swizzle128 = false, bool padded4 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !op.ptr) return false;
  const int64_t rb = op.row_stride / 2;  // bytes per row
  const int64_t depth_stride = op.depth > 1 ? op.depth_stride / 2 : op.rows * rb;
  cuuint64_t dims[3] = {(cuuint64_t)(padded4 ? op.cols : op.cols / 2), (cuuint64_t)op.rows, (cuuint64_t)op.depth};
  cuuint64_t strides[2] = {(cuuint64_t)rb, (cuuint64_t)depth_stride};
  cuuint32_t box[3] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, padded4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
             const_cast<void*>(op.ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace tc
}  // namespace lmoe
