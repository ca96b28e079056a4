// Three-term MXFP4 activation records for the block-scaled (kind::mxf4) expert GEMMs.
//
// tcgen05.mma kind::mxf4 multiplies E2M1 by E2M1, each with an E8M0 scale per 32 elements along
// K (OCP Microscaling v1.0).  The routed experts' weights are stored that way (page "What K3
// actually is", srikanthmalla.com, the MXFP4 passage); the activations are not, so each row of
// them is split into three MXFP4 terms whose sum approximates it:
//
//   v ~= q_0 + q_1 + q_2,   q_t = E2M1(r_t / s_t) * s_t,   r_0 = v,  r_{t+1} = r_t - q_t,
//
// per 32-element block, with s_t the smallest power of two >= max|r_t| / 6 (no element
// saturates) and E2M1 rounding to nearest, ties to the even code.  Each term removes most of
// what the previous one left (relative error after three terms ~2e-3 for normal data), and one
// MMA per term against the same weight tile sums them in the fp32 accumulator.
//
// Record of one row of K values (K % 512 == 0), mx3_row_bytes(K) bytes:
//   [term 0: K/2 bytes][term 1: K/2][term 2: K/2][scales of term 0: K/32][term 1: K/32][term 2: K/32]
// with E2M1 element 2i in the low nibble of byte i (the weights' convention) and scale byte e
// meaning 2^(e - 127).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace lmoe {

constexpr int kMxTerms = 3;

__host__ __device__ constexpr int64_t mx3_row_bytes(int64_t K) { return kMxTerms * (K / 2) + kMxTerms * (K / 32); }
__host__ __device__ constexpr int64_t mx3_scale_offset(int64_t K) { return kMxTerms * (K / 2); }

namespace mx {

// Biased E8M0 exponent of the smallest power of two s with amax <= 6 s, clamped to [1, 253]
// (amax = 0 gives 1; every code is then 0).  With amax = m 2^E, m in [1, 2): 6 * 2^(E-2) =
// 1.5 * 2^E covers m <= 1.5, else 2^(E-1) is needed.
__device__ __forceinline__ uint32_t scale_byte(float amax) {
  const uint32_t b = __float_as_uint(amax);
  int e = (int)((b >> 23) & 0xFFu) - 2 + ((b & 0x7FFFFFu) > 0x400000u ? 1 : 0);
  e = e < 1 ? 1 : (e > 253 ? 253 : e);
  return (uint32_t)e;
}

// 8 fp32 values x[0..7] (already divided by the scale, |x| <= 6) -> E2M1 nibbles, element i at
// bits 4i of the returned word (round to nearest, ties to the even code: cvt.rn.satfinite), and
// the E2M1 values back as 4 f16x2 words (dec[j] holds elements 2j, 2j+1; exact in fp16).
__device__ __forceinline__ uint32_t e2m1x8_round(const float (&x)[8], uint32_t (&dec)[4]) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %6, %5;\n\t"   // the second source lands in the low nibble
      "cvt.rn.satfinite.e2m1x2.f32 b1, %8, %7;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %10, %9;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %12, %11;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %4, b3;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w), "=r"(dec[0]), "=r"(dec[1]), "=r"(dec[2]), "=r"(dec[3])
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  // a negative value that rounds to zero keeps its sign bit; store +0 (code 0) instead
  const uint32_t mag = w & 0x77777777u;
  const uint32_t nonzero = (mag + 0x77777777u) & 0x88888888u;  // bit 3 of a nibble: magnitude != 0
  return mag | (w & nonzero);
}

// Split one 32-element block r[] (overwritten with the final residual) into kMxTerms MXFP4
// terms: packed[t][w] holds elements 8w .. 8w+7 (element i at bits 4*(i%8)), sc[t] the scale byte.
__device__ __forceinline__ void quantize_block(float (&r)[32], uint32_t (&packed)[kMxTerms][4],
                                               uint32_t (&sc)[kMxTerms]) {
#pragma unroll
  for (int t = 0; t < kMxTerms; ++t) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(r[i]));
    const uint32_t e = scale_byte(amax);
    const float s = __uint_as_float(e << 23);            // 2^(e - 127)
    const float inv = __uint_as_float((254u - e) << 23);  // 2^(127 - e), exact
    sc[t] = e;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = r[8 * w + i] * inv;  // exact: a power of two
      uint32_t dec[4];
      packed[t][w] = e2m1x8_round(x, dec);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 q = __half22float2(*reinterpret_cast<const __half2*>(&dec[j]));
        r[8 * w + 2 * j] = fmaf(-q.x, s, r[8 * w + 2 * j]);  // q * s is exact; the residual keeps what is left
        r[8 * w + 2 * j + 1] = fmaf(-q.y, s, r[8 * w + 2 * j + 1]);
      }
    }
  }
}

// ---------------------------------------------------------------- MXFP8 activation records
// One term: E4M3 elements with an E8M0 scale per 32 (OCP Microscaling v1.0), for the
// kind::mxf8f6f4 expert GEMMs (E2M1 weights x E4M3 activations; page "What K3 actually is",
// srikanthmalla.com: K3's quantization-aware training with MXFP8 activations).  Scale: the
// smallest power of two s with amax <= 448 s (no element saturates); elements round to nearest,
// ties to the even code; a value that rounds to zero is stored as +0.  Record of one row of K
// values, mx8_row_bytes(K) bytes: [K E4M3 codes][K/32 scale bytes].

// Biased E8M0 exponent of the smallest power of two s with amax <= 448 s, clamped to [1, 253]:
// with amax = m 2^E, m in [1, 2), 448 * 2^(E-8) = 1.75 * 2^E covers m <= 1.75.
__device__ __forceinline__ uint32_t scale_byte8(float amax) {
  const uint32_t b = __float_as_uint(amax);
  int e = (int)((b >> 23) & 0xFFu) - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  e = e < 1 ? 1 : (e > 253 ? 253 : e);
  return (uint32_t)e;
}

// 32 values r[] -> 32 E4M3 codes (element i in byte i of codes[i / 4]) and the scale byte.
__device__ __forceinline__ void quantize_block8(const float (&r)[32], uint32_t (&codes)[8], uint32_t& sc) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(r[i]));
  const uint32_t e = scale_byte8(amax);
  const float inv = __uint_as_float((254u - e) << 23);  // 2^(127 - e), exact
  sc = e;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t lo, hi;
    // cvt.rn.satfinite.e4m3x2.f32 d, a, b: b lands in the low byte
    asm("{\n\t.reg .b16 h;\n\tcvt.rn.satfinite.e4m3x2.f32 h, %2, %1;\n\tcvt.u32.u16 %0, h;\n\t}"
        : "=r"(lo) : "f"(r[4 * w] * inv), "f"(r[4 * w + 1] * inv));
    asm("{\n\t.reg .b16 h;\n\tcvt.rn.satfinite.e4m3x2.f32 h, %2, %1;\n\tcvt.u32.u16 %0, h;\n\t}"
        : "=r"(hi) : "f"(r[4 * w + 2] * inv), "f"(r[4 * w + 3] * inv));
    uint32_t v = lo | (hi << 16);
    // -0 (sign bit over a zero magnitude) -> +0
    const uint32_t mag = v & 0x7F7F7F7Fu;
    const uint32_t nonzero = ((mag + 0x7F7F7F7Fu) & 0x80808080u);  // bit 7 of a byte: magnitude != 0
    codes[w] = mag | (v & nonzero);
  }
}

}  // namespace mx

__host__ __device__ constexpr int64_t mx8_row_bytes(int64_t K) { return K + K / 32; }
__host__ __device__ constexpr int64_t mx8_scale_offset(int64_t K) { return K; }

}  // namespace lmoe
