// NVFP4 quantisation of activations (the W4A4 mode's reading of the NVFP4
// checkpoint format named on "Reflection Releases Beam ...", section "Where
// Beam Saves and Where the Memory Bill Comes In": one E4M3 scale per 16
// consecutive values of a row and a static fp32 global scale g per tensor).
// For one block of 16 values v, in fp32 with IEEE rounding:
//   amax = max |v|,  s = e4m3_rne_satfinite(amax / (6 g)),  scale = e4m3(s) * g,
//   code_i = e2m1_rne_satfinite(v_i / scale),  all codes 0 when scale == 0.
// Two codes per byte, the even index in the low nibble.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace beam {

// e4m3 code -> fp32 (exact: every E4M3 value is an f16 value)
__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
  uint32_t h2;
  const uint16_t c16 = (uint16_t)(code & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c16));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// fp32 -> e4m3 code, round to nearest even, saturating at 448
__device__ __forceinline__ uint32_t float_to_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// two fp32 values -> one byte of e2m1 codes (lo in bits 0..3), nearest even, saturating at 6
__device__ __forceinline__ uint32_t float2_to_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// Quantises one block of 16 values; returns the scale code and sets the eight
// code bytes (little-endian: byte i holds values 2i and 2i+1) in codes.
__device__ __forceinline__ uint32_t nvfp4_quantize_block(const float (&v)[16], float six_g, float g,
                                                         uint2 &codes) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t sc = float_to_e4m3(__fdiv_rn(amax, six_g));
  const float scale = __fmul_rn(e4m3_to_float(sc), g);
  uint32_t w[2] = {0u, 0u};
  if (scale != 0.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t b = float2_to_e2m1x2(__fdiv_rn(v[2 * i], scale), __fdiv_rn(v[2 * i + 1], scale));
      w[i >> 2] |= b << (8 * (i & 3));
    }
  }
  codes = make_uint2(w[0], w[1]);
  return sc;
}

}  // namespace beam
