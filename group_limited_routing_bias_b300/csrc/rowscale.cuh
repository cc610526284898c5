// Activations of the packed-weight GEMMs as f16 with one power-of-two scale
// per token row.  The packed weights (e2m1 x e4m3 products, e4m3 codes) are
// exact in f16, and f16 operands halve the dequantisation work against bf16
// ones, but f16 lacks bf16's range.  So each row of x_perm, and each row of h,
// is multiplied by the power of two that puts its largest magnitude in
// [2^14, 2^15): every bf16 value of the row is then exact in f16, except
// values below 2^-28 of the row's largest, which become f16 subnormals
// (absolute error at most 2^-39 of it).  The MMAs see the scaled rows; the
// epilogues multiply the row's inverse factor back into the fp32 accumulator
// (exactly, a power of two) before the weight scales.  The products are exact
// and the tensor cores' accumulation is invariant under such a scaling, so the
// results are those of bf16 operands.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace beam {

// The power of two that brings a row whose largest magnitude has the fp32
// exponent field e32 into [2^14, 2^15): 2^(141 - e32), at most 2^127 (rows of
// zeros or of values below 2^-113).  Returns its exponent.  bf16 shares the
// fp32 exponent field, so a bf16 magnitude's bits >> 7 serve as e32 as well.
__device__ __forceinline__ int row_scale_exp(uint32_t e32) {
  return min(127, 141 - (int)e32);
}

// Largest |value| of 8 bf16 values (16 bytes), as bf16 magnitude bits.
__device__ __forceinline__ uint32_t bf16x8_absmax_bits(uint4 v, uint32_t m) {
  m = __vmaxu2(m, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                           __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
  return m;
}

// bf16 pairs -> the same values times s (a power of two) as f16 pairs (exact
// but for the subnormal tail); 8 values per 16-byte vector.
__device__ __forceinline__ uint4 bf16x8_to_f16x8_scaled(uint4 v, float s) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16) * s;
    const float hi = __uint_as_float(w[i] & 0xFFFF0000u) * s;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w[i]) : "f"(hi), "f"(lo));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One warp rescales one row of h (bf16 [K], in place) by the factor its
// largest magnitude `hmax_bits` (fp32 bits) asks for; returns the inverse
// factor.  Eight 16-byte loads in flight per lane.
__device__ __forceinline__ float rescale_row_inplace(__nv_bfloat16 *h_row, int K, uint32_t hmax_bits,
                                                     int lane) {
  const int sx = row_scale_exp(hmax_bits >> 23);
  const float sc = ldexpf(1.0f, sx);
  uint4 *row = reinterpret_cast<uint4 *>(h_row);
  const int n4 = K / 8;
  for (int i0 = 0; i0 < n4; i0 += 32 * 8) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * 32 + lane;
      if (i < n4) v[u] = __ldcg(row + i);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * 32 + lane;
      if (i < n4) row[i] = bf16x8_to_f16x8_scaled(v[u], sc);
    }
  }
  return ldexpf(1.0f, -sx);
}

}  // namespace beam
