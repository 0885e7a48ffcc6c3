// nvfp4q.cuh — NVFP4 quantisation of query heads for the FP4-MMA scoring mode.
//
// The header comment of "indexer_score_topk.cu" plans a phase in which the
// dot products run on the FP4 tensor-core MMA, which takes both operands in
// FP4; the page's query inputs are already "dequantized from FP4". A head row
// of D = 128 values x becomes, in the NVFP4 scheme of the keys (E2M1 elements,
// one E4M3 scale per 16 elements), plus one float32 scale per head that maps
// the head's largest |x| onto 6 * 448 = 2688, the top of the E2M1 x E4M3 range:
//   amax = max |x|;  gq = amax / 2688 (0 when amax == 0)
//   group g of 16:   s_g = E4M3(ag / (6 gq))          (ag = the group's max |x|)
//   element:         c = E2M1(x / (gq s_g)), 0 when s_g == 0
// and dequantises to gq * s_g * e2m1(c). Each operation is one float32
// operation rounded to nearest (division included, whatever the compiler's
// fast-math settings); E4M3() and E2M1() round to the nearest representable
// value, ties to the even code, saturating at 448 and 6; a value rounding to
// zero gets code 0 (no negative zero).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace idx {

constexpr float kNvfp4QRange = 2688.0f;  // 6 (largest E2M1) * 448 (largest finite E4M3)

// E4M3 byte of v >= 0: nearest finite value, ties to the even code, 448 at
// and above 448.
__device__ __forceinline__ uint32_t e4m3_encode_rn(float v) {
  if (!(v > 0.0f)) return 0u;
  if (v >= 448.0f) return 0x7Eu;
  if (v < 0.015625f)   // below 2^-6: the subnormal grid m * 2^-9 (m = 8 is 2^-6 itself, code 8)
    return static_cast<uint32_t>(__float2int_rn(__fmul_rn(v, 512.0f)));
  uint32_t b = __float_as_uint(v);
  b += 0x7FFFFu + ((b >> 20) & 1u);   // round the 23-bit mantissa to 3 bits, ties to even
  const uint32_t e = ((b >> 23) & 0xFFu) - 127u + 7u;
  return (e << 3) | ((b >> 20) & 7u);
}

// Value of a non-negative E4M3 byte (exact).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  if (e == 0u) return __fmul_rn(static_cast<float>(m), 0.001953125f);   // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));               // (1 + m/8) 2^(e-7)
}

// E2M1 code of y: nearest of {0, .5, 1, 1.5, 2, 3, 4, 6} in magnitude, ties to
// the even code, 6 beyond 6; bit 3 is the sign of a non-zero result.
__device__ __forceinline__ uint32_t e2m1_encode_rn(float y) {
  const float a = fabsf(y);
  const uint32_t c = static_cast<uint32_t>(a > 0.25f) + static_cast<uint32_t>(a >= 0.75f) +
                     static_cast<uint32_t>(a > 1.25f) + static_cast<uint32_t>(a >= 1.75f) +
                     static_cast<uint32_t>(a > 2.5f) + static_cast<uint32_t>(a >= 3.5f) +
                     static_cast<uint32_t>(a > 5.0f);
  return (y < 0.0f && c != 0u) ? (c | 8u) : c;
}

// One warp quantises one head row; this lane holds elements 4 lane .. 4 lane + 3
// (x.x first). Gives the lane's four codes in 16 bits (element 4 lane in bits
// 0-3: in each byte the low nibble is the even element), the E4M3 scale of the
// lane's group (lanes 4g .. 4g+3 hold group g) and gq (every lane).
__device__ __forceinline__ void nvfp4_quantize_lane(float4 x, uint32_t &codes16, uint32_t &scale, float &gq) {
  float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
  float ag = amax;
  ag = fmaxf(ag, __shfl_xor_sync(0xFFFFFFFFu, ag, 1));
  ag = fmaxf(ag, __shfl_xor_sync(0xFFFFFFFFu, ag, 2));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  gq = (amax > 0.0f) ? __fdiv_rn(amax, kNvfp4QRange) : 0.0f;
  scale = (ag > 0.0f) ? e4m3_encode_rn(__fdiv_rn(ag, __fmul_rn(6.0f, gq))) : 0u;
  codes16 = 0u;
  if (scale != 0u) {
    const float m = __fmul_rn(gq, e4m3_value(scale));
    codes16 = e2m1_encode_rn(__fdiv_rn(x.x, m)) | (e2m1_encode_rn(__fdiv_rn(x.y, m)) << 4) |
              (e2m1_encode_rn(__fdiv_rn(x.z, m)) << 8) | (e2m1_encode_rn(__fdiv_rn(x.w, m)) << 12);
  }
}

}  // namespace idx
