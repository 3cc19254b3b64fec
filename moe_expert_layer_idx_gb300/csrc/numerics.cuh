// Block-scale arithmetic shared by the quantiser and the L1 epilogue.
//
// Scale rule: for a block of 32 values with largest magnitude a, the UE8M0
// exponent s is the smallest integer with a <= F * 2^s (F = 448 for E4M3, 6
// for E2M1), clamped to [-127, 127]; an all-zero block takes s = 0.  It is
// computed exactly from the fp32 bit pattern of a: with a = m * 2^P,
// m in [1, 2), s = P - 8 if m <= 1.75 else P - 7 (E4M3), and s = P - 2 if
// m <= 1.5 else P - 1 (E2M1).  Elements are RNE(v / 2^s); the division by a
// power of two is exact in fp32 except where the quotient is far below the
// smallest element step, where every rounding gives zero anyway.
#pragma once
#include <cstdint>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

namespace mm {

template <bool kE4M3>
__device__ __forceinline__ int block_scale_exp(float amax) {
  const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  const uint32_t e = b >> 23, m = b & 0x7FFFFFu;
  if (e == 0) return (m == 0) ? 0 : -127;     // zero block; subnormal amax -> below -127
  const int P = (int)e - 127;
  int s;
  if (kE4M3) s = (m <= 0x600000u) ? P - 8 : P - 7;    // 1.75 = 1 + 0x600000 / 2^23
  else       s = (m <= 0x400000u) ? P - 2 : P - 1;    // 1.5  = 1 + 0x400000 / 2^23
  return max(-127, min(127, s));
}

// 2^-s as an fp32 value, s in [-127, 127].
__device__ __forceinline__ float exp2_neg(int s) {
  const int ef = 127 - s;
  return ef >= 1 ? __uint_as_float((uint32_t)ef << 23) : __uint_as_float(1u << (22 + ef));
}

// Round-to-nearest-even into E4M3 (saturating); the sign bit follows v, so a
// negative value that rounds to zero is negative zero.
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  const uint32_t c = (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
  return (c | ((__float_as_uint(v) >> 24) & 0x80u)) & 0xFFu;
}

// Round-to-nearest-even into E2M1 (saturating), sign bit as above.
__device__ __forceinline__ uint32_t e2m1_code(float v) {
  const uint32_t c = (uint32_t)__nv_cvt_float_to_fp4(v, __NV_E2M1, cudaRoundNearest);
  return (c | ((__float_as_uint(v) >> 28) & 0x8u)) & 0xFu;
}

}  // namespace mm
