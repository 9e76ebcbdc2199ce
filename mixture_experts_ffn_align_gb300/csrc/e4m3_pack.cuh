// Packing of fp32 values into e4m3fn codes, two per conversion instruction.
// Same rounding as f32_to_e4m3 in moe_common.cuh (round to nearest even,
// saturating to +-448): __nv_cvt_float2_to_fp8x2 converts a pair at once,
// the first value into the low byte.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

// v / s rounded to nearest fp32, for many v sharing one positive normal
// divisor s with r = __frcp_rn(s): q0 = v * r is within an ulp or two of
// v / s, the remainder v - s * q0 is exact under an FMA, and one correction
// step q0 + rem * r gives the correctly rounded quotient (Markstein's
// division correction).  A zero remainder means q0 is already exact; it is
// returned as is, which also keeps the sign of a -0 quotient (the correction
// would add +0 and turn it into +0, unlike IEEE division).
__device__ __forceinline__ float quot_rn(float v, float s, float r) {
  const float q0 = v * r;
  const float rem = fmaf(-q0, s, v);
  return rem == 0.0f ? q0 : fmaf(rem, r, q0);
}

// Four values -> one 32-bit word, value j in byte j.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | hi << 16;
}

}  // namespace moe
