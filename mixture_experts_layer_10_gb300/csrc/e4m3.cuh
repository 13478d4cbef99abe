// The e4m3 row quantisation step of the FP8 expert GEMMs, shared by the kernels that quantise rows
// (the row quantiser, and the backward's dispatch gather that quantises each token row once while
// it copies it): per row, scale = amax / 448 in fp32 (1 for an all-zero row), codes =
// e4m3(v / scale) rounded to nearest even and saturated.
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

// The row's scale from its largest magnitude.
__device__ __forceinline__ float e4m3_row_scale(float amax) { return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f; }

// Scales whose reciprocal-based quotient is exact (div_by_scale); other rows take the IEEE division.
__device__ __forceinline__ bool e4m3_recip_ok(float scale) { return scale >= 0x1p-80f && scale <= 0x1p80f; }

// v / scale rounded to nearest in fp32, from the row's reciprocal y = RN(1 / scale): q0 = RN(v y) is
// within one ulp of the quotient, the residual v - q0 scale is exact in one fma, and RN(q0 + r y) is
// the correctly rounded quotient (Markstein's theorem on the final correction of a division; it
// needs no underflow or overflow in the steps, which holds for scales in [2^-80, 2^80] whenever the
// quotient is large enough to give a nonzero e4m3 code; rows with other scales use the IEEE
// division).  A zero keeps its sign.
__device__ __forceinline__ float div_by_scale(float v, float scale, float y) {
  const float q0 = v * y;
  const float r = fmaf(-q0, scale, v);
  return copysignf(fmaf(r, y, q0), v);
}

// Eight bf16 values (one 16-byte vector) to eight e4m3 codes.
template <bool kRecip>
__device__ __forceinline__ uint2 encode8_e4m3(const uint4& u, float scale, float y) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t c[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float lo = bf16_lo(w[m]), hi = bf16_hi(w[m]);
    const float2 f2 = kRecip ? make_float2(div_by_scale(lo, scale, y), div_by_scale(hi, scale, y))
                             : make_float2(__fdiv_rn(lo, scale), __fdiv_rn(hi, scale));
    c[m] = (uint32_t)__nv_cvt_float2_to_fp8x2(f2, __NV_SATFINITE, __NV_E4M3);   // .x in the low byte
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

__device__ __forceinline__ uint2 encode8_e4m3(const uint4& u, float scale) {
  return e4m3_recip_ok(scale) ? encode8_e4m3<true>(u, scale, __frcp_rn(scale)) : encode8_e4m3<false>(u, scale, 0.f);
}

// The largest magnitude of eight bf16 values.
__device__ __forceinline__ float amax8_bf16(const uint4& u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float a = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[m])), fabsf(bf16_hi(w[m]))));
  return a;
}

}  // namespace moe
