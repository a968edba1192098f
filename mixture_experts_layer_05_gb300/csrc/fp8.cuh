// e4m3 (float8_e4m3fn) helpers of the FP8 w8a8 path: the per-group scale and the
// conversion of fp32 values to packed e4m3 bytes.
//
// The per-token-group-128 quant of the sglang `models/deepseek_v2.py` page
// (`DeepseekV2MoE._maybe_quant_moe_input_once`, the post-SiLU quant of
// `DeepseekV2MLP.forward`): s = max(amax, 1e-10) / 448 and q = e4m3(x / s), both the
// scale and the quotient one IEEE fp32 division, the conversion round-to-nearest-even
// and saturating at +-448 (448 is the largest finite e4m3fn value).
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace gbmoe {

constexpr float kE4m3Max = 448.f;
constexpr float kQuantScaleFloor = 1e-10f;

__device__ __forceinline__ float fp8_group_scale(float amax) {
  return __fdiv_rn(fmaxf(amax, kQuantScaleFloor), kE4m3Max);
}

// Four e4m3 bytes of (a, b, c, d) / s, a in the lowest byte.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d, float s) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
      make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s)), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
      make_float2(__fdiv_rn(c, s), __fdiv_rn(d, s)), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

}  // namespace gbmoe
