// NVFP4 helpers: the block quantization of the FlashInferFP4MoE layer (sglang
// `fused_moe_triton/layer.py` page: `fp4_quantize(x, global_scale, 16, ...)` on the hidden
// states, the same quantization on the activation before the second GEMM) and the e2m1 /
// e4m3 -> f16 expansions of the expert GEMMs.
//
// Per block of 16 consecutive values, every step one IEEE fp32 operation:
//   amax = max |x|;  sf = e4m3(g * (amax / 6))  (round to nearest even, saturating at 448);
//   r = g / sf (0 when sf is 0);  q = e2m1(x * r)  (round to nearest even, saturating at 6).
// Dequantized the block holds q * sf / g. q * sf is exact in f16 (at most 6 significant
// bits, magnitudes in [2^-10, 2688]), so the GEMMs take q * sf as their f16 operands and
// apply the per-tensor scales in the epilogue.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace gbmoe {

constexpr int kFp4Block = 16;   // values per block scale
constexpr float kE2m1Max = 6.f;

// The fp32 block scale (an e4m3 value) and its byte, from the block's amax.
__device__ __forceinline__ float fp4_block_scale(float amax, float g, uint8_t& code) {
  const float sfv = __fmul_rn(g, __fdiv_rn(amax, kE2m1Max));
  code = (uint8_t)__nv_cvt_float_to_fp8(sfv, __NV_SATFINITE, __NV_E4M3);
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(__half(h));
}

// The e2m1 byte of (a, b): a in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest);
}

// f16x2 of the two e2m1 codes of a byte (low nibble in the low half).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  const __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)byte, __NV_E2M1);
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}

// Quantizes one block of 16 fp32 values with per-tensor scale g: the 16 codes packed low
// nibble first into q[0..1] (element 0 in bits 0..3 of q[0]), the scale byte, and the f16
// values q * sf packed in pairs into v[0..7] (element 0 in the low half of v[0]).
__device__ __forceinline__ void fp4_quant_block(const float (&x)[16], float g, uint32_t (&q)[2],
                                                uint8_t& sf_code, uint32_t (&v)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const float sf = fp4_block_scale(amax, g, sf_code);
  const float r = sf > 0.f ? __fdiv_rn(g, sf) : 0.f;
  const __half2 s2 = __float2half2_rn(sf);  // exact: sf is an e4m3 value
  q[0] = q[1] = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t b = e2m1x2(__fmul_rn(x[2 * i], r), __fmul_rn(x[2 * i + 1], r));
    q[i >> 2] |= b << (8 * (i & 3));
    const uint32_t h = e2m1x2_to_f16x2(b);
    __half2 hv;
    memcpy(&hv, &h, 4);
    hv = __hmul2(hv, s2);  // exact: both operands have few significant bits
    memcpy(&v[i], &hv, 4);
  }
}

}  // namespace gbmoe
