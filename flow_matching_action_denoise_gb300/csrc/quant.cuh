// Activation quantisers of the consumer kernels (row kernel, attention epilogue,
// NVFP4-weight GEMM epilogue).
//
// Four-bit activations (news article "FlashRT-PAI", the four-bit inference path):
// a row is cut into blocks of 16 consecutive K elements; with the static fp32 tensor
// scale ts of the quant point, each block gets its own E4M3 block scale
// bs = E4M3_RNE_sat(amax_block / fp32(6 ts)) and each element the E2M1 code
// e = E2M1_RNE_sat(h / fp32(bs ts)) (0 where bs ts = 0). The GEMM operand is stored as
// the f16 value e * bs, which is exact (at most six significant bits, magnitude within
// [2^-10, 2688]); ts joins the weight's tensor scale in the consumer's dequantisation.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

namespace fm {

// value of E4M3_RNE_sat(x) (OCP E4M3FN, saturating at +-448)
__device__ __forceinline__ float e4m3_round(float x) {
  const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(c, __NV_E4M3)));
}

// Block scale value bs and the divisor fp32(bs * ts) of a block with the given amax.
__device__ __forceinline__ float nvfp4_block(float amax, float ts, float* den) {
  const float bs = e4m3_round(__fdiv_rn(amax, __fmul_rn(6.0f, ts)));
  *den = __fmul_rn(bs, ts);
  return bs;
}

// f16 values e * bs of two elements of a block (den = fp32(bs * ts) from nvfp4_block).
__device__ __forceinline__ __half2 nvfp4_pair(float a, float b, float bs, float den) {
  if (!(den > 0.f)) return __floats2half2_rn(0.f, 0.f);
  const __nv_fp4x2_storage_t e =
      __nv_cvt_float2_to_fp4x2(make_float2(__fdiv_rn(a, den), __fdiv_rn(b, den)), __NV_E2M1, cudaRoundNearest);
  const __half2_raw r = __nv_cvt_fp4x2_to_halfraw2(e, __NV_E2M1);
  const __half hb = __float2half_rn(bs);   // exact: bs is an E4M3 value
  return __hmul2(__half2(r), __half2(hb, hb));
}

// f16 value e * bs of one element of a block.
__device__ __forceinline__ __half nvfp4_one(float a, float bs, float den) {
  if (!(den > 0.f)) return __float2half_rn(0.f);
  const __nv_fp4x2_storage_t e =
      __nv_cvt_float2_to_fp4x2(make_float2(__fdiv_rn(a, den), 0.f), __NV_E2M1, cudaRoundNearest);
  const __half2_raw r = __nv_cvt_fp4x2_to_halfraw2(e, __NV_E2M1);
  return __hmul(__low2half(__half2(r)), __float2half_rn(bs));
}

}  // namespace fm
