// Device helpers shared by the GEMM engines: GELU and its derivative, bf16
// conversion, and the per-element epilogue of the fp32 engine.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "tp_internal.h"

namespace tp {

// GELU(z) = z * Phi(z), Phi(z) = (1 + erf(z / sqrt 2)) / 2 (exact erf form; the
// activation between the column- and row-parallel linears of the MLP block,
// "Megatron tensor / model parallelism" notes, section MLP层).
__device__ __forceinline__ float gelu_f(float z) {
  return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
}

// d GELU / dz = Phi(z) + z * phi(z), phi(z) = exp(-z^2 / 2) / sqrt(2 pi).
__device__ __forceinline__ float gelu_grad_f(float z) {
  const float cdf = 0.5f * (1.0f + erff(z * 0.70710678118654752f));
  const float pdf = expf(-0.5f * z * z) * 0.39894228040143268f;
  return fmaf(z, pdf, cdf);
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void unpack_bf16x2(uint32_t u, float& lo, float& hi) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  lo = __low2float(v);
  hi = __high2float(v);
}

}  // namespace tp
