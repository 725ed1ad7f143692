// Device helpers shared by the GEMM engines: GELU and its derivative, bf16
// conversion, and the per-element epilogue of the fp32 engine.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "tp_internal.h"

namespace tp {

// Hardware approximations (PTX ex2.approx.ftz / rcp.approx.ftz: one MUFU
// operation each, results that would be denormal flush to zero).  Measured on
// GB300, the non-ftz forms add fix-up instructions that cost about a third of
// the GELU epilogue's time.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_ftz(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// erf(x) by Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26: erf(x) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) e^{-x^2},
// t = 1 / (1 + p x) for x >= 0, odd in x, |error| <= 1.5e-7.  e^{-x^2} is
// 2^{-x^2 log2 e}.  The factor e^{-x^2} is returned too: with x = z / sqrt 2
// it is the e^{-z^2/2} of the normal density, so GELU' reuses it.
__device__ __forceinline__ float erf_as7126(float x, float& e_mx2) {
  const float ax = fabsf(x);
  const float t = rcp_ftz(fmaf(0.3275911f, ax, 1.0f));
  float q = fmaf(1.061405429f, t, -1.453152027f);
  q = fmaf(q, t, 1.421413741f);
  q = fmaf(q, t, -0.284496736f);
  q = fmaf(q, t, 0.254829592f);
  e_mx2 = ex2_ftz(ax * (ax * -1.4426950408889634f));
  return copysignf(fmaf(-q * t, e_mx2, 1.0f), x);
}

// GELU(z) = z * Phi(z), Phi(z) = (1 + erf(z / sqrt 2)) / 2 (exact erf form; the
// activation between the column- and row-parallel linears of the MLP block,
// "Megatron tensor / model parallelism" notes, section MLP层).
__device__ __forceinline__ float gelu_f(float z) {
  float e;
  const float r = erf_as7126(z * 0.70710678118654752f, e);
  return 0.5f * z * (1.0f + r);
}

// d GELU / dz = Phi(z) + z * phi(z), phi(z) = exp(-z^2 / 2) / sqrt(2 pi).
__device__ __forceinline__ float gelu_grad_f(float z) {
  float e;
  const float r = erf_as7126(z * 0.70710678118654752f, e);
  return fmaf(z * 0.39894228040143268f, e, 0.5f * (1.0f + r));
}

// The same two functions through CUDA's erff / expf, for the fp32 engine:
// its 1e-4 bar is also met element by element, which the approximation's
// 1.5e-7 absolute error in erf does not allow near the zero of GELU'.
__device__ __forceinline__ float gelu_exact_f(float z) {
  return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
}
__device__ __forceinline__ float gelu_grad_exact_f(float z) {
  return fmaf(z * 0.39894228040143268f, expf(-0.5f * z * z), 0.5f * (1.0f + erff(z * 0.70710678118654752f)));
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
