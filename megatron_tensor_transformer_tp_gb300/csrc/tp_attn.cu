// Row kernels of the attention core (the GEMMs run on the tensor-core engine):
//   attn_lse_kernel     merges the per-64-key (max, sum exp) parts of every
//                       score row into its log-sum-exp, in a fixed order;
//   attn_rowdot_kernel  D = sum over a head's columns of dC * C per token,
//                       the softmax backward's row term (sum_keys P dP).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "tp_internal.h"

namespace tp {
namespace {

// rows = pairs * s; part p of row r of pair g at part[(g * P + p) * s + r].
// A block takes 32 rows (lane = row) and 8 slices (warp = slice): slice w
// merges parts w, w + 8, ... of its row, then slice 0 merges the 8 slices in
// order.  Causal rows stop at the part of their own position.
constexpr int kLseSlices = 8;

__device__ __forceinline__ void lse_merge(float& m, float& sum, float xm, float xs) {
  if (xm == -INFINITY) return;  // nothing counted there
  const float nm = fmaxf(m, xm);
  sum = sum * expf(m - nm) + xs * expf(xm - nm);
  m = nm;
}

// Grid: x = 32-row blocks of a pair's rows, y = pair (no 64-bit divisions).
__global__ void __launch_bounds__(32 * kLseSlices) attn_lse_kernel(const float2* __restrict__ part, int P,
                                                                    int64_t s, int64_t g0, int causal,
                                                                    float* __restrict__ lse) {
  __shared__ float sm[kLseSlices][32], ss[kLseSlices][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const int64_t g = g0 + blockIdx.y;
  float m = -INFINITY, sum = 0.f;
  if (r < s) {
    const int plim = causal ? static_cast<int>(r / 64) + 1 : P;
    const float2* q = part + g * P * s + r;
    for (int p = w; p < plim; p += kLseSlices) {
      const float2 x = q[static_cast<int64_t>(p) * s];
      lse_merge(m, sum, x.x, x.y);
    }
  }
  sm[w][lane] = m;
  ss[w][lane] = sum;
  __syncthreads();
  if (w == 0 && r < s) {
    float M = sm[0][lane], S = ss[0][lane];
    for (int k = 1; k < kLseSlices; ++k) lse_merge(M, S, sm[k][lane], ss[k][lane]);
    lse[g * s + r] = M + logf(S);
  }
}

// One warp per (pair, token): D[g * s + t] = sum_c dC[row, c0 + c] C[row, c0 + c]
// over the head's d columns (16-byte loads when d and the offsets allow).
// Grid: x = blocks of 8 tokens, y = pair.
__global__ void __launch_bounds__(256) attn_rowdot_kernel(const __nv_bfloat16* __restrict__ C,
                                                           const __nv_bfloat16* __restrict__ dC,
                                                           int64_t h, int64_t s, int n_heads, int d,
                                                           int64_t g0, int vec, float* __restrict__ D) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= s) return;
  const int64_t g = g0 + blockIdx.y;
  const int64_t b = g / n_heads, j = g - b * n_heads;
  const int64_t off = (b * s + t) * h + j * d;
  float acc = 0.f;
  if (vec) {
    const uint4* c4 = reinterpret_cast<const uint4*>(C + off);
    const uint4* g4 = reinterpret_cast<const uint4*>(dC + off);
    for (int k = lane; k < d / 8; k += 32) {
      const uint4 a = __ldg(c4 + k), e = __ldg(g4 + k);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* e2 = reinterpret_cast<const __nv_bfloat162*>(&e);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 x = __bfloat1622float2(a2[q]), y = __bfloat1622float2(e2[q]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
  } else {
    for (int k = lane; k < d; k += 32) acc = fmaf(__bfloat162float(C[off + k]), __bfloat162float(dC[off + k]), acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) D[g * s + t] = acc;
}

}  // namespace

// Pairs go in grid y, at most 65535 per launch.
constexpr int64_t kMaxGridY = 65535;

cudaError_t launch_attn_lse(const void* part, int P, int64_t s, int64_t rows, int causal, float* lse,
                            cudaStream_t st) {
  const int64_t pairs = rows / s;
  for (int64_t g0 = 0; g0 < pairs; g0 += kMaxGridY) {
    const dim3 grid(static_cast<unsigned>((s + 31) / 32),
                    static_cast<unsigned>(pairs - g0 < kMaxGridY ? pairs - g0 : kMaxGridY));
    attn_lse_kernel<<<grid, 32 * kLseSlices, 0, st>>>(static_cast<const float2*>(part), P, s, g0, causal, lse);
    count_launches(1);
  }
  return cudaGetLastError();
}

cudaError_t launch_attn_rowdot(const void* C, const void* dC, int64_t h, int64_t s, int n_heads, int d,
                               int64_t pairs, float* D, cudaStream_t st) {
  const int vec = (d % 8 == 0) && (h % 8 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0) &&
                  ((reinterpret_cast<uintptr_t>(dC) & 15u) == 0);
  for (int64_t g0 = 0; g0 < pairs; g0 += kMaxGridY) {
    const dim3 grid(static_cast<unsigned>((s + 7) / 8),
                    static_cast<unsigned>(pairs - g0 < kMaxGridY ? pairs - g0 : kMaxGridY));
    attn_rowdot_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(C),
                                             static_cast<const __nv_bfloat16*>(dC), h, s, n_heads, d, g0, vec, D);
    count_launches(1);
  }
  return cudaGetLastError();
}

}  // namespace tp
