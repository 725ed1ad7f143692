// fp32 GEMM engine (CUDA cores, fp32 FMA) with the same group / segment /
// epilogue model as the tensor-core engine.  It serves the fp32 dtype, whose
// 1e-4 tolerance rules out tensor-core tf32 rounding.  Operands are addressed
// through explicit (row, column) strides, so K-major and MN-major storage are
// both plain strided reads.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tp_device.cuh"
#include "tp_internal.h"

namespace tp {
namespace {

constexpr int SB = 64;   // output tile edge
constexpr int SK = 16;   // k step
constexpr int STHREADS = 256;

__device__ __forceinline__ void epilogue_elem(const GemmGroup& G, int m, int n, float v) {
  if (m >= G.M || n >= G.N) return;
  switch (G.epi) {
    case EPI_STORE:
    case EPI_BIAS_GELU: {
      if (G.bias != nullptr) v += static_cast<const float*>(G.bias)[n];
      static_cast<float*>(G.out)[static_cast<int64_t>(m) * G.ldo + n] = v;
      if (G.epi == EPI_BIAS_GELU)
        static_cast<float*>(G.out2)[static_cast<int64_t>(m) * G.ldo + n] = gelu_exact_f(v);
      break;
    }
    case EPI_DGELU: {
      const float z = static_cast<const float*>(G.aux)[static_cast<int64_t>(m) * G.ld_aux + n];
      static_cast<float*>(G.out)[static_cast<int64_t>(m) * G.ldo + n] = v * gelu_grad_exact_f(z);
      break;
    }
    case EPI_F32:
    case EPI_SEGSUM: {
      if (G.epi == EPI_SEGSUM) {
        const int64_t id = G.seg_row0 + m;
        const int b = G.seg_offsets[id], e = G.seg_offsets[id + 1];
        float s = 0.f;
        for (int t = b; t < e; ++t)
          s += static_cast<const float*>(G.seg_src)[static_cast<int64_t>(G.seg_perm[t]) * G.ld_seg + n];
        v += s;
      }
      float* o = static_cast<float*>(G.out) + static_cast<int64_t>(m) * G.ldo + n;
      if (G.accumulate) v += *o;
      *o = v;
      break;
    }
    default:
      break;
  }
}

__global__ void __launch_bounds__(STHREADS) simt_gemm_kernel(const __grid_constant__ SimtGemmParams p) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[SK][SB + 1];
  __shared__ float Bs[SK][SB + 1];
  const int tile = blockIdx.x;
  int g = 0;
  while (g + 1 < p.num_groups && tile >= p.grp[g + 1].tile_begin) ++g;
  const GemmGroup& G = p.grp[g];
  const int local = tile - G.tile_begin;
  const int m0 = (local % G.tiles_m) * SB;
  const int n0 = (local / G.tiles_m) * SB;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int s = G.seg_begin; s < G.seg_end; ++s) {
    const SimtSeg& S = p.seg[s];
    for (int k0 = 0; k0 < S.K; k0 += SK) {
      for (int idx = threadIdx.x; idx < SB * SK; idx += STHREADS) {
        const int r = idx / SK, kk = idx % SK;
        const int m = m0 + r, n = n0 + r, k = k0 + kk;
        As[kk][r] = (m < G.M && k < S.K) ? S.A[m * S.sam + k * S.sak] : 0.f;
        Bs[kk][r] = (n < G.N && k < S.K) ? S.B[n * S.sbn + k * S.sbk] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < SK; ++kk) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) epilogue_elem(G, m0 + ty * 4 + i, n0 + tx * 4 + j, acc[i][j]);
}

// Evaluates the epilogues' GELU and GELU' on an array (test hook for the
// device math).
__global__ void gelu_eval_kernel(const float* __restrict__ z, float* __restrict__ y,
                                 float* __restrict__ dy, int64_t n) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float v = z[i];
    if (y) y[i] = gelu_f(v);
    if (dy) dy[i] = gelu_grad_f(v);
  }
}

}  // namespace

cudaError_t launch_gelu_eval(const float* z, float* y, float* dy, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  launch_k(gelu_eval_kernel, static_cast<int>(blocks), 256, 0, s, z, y, dy, n);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_simt_gemm(const SimtGemmParams& p, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  launch_k(simt_gemm_kernel, p.total_tiles, STHREADS, 0, s, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace tp
