// Row kernels of the attention core (the GEMMs run on the tensor-core engine):
//   attn_norm_kernel    merges the per-64-key (max, sum exp) parts of every
//                       score row into its log-sum-exp, in a fixed order, and
//                       turns the row's stored exponentials into P;
//   attn_rowdot_kernel  D = sum over a head's columns of dC * C per token,
//                       the softmax backward's row term (sum_keys P dP).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "tp_internal.h"
#include "tp_philox.cuh"

namespace tp {
namespace {

// One warp per score row (query) of a pair; part p of row r of pair g at
// part[(g * P + p) * s + r].  The row's log-sum-exp: lane l merges parts l,
// l + 32, ... in order, then the lanes merge by a butterfly over lane
// distances 16, 8, 4, 2, 1 (each merge is commutative, so every lane ends with
// the same value).  Causal rows stop at the part of their own position.  The
// probabilities: lane l takes the row's 8-column chunks l, l + 32, ...
// (16-byte accesses; s % 8 == 0), P = e exp(m_part - lse) over the stored e
// of the scores launch (a chunk that starts after the row's position is
// written as zeros without being read; inside the row's last chunk the scores
// launch already wrote zeros).  The first chunks' loads are issued before the
// statistics, so their latency overlaps the merge.
// With attention dropout (DROP) the kernel also draws the keep bits, one
// Philox4x32-10 block per 8-column chunk, stores them as the keep words
// (32 keys per word; a word whose first key lies after the row's position is
// zero, as the keep-word kernel writes it) and writes Pd = P keep / (1 - p).
constexpr int kNormWarps = 8;  // rows per block
constexpr int kNormBatch = 4;  // chunks a lane loads before it stores

__device__ __forceinline__ void lse_merge(float& m, float& sum, float xm, float xs) {
  if (xm == -INFINITY) return;  // nothing counted there
  const float nm = fmaxf(m, xm);
  sum = sum * expf(m - nm) + xs * expf(xm - nm);
  m = nm;
}

__device__ __forceinline__ void scale8(uint4 e, float f, float* v) {
  const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(&e);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 x = __bfloat1622float2(a[k]);
    v[2 * k] = x.x * f;
    v[2 * k + 1] = x.y * f;
  }
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 q;
  __nv_bfloat162* a = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
  for (int k = 0; k < 4; ++k) a[k] = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
  return q;
}

struct NormDrop {
  uint8_t* keep;  // the keep words as bytes: byte 4 w + k of a row holds keys 32 w + 8 k .. + 7
  uint64_t seed, stream0;
  uint32_t thr;
  int n_heads, heads_per_shard, wpr;
  float scale;
};

// Grid: x = blocks of kNormWarps rows of a pair, y = pair (no 64-bit divisions).
template <bool DROP>
__global__ void __launch_bounds__(32 * kNormWarps, 4) attn_norm_kernel(const float2* __restrict__ part, int P,
                                                                     int64_t s, int64_t g0, int causal,
                                                                     float* __restrict__ lse,
                                                                     __nv_bfloat16* __restrict__ Pm,
                                                                     __nv_bfloat16* __restrict__ Pd,
                                                                     NormDrop dr) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kNormWarps + (threadIdx.x >> 5);
  if (row >= s) return;  // warp-uniform
  const int64_t g = g0 + blockIdx.y;
  const float2* pg = part + g * P * s + row;  // part p of this row at pg[p * s]
  const int64_t nch = s / 8, lim = causal ? row + 1 : s;  // chunks; columns < lim are kept
  const int64_t rbase = (g * s + row) * s;
  uint4 e[kNormBatch];
  float mp[kNormBatch];
  auto load_batch = [&](int64_t ch0) {
#pragma unroll
    for (int u = 0; u < kNormBatch; ++u) {
      const int64_t c = (ch0 + u * 32 + lane) * 8;
      if (c < lim) {
        e[u] = *reinterpret_cast<const uint4*>(Pm + rbase + c);
        mp[u] = pg[(c / 64) * s].x;
      }
    }
  };
  load_batch(0);
  float m = -INFINITY, sum = 0.f;
  const int plim = causal ? static_cast<int>(row / 64) + 1 : P;
  for (int p = lane; p < plim; p += 32) {
    const float2 x = pg[static_cast<int64_t>(p) * s];
    lse_merge(m, sum, x.x, x.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, sum, o);
    lse_merge(m, sum, om, os);
  }
  const float L = m + logf(sum);
  if (lane == 0) lse[g * s + row] = L;
  const uint64_t stream = DROP ? dr.stream0 + static_cast<uint64_t>((g % dr.n_heads) / dr.heads_per_shard) : 0;
  for (int64_t ch0 = 0; ch0 < nch; ch0 += 32 * kNormBatch) {
    if (ch0 != 0) load_batch(ch0);
    uint32_t bits[kNormBatch];
    if constexpr (DROP) {
      // drawn while the loads are in flight
#pragma unroll
      for (int u = 0; u < kNormBatch; ++u) {
        const int64_t ch = ch0 + u * 32 + lane, c = ch * 8;
        bits[u] = 0u;
        if (ch < nch) {
          if (!causal || (c & ~static_cast<int64_t>(31)) <= row)
            bits[u] = keep8(static_cast<uint64_t>((rbase + c) / 8), dr.seed, stream, dr.thr);
          uint8_t* kb = dr.keep + (g * s + row) * dr.wpr * 4 + ch;
          kb[0] = static_cast<uint8_t>(bits[u]);
          if (c + 8 == s && (s & 31) == 16) kb[1] = kb[2] = 0;  // the last word's keys past s
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kNormBatch; ++u) {
      const int64_t c = (ch0 + u * 32 + lane) * 8;
      if (c >= s) break;
      float v[8];
      if (c < lim) {
        scale8(e[u], expf(mp[u] - L), v);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = 0.f;
      }
      *reinterpret_cast<uint4*>(Pm + rbase + c) = pack8(v);
      if constexpr (DROP) {
        // attention dropout: the kept probabilities, scaled, for the P V product
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = (bits[u] >> k) & 1u ? v[k] * dr.scale : 0.f;
        *reinterpret_cast<uint4*>(Pd + rbase + c) = pack8(v);
      }
    }
  }
}

// One warp per (pair, token): D[g * s + t] = sum_c dC[row, c0 + c] C[row, c0 + c]
// over the head's d columns (16-byte loads when d and the offsets allow).
// Grid: x = blocks of 8 tokens, y = pair.
__global__ void __launch_bounds__(256) attn_rowdot_kernel(const __nv_bfloat16* __restrict__ C,
                                                           const __nv_bfloat16* __restrict__ dC,
                                                           int64_t h, int64_t s, int n_heads, int d,
                                                           int64_t g0, int vec, float* __restrict__ D) {
  pdl_wait();
  pdl_trigger();
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

cudaError_t launch_attn_norm(const void* part, int P, int64_t s, int64_t pairs, int causal, float* lse,
                             void* Pm, void* Pd, uint32_t* keep, float p_drop, uint64_t seed,
                             uint64_t stream0, int n_heads, int heads_per_shard, cudaStream_t st) {
  if (s % 8 != 0 || (reinterpret_cast<uintptr_t>(Pm) & 15u) != 0 ||
      (Pd != nullptr && ((reinterpret_cast<uintptr_t>(Pd) & 15u) != 0 || keep == nullptr || s % 16 != 0)))
    return cudaErrorInvalidValue;
  NormDrop dr{reinterpret_cast<uint8_t*>(keep), seed, stream0, dropout_threshold(p_drop), n_heads,
              heads_per_shard, static_cast<int>((s + 31) / 32), p_drop > 0.f ? 1.f / (1.f - p_drop) : 1.f};
  for (int64_t g0 = 0; g0 < pairs; g0 += kMaxGridY) {
    const dim3 grid(static_cast<unsigned>((s + kNormWarps - 1) / kNormWarps),
                    static_cast<unsigned>(pairs - g0 < kMaxGridY ? pairs - g0 : kMaxGridY));
    if (Pd != nullptr)
      launch_k(attn_norm_kernel<true>, grid, 32 * kNormWarps, 0, st, static_cast<const float2*>(part), P, s,
               g0, causal, lse, static_cast<__nv_bfloat16*>(Pm), static_cast<__nv_bfloat16*>(Pd), dr);
    else
      launch_k(attn_norm_kernel<false>, grid, 32 * kNormWarps, 0, st, static_cast<const float2*>(part), P, s,
               g0, causal, lse, static_cast<__nv_bfloat16*>(Pm), nullptr, dr);
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
    launch_k(attn_rowdot_kernel, grid, 256, 0, st, static_cast<const __nv_bfloat16*>(C),
             static_cast<const __nv_bfloat16*>(dC), h, s, n_heads, d, g0, vec, D);
    count_launches(1);
  }
  return cudaGetLastError();
}

}  // namespace tp
