// Row kernels of the transformer layer ("Megatron" walkthrough,
// §ParallelTransformerLayer; "Megatron / ZeRO" study notes on fp32 LayerNorm
// parameters):
//   ln_fwd_kernel        LayerNorm of bf16 rows with fp32 gain and bias,
//                        saving the row mean and 1/std;
//   ln_bwd_kernel        its input gradient (plus an optional residual gradient)
//                        and the gain and bias gradient parts of 8-row groups,
//                        in one pass over dy and x;
//   ln_param_grad_sum    the groups' parts summed in order (deterministic);
//   dropout_add_kernel   out = res + x * keep / (1 - p) and its backward;
//   pos_embed_dropout    (word + position embedding) with dropout;
//   attn_keep_kernel     attention-dropout keep bits, 32 keys per word.
// Dropout draws its keep bits from Philox4x32-10 (tp_philox.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "tp_internal.h"
#include "tp_philox.cuh"

namespace tp {
namespace {

constexpr int kLnThreads = 256;  // rows up to 256 x 32 = 8192 wide

// Fixed-order block sum of one float (all threads receive it).
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red is reused between calls
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < kLnThreads / 32; ++i) t += red[i];
  return t;
}

// Eight floats to eight consecutive bf16 of a row (one 16-byte store).
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float* v) {
  uint4 q;
  __nv_bfloat162* a = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
  for (int k = 0; k < 4; ++k) a[k] = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
  *reinterpret_cast<uint4*>(p) = q;
}
__device__ __forceinline__ void load8f(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
// The eight bf16 of one 16-byte load as floats.
__device__ __forceinline__ void unpack8(const uint4& q, float* v) {
  const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(a[k]);
    v[2 * k] = f.x;
    v[2 * k + 1] = f.y;
  }
}

// A thread owns PER values of a row in groups of eight consecutive columns:
// group k covers columns 8 (k kLnThreads + tid) .. + 7 (h % 8 == 0).  A block
// takes kLnFwdRows consecutive rows in order; the next row is loaded while
// this row's sums run.
constexpr int kLnFwdRows = 4;

template <int PER>
__global__ void __launch_bounds__(kLnThreads) ln_fwd_kernel(const __nv_bfloat16* __restrict__ x,
                                                            const float* __restrict__ g,
                                                            const float* __restrict__ b, int64_t T,
                                                            int64_t h, float eps,
                                                            __nv_bfloat16* __restrict__ y,
                                                            float* __restrict__ mean_out,
                                                            float* __restrict__ rstd_out) {
  pdl_wait();
  pdl_trigger();
  constexpr int NV = PER / 8;
  __shared__ float red[kLnThreads / 32];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kLnFwdRows;
  const int64_t r1 = min(T, r0 + kLnFwdRows);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 cur[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t c = (static_cast<int64_t>(k) * kLnThreads + threadIdx.x) * 8;
    cur[k] = c < h ? *reinterpret_cast<const uint4*>(x + r0 * h + c) : zero;
  }
  for (int64_t r = r0; r < r1; ++r) {
    uint4 nxt[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t c = (static_cast<int64_t>(k) * kLnThreads + threadIdx.x) * 8;
      nxt[k] = (c < h && r + 1 < r1) ? *reinterpret_cast<const uint4*>(x + (r + 1) * h + c) : zero;
    }
    float v[PER];  // zero past h
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      unpack8(cur[k], v + 8 * k);
#pragma unroll
      for (int t = 0; t < 8; ++t) s += v[8 * k + t];
    }
    const float mean = block_sum(s, red) / static_cast<float>(h);
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t c = (static_cast<int64_t>(k) * kLnThreads + threadIdx.x) * 8;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const float dlt = c < h ? v[8 * k + t] - mean : 0.f;
        q += dlt * dlt;
      }
    }
    const float rstd = rsqrtf(block_sum(q, red) / static_cast<float>(h) + eps);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t c = (static_cast<int64_t>(k) * kLnThreads + threadIdx.x) * 8;
      if (c < h) {
        float gg[8], bb[8], o[8];
        load8f(g + c, gg);
        load8f(b + c, bb);
#pragma unroll
        for (int t = 0; t < 8; ++t) o[t] = (v[8 * k + t] - mean) * rstd * gg[t] + bb[t];
        store8(y + r * h + c, o);
      }
      cur[k] = nxt[k];
    }
    if (threadIdx.x == 0) {
      mean_out[r] = mean;
      rstd_out[r] = rstd;
    }
  }
}

// A block takes kLnRows consecutive rows, in order: for each,
// dx = rstd (dxhat - mean(dxhat) - xhat mean(dxhat xhat)) (+ dres), dxhat = dy g,
// while the gain and bias gradient parts of the block's rows (sums of dy xhat
// and of dy, rows in order) gather in registers; they go to
// partial[block][0..h) and partial[block][h..2h).  The next row's dy and x and
// this row's dres are loaded before this row's sums, so one pass over dy and x
// gives both gradients.
constexpr int kLnRows = 8;

// Fixed-order block sums of two floats at once (all threads receive them).
__device__ __forceinline__ float2 block_sum2(float a, float b, float2* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red is reused between rows
  if (lane == 0) red[w] = make_float2(a, b);
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
  for (int i = 0; i < kLnThreads / 32; ++i) {
    t.x += red[i].x;
    t.y += red[i].y;
  }
  return t;
}

template <int PER>
__global__ void __launch_bounds__(kLnThreads) ln_bwd_kernel(
    const __nv_bfloat16* __restrict__ dy, const __nv_bfloat16* __restrict__ x,
    const float* __restrict__ g, const float* __restrict__ mean_in, const float* __restrict__ rstd_in,
    const __nv_bfloat16* __restrict__ dres, int64_t T, int64_t h, __nv_bfloat16* __restrict__ dx,
    float* __restrict__ partial) {
  pdl_wait();
  pdl_trigger();
  constexpr int NV = PER / 8;
  __shared__ float2 red[kLnThreads / 32];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kLnRows;
  const int64_t r1 = min(T, r0 + kLnRows);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  float gg[PER], ag[PER], ab[PER];
  uint4 cd[NV], cx[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t c = (static_cast<int64_t>(k) * kLnThreads + threadIdx.x) * 8;
    cd[k] = cx[k] = zero;
    if (c < h) {
      load8f(g + c, gg + 8 * k);
      cd[k] = *reinterpret_cast<const uint4*>(dy + r0 * h + c);
      cx[k] = *reinterpret_cast<const uint4*>(x + r0 * h + c);
    } else {
#pragma unroll
      for (int t = 0; t < 8; ++t) gg[8 * k + t] = 0.f;
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) ag[8 * k + t] = ab[8 * k + t] = 0.f;
  }
  float mean = mean_in[r0], rstd = rstd_in[r0];
  for (int64_t r = r0; r < r1; ++r) {
    const bool more = r + 1 < r1;
    uint4 nd[NV], nx[NV], rr[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t c = (static_cast<int64_t>(k) * kLnThreads + threadIdx.x) * 8;
      nd[k] = nx[k] = rr[k] = zero;
      if (c < h) {
        if (more) {
          nd[k] = *reinterpret_cast<const uint4*>(dy + (r + 1) * h + c);
          nx[k] = *reinterpret_cast<const uint4*>(x + (r + 1) * h + c);
        }
        if (dres) rr[k] = *reinterpret_cast<const uint4*>(dres + r * h + c);
      }
    }
    const float nmean = more ? mean_in[r + 1] : 0.f, nrstd = more ? rstd_in[r + 1] : 0.f;
    // columns past h hold dy = 0 and g = 0, so they add nothing below
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      float d[8], xv[8];
      unpack8(cd[k], d);
      unpack8(cx[k], xv);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const float xn = (xv[t] - mean) * rstd, e = d[t] * gg[8 * k + t];
        s1 += e;
        s2 += e * xn;
        ag[8 * k + t] += d[t] * xn;
        ab[8 * k + t] += d[t];
      }
    }
    const float2 m = block_sum2(s1, s2, red);
    const float m1 = m.x / static_cast<float>(h), m2 = m.y / static_cast<float>(h);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t c = (static_cast<int64_t>(k) * kLnThreads + threadIdx.x) * 8;
      if (c < h) {
        float d[8], xv[8], res[8], o[8];
        unpack8(cd[k], d);
        unpack8(cx[k], xv);
        unpack8(rr[k], res);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float xn = (xv[t] - mean) * rstd;
          o[t] = rstd * (d[t] * gg[8 * k + t] - m1 - xn * m2) + res[t];
        }
        store8(dx + r * h + c, o);
      }
      cd[k] = nd[k];
      cx[k] = nx[k];
    }
    mean = nmean;
    rstd = nrstd;
  }
  float* pp = partial + static_cast<int64_t>(blockIdx.x) * 2 * h;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t c = (static_cast<int64_t>(k) * kLnThreads + threadIdx.x) * 8;
    if (c < h) {
#pragma unroll
      for (int t = 0; t < 8; t += 4) {
        *reinterpret_cast<float4*>(pp + c + t) =
            make_float4(ag[8 * k + t], ag[8 * k + t + 1], ag[8 * k + t + 2], ag[8 * k + t + 3]);
        *reinterpret_cast<float4*>(pp + h + c + t) =
            make_float4(ab[8 * k + t], ab[8 * k + t + 1], ab[8 * k + t + 2], ab[8 * k + t + 3]);
      }
    }
  }
}

// The groups' partials summed into dg and db (+ the existing values when
// accumulating); 2h columns.  A block takes 32 columns (lane = column) and
// kLnSumSlices slices (warp = slice): slice w sums groups w, w + kLnSumSlices,
// ... in order, then warp 0 adds the slices in order (fixed order,
// deterministic).
constexpr int kLnSumSlices = 32;
__global__ void __launch_bounds__(32 * kLnSumSlices) ln_param_grad_sum_kernel(const float* __restrict__ part2,
                                                                             int ngroups, int64_t h,
                                                                             float* __restrict__ dg,
                                                                             float* __restrict__ db,
                                                                             int accumulate) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[kLnSumSlices][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  float s = 0.f;
  if (c < 2 * h) {
#pragma unroll 4
    for (int k = w; k < ngroups; k += kLnSumSlices) s += part2[static_cast<int64_t>(k) * 2 * h + c];
  }
  red[w][lane] = s;
  __syncthreads();
  if (w != 0 || c >= 2 * h) return;
  float t = red[0][lane];
  for (int k = 1; k < kLnSumSlices; ++k) t += red[k][lane];
  float* out = c < h ? dg + c : db + (c - h);
  *out = accumulate ? *out + t : t;
}

// 16 elements per thread (two generator blocks): out = res + x * keep * scale, or
// (res == null) out = x * keep * scale.  n is a multiple of 16.
__global__ void __launch_bounds__(256) dropout_add_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const __nv_bfloat16* __restrict__ res,
                                                          int64_t nblk, uint64_t seed, uint64_t stream,
                                                          uint32_t thr, float scale,
                                                          __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (blk >= nblk) return;
  // the loads go out first; the Philox rounds run while they are in flight
  const uint4* x4 = reinterpret_cast<const uint4*>(x) + blk * 2;
  uint4 xv[2] = {x4[0], x4[1]};
  uint4 rv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
  if (res) {
    const uint4* r4 = reinterpret_cast<const uint4*>(res) + blk * 2;
    rv[0] = r4[0];
    rv[1] = r4[1];
  }
  const uint32_t bits = keep16(static_cast<uint64_t>(blk), seed, stream, thr);
  uint4 ov[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const __nv_bfloat162* xa = reinterpret_cast<const __nv_bfloat162*>(&xv[q]);
    const __nv_bfloat162* ra = reinterpret_cast<const __nv_bfloat162*>(&rv[q]);
    __nv_bfloat162* oa = reinterpret_cast<__nv_bfloat162*>(&ov[q]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int f = q * 8 + 2 * k;
      const float2 a = __bfloat1622float2(xa[k]), r = __bfloat1622float2(ra[k]);
      const float k0 = (bits >> f) & 1u ? scale : 0.f, k1 = (bits >> (f + 1)) & 1u ? scale : 0.f;
      oa[k] = __floats2bfloat162_rn(r.x + a.x * k0, r.y + a.y * k1);
    }
  }
  uint4* o4 = reinterpret_cast<uint4*>(out) + blk * 2;
  o4[0] = ov[0];
  o4[1] = ov[1];
}

// Input of the first layer: out = (words + pos_table[positions[row]]) * keep *
// scale, 16 elements of one row per thread (h % 16 == 0).
__global__ void __launch_bounds__(256) pos_embed_dropout_kernel(
    const __nv_bfloat16* __restrict__ words, const __nv_bfloat16* __restrict__ pos_table,
    const int64_t* __restrict__ positions, int64_t h, int64_t max_pos, int64_t nblk, uint64_t seed,
    uint64_t stream, uint32_t thr, float scale, __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (blk >= nblk) return;
  const int64_t e = blk * 16, row = e / h, col = e - row * h;
  const uint4* w4 = reinterpret_cast<const uint4*>(words + e);
  const int64_t pos = positions[row];
  const bool pos_ok = pos >= 0 && pos < max_pos;  // a position outside the table adds zeros
  const uint4* p4 = reinterpret_cast<const uint4*>(pos_table + (pos_ok ? pos : 0) * h + col);
  const uint4 wv2[2] = {w4[0], w4[1]};
  const uint4 pv2[2] = {pos_ok ? p4[0] : make_uint4(0, 0, 0, 0), pos_ok ? p4[1] : make_uint4(0, 0, 0, 0)};
  const uint32_t bits = keep16(static_cast<uint64_t>(blk), seed, stream, thr);
  uint4 ov[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint4 wv = wv2[q], pv = pv2[q];
    const __nv_bfloat162* wa = reinterpret_cast<const __nv_bfloat162*>(&wv);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&pv);
    __nv_bfloat162* oa = reinterpret_cast<__nv_bfloat162*>(&ov[q]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int f = q * 8 + 2 * k;
      const float2 a = __bfloat1622float2(wa[k]), b = __bfloat1622float2(pa[k]);
      const float k0 = (bits >> f) & 1u ? scale : 0.f, k1 = (bits >> (f + 1)) & 1u ? scale : 0.f;
      oa[k] = __floats2bfloat162_rn((a.x + b.x) * k0, (a.y + b.y) * k1);
    }
  }
  uint4* o4 = reinterpret_cast<uint4*>(out + e);
  o4[0] = ov[0];
  o4[1] = ov[1];
}

// Keep bits of attention dropout: word w of row q of pair g covers keys
// 32 w .. 32 w + 31 of element block ((g s + q) s + 32 w) / 16 (s % 16 == 0);
// pair g = sequence * heads + head draws from stream stream0 + shard(head).
// Grid: x over the words of a row, y = q, z = g (no integer divisions).
__global__ void __launch_bounds__(256) attn_keep_kernel(int64_t s, int wpr, int n_heads, int heads_per_shard,
                                                        int causal, uint64_t seed, uint64_t stream0,
                                                        uint32_t thr, uint32_t* __restrict__ words) {
  pdl_wait();
  pdl_trigger();
  const int w = blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= wpr) return;
  const int64_t q = blockIdx.y, g = blockIdx.z;
  uint32_t* out = words + (g * s + q) * wpr + w;
  if (causal && 32 * static_cast<int64_t>(w) > q) {  // every key of the word lies after the query: never read
    *out = 0u;
    return;
  }
  const int j = static_cast<int>(blockIdx.z % static_cast<unsigned>(n_heads));
  const uint64_t stream = stream0 + static_cast<uint64_t>(j / heads_per_shard);
  const uint64_t blk = static_cast<uint64_t>(((g * s + q) * s) / 16) + 2 * static_cast<uint64_t>(w);
  uint32_t bits = keep16(blk, seed, stream, thr);
  if (32 * static_cast<int64_t>(w) + 16 < s) bits |= keep16(blk + 1, seed, stream, thr) << 16;
  *out = bits;
}

}  // namespace

uint32_t dropout_threshold(float p) {
  const double t = floor(static_cast<double>(p) * 65536.0);
  return t < 0 ? 0u : (t > 65536.0 ? 65536u : static_cast<uint32_t>(t));
}

// Values per thread for a row of h: the smallest of 8, 16, 32 that covers it.
static int ln_per(int64_t h) {
  for (int p = 8; p <= 32; p *= 2)
    if (h <= static_cast<int64_t>(p) * kLnThreads) return p;
  return 0;
}

cudaError_t launch_ln_fwd(const void* x, const float* g, const float* b, int64_t T, int64_t h, float eps,
                          void* y, float* mean, float* rstd, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  auto* yb = static_cast<__nv_bfloat16*>(y);
  const unsigned grid = static_cast<unsigned>((T + kLnFwdRows - 1) / kLnFwdRows);
  switch (ln_per(h)) {
    case 8: launch_k(ln_fwd_kernel<8>, grid, kLnThreads, 0, st, xb, g, b, T, h, eps, yb, mean, rstd); break;
    case 16: launch_k(ln_fwd_kernel<16>, grid, kLnThreads, 0, st, xb, g, b, T, h, eps, yb, mean, rstd); break;
    case 32: launch_k(ln_fwd_kernel<32>, grid, kLnThreads, 0, st, xb, g, b, T, h, eps, yb, mean, rstd); break;
    default: return cudaErrorInvalidValue;
  }
  count_launches(1);
  return cudaGetLastError();
}

int ln_bwd_blocks(int64_t T) { return static_cast<int>((T + kLnRows - 1) / kLnRows); }

size_t ln_bwd_scratch_floats(int64_t T, int64_t h) {
  return static_cast<size_t>(ln_bwd_blocks(T)) * 2 * static_cast<size_t>(h);
}

cudaError_t launch_ln_bwd(const void* dy, const void* x, const float* g, const float* mean,
                          const float* rstd, const void* dres, int64_t T, int64_t h, void* dx,
                          float* dg, float* db, int accumulate, float* partial, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const auto* dyb = static_cast<const __nv_bfloat16*>(dy);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  const auto* rb = static_cast<const __nv_bfloat16*>(dres);
  auto* dxb = static_cast<__nv_bfloat16*>(dx);
  const int ngroups = ln_bwd_blocks(T);
  const unsigned grid = static_cast<unsigned>(ngroups);
#define TP_LNB(P) \
  launch_k(ln_bwd_kernel<P>, grid, kLnThreads, 0, st, dyb, xb, g, mean, rstd, rb, T, h, dxb, partial)
  switch (ln_per(h)) {
    case 8: TP_LNB(8); break;
    case 16: TP_LNB(16); break;
    case 32: TP_LNB(32); break;
    default: return cudaErrorInvalidValue;
  }
#undef TP_LNB
  launch_k(ln_param_grad_sum_kernel, static_cast<unsigned>((2 * h + 31) / 32), 32 * kLnSumSlices, 0, st,
           partial, ngroups, h, dg, db, accumulate);
  count_launches(2);
  return cudaGetLastError();
}

cudaError_t launch_dropout_add(const void* x, const void* res, int64_t n, uint64_t seed, uint64_t stream,
                               float p, void* out, cudaStream_t st) {
  const int64_t nblk = n / 16;
  if (nblk == 0) return cudaSuccess;
  launch_k(dropout_add_kernel, static_cast<unsigned>((nblk + 255) / 256), 256, 0, st,
           static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(res), nblk, seed, stream,
           dropout_threshold(p), 1.0f / (1.0f - p), static_cast<__nv_bfloat16*>(out));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_pos_embed_dropout(const void* words, const void* pos_table, const int64_t* positions,
                                     int64_t T, int64_t h, int64_t max_pos, uint64_t seed, uint64_t stream,
                                     float p, void* out, cudaStream_t st) {
  const int64_t nblk = T * h / 16;
  if (nblk == 0) return cudaSuccess;
  launch_k(pos_embed_dropout_kernel, static_cast<unsigned>((nblk + 255) / 256), 256, 0, st,
           static_cast<const __nv_bfloat16*>(words), static_cast<const __nv_bfloat16*>(pos_table), positions, h,
           max_pos, nblk, seed, stream, dropout_threshold(p), 1.0f / (1.0f - p),
           static_cast<__nv_bfloat16*>(out));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_attn_keep(int64_t pairs, int64_t s, int n_heads, int heads_per_shard, int causal,
                             uint64_t seed, uint64_t stream0, float p, uint32_t* words, cudaStream_t st) {
  const int wpr = static_cast<int>((s + 31) / 32);
  if (pairs == 0 || s == 0) return cudaSuccess;
  if (s > 65535 || pairs > 65535) return cudaErrorInvalidValue;  // grid y / z limits
  const int bx = wpr < 256 ? wpr : 256;
  const dim3 grid(static_cast<unsigned>((wpr + bx - 1) / bx), static_cast<unsigned>(s),
                  static_cast<unsigned>(pairs));
  launch_k(attn_keep_kernel, grid, bx, 0, st, s, wpr, n_heads, heads_per_shard, causal, seed, stream0,
           dropout_threshold(p), words);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace tp
