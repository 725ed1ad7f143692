// HBM-bound kernels of the block: the vocab-parallel embedding gather, the
// deterministic grouping of tokens by id (counting sort, stable in token
// order) and the input-side embedding gradient as ordered segment sums.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tp_device.cuh"
#include "tp_internal.h"

namespace tp {
namespace {

// ---------------------------------------------------------------------------
// Vocab-parallel embedding gather ("Megatron" walkthrough, section
// VocabParallelEmbedding: each range looks up the ids it owns and zeroes the
// others, then the ranges are summed).  Exactly one range owns an id in
// [0, V), so the sum over ranges is the owner's row: one 16-byte vectorised,
// bit-exact copy per row chunk.  One warp per token row.
// ---------------------------------------------------------------------------
__device__ __forceinline__ const uint8_t* owner_row(const RangeTable& rt, int64_t id,
                                                    int64_t row_bytes) {
  if (id < rt.start[0] || id >= rt.start[rt.n]) return nullptr;
  int lo = 0, hi = rt.n - 1;  // find r with start[r] <= id < start[r+1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (rt.start[mid] <= id) lo = mid; else hi = mid - 1;
  }
  return static_cast<const uint8_t*>(rt.ptr[lo]) + (id - rt.start[lo]) * row_bytes;
}

constexpr int GATHER_UNROLL = 4;

__global__ void __launch_bounds__(256) embed_gather_vec16(const int64_t* __restrict__ ids, int64_t T,
                                                          int64_t row_bytes,
                                                          const __grid_constant__ RangeTable rt,
                                                          uint8_t* __restrict__ out) {
  // No early trigger: the gather's blocks all fit in one wave, so a trigger at
  // entry would start the next kernel's blocks at once, left waiting beside
  // the gather's (measured 4% slower for back-to-back gathers); the next
  // kernel launches as the gather's blocks exit.
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t nvec = row_bytes >> 4;
  for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < T;
       t += nwarps) {
    const uint8_t* src = owner_row(rt, __ldg(ids + t), row_bytes);
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(out + t * row_bytes);
    for (int64_t i = lane; i < nvec; i += 32 * GATHER_UNROLL) {
      uint4 v[GATHER_UNROLL];
#pragma unroll
      for (int u = 0; u < GATHER_UNROLL; ++u) {
        const int64_t j = i + 32 * u;
        v[u] = (src != nullptr && j < nvec) ? __ldg(s4 + j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < GATHER_UNROLL; ++u) {
        const int64_t j = i + 32 * u;
        if (j < nvec) __stcs(d4 + j, v[u]);
      }
    }
  }
}

// Byte-granular fallback for rows that are not 16-byte multiples or aligned.
__global__ void embed_gather_bytes(const int64_t* __restrict__ ids, int64_t T, int64_t row_bytes,
                                   const __grid_constant__ RangeTable rt, uint8_t* __restrict__ out) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < T;
       t += nwarps) {
    const uint8_t* src = owner_row(rt, ids[t], row_bytes);
    for (int64_t j = lane; j < row_bytes; j += 32) out[t * row_bytes + j] = src ? src[j] : 0;
  }
}

// ---------------------------------------------------------------------------
// Grouping of tokens by id: offsets[V+1] and perm[T] such that the tokens of
// id v are perm[offsets[v] .. offsets[v+1]) in increasing position.
// ---------------------------------------------------------------------------
__global__ void sort_histogram(const int64_t* __restrict__ ids, int64_t T, int64_t V,
                               int* __restrict__ counts) {
  pdl_wait();
  pdl_trigger();
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < T;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t v = ids[t];
    if (v >= 0 && v < V) atomicAdd(counts + v, 1);
  }
}

// Single-CTA exclusive scan of counts[0..V) into offsets[0..V]; counts is
// reset to zero for reuse as the scatter cursor.  The counts go through in
// chunks of 4 x SCAN_THREADS (four consecutive per thread, one 16-byte load),
// SCAN_DEPTH chunks in flight ahead of the one being scanned; a running total
// carries from chunk to chunk.
constexpr int SCAN_THREADS = 1024;
constexpr int SCAN_CHUNK = 4 * SCAN_THREADS;
constexpr int SCAN_DEPTH = 4;

__device__ __forceinline__ int4 scan_load4(const int* counts, int64_t V, int64_t v) {
  if (v + 3 < V) return *reinterpret_cast<const int4*>(counts + v);  // v % 4 == 0, base 256-aligned
  int4 q = make_int4(0, 0, 0, 0);
  if (v < V) q.x = counts[v];
  if (v + 1 < V) q.y = counts[v + 1];
  if (v + 2 < V) q.z = counts[v + 2];
  return q;
}

__global__ void __launch_bounds__(SCAN_THREADS) sort_scan(int* __restrict__ counts, int64_t V,
                                                          int* __restrict__ offsets) {
  pdl_wait();
  pdl_trigger();
  __shared__ int warp_sums[SCAN_THREADS / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t nch = (V + SCAN_CHUNK - 1) / SCAN_CHUNK;
  int4 q[SCAN_DEPTH];
#pragma unroll
  for (int d = 0; d < SCAN_DEPTH; ++d)
    q[d] = scan_load4(counts, V, static_cast<int64_t>(d) * SCAN_CHUNK + 4 * threadIdx.x);
  int carry = 0;
  for (int64_t c0 = 0; c0 < nch; c0 += SCAN_DEPTH) {
#pragma unroll
    for (int d = 0; d < SCAN_DEPTH; ++d) {
      const int64_t c = c0 + d;
      if (c >= nch) break;  // the same for every thread
      const int64_t v = c * SCAN_CHUNK + 4 * threadIdx.x;
      const int4 x = q[d];
      q[d] = scan_load4(counts, V, v + static_cast<int64_t>(SCAN_DEPTH) * SCAN_CHUNK);
      const int s0 = x.x, s1 = s0 + x.y, s2 = s1 + x.z, tot = s2 + x.w;
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) warp_sums[w] = incl;
      __syncthreads();
      if (w == 0) {
        int y = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int z = __shfl_up_sync(0xffffffffu, y, o);
          if (lane >= o) y += z;
        }
        warp_sums[lane] = y;  // inclusive over warps
      }
      __syncthreads();
      const int e = carry + incl - tot + (w > 0 ? warp_sums[w - 1] : 0);
      const int chunk_total = warp_sums[SCAN_THREADS / 32 - 1];
      if (v + 3 < V) {
        *reinterpret_cast<int4*>(offsets + v) = make_int4(e, e + s0, e + s1, e + s2);
        *reinterpret_cast<int4*>(counts + v) = make_int4(0, 0, 0, 0);
      } else {
        const int ev[3] = {e, e + s0, e + s1};
        for (int j = 0; j < 3; ++j)
          if (v + j < V) {
            offsets[v + j] = ev[j];
            counts[v + j] = 0;
          }
      }
      carry += chunk_total;
      __syncthreads();  // warp_sums is rewritten by the next chunk
    }
  }
  if (threadIdx.x == 0) offsets[V] = carry;
}

__global__ void sort_scatter(const int64_t* __restrict__ ids, int64_t T, int64_t V,
                             const int* __restrict__ offsets, int* __restrict__ cursor,
                             int* __restrict__ perm) {
  pdl_wait();
  pdl_trigger();
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < T;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t v = ids[t];
    if (v >= 0 && v < V) perm[offsets[v] + atomicAdd(cursor + v, 1)] = static_cast<int>(t);
  }
}

// The scatter placed each segment's tokens in arbitrary order; sorting each
// segment by position makes the result unique (hence deterministic).
__global__ void sort_segments(const int* __restrict__ offsets, int64_t V, int* __restrict__ perm) {
  pdl_wait();
  pdl_trigger();
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < V;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = offsets[v], e = offsets[v + 1];
    for (int i = b + 1; i < e; ++i) {
      const int x = perm[i];
      int j = i - 1;
      while (j >= b && perm[j] > x) {
        perm[j + 1] = perm[j];
        --j;
      }
      perm[j + 1] = x;
    }
  }
}

// ---------------------------------------------------------------------------
// Input-side embedding gradient alone (no output-layer term): one warp per
// vocabulary row; the row's tokens are summed in position order in fp32.
// ---------------------------------------------------------------------------
__global__ void segment_sum_rows(const int* __restrict__ offsets, const int* __restrict__ perm,
                                 int64_t V, const void* __restrict__ dEmb, int in_f32, int64_t h,
                                 const __grid_constant__ RangeTable dE, int accumulate) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t v = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; v < V;
       v += nwarps) {
    int r = 0;
    while (v >= dE.start[r + 1]) ++r;
    float* row = static_cast<float*>(const_cast<void*>(dE.ptr[r])) + (v - dE.start[r]) * h;
    const int b = offsets[v], e = offsets[v + 1];
    for (int64_t c = lane; c < h; c += 32) {
      float s = 0.f;
      for (int t = b; t < e; ++t) {
        const int64_t idx = static_cast<int64_t>(perm[t]) * h + c;
        s += in_f32 ? static_cast<const float*>(dEmb)[idx]
                    : bf2f(static_cast<const __nv_bfloat16*>(dEmb)[idx]);
      }
      row[c] = accumulate ? row[c] + s : s;
    }
  }
}

inline int blocks_for(int64_t n, int threads, int cap = 65535 * 8) {
  int64_t b = (n + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > cap) b = cap;
  return static_cast<int>(b);
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

cudaError_t launch_embed_gather(const int64_t* ids, int64_t T, int64_t row_bytes,
                                const RangeTable& rt, void* out, cudaStream_t s) {
  if (T <= 0 || row_bytes <= 0) return cudaSuccess;
  bool vec = (row_bytes % 16) == 0 && (reinterpret_cast<uintptr_t>(out) % 16) == 0;
  for (int r = 0; r < rt.n; ++r) vec = vec && (reinterpret_cast<uintptr_t>(rt.ptr[r]) % 16) == 0;
  const int blocks = blocks_for(T * 32, 256);
  if (vec)
    launch_k(embed_gather_vec16, blocks, 256, 0, s, ids, T, row_bytes, rt, static_cast<uint8_t*>(out));
  else
    launch_k(embed_gather_bytes, blocks, 256, 0, s, ids, T, row_bytes, rt, static_cast<uint8_t*>(out));
  count_launches(1);
  return cudaGetLastError();
}

size_t sort_workspace_bytes(int64_t T, int64_t V) {
  return align256(static_cast<size_t>(V + 1) * 4) + align256(static_cast<size_t>(T > 0 ? T : 1) * 4) +
         align256(static_cast<size_t>(V) * 4);
}

int* sort_offsets(void* ws) { return static_cast<int*>(ws); }
int* sort_perm(void* ws, int64_t V) {
  return reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + align256(static_cast<size_t>(V + 1) * 4));
}
static int* sort_counts(void* ws, int64_t T, int64_t V) {
  return reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + align256(static_cast<size_t>(V + 1) * 4) +
                                align256(static_cast<size_t>(T > 0 ? T : 1) * 4));
}

cudaError_t launch_embed_sort(const int64_t* ids, int64_t T, int64_t V, void* ws, cudaStream_t s) {
  int* offsets = sort_offsets(ws);
  int* perm = sort_perm(ws, V);
  int* counts = sort_counts(ws, T, V);
  cudaError_t e = cudaMemsetAsync(counts, 0, static_cast<size_t>(V) * 4, s);
  if (e != cudaSuccess) return e;
  if (T > 0) launch_k(sort_histogram, blocks_for(T, 256), 256, 0, s, ids, T, V, counts);
  launch_k(sort_scan, 1, SCAN_THREADS, 0, s, counts, V, offsets);
  if (T > 0) {
    launch_k(sort_scatter, blocks_for(T, 256), 256, 0, s, ids, T, V, offsets, counts, perm);
    launch_k(sort_segments, blocks_for(V, 256), 256, 0, s, offsets, V, perm);
  }
  count_launches(T > 0 ? 4 : 1);
  return cudaGetLastError();
}

cudaError_t launch_segment_sum(const void* ws, int64_t V, int64_t T, const void* dEmb, int in_f32,
                               int64_t h, const RangeTable& dE, int accumulate, cudaStream_t s) {
  (void)T;
  const int* offsets = sort_offsets(const_cast<void*>(ws));
  const int* perm = sort_perm(const_cast<void*>(ws), V);
  launch_k(segment_sum_rows, blocks_for(V * 32, 256), 256, 0, s, offsets, perm, V, dEmb, in_f32, h, dE,
                                                           accumulate);
  count_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Vocab-parallel cross-entropy: combine the per-part (max, sum exp) pairs of
// each row in fixed part order (the on-chip form of the all-reduce MAX and the
// all-reduce SUM of [Walkthrough] §_VocabParallelCrossEntropy), then
// loss = log(sum) - (target logit - max) and lse = max + log(sum).  A block
// covers 32 rows with 32 slices of the parts each; slices merge in order.
// ---------------------------------------------------------------------------
namespace {

__device__ __forceinline__ void lse_merge(float& m, float& s, float mj, float sj) {
  if (mj == -INFINITY) return;  // an empty slice (no parts)
  if (mj > m) {
    s = s * expf(m - mj) + sj;
    m = mj;
  } else {
    s += sj * expf(mj - m);
  }
}

constexpr int CE_SLICES = 32;

__global__ void __launch_bounds__(32 * CE_SLICES) ce_reduce_kernel(const float2* __restrict__ part, int P, int64_t T,
                                                        const int64_t* __restrict__ targets, int64_t V,
                                                        const float* __restrict__ target_logit,
                                                        float* __restrict__ loss, float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sm[CE_SLICES][32], ss[CE_SLICES][32];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 32 + tx;
  float m = -INFINITY, s = 0.f;
  if (row < T) {
    const int p0 = static_cast<int>(static_cast<int64_t>(P) * ty / CE_SLICES);
    const int p1 = static_cast<int>(static_cast<int64_t>(P) * (ty + 1) / CE_SLICES);
    for (int p = p0; p < p1; ++p) {
      const float2 v = part[static_cast<int64_t>(p) * T + row];
      lse_merge(m, s, v.x, v.y);
    }
  }
  sm[ty][tx] = m;
  ss[ty][tx] = s;
  __syncthreads();
  if (ty == 0 && row < T) {
    float M = sm[0][tx], S = ss[0][tx];
    for (int k = 1; k < CE_SLICES; ++k) lse_merge(M, S, sm[k][tx], ss[k][tx]);
    const float log_s = logf(S);
    const int64_t t = targets[row];
    // a target in no range: predicted (shifted) logit 0, so loss = log(sum)
    loss[row] = (t >= 0 && t < V) ? log_s - (target_logit[row] - M) : log_s;
    lse[row] = M + log_s;
  }
}

}  // namespace

cudaError_t launch_ce_reduce(const void* part, int P, int64_t T, const int64_t* targets, int64_t V,
                             const float* target_logit, float* loss, float* lse, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  launch_k(ce_reduce_kernel, static_cast<unsigned>((T + 31) / 32), 32 * CE_SLICES, 0, s, static_cast<const float2*>(part), P, T, targets, V, target_logit, loss, lse);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace tp
