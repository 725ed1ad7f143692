// Mixed-precision Adam step over flat fp32 parameter groups ("Megatron"
// walkthrough, section MixedPrecisionOptimizer.step and DynamicGradScaler;
// "Megatron / ZeRO" study notes, sections on gradient clipping and on Adam's
// momentum and variance).  Two kernels, both HBM-bound streams:
//   opt_norm_kernel      unscaled gradients' sum of squares and overflow flag,
//                        one fp64 partial per block (fixed chunk assignment);
//                        the last block to finish (a completion counter) then
//                        sums the partials in fixed order, updates the loss
//                        scale, prepares the clip coefficient and the bias
//                        corrections, and marks the step skipped on overflow;
//   opt_adam_kernel      unscale + clip + weight decay + Adam + bf16 copy of
//                        every element, in one pass.
// Deterministic: every sum has a fixed order for a given device.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "tp_internal.h"

namespace tp {
namespace {

// Completion counters of the norm launches, one per launch slot; launches
// rotate over the slots and the last block of a launch resets its counter.
constexpr int kOptSlots = 64;
__device__ int g_opt_done[kOptSlots];
std::atomic<unsigned> g_opt_slot_seq{0};

constexpr int kOptThreads = 256;
constexpr int64_t kOptChunk = 16384;  // elements per chunk (a multiple of 4 x kOptThreads)
static_assert(kOptChunk % (4 * kOptThreads) == 0, "chunk = whole float4 rows of the block");

// Scalars the finalize kernel hands to the update kernel (workspace head).
struct OptControl {
  int skip;          // overflow: no update this step
  float grad_mul;    // 1/scale (of the scale the gradients carry) x clip coefficient
  float step_size;   // lr / (1 - beta1^step)
  float inv_bc2;     // 1 / (1 - beta2^step)
};

// Binary search over the groups' first chunks (chunk_begin is non-decreasing).
__device__ __forceinline__ void group_of_chunk(const OptParams& P, int64_t c, int& g, int64_t& off,
                                               int64_t& len) {
  int lo = 0, hi = P.ngroups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.group[mid].chunk_begin <= c) lo = mid;
    else hi = mid - 1;
  }
  g = lo;
  off = (c - P.group[g].chunk_begin) * kOptChunk;
  const int64_t rem = P.group[g].n - off;
  len = rem < kOptChunk ? rem : kOptChunk;
}

__device__ __forceinline__ float inv_scale_of(const OptParams& P) {
  return P.use_scaler ? 1.0f / P.state->scale : 1.0f;
}

// The finalize step, run by the last block of the norm launch: partials
// summed in a fixed order (thread i takes i, i + 256, ..., then a fixed tree),
// then the scaler update, the skip decision, the clip coefficient and the bias
// corrections.
__device__ void opt_finalize_block(const OptParams& P, const double* partial, const int* flag,
                                   int nparts, OptControl* ctl, double* red, int* bred) {
  double acc = 0.0;
  int bad = 0;
  for (int i = threadIdx.x; i < nparts; i += kOptThreads) {
    acc += __ldcg(partial + i);
    bad |= __ldcg(flag + i);
  }
  red[threadIdx.x] = acc;
  bred[threadIdx.x] = bad;
  __syncthreads();
  for (int w = kOptThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      red[threadIdx.x] += red[threadIdx.x + w];
      bred[threadIdx.x] |= bred[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x != 0) return;
  tp_optimizer_state* st = P.state;
  const double norm_sq = red[0];
  const int found_inf = bred[0] != 0 || !isfinite(norm_sq);
  const float grad_mul0 = inv_scale_of(P);
  // dynamic loss scale ("Megatron" walkthrough, DynamicGradScaler.update)
  if (P.use_scaler) {
    if (found_inf) {
      st->growth_tracker = 0;
      st->hysteresis_tracker -= 1;
      if (st->hysteresis_tracker <= 0) st->scale = fmaxf(st->scale * P.backoff_factor, P.min_scale);
    } else {
      st->growth_tracker += 1;
      if (st->growth_tracker == P.growth_interval) {
        st->growth_tracker = 0;
        st->hysteresis_tracker = P.hysteresis;
        st->scale = st->scale * P.growth_factor;
      }
    }
  }
  const double norm = sqrt(norm_sq);
  st->found_inf = found_inf;
  st->grad_norm = static_cast<float>(norm);
  ctl->skip = found_inf;
  if (found_inf) return;
  // global-norm clip: g * max_norm / ||g|| when ||g|| > max_norm
  const double coef = (P.max_norm > 0.0 && norm > P.max_norm) ? P.max_norm / norm : 1.0;
  const int step = st->step + 1;
  st->step = step;
  ctl->grad_mul = static_cast<float>(grad_mul0 * coef);
  ctl->step_size = static_cast<float>(P.lr / (1.0 - pow(P.beta1_d, step)));
  ctl->inv_bc2 = static_cast<float>(1.0 / (1.0 - pow(P.beta2_d, step)));
}

__global__ void __launch_bounds__(kOptThreads) opt_norm_kernel(const __grid_constant__ OptParams P,
                                                               double* __restrict__ partial,
                                                               int* __restrict__ flag,
                                                               OptControl* __restrict__ ctl, int slot) {
  pdl_wait();
  pdl_trigger();
  const float inv_scale = inv_scale_of(P);
  double acc = 0.0;
  int bad = 0;
  for (int64_t c = blockIdx.x; c < P.nchunks; c += gridDim.x) {
    int g;
    int64_t off, len;
    group_of_chunk(P, c, g, off, len);
    const float* src = P.group[g].grad + off;
    float part = 0.f;
    const int64_t nv = len >> 2;
    auto add4 = [&](const float4 q) {
      const float a = q.x * inv_scale, b = q.y * inv_scale, d = q.z * inv_scale, e = q.w * inv_scale;
      bad |= !(isfinite(a) && isfinite(b) && isfinite(d) && isfinite(e));
      part = fmaf(a, a, part);
      part = fmaf(b, b, part);
      part = fmaf(d, d, part);
      part = fmaf(e, e, part);
    };
    if (len == kOptChunk) {
      // full chunk: all of the thread's loads in flight at once, then the
      // same summation order as the general loop
      constexpr int kPer = static_cast<int>(kOptChunk / 4 / kOptThreads);
      const float4* s4 = reinterpret_cast<const float4*>(src) + threadIdx.x;
      float4 q[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) q[j] = __ldcs(s4 + j * kOptThreads);
#pragma unroll
      for (int j = 0; j < kPer; ++j) add4(q[j]);
    } else {
      for (int64_t i = threadIdx.x; i < nv; i += kOptThreads)
        add4(__ldcs(reinterpret_cast<const float4*>(src) + i));
    }
    for (int64_t i = (nv << 2) + threadIdx.x; i < len; i += kOptThreads) {
      const float a = src[i] * inv_scale;
      bad |= !isfinite(a);
      part = fmaf(a, a, part);
    }
    acc += static_cast<double>(part);  // at most 64 fp32 squares per thread per chunk
  }
  // block sum in a fixed tree
  __shared__ double red[kOptThreads];
  __shared__ int bred[kOptThreads];
  red[threadIdx.x] = acc;
  bred[threadIdx.x] = bad;
  __syncthreads();
  for (int w = kOptThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      red[threadIdx.x] += red[threadIdx.x + w];
      bred[threadIdx.x] |= bred[threadIdx.x + w];
    }
    __syncthreads();
  }
  __shared__ int last;
  if (threadIdx.x == 0) {
    partial[blockIdx.x] = red[0];
    flag[blockIdx.x] = bred[0];
    // publish this block's partial, then count it; the block that counts
    // last sees every partial
    __threadfence();
    last = atomicAdd(g_opt_done + slot, 1) == static_cast<int>(gridDim.x) - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  opt_finalize_block(P, partial, flag, gridDim.x, ctl, red, bred);
  if (threadIdx.x == 0) g_opt_done[slot] = 0;  // the slot's next launch counts from zero
}

__device__ __forceinline__ float adam_elem(float p, float g, float& m, float& v, float wd,
                                           const OptParams& P, const OptControl& c) {
  g = fmaf(wd, p, g * c.grad_mul);
  m = fmaf(P.beta1, m, P.one_minus_beta1 * g);
  v = fmaf(P.beta2, v, P.one_minus_beta2 * g * g);
  const float denom = sqrtf(v * c.inv_bc2) + P.eps;
  return p - c.step_size * (m / denom);
}

__global__ void __launch_bounds__(kOptThreads) opt_adam_kernel(const __grid_constant__ OptParams P,
                                                               const OptControl* __restrict__ ctl) {
  pdl_wait();
  pdl_trigger();
  const OptControl c = *ctl;
  if (c.skip) return;
  for (int64_t ch = blockIdx.x; ch < P.nchunks; ch += gridDim.x) {
    int g;
    int64_t off, len;
    group_of_chunk(P, ch, g, off, len);
    const OptGroup& G = P.group[g];
    float* p = G.param + off;
    const float* gr = G.grad + off;
    float* m = G.exp_avg + off;
    float* v = G.exp_avg_sq + off;
    __nv_bfloat16* mp = G.model_param ? static_cast<__nv_bfloat16*>(G.model_param) + off : nullptr;
    const int64_t nv = len >> 2;
    for (int64_t i = threadIdx.x; i < nv; i += kOptThreads) {
      float4 pp = reinterpret_cast<float4*>(p)[i];
      const float4 gg = __ldcs(reinterpret_cast<const float4*>(gr) + i);
      float4 mm = reinterpret_cast<float4*>(m)[i];
      float4 vv = reinterpret_cast<float4*>(v)[i];
      pp.x = adam_elem(pp.x, gg.x, mm.x, vv.x, G.weight_decay, P, c);
      pp.y = adam_elem(pp.y, gg.y, mm.y, vv.y, G.weight_decay, P, c);
      pp.z = adam_elem(pp.z, gg.z, mm.z, vv.z, G.weight_decay, P, c);
      pp.w = adam_elem(pp.w, gg.w, mm.w, vv.w, G.weight_decay, P, c);
      reinterpret_cast<float4*>(p)[i] = pp;
      __stcs(reinterpret_cast<float4*>(m) + i, mm);
      __stcs(reinterpret_cast<float4*>(v) + i, vv);
      if (mp) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(pp.x, pp.y), hi = __floats2bfloat162_rn(pp.z, pp.w);
        uint2 w;
        w.x = *reinterpret_cast<uint32_t*>(&lo);
        w.y = *reinterpret_cast<uint32_t*>(&hi);
        reinterpret_cast<uint2*>(mp)[i] = w;
      }
    }
    for (int64_t i = (nv << 2) + threadIdx.x; i < len; i += kOptThreads) {
      float mm = m[i], vv = v[i];
      const float np = adam_elem(p[i], gr[i], mm, vv, G.weight_decay, P, c);
      p[i] = np;
      m[i] = mm;
      v[i] = vv;
      if (mp) mp[i] = __float2bfloat16_rn(np);
    }
  }
}

}  // namespace

int64_t opt_chunk_elems() { return kOptChunk; }

// [0, 256): OptControl; then kMaxOptGrid fp64 partials and kMaxOptGrid flags.
size_t opt_workspace_bytes() {
  return 256 + static_cast<size_t>(kMaxOptGrid) * (sizeof(double) + sizeof(int));
}

// One wave: as many blocks as fit on all SMs at once (so every block gets the
// same share of chunks and no partial second wave), never more than chunks.
template <class K>
int opt_grid(K kernel, int64_t nchunks, int num_sms) {
  // Blocks per SM depend on the kernel's resources and the architecture
  // only (one build, one GPU model): computed on first use; threads racing on
  // it compute the same value.
  static std::atomic<int> per_sm{0};
  int b = per_sm.load(std::memory_order_relaxed);
  if (b == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kOptThreads, 0) != cudaSuccess || b < 1)
      b = 1;
    per_sm.store(b, std::memory_order_relaxed);
  }
  int64_t g = static_cast<int64_t>(num_sms) * b;
  if (g > kMaxOptGrid) g = kMaxOptGrid;
  if (g > nchunks) g = nchunks;
  return g < 1 ? 1 : static_cast<int>(g);
}

static double* ws_partial(void* ws) {
  return reinterpret_cast<double*>(static_cast<uint8_t*>(ws) + 256);
}
static int* ws_flag(void* ws) { return reinterpret_cast<int*>(ws_partial(ws) + kMaxOptGrid); }

cudaError_t launch_adam_norm(const OptParams& P, int num_sms, void* ws, cudaStream_t s) {
  const int grid = opt_grid(opt_norm_kernel, P.nchunks, num_sms);
  const int slot = static_cast<int>(g_opt_slot_seq.fetch_add(1) % kOptSlots);
  launch_k(opt_norm_kernel, grid, kOptThreads, 0, s, P, ws_partial(ws), ws_flag(ws), static_cast<OptControl*>(ws),
           slot);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_adam_update(const OptParams& P, int num_sms, void* ws, cudaStream_t s) {
  const int grid = opt_grid(opt_adam_kernel, P.nchunks, num_sms);
  launch_k(opt_adam_kernel, grid, kOptThreads, 0, s, P, static_cast<const OptControl*>(ws));
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace tp
