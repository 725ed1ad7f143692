// Allocation-free variant of tied_embed_grad.
//
// tied_embed_grad needs a small device workspace for grouping tokens by id
// (segment offsets, the token permutation and per-id counters).  Some callers
// cannot hand one over: code that runs under a memory manager which owns every
// device allocation (a serving runtime that reserves HBM up front and forbids
// libraries from allocating), or code that must not call cudaMalloc because it
// synchronises the device in the middle of their stream work.  For them this
// file keeps the scratch in a fixed-size static device array that every GPU
// loading the library holds until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "tp.h"
#include "tp_internal.h"

namespace {

constexpr size_t kScratchBytes = 1536u * 1024u;  // 1.5 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_tied_grad_scratch[kScratchBytes];

// Device address of the scratch array per device.  In host code the array's
// name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress with the device current.
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

tp_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TP_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tied_grad_scratch) != cudaSuccess || p == nullptr)
      return TP_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TP_OK;
}

}  // namespace

extern "C" TP_API tp_status tied_embed_grad_noalloc(tp_dtype dt, int64_t T, int64_t h, int64_t V,
                                                    int N, const int64_t* ids, const void* dEmb,
                                                    const void* X, const void* const* dLogits,
                                                    const int64_t* ld_dlogits,
                                                    const int64_t* range_starts, void* const* dE,
                                                    int accumulate, void* stream) {
  // Argument errors first, then the size limit, and only then the device: an
  // invalid call returns its argument error even without a usable GPU.
  const tp_status chk =
      tp::tied_embed_grad_check(dt, T, h, V, N, ids, dEmb, X, dLogits, ld_dlogits, range_starts, dE);
  if (chk != TP_OK) return chk;
  if (tied_embed_grad_workspace_size(T, V) > kScratchBytes) return TP_ERR_WORKSPACE;
  void* scratch = nullptr;
  const tp_status st = scratch_for_current_device(&scratch);
  if (st != TP_OK) return st;
  // The grouping kernels clear the per-id counters they use on every call, so
  // whatever an earlier call left in the array does not matter.
  return tied_embed_grad(dt, T, h, V, N, ids, dEmb, X, dLogits, ld_dlogits, range_starts, dE,
                         accumulate, scratch, kScratchBytes, stream);
}
