// C ABI of the tensor-parallel block library: argument validation, TMA
// descriptor encoding, GEMM planning (groups = output matrices, segments =
// shards summed into them), launches, status and profiling.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "tp.h"
#include "tp_internal.h"

using namespace tp;

// Device error word: bit kErrTimeout is set by a kernel whose bounded wait
// expired.  A static device variable, so the library allocates nothing.
__device__ unsigned int g_tp_error_word;

namespace {

// ---------------------------------------------------------------------------
// Per-device state: SM count and the error word's device address
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;
struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  unsigned* err = nullptr;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

int g_fault_kind = 0;
unsigned long long g_wait_limit_ns = 1000ull * 1000ull * 1000ull;

tp_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TP_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return TP_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tp_error_word) != cudaSuccess) return TP_ERR_CUDA;
    d.err = static_cast<unsigned*>(p);
    d.ready = true;
  }
  *out = &d;
  return TP_OK;
}

// ---------------------------------------------------------------------------
// Profiling: optional CUDA events around every launch
// ---------------------------------------------------------------------------
struct ProfRec {
  const char* name;
  cudaEvent_t e0, e1;
};
bool g_prof_on = false;
std::vector<ProfRec> g_prof_pending;
std::vector<cudaEvent_t> g_event_pool;
struct ProfAgg {
  const char* name;
  int64_t launches;
  double ms;
};
std::vector<ProfAgg> g_prof_agg;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

template <class F>
cudaError_t timed(const char* name, cudaStream_t s, F&& launch) {
  if (!g_prof_on) return launch();
  std::lock_guard<std::mutex> lk(g_mu);
  ProfRec r{name, take_event(), take_event()};
  cudaEventRecord(r.e0, s);
  cudaError_t e = launch();
  cudaEventRecord(r.e1, s);
  g_prof_pending.push_back(r);
  return e;
}

void prof_flush_locked() {
  if (g_prof_pending.empty()) return;
  cudaDeviceSynchronize();
  for (auto& r : g_prof_pending) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.e0, r.e1);
    bool found = false;
    for (auto& a : g_prof_agg)
      if (strcmp(a.name, r.name) == 0) {
        a.launches += 1;
        a.ms += ms;
        found = true;
      }
    if (!found) g_prof_agg.push_back(ProfAgg{r.name, 1, ms});
    g_event_pool.push_back(r.e0);
    g_event_pool.push_back(r.e1);
  }
  g_prof_pending.clear();
}

// ---------------------------------------------------------------------------
// TMA descriptor encoding (driver entry point fetched through the runtime)
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool get_encode() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return true;
}

// A stored bf16 matrix (rows x cols, row pitch ld elements) as a 2D tensor
// map with a (64 columns x box_rows) box and 128-byte swizzle.
bool encode_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                uint32_t box_rows) {
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), gdim, gstride, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// GEMM planning
// ---------------------------------------------------------------------------
// A stored operand.  K-major: rows = M (or N), cols = K.  MN-major: rows = K,
// cols = M (or N).
struct Operand {
  const void* ptr;
  int mn;
  int64_t rows, cols, ld;
};
inline Operand kmajor(const void* p, int64_t mn_extent, int64_t K, int64_t ld) {
  return Operand{p, 0, mn_extent, K, ld};
}
inline Operand mnmajor(const void* p, int64_t K, int64_t mn_extent, int64_t ld) {
  return Operand{p, 1, K, mn_extent, ld};
}

struct Plan {
  struct Seg {
    Operand A, B;
    int64_t K;
  };
  Seg seg[kMaxSegs];
  GemmGroup grp[kMaxGroups];
  int ns = 0, ng = 0;
  bool overflow = false;

  int add_seg(const Operand& A, const Operand& B, int64_t K) {
    if (ns >= kMaxSegs) {
      overflow = true;
      return 0;
    }
    seg[ns] = Seg{A, B, K};
    return ns++;
  }
  GemmGroup& add_group(int64_t M, int64_t N, int sb, int se, int epi, int out_type, void* out,
                       int64_t ldo) {
    static GemmGroup dummy;
    if (ng >= kMaxGroups) {
      overflow = true;
      return dummy;
    }
    GemmGroup& g = grp[ng++];
    memset(&g, 0, sizeof(g));
    g.M = static_cast<int>(M);
    g.N = static_cast<int>(N);
    g.seg_begin = sb;
    g.seg_end = se;
    g.epi = epi;
    g.out_type = out_type;
    g.out = out;
    g.ldo = ldo;
    return g;
  }
};

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool group_vec_ok(const GemmGroup& g, int in_esize) {
  const int oes = g.out_type == OUT_F32 ? 4 : 2;
  bool ok = al16(g.out) && (g.ldo * oes) % 16 == 0;
  if (g.out2) ok = ok && al16(g.out2);
  if (g.bias) ok = ok && al16(g.bias);
  if (g.aux) ok = ok && al16(g.aux) && (g.ld_aux * in_esize) % 16 == 0;
  if (g.seg_src) ok = ok && al16(g.seg_src) && (g.ld_seg * in_esize) % 16 == 0;
  return ok;
}

tp_status run_plan(Plan& pl, tp_dtype dt, const char* name, cudaStream_t s) {
  if (pl.overflow) return TP_ERR_INVALID;
  // Drop empty outputs; mark outputs with no k-blocks and the segments that
  // kept outputs use.
  GemmGroup groups[kMaxGroups];
  bool used[kMaxSegs] = {};
  int ng = 0;
  for (int i = 0; i < pl.ng; ++i) {
    GemmGroup g = pl.grp[i];
    if (g.M <= 0 || g.N <= 0) continue;
    int64_t ktot = 0;
    for (int sidx = g.seg_begin; sidx < g.seg_end; ++sidx) {
      ktot += pl.seg[sidx].K;
      used[sidx] = pl.seg[sidx].K > 0;
    }
    g.k_empty = ktot == 0;
    groups[ng++] = g;
  }
  if (ng == 0) return TP_OK;
  // Host-side checks before anything touches the GPU.
  if (dt == TP_BF16) {
    for (int i = 0; i < pl.ns; ++i) {
      if (!used[i]) continue;
      const Plan::Seg& S = pl.seg[i];
      const Operand* ops[2] = {&S.A, &S.B};
      for (int j = 0; j < 2; ++j) {
        const Operand& o = *ops[j];
        if (!al16(o.ptr) || (o.ld % 8) != 0) return TP_ERR_ALIGN;
        if (o.rows <= 0 || o.cols <= 0) return TP_ERR_INVALID;
      }
    }
  }
  DeviceState* dev = nullptr;
  tp_status st = device_state(&dev);
  if (st != TP_OK) return st;

  if (dt == TP_F32) {
    static SimtGemmParams p;
    memset(&p, 0, sizeof(p));
    for (int i = 0; i < pl.ns; ++i) {
      const Plan::Seg& S = pl.seg[i];
      SimtSeg& q = p.seg[i];
      q.A = static_cast<const float*>(S.A.ptr);
      q.B = static_cast<const float*>(S.B.ptr);
      q.sam = S.A.mn ? 1 : S.A.ld;
      q.sak = S.A.mn ? S.A.ld : 1;
      q.sbn = S.B.mn ? 1 : S.B.ld;
      q.sbk = S.B.mn ? S.B.ld : 1;
      q.K = static_cast<int>(S.K);
    }
    int tiles = 0;
    for (int i = 0; i < ng; ++i) {
      GemmGroup& g = groups[i];
      g.tiles_m = (g.M + 63) / 64;
      g.tiles_n = (g.N + 63) / 64;
      g.tile_begin = tiles;
      tiles += g.tiles_m * g.tiles_n;
      p.grp[i] = g;
    }
    p.num_groups = ng;
    p.num_segs = pl.ns;
    p.total_tiles = tiles;
    cudaError_t e = timed(name, s, [&] { return launch_simt_gemm(p, s); });
    return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
  }

  if (!get_encode()) return TP_ERR_CUDA;
  static TcGemmParams p;
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < pl.ns; ++i) {
    const Plan::Seg& S = pl.seg[i];
    p.seg[i].K = static_cast<int>(S.K);
    p.seg[i].a_mn = S.A.mn;
    p.seg[i].b_mn = S.B.mn;
    if (!used[i]) continue;
    // K-major boxes are (64 K) x (128 or 256 rows); MN-major boxes (64 MN) x (64 K).
    if (!encode_map(&p.mapA[i], S.A.ptr, S.A.rows, S.A.cols, S.A.ld, S.A.mn ? 64 : 128))
      return TP_ERR_CUDA;
    if (!encode_map(&p.mapB[i], S.B.ptr, S.B.rows, S.B.cols, S.B.ld, S.B.mn ? 64 : 256))
      return TP_ERR_CUDA;
  }
  int tiles = 0;
  for (int i = 0; i < ng; ++i) {
    GemmGroup& g = groups[i];
    g.tiles_m = (g.M + 127) / 128;
    g.tiles_n = (g.N + 255) / 256;
    g.tile_begin = tiles;
    g.vec_ok = group_vec_ok(g, 2);
    tiles += g.tiles_m * g.tiles_n;
    p.grp[i] = g;
  }
  p.num_groups = ng;
  p.num_segs = pl.ns;
  p.total_tiles = tiles;
  p.err = dev->err;
  p.wait_limit_ns = g_wait_limit_ns;
  p.fault_skip = g_fault_kind == 1;
  g_fault_kind = 0;
  cudaError_t e = timed(name, s, [&] { return launch_tc_gemm(p, dev->num_sms, s); });
  return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

inline size_t esize(tp_dtype dt) { return dt == TP_F32 ? 4 : 2; }
inline const uint8_t* cb(const void* p) { return static_cast<const uint8_t*>(p); }
inline uint8_t* bb(void* p) { return static_cast<uint8_t*>(p); }

bool dtype_ok(tp_dtype dt) { return dt == TP_F32 || dt == TP_BF16; }

bool shards_ok(const void* const* a, int N) {
  if (a == nullptr) return false;
  for (int i = 0; i < N; ++i)
    if (a[i] == nullptr) return false;
  return true;
}

bool opt_shards_ok(const void* const* a, int N) { return a == nullptr || shards_ok(a, N); }

}  // namespace

// ===========================================================================
// MLP block
// ===========================================================================
extern "C" tp_status tp_mlp_fwd(tp_dtype dt, int64_t M, int64_t h, int64_t hp, int N,
                                const void* X, const void* const* W, const void* const* a,
                                const void* const* U, const void* b, void* Z, void* Y, void* Out,
                                void* stream) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (M < 0 || h <= 0 || hp <= 0 || N < 1 || N > 8 || hp % N != 0) return TP_ERR_INVALID;
  if (M > INT32_MAX || h > INT32_MAX || hp > INT32_MAX) return TP_ERR_INVALID;
  if (!shards_ok(W, N) || !shards_ok(U, N) || !opt_shards_ok(a, N)) return TP_ERR_INVALID;
  if (M > 0 && (!X || !Z || !Y || !Out)) return TP_ERR_INVALID;
  if (M == 0) return TP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t ns = hp / N;
  const size_t es = esize(dt);
  const int ot = dt == TP_F32 ? OUT_F32 : OUT_BF16;

  // Column-parallel linear + bias + GELU: one output block per shard.
  Plan p1;
  for (int i = 0; i < N; ++i) {
    const int si = p1.add_seg(kmajor(X, M, h, h), kmajor(W[i], ns, h, h), h);
    GemmGroup& g = p1.add_group(M, ns, si, si + 1, EPI_BIAS_GELU, ot, bb(Z) + i * ns * es, hp);
    g.out2 = bb(Y) + i * ns * es;
    g.bias = a ? a[i] : nullptr;
  }
  tp_status st = run_plan(p1, dt, "gemm_column_gelu", s);
  if (st != TP_OK) return st;

  // Row-parallel linear: the shards are the segments of one output (g = sum).
  Plan p2;
  for (int i = 0; i < N; ++i)
    p2.add_seg(kmajor(cb(Y) + i * ns * es, M, ns, hp), kmajor(U[i], h, ns, ns), ns);
  GemmGroup& g = p2.add_group(M, h, 0, N, EPI_STORE, ot, Out, h);
  g.bias = b;
  return run_plan(p2, dt, "gemm_row_shardsum", s);
}

extern "C" size_t tp_mlp_bwd_workspace_size(int64_t M, int64_t h, int64_t hp) {
  if (M < 0 || h <= 0 || hp <= 0) return 0;
  return colsum_workspace_bytes(M, hp) + colsum_workspace_bytes(M, h);
}

extern "C" tp_status tp_mlp_bwd(tp_dtype dt, int64_t M, int64_t h, int64_t hp, int N,
                                const void* dOut, const void* X, const void* const* W,
                                const void* const* U, const void* Z, const void* Y, void* dZ,
                                void* dX, void* const* dW, void* const* da, void* const* dU,
                                void* db, int accumulate, void* workspace, size_t ws_bytes,
                                void* stream) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (M < 0 || h <= 0 || hp <= 0 || N < 1 || N > 8 || hp % N != 0) return TP_ERR_INVALID;
  if (M > INT32_MAX || h > INT32_MAX || hp > INT32_MAX) return TP_ERR_INVALID;
  if (!shards_ok(W, N) || !shards_ok(U, N) || !shards_ok(dW, N) || !shards_ok(dU, N) ||
      !opt_shards_ok(da, N))
    return TP_ERR_INVALID;
  if (M > 0 && (!dOut || !X || !Z || !Y || !dZ || !dX)) return TP_ERR_INVALID;
  const bool bias_grads = da != nullptr || db != nullptr;
  if (bias_grads && (workspace == nullptr || ws_bytes < tp_mlp_bwd_workspace_size(M, h, hp)))
    return TP_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t ns = hp / N;
  const size_t es = esize(dt);
  const int ot = dt == TP_F32 ? OUT_F32 : OUT_BF16;

  // Launch 1: dU_i = dOut^T Y_i (contraction over tokens) and
  //           dZ_i = (dOut U_i) * GELU'(Z_i)  (g backward is the identity).
  Plan p1;
  for (int i = 0; i < N; ++i) {
    const int si = p1.add_seg(mnmajor(dOut, M, h, h), mnmajor(cb(Y) + i * ns * es, M, ns, hp), M);
    GemmGroup& g = p1.add_group(h, ns, si, si + 1, EPI_F32, OUT_F32, dU[i], ns);
    g.accumulate = accumulate;
  }
  for (int i = 0; i < N; ++i) {
    const int si = p1.add_seg(kmajor(dOut, M, h, h), mnmajor(U[i], h, ns, ns), h);
    GemmGroup& g = p1.add_group(M, ns, si, si + 1, EPI_DGELU, ot, bb(dZ) + i * ns * es, hp);
    g.aux = cb(Z) + i * ns * es;
    g.ld_aux = hp;
  }
  tp_status st = run_plan(p1, dt, "gemm_dU_dgelu", s);
  if (st != TP_OK) return st;

  // Launch 2: dX = sum_i dZ_i W_i (f backward = sum over shards, fused) and
  //           dW_i = dZ_i^T X.
  Plan p2;
  for (int i = 0; i < N; ++i)
    p2.add_seg(kmajor(cb(dZ) + i * ns * es, M, ns, hp), mnmajor(W[i], ns, h, h), ns);
  p2.add_group(M, h, 0, N, EPI_STORE, ot, dX, h);
  for (int i = 0; i < N; ++i) {
    const int si = p2.add_seg(mnmajor(cb(dZ) + i * ns * es, M, ns, hp), mnmajor(X, M, h, h), M);
    GemmGroup& g = p2.add_group(ns, h, si, si + 1, EPI_F32, OUT_F32, dW[i], h);
    g.accumulate = accumulate;
  }
  st = run_plan(p2, dt, "gemm_dX_shardsum_dW", s);
  if (st != TP_OK) return st;

  // Bias gradients: deterministic column sums.
  if (bias_grads) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int in_f32 = dt == TP_F32;
    if (da) {
      ShardOut o{};
      for (int i = 0; i < N; ++i) o.p[i] = static_cast<float*>(da[i]);
      o.cols_per_shard = ns;
      o.n = N;
      cudaError_t e = timed("colsum_da", s, [&] {
        return launch_colsum(dZ, in_f32, M, hp, hp, o, accumulate, ws, s);
      });
      if (e != cudaSuccess) return TP_ERR_CUDA;
    }
    if (db) {
      ShardOut o{};
      o.p[0] = static_cast<float*>(db);
      o.cols_per_shard = h;
      o.n = 1;
      cudaError_t e = timed("colsum_db", s, [&] {
        return launch_colsum(dOut, in_f32, M, h, h, o, accumulate,
                             ws + colsum_workspace_bytes(M, hp), s);
      });
      if (e != cudaSuccess) return TP_ERR_CUDA;
    }
  }
  return TP_OK;
}

// ===========================================================================
// Attention projections
// ===========================================================================
extern "C" tp_status tp_attn_proj_fwd(tp_dtype dt, int64_t M, int64_t h, int n_heads, int N,
                                      const void* X, const void* const* Wqkv,
                                      const void* const* bqkv, const void* C,
                                      const void* const* Wo, const void* bo, void* QKV, void* O,
                                      void* stream) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (M < 0 || h <= 0 || N < 1 || N > 8 || n_heads < 1 || n_heads % N != 0 || h % n_heads != 0)
    return TP_ERR_INVALID;
  if (M > INT32_MAX || 3 * h > INT32_MAX) return TP_ERR_INVALID;
  if (!shards_ok(Wqkv, N) || !shards_ok(Wo, N) || !opt_shards_ok(bqkv, N)) return TP_ERR_INVALID;
  if (M > 0 && (!X || !C || !QKV || !O)) return TP_ERR_INVALID;
  if (M == 0) return TP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t d = h / N;  // context columns per shard
  const size_t es = esize(dt);
  const int ot = dt == TP_F32 ? OUT_F32 : OUT_BF16;

  Plan p;
  // Output projection first: O = sum_i C_i Wo_i^T + bo.
  for (int i = 0; i < N; ++i) p.add_seg(kmajor(cb(C) + i * d * es, M, d, h), kmajor(Wo[i], h, d, d), d);
  GemmGroup& go = p.add_group(M, h, 0, N, EPI_STORE, ot, O, h);
  go.bias = bo;
  // QKV_i = X Wqkv_i^T + bqkv_i, one block per shard.
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(kmajor(X, M, h, h), kmajor(Wqkv[i], 3 * d, h, h), h);
    GemmGroup& g = p.add_group(M, 3 * d, si, si + 1, EPI_STORE, ot, bb(QKV) + i * 3 * d * es, 3 * h);
    g.bias = bqkv ? bqkv[i] : nullptr;
  }
  return run_plan(p, dt, "gemm_attn_fwd", s);
}

extern "C" size_t tp_attn_proj_bwd_workspace_size(int64_t M, int64_t h) {
  if (M < 0 || h <= 0) return 0;
  return colsum_workspace_bytes(M, 3 * h) + colsum_workspace_bytes(M, h);
}

extern "C" tp_status tp_attn_proj_bwd(tp_dtype dt, int64_t M, int64_t h, int n_heads, int N,
                                      const void* dQKV, const void* dO, const void* X,
                                      const void* C, const void* const* Wqkv,
                                      const void* const* Wo, void* dX, void* dC,
                                      void* const* dWqkv, void* const* dbqkv, void* const* dWo,
                                      void* dbo, int accumulate, void* workspace, size_t ws_bytes,
                                      void* stream) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (M < 0 || h <= 0 || N < 1 || N > 8 || n_heads < 1 || n_heads % N != 0 || h % n_heads != 0)
    return TP_ERR_INVALID;
  if (M > INT32_MAX || 3 * h > INT32_MAX) return TP_ERR_INVALID;
  if (!shards_ok(Wqkv, N) || !shards_ok(Wo, N) || !shards_ok(dWqkv, N) || !shards_ok(dWo, N) ||
      !opt_shards_ok(dbqkv, N))
    return TP_ERR_INVALID;
  if (M > 0 && (!dQKV || !dO || !X || !C || !dX || !dC)) return TP_ERR_INVALID;
  const bool bias_grads = dbqkv != nullptr || dbo != nullptr;
  if (bias_grads && (workspace == nullptr || ws_bytes < tp_attn_proj_bwd_workspace_size(M, h)))
    return TP_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t d = h / N;
  const int64_t w = 3 * d;
  const size_t es = esize(dt);
  const int ot = dt == TP_F32 ? OUT_F32 : OUT_BF16;

  // Weight gradients (contractions over tokens), one launch.
  Plan p1;
  for (int i = 0; i < N; ++i) {
    const int si = p1.add_seg(mnmajor(cb(dQKV) + i * w * es, M, w, 3 * h), mnmajor(X, M, h, h), M);
    GemmGroup& g = p1.add_group(w, h, si, si + 1, EPI_F32, OUT_F32, dWqkv[i], h);
    g.accumulate = accumulate;
  }
  for (int i = 0; i < N; ++i) {
    const int si = p1.add_seg(mnmajor(dO, M, h, h), mnmajor(cb(C) + i * d * es, M, d, h), M);
    GemmGroup& g = p1.add_group(h, d, si, si + 1, EPI_F32, OUT_F32, dWo[i], d);
    g.accumulate = accumulate;
  }
  tp_status st = run_plan(p1, dt, "gemm_attn_dW", s);
  if (st != TP_OK) return st;

  // Activation gradients: dX = sum_i dQKV_i Wqkv_i (shard sum), dC_i = dO Wo_i.
  Plan p2;
  for (int i = 0; i < N; ++i)
    p2.add_seg(kmajor(cb(dQKV) + i * w * es, M, w, 3 * h), mnmajor(Wqkv[i], w, h, h), w);
  p2.add_group(M, h, 0, N, EPI_STORE, ot, dX, h);
  for (int i = 0; i < N; ++i) {
    const int si = p2.add_seg(kmajor(dO, M, h, h), mnmajor(Wo[i], h, d, d), h);
    p2.add_group(M, d, si, si + 1, EPI_STORE, ot, bb(dC) + i * d * es, h);
  }
  st = run_plan(p2, dt, "gemm_attn_dX_dC", s);
  if (st != TP_OK) return st;

  if (bias_grads) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int in_f32 = dt == TP_F32;
    if (dbqkv) {
      ShardOut o{};
      for (int i = 0; i < N; ++i) o.p[i] = static_cast<float*>(dbqkv[i]);
      o.cols_per_shard = w;
      o.n = N;
      cudaError_t e = timed("colsum_dbqkv", s, [&] {
        return launch_colsum(dQKV, in_f32, M, 3 * h, 3 * h, o, accumulate, ws, s);
      });
      if (e != cudaSuccess) return TP_ERR_CUDA;
    }
    if (dbo) {
      ShardOut o{};
      o.p[0] = static_cast<float*>(dbo);
      o.cols_per_shard = h;
      o.n = 1;
      cudaError_t e = timed("colsum_dbo", s, [&] {
        return launch_colsum(dO, in_f32, M, h, h, o, accumulate,
                             ws + colsum_workspace_bytes(M, 3 * h), s);
      });
      if (e != cudaSuccess) return TP_ERR_CUDA;
    }
  }
  return TP_OK;
}

// ===========================================================================
// Vocab-parallel embedding, logits, tied gradient
// ===========================================================================
namespace {
bool ranges_ok(const int64_t* rs, int N, int64_t V) {
  if (rs == nullptr || N < 1 || N > kMaxRanges) return false;
  if (rs[0] != 0 || rs[N] != V) return false;
  for (int r = 0; r < N; ++r)
    if (rs[r + 1] <= rs[r]) return false;
  return true;
}
}  // namespace

extern "C" tp_status vocab_parallel_embed(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                                          const int64_t* ids, const void* const* E,
                                          const int64_t* range_starts, void* out, void* stream) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (T < 0 || h <= 0 || V <= 0 || !ranges_ok(range_starts, N, V) || !shards_ok(E, N))
    return TP_ERR_INVALID;
  if (T > 0 && (!ids || !out)) return TP_ERR_INVALID;
  if (T == 0) return TP_OK;
  RangeTable rt{};
  for (int r = 0; r <= N; ++r) rt.start[r] = range_starts[r];
  for (int r = 0; r < N; ++r) rt.ptr[r] = E[r];
  rt.n = N;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t row_bytes = h * static_cast<int64_t>(esize(dt));
  cudaError_t e = timed("embed_gather", s, [&] { return launch_embed_gather(ids, T, row_bytes, rt, out, s); });
  return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

extern "C" tp_status tp_vocab_logits(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                                     const void* X, const void* const* E,
                                     const int64_t* range_starts, void* const* logits,
                                     const int64_t* ld_logits, void* stream) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (T < 0 || h <= 0 || V <= 0 || N > kMaxGroups || !ranges_ok(range_starts, N, V) ||
      !shards_ok(E, N) || ld_logits == nullptr || (T > 0 && !shards_ok(logits, N)))
    return TP_ERR_INVALID;
  if (T > INT32_MAX || V > INT32_MAX || h > INT32_MAX) return TP_ERR_INVALID;
  for (int r = 0; r < N; ++r)
    if (ld_logits[r] < range_starts[r + 1] - range_starts[r]) return TP_ERR_INVALID;
  if (T > 0 && !X) return TP_ERR_INVALID;
  if (T == 0) return TP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int ot = dt == TP_F32 ? OUT_F32 : OUT_BF16;
  Plan p;
  for (int r = 0; r < N; ++r) {
    const int64_t nr = range_starts[r + 1] - range_starts[r];
    const int si = p.add_seg(kmajor(X, T, h, h), kmajor(E[r], nr, h, h), h);
    p.add_group(T, nr, si, si + 1, EPI_STORE, ot, logits[r], ld_logits[r]);
  }
  return run_plan(p, dt, "gemm_logits", s);
}

extern "C" size_t tied_embed_grad_workspace_size(int64_t T, int64_t V) {
  if (T < 0 || V <= 0) return 0;
  return sort_workspace_bytes(T, V);
}

extern "C" tp_status tied_embed_grad(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                                     const int64_t* ids, const void* dEmb, const void* X,
                                     const void* const* dLogits, const int64_t* ld_dlogits,
                                     const int64_t* range_starts, void* const* dE, int accumulate,
                                     void* workspace, size_t ws_bytes, void* stream) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (T < 0 || h <= 0 || V <= 0 || N > kMaxGroups || !ranges_ok(range_starts, N, V) ||
      !shards_ok(dE, N))
    return TP_ERR_INVALID;
  if (T > INT32_MAX || V > INT32_MAX || h > INT32_MAX) return TP_ERR_INVALID;
  if (dLogits != nullptr) {
    if ((T > 0 && !shards_ok(dLogits, N)) || ld_dlogits == nullptr) return TP_ERR_INVALID;
    for (int r = 0; r < N; ++r)
      if (ld_dlogits[r] < range_starts[r + 1] - range_starts[r]) return TP_ERR_INVALID;
    if (T > 0 && !X) return TP_ERR_INVALID;
  }
  if (T > 0 && (!ids || !dEmb)) return TP_ERR_INVALID;
  if (workspace == nullptr || ws_bytes < tied_embed_grad_workspace_size(T, V)) return TP_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  cudaError_t e = timed("embed_sort", s, [&] { return launch_embed_sort(ids, T, V, workspace, s); });
  if (e != cudaSuccess) return TP_ERR_CUDA;

  if (dLogits == nullptr) {
    RangeTable rt{};
    for (int r = 0; r <= N; ++r) rt.start[r] = range_starts[r];
    for (int r = 0; r < N; ++r) rt.ptr[r] = dE[r];
    rt.n = N;
    e = timed("segment_sum", s, [&] {
      return launch_segment_sum(workspace, V, T, dEmb, dt == TP_F32, h, rt, accumulate, s);
    });
    return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
  }

  // dE_r = dLogits_r^T X (contraction over tokens) + ordered segment sums of
  // dEmb, fused in the epilogue.
  Plan p;
  const int* offsets = sort_offsets(workspace);
  const int* perm = sort_perm(workspace, V);
  for (int r = 0; r < N; ++r) {
    const int64_t nr = range_starts[r + 1] - range_starts[r];
    const int si = p.add_seg(mnmajor(dLogits[r], T, nr, ld_dlogits[r]), mnmajor(X, T, h, h), T);
    GemmGroup& g = p.add_group(nr, h, si, si + 1, EPI_SEGSUM, OUT_F32, dE[r], h);
    g.accumulate = accumulate;
    g.seg_offsets = offsets;
    g.seg_perm = perm;
    g.seg_src = dEmb;
    g.ld_seg = h;
    g.seg_row0 = range_starts[r];
  }
  return run_plan(p, dt, "gemm_tied_grad_segsum", s);
}

// ===========================================================================
// Status, profiling, debugging
// ===========================================================================
extern "C" tp_status tp_get_status(void* stream) {
  DeviceState* dev = nullptr;
  if (device_state(&dev) != TP_OK) return TP_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TP_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return TP_ERR_CUDA;
  unsigned w = 0;
  if (cudaMemcpyFromSymbol(&w, g_tp_error_word, sizeof(w)) != cudaSuccess) return TP_ERR_CUDA;
  if (w != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_tp_error_word, &zero, sizeof(zero)) != cudaSuccess) return TP_ERR_CUDA;
    if (w & kErrTimeout) return TP_ERR_TIMEOUT;
  }
  return TP_OK;
}

extern "C" const char* tp_status_string(tp_status s) {
  switch (s) {
    case TP_OK: return "TP_OK";
    case TP_ERR_INVALID: return "TP_ERR_INVALID";
    case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED";
    case TP_ERR_CUDA: return "TP_ERR_CUDA";
    case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT";
    case TP_ERR_WORKSPACE: return "TP_ERR_WORKSPACE";
    case TP_ERR_ALIGN: return "TP_ERR_ALIGN";
  }
  return "TP_ERR_UNKNOWN";
}

extern "C" int tp_num_sms(void) {
  DeviceState* dev = nullptr;
  if (device_state(&dev) != TP_OK) return 0;
  return dev->num_sms;
}

extern "C" void tp_profile_enable(int on) { g_prof_on = on != 0; }

extern "C" void tp_profile_reset(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  prof_flush_locked();
  g_prof_agg.clear();
}

extern "C" int tp_profile_read(const char** names, int64_t* launches, double* total_ms, int cap) {
  std::lock_guard<std::mutex> lk(g_mu);
  prof_flush_locked();
  const int n = static_cast<int>(g_prof_agg.size());
  for (int i = 0; i < n && i < cap; ++i) {
    if (names) names[i] = g_prof_agg[i].name;
    if (launches) launches[i] = g_prof_agg[i].launches;
    if (total_ms) total_ms[i] = g_prof_agg[i].ms;
  }
  return n;
}

extern "C" void tp_debug_inject_fault(int kind) { g_fault_kind = kind; }

extern "C" void tp_debug_set_wait_limit_ms(int ms) {
  g_wait_limit_ns = static_cast<unsigned long long>(ms > 0 ? ms : 1000) * 1000000ull;
}
