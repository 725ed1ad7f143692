// C ABI of the tensor-parallel block library: argument validation, TMA
// descriptor encoding, GEMM planning (groups = output matrices, segments =
// shards summed into them), launches, status and profiling.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <math.h>
#include <mutex>
#include <vector>

#include "tp.h"
#include "tp_internal.h"

using namespace tp;

// Device error word: bit kErrTimeout is set by a kernel whose bounded wait
// expired.  A static device variable, so the library allocates nothing.
__device__ unsigned int g_tp_error_word;

// Ones operands for column sums computed as GEMMs (colsum(A) = A^T 1): a
// 16 x 64 bf16 block of ones read by TMA for the tensor-core engine (every
// k-block reads the same box), and one fp32 1.0 read with zero strides by the
// fp32 engine.
__device__ __align__(128) unsigned short g_ones_bf16[16 * 64];
__device__ float g_one_f32 = 1.0f;

namespace {

// ---------------------------------------------------------------------------
// Per-device state: SM count and the error word's device address
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;
struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  unsigned* err = nullptr;
  void* ones_bf16 = nullptr;
  void* one_f32 = nullptr;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

int g_fault_kind = 0;
int g_gemm_mode = 2;  // 0: one-SM kernel, 1: two-SM kernel, 2: choose per launch
int g_split_tiles_per_sm = 8;  // plans with dependent tiles and more tiles per SM run as two launches
unsigned long long g_wait_limit_ns = 1000ull * 1000ull * 1000ull;
int g_pdl = 1;  // programmatic dependent launch of the library's kernels

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
    if (cudaGetSymbolAddress(&d.ones_bf16, g_ones_bf16) != cudaSuccess) return TP_ERR_CUDA;
    if (cudaGetSymbolAddress(&d.one_f32, g_one_f32) != cudaSuccess) return TP_ERR_CUDA;
    unsigned short ones[16 * 64];
    for (int i = 0; i < 16 * 64; ++i) ones[i] = 0x3F80;  // bf16 1.0
    if (cudaMemcpyToSymbol(g_ones_bf16, ones, sizeof(ones)) != cudaSuccess) return TP_ERR_CUDA;
    d.ready = true;
  }
  *out = &d;
  return TP_OK;
}

// ---------------------------------------------------------------------------
// Profiling: optional CUDA events around every library call's device work
// ---------------------------------------------------------------------------
struct ProfRec {
  const char* name;
  cudaEvent_t e0, e1;
  long long kernels;
};
bool g_prof_on = false;
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof_pending;
std::vector<cudaEvent_t> g_event_pool;
struct ProfAgg {
  const char* name;
  int64_t calls, kernels;
  double ms;
};
std::vector<ProfAgg> g_prof_agg;
std::atomic<long long> g_kernel_launches{0};

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

// Runs `work` (which enqueues kernels on s); when profiling is on, brackets it
// with events on s and records how many kernels it launched.
template <class F>
auto timed(const char* name, cudaStream_t s, F&& work) -> decltype(work()) {
  if (!g_prof_on) return work();
  cudaEvent_t e0, e1;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    e0 = take_event();
    e1 = take_event();
  }
  const long long k0 = g_kernel_launches.load();
  cudaEventRecord(e0, s);
  auto r = work();
  cudaEventRecord(e1, s);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_pending.push_back(ProfRec{name, e0, e1, g_kernel_launches.load() - k0});
  return r;
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
        a.calls += 1;
        a.kernels += r.kernels;
        a.ms += ms;
        found = true;
      }
    if (!found) g_prof_agg.push_back(ProfAgg{r.name, 1, r.kernels, ms});
    g_event_pool.push_back(r.e0);
    g_event_pool.push_back(r.e1);
  }
  g_prof_pending.clear();
}

}  // namespace

void tp::count_launches(int n) { g_kernel_launches.fetch_add(n); }
bool tp::pdl_on() { return g_pdl != 0; }

namespace {

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

// An MN-major bf16 matrix (rows = K, cols = MN, MN a multiple of 64) as a 3D
// map (64 MN, K rows, MN / 64 blocks) whose (64, 64, nblocks) box lands in
// shared memory as nblocks consecutive (64 x 64) blocks, the layout of the
// per-block 2D boxes.  Returns false if the driver rejects the map.
bool encode_map_mn3d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                     uint32_t nblocks) {
  if (cols % 64 != 0) return false;
  cuuint64_t gdim[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
  cuuint64_t gstride[2] = {static_cast<cuuint64_t>(ld) * 2, 128};
  cuuint32_t box[3] = {64, 64, nblocks};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), gdim, gstride, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An output (rows x cols, row pitch ld elements, bf16 or fp32) as a 2D map for
// the epilogue's bulk tensor stores: one box is a 32-row chunk of 64-byte
// rows (32 bf16 or 16 fp32 columns) in the 64-byte swizzle of the stage.
bool encode_store_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, bool f32) {
  const int es = f32 ? 4 : 2;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ld) * es};
  cuuint32_t box[2] = {f32 ? 16u : 32u, 32u};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(ptr), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// GEMM planning
// ---------------------------------------------------------------------------
// A stored operand.  K-major: rows = M (or N), cols = K.  MN-major: rows = K,
// cols = M (or N).  `ones` marks the ones block of a column sum.
struct Operand {
  const void* ptr;
  int mn;
  int64_t rows, cols, ld;
  int ones;
};
inline Operand kmajor(const void* p, int64_t mn_extent, int64_t K, int64_t ld) {
  return Operand{p, 0, mn_extent, K, ld, 0};
}
inline Operand mnmajor(const void* p, int64_t K, int64_t mn_extent, int64_t ld) {
  return Operand{p, 1, K, mn_extent, ld, 0};
}
inline Operand ones_operand() { return Operand{nullptr, 0, 16, 64, 64, 1}; }

struct Plan {
  struct Seg {
    Operand A, B;
    int64_t K;
  };
  Seg seg[kMaxSegs];
  GemmGroup grp[kMaxGroups];
  int ns = 0, ng = 0;
  int interleave = 0;   // leading groups enumerated by row block
  int ncounters = 0;
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
    g.prod_row = -1;
    g.prod_col = -1;
    g.alpha = 1.f;
    g.out_map = -1;
    g.out2_map = -1;
    g.aux_map = -1;
    return g;
  }
  // Counter block for row- or column-tile completion of producing groups.
  int counters(int64_t n) {
    const int b = ncounters;
    ncounters += static_cast<int>(n);
    if (ncounters > kMaxCounters) overflow = true;
    return b;
  }
  // Column sums of a stored MN-major matrix src (rows = K tokens, cols = n)
  // into fp32 out[n]: one GEMM against the ones block.
  GemmGroup& add_colsum(const void* src, int64_t K, int64_t n, int64_t ld, void* out, int accumulate) {
    const int si = add_seg(mnmajor(src, K, n, ld), ones_operand(), K);
    GemmGroup& g = add_group(n, 1, si, si + 1, EPI_F32, OUT_F32, out, 1);
    g.accumulate = accumulate;
    return g;
  }
};

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline size_t round256(size_t b) { return (b + 255) / 256 * 256; }

bool group_vec_ok(const GemmGroup& g, int in_esize) {
  const int oes = g.out_type == OUT_F32 ? 4 : 2;
  bool ok = al16(g.out) && (g.ldo * oes) % 16 == 0;
  if (g.out2) ok = ok && al16(g.out2);
  if (g.bias) ok = ok && al16(g.bias);
  if (g.aux) ok = ok && al16(g.aux) && (g.ld_aux * in_esize) % 16 == 0;
  if (g.seg_src) ok = ok && al16(g.seg_src) && (g.ld_seg * in_esize) % 16 == 0;
  return ok;
}

// Targets of the dependency counters: a consumer waits until every producer
// tile feeding its counter has been stored by all epilogue warps.
// A producer tile counts epi_parts times per CTA that stores part of it (once
// in the one-SM kernel, once per epilogue warp in the two-SM kernel): per
// 128-row block for row counters, per CTA half (`halves` = 2 for the two-SM
// kernel's 256-row tiles) for column counters.
void set_dep_targets(GemmGroup* groups, int ng, int epi_parts, int halves) {
  for (int i = 0; i < ng; ++i) {
    GemmGroup& c = groups[i];
    if (c.dep_kind == DEP_NONE) continue;
    int tiles = 0;
    for (int j = 0; j < ng; ++j) {
      const GemmGroup& q = groups[j];
      if (c.dep_kind == DEP_ROW && q.prod_row == c.dep_base) tiles += q.tiles_n;
      if (c.dep_kind == DEP_COL && q.prod_col == c.dep_base) tiles += q.tiles_m * halves;
    }
    c.dep_target = tiles * epi_parts;
  }
}

tp_status launch_simt_groups(const Plan& pl, const GemmGroup* groups, int ng, const DeviceState* dev,
                             const char* name, cudaStream_t s) {
  static thread_local SimtGemmParams p;
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < pl.ns; ++i) {
    const Plan::Seg& S = pl.seg[i];
    SimtSeg& q = p.seg[i];
    q.A = static_cast<const float*>(S.A.ptr);
    q.sam = S.A.mn ? 1 : S.A.ld;
    q.sak = S.A.mn ? S.A.ld : 1;
    if (S.B.ones) {
      q.B = static_cast<const float*>(dev->one_f32);
      q.sbn = 0;
      q.sbk = 0;
    } else {
      q.B = static_cast<const float*>(S.B.ptr);
      q.sbn = S.B.mn ? 1 : S.B.ld;
      q.sbk = S.B.mn ? S.B.ld : 1;
    }
    q.K = static_cast<int>(S.K);
  }
  int tiles = 0;
  for (int i = 0; i < ng; ++i) {
    GemmGroup g = groups[i];
    g.tiles_m = (g.M + 63) / 64;
    g.tiles_n = (g.N + 63) / 64;
    g.tile_begin = tiles;
    g.dep_kind = DEP_NONE;  // phases are ordered by separate launches instead
    tiles += g.tiles_m * g.tiles_n;
    p.grp[i] = g;
  }
  p.num_groups = ng;
  p.num_segs = pl.ns;
  p.total_tiles = tiles;
  (void)name;
  const cudaError_t e = launch_simt_gemm(p, s);
  return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

// K of an output (the sum over its segments): the length of its tiles' main loop.
int64_t group_k(const Plan& pl, const GemmGroup& g) {
  int64_t k = 0;
  for (int s = g.seg_begin; s < g.seg_end; ++s) k += pl.seg[s].K;
  return k;
}

tp_status launch_tc_groups(const Plan& pl, const bool* used, GemmGroup* groups, int ng,
                           int interleave, int ncounters, const DeviceState* dev, const char* name,
                           cudaStream_t s, bool longest_first) {
  if (ng == 0) return TP_OK;
  // Kernel choice (measured on GB300): the two-SM kernel (256 x 256 pair
  // tiles, 6-stage ring, 32 KB loaded per SM per k-block instead of 48 KB) is
  // faster on large launches (over 5 one-SM tiles per SM; 6 for causal
  // ranges, whose short tiles balance better at one SM; 8 when tiles of the
  // launch wait on other tiles of it), K-major or MN-major; the one-SM
  // kernel (128 x 256 tiles) on small ones, where its finer tiles balance
  // better across SMs.
  // Causal attention outputs count the tiles that hold work: about half, plus
  // the diagonal.  Launches of very long contractions (over 500 k-blocks of
  // tiles per SM, e.g. a shard sum over a whole vocabulary range or over the
  // model-width FFN) also take
  // the two-SM kernel once they hold two one-SM tiles per SM: there the lower
  // operand traffic per SM pays and the tile count no longer sets the balance.
  // So do launches of at least one one-SM tile per SM whose tiles average 48
  // k-blocks or more (without causal ranges): both kernels then need the same
  // number of rounds, and the pair tiles' long main loops hide their epilogue
  // (the H = 4096 layer's output projection, 256 one-SM tiles of 64 k-blocks:
  // 62.4 -> 59.1 us).
  bool pair = g_gemm_mode == 1;
  if (g_gemm_mode == 2) {
    int64_t tiles128 = 0, kb_tiles = 0;
    bool deps = false, ranges = false;
    for (int i = 0; i < ng; ++i) {
      deps = deps || groups[i].dep_kind != DEP_NONE;
      ranges = ranges || groups[i].kr_mode != KR_NONE;
      const int64_t rb = (groups[i].M + 127) / 128, t = rb * ((groups[i].N + 255) / 256);
      const int64_t tw = groups[i].kr_mode != KR_NONE ? (t + rb) / 2 : t;
      int64_t kb = 0;
      for (int sidx = groups[i].seg_begin; sidx < groups[i].seg_end; ++sidx) kb += (pl.seg[sidx].K + 63) / 64;
      tiles128 += tw;
      kb_tiles += tw * kb;
    }
    const int64_t sms = dev->num_sms;
    pair = tiles128 > (deps ? 8 : (ranges ? 6 : 5)) * sms || (tiles128 >= 2 * sms && kb_tiles > 500 * sms) ||
           (!ranges && tiles128 >= sms && kb_tiles >= 48 * tiles128);
  }
  // Tile width: 256 for every output.  (128-wide tiles for the long dependent
  // contractions of small fused launches were measured slower on GB300: a
  // 128-wide MMA is bound by shared-memory bandwidth and doubles A traffic.)
  int seg_bn[kMaxSegs];
  for (int i = 0; i < pl.ns; ++i) seg_bn[i] = 256;
  for (int i = 0; i < ng; ++i) groups[i].bn = 256;
  if (longest_first) {
    // stable: longest contraction first
    for (int i = 1; i < ng; ++i) {
      GemmGroup g = groups[i];
      const int64_t k = group_k(pl, g);
      int j = i - 1;
      while (j >= 0 && group_k(pl, groups[j]) < k) {
        groups[j + 1] = groups[j];
        --j;
      }
      groups[j + 1] = g;
    }
  }
  static thread_local TcGemmParams p;  // per host thread: calls from several threads do not share it
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < pl.ns; ++i) {
    const Plan::Seg& S = pl.seg[i];
    p.seg[i].K = static_cast<int>(S.K);
    p.seg[i].a_mn = S.A.mn;
    p.seg[i].b_mn = S.B.mn;
    p.seg[i].n_mma = S.B.ones ? 16 : seg_bn[i];
    p.seg[i].b_fixed = S.B.ones;
    if (!used[i]) continue;
    // K-major boxes are (64 K) x (128 or 256 rows); MN-major operands use one 3D
    // box per stage when their width is a multiple of 64, else (64 MN) x (64 K)
    // 2D boxes; the ones block is one (64 K) x (16 rows) box.  The two-SM
    // kernel stages half of a 256-wide B tile per CTA.
    const uint32_t b_rows = pair ? 128 : static_cast<uint32_t>(seg_bn[i]);
    if (S.A.mn && encode_map_mn3d(&p.mapA[i], S.A.ptr, S.A.rows, S.A.cols, S.A.ld, 2)) {
      p.seg[i].a_3d = 1;
    } else if (!encode_map(&p.mapA[i], S.A.ptr, S.A.rows, S.A.cols, S.A.ld, S.A.mn ? 64 : 128)) {
      return TP_ERR_CUDA;
    }
    if (S.B.ones) {
      if (!encode_map(&p.mapB[i], dev->ones_bf16, 16, 64, 64, 16)) return TP_ERR_CUDA;
    } else if (S.B.mn && encode_map_mn3d(&p.mapB[i], S.B.ptr, S.B.rows, S.B.cols, S.B.ld, b_rows / 64)) {
      p.seg[i].b_3d = 1;
    } else if (!encode_map(&p.mapB[i], S.B.ptr, S.B.rows, S.B.cols, S.B.ld, S.B.mn ? 64 : b_rows)) {
      return TP_ERR_CUDA;
    }
    if (pair && S.B.ones) p.seg[i].n_mma = 32;  // 16 rows of ones per CTA
  }
  int tiles = 0, inter_nt = 0;
  double inter_b_bytes = 0;  // B operand bytes of the interleaved groups
  const int rows_per_tile = pair ? 256 : 128;
  for (int i = 0; i < ng; ++i) {
    GemmGroup& g = groups[i];
    g.tiles_m = (g.M + rows_per_tile - 1) / rows_per_tile;
    g.tiles_n = (g.N + g.bn - 1) / g.bn;
    g.vec_ok = group_vec_ok(g, 2);
    if (i < interleave) {
      if (g.tiles_m != groups[0].tiles_m) return TP_ERR_INVALID;
      inter_nt += g.tiles_n;
      inter_b_bytes += 2.0 * static_cast<double>(g.N) * static_cast<double>(group_k(pl, g));
    }
  }
  // Tile order: row blocks fastest (consecutive tiles share B's column tile),
  // except for independent, non-causal outputs taller than wide whose A
  // operand is far larger than B and does not stay in L2 (for example the
  // tied gradient's dLogits range, contracted over the tokens): there
  // consecutive tiles share A's row block, which is then read from DRAM once
  // instead of once per column tile.
  for (int i = 0; i < ng; ++i) {
    GemmGroup& g = groups[i];
    const double a_bytes = 2.0 * static_cast<double>(g.M) * static_cast<double>(group_k(pl, g));
    g.n_fastest = i >= interleave && g.kr_mode == KR_NONE && g.dep_kind == DEP_NONE && g.prod_row < 0 &&
                  g.prod_col < 0 && g.M > g.N && a_bytes > 128.0 * (1 << 20);
  }
  // Stripes: in launches without dependent tiles, consecutive groups with
  // causal contraction ranges (P V, dV, dQ, dK of the attention core: one
  // group per head, each tile's length set by its row block) and the same
  // tiling are enumerated together, so the longest tiles of every head come
  // first and the launch does not end on one head's long tiles.
  for (int i = 0; i < ng; ++i) groups[i].stripe_first = i, groups[i].stripe_n = 1;
  bool any_dep = false;
  for (int i = 0; i < ng; ++i) any_dep = any_dep || groups[i].dep_kind != DEP_NONE;
  if (!any_dep) {
    auto stripable = [&](const GemmGroup& g) {
      return (g.kr_mode == KR_END || g.kr_mode == KR_BEGIN) && g.kr_mode != KR_TRI && !g.n_fastest &&
             g.prod_row < 0 && g.prod_col < 0;
    };
    for (int i = interleave; i < ng;) {
      int j = i + 1;
      if (stripable(groups[i]))
        while (j < ng && j - i < 255 && stripable(groups[j]) && groups[j].tiles_m == groups[i].tiles_m &&
               groups[j].tiles_n == groups[i].tiles_n)
          ++j;
      if (j - i > 1)
        for (int k = i; k < j; ++k) groups[k].stripe_first = i, groups[k].stripe_n = j - i;
      i = j;
    }
  }
  for (int i = 0; i < ng; ++i) {
    GemmGroup& g = groups[i];
    g.tile_begin = tiles;
    // causal groups whose empty tiles need not run (and that count no tiles
    // for dependants) enumerate only their causal tiles
    g.tri = g.kr_mode == KR_TRI && g.tri_ok && g.prod_row < 0 && g.prod_col < 0 && i >= interleave;
    if (g.tri) {
      for (int mt = 0; mt < g.tiles_m; ++mt)
        tiles += std::min(g.tiles_n, (mt * rows_per_tile + rows_per_tile - 1) / g.bn + 1);
    } else {
      tiles += g.tiles_m * g.tiles_n;
    }
  }
  // Bulk tensor-store maps for the bf16 outputs the epilogue stores whole
  // (16-byte aligned rows) and bulk-load maps for its bf16 operands, as long
  // as map slots last.
  int nmaps = 0;
  for (int i = 0; i < ng; ++i) {
    GemmGroup& g = groups[i];
    g.out_map = g.out2_map = g.aux_map = -1;
    if (!g.vec_ok || g.out == nullptr || g.k_empty) continue;
    // the dGELU / softmax-backward operand comes in through one bulk load per chunk
    if ((g.epi == EPI_DGELU || g.epi == EPI_SMAX_BWD) && g.aux != nullptr && nmaps < kMaxStoreMaps &&
        encode_store_map(&p.mapO[nmaps], g.aux, g.M, g.N, g.ld_aux, false))
      g.aux_map = nmaps++;
    const bool f32 = g.out_type == OUT_F32;
    bool ok = false;
    switch (g.epi) {
      case EPI_STORE: case EPI_BIAS_GELU: case EPI_DGELU: case EPI_CE_BWD: case EPI_SMAX_BWD:
      case EPI_SMAX_PARTS:
        ok = true;
        break;
      case EPI_F32: case EPI_SEGSUM:
        ok = !g.accumulate;
        break;
      default:
        break;
    }
    // the stores of these epilogues are bf16 whatever out_type says
    const bool out_f32 = f32 && !(g.epi == EPI_CE_BWD || g.epi == EPI_SMAX_BWD || g.epi == EPI_SMAX_PARTS);
    // fp32 outputs keep the lanes' stores: their two 64-byte halves per chunk
    // would wait on each other's bulk read (measured slower on the backward)
    if (!ok || out_f32) continue;
    const bool two = g.out2 != nullptr && g.epi == EPI_BIAS_GELU;
    if (nmaps + (two ? 2 : 1) > kMaxStoreMaps) break;
    if (!encode_store_map(&p.mapO[nmaps], g.out, g.M, g.N, g.ldo, out_f32)) continue;
    g.out_map = nmaps++;
    if (two) {
      if (encode_store_map(&p.mapO[nmaps], g.out2, g.M, g.N, g.ldo, out_f32)) g.out2_map = nmaps++;
      else g.out_map = -1, --nmaps;
    }
  }
  // one count per producer tile (one-SM kernel), one per epilogue warp and CTA (two-SM kernel)
  set_dep_targets(groups, ng, pair ? kEpiWarps : 1, pair ? 2 : 1);
  for (int i = 0; i < ng; ++i) p.grp[i] = groups[i];
  p.pair = pair ? 1 : 0;
  p.has_dep = 0;
  for (int i = 0; i < ng; ++i)
    if (groups[i].dep_kind != DEP_NONE) p.has_dep = 1;
  p.attn = 0;
  for (int i = 0; i < ng; ++i)
    if (groups[i].kr_mode != KR_NONE || groups[i].causal || groups[i].alpha != 1.f ||
        groups[i].epi == EPI_SMAX_BWD || groups[i].epi == EPI_SMAX_PARTS)
      p.attn = 1;
  p.num_groups = ng;
  p.num_segs = pl.ns;
  p.total_tiles = tiles;
  p.interleave_groups = interleave;
  p.interleave_nt = inter_nt;
  p.interleave_tiles = interleave > 0 ? groups[0].tiles_m * inter_nt : 0;
  // Row-block order when the column operands are small enough to stay in L2
  // across the whole sweep (their dependants then start early); otherwise the
  // whole height per column tile, which streams each column operand once.
  p.interleave_gm =
      interleave > 0 ? (inter_b_bytes <= 32.0 * 1024 * 1024 ? 1 : groups[0].tiles_m) : 1;
  p.num_counters = ncounters;
  p.err = dev->err;
  p.wait_limit_ns = g_wait_limit_ns;
  p.fault_skip = g_fault_kind == 1;
  g_fault_kind = 0;
  (void)name;
  const cudaError_t e = launch_tc_gemm(p, dev->num_sms, s);
  return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

tp_status run_plan_impl(Plan& pl, tp_dtype dt, const char* name, cudaStream_t s) {
  if (pl.overflow) return TP_ERR_INVALID;
  // Drop empty outputs; mark outputs with no k-blocks and the segments that
  // kept outputs use.
  GemmGroup groups[kMaxGroups];
  bool used[kMaxSegs] = {};
  int ng = 0, interleave = 0;
  for (int i = 0; i < pl.ng; ++i) {
    GemmGroup g = pl.grp[i];
    if (g.M <= 0 || g.N <= 0) continue;
    int64_t ktot = 0;
    for (int sidx = g.seg_begin; sidx < g.seg_end; ++sidx) {
      ktot += pl.seg[sidx].K;
      used[sidx] = pl.seg[sidx].K > 0;
    }
    g.k_empty = ktot == 0;
    if (i < pl.interleave) ++interleave;
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
        if (o.ones) continue;
        if (!al16(o.ptr) || (o.ld % 8) != 0) return TP_ERR_ALIGN;
        if (o.rows <= 0 || o.cols <= 0) return TP_ERR_INVALID;
      }
    }
  }
  DeviceState* dev = nullptr;
  tp_status st = device_state(&dev);
  if (st != TP_OK) return st;

  if (dt == TP_F32) {
    // The fp32 engine is not persistent: dependent outputs go in a second launch.
    GemmGroup first[kMaxGroups], second[kMaxGroups];
    int n1 = 0, n2 = 0;
    for (int i = 0; i < ng; ++i) {
      if (groups[i].dep_kind == DEP_NONE) first[n1++] = groups[i];
      else second[n2++] = groups[i];
    }
    if (n1 > 0) {
      st = launch_simt_groups(pl, first, n1, dev, name, s);
      if (st != TP_OK) return st;
    }
    if (n2 > 0) st = launch_simt_groups(pl, second, n2, dev, name, s);
    return st;
  }

  if (!get_encode()) return TP_ERR_CUDA;
  // Small plans run as one launch in which dependent tiles wait for the tiles
  // they read (no launch boundary, no tail between the phases).  Large plans
  // have enough tiles per SM that the boundary costs little; there the
  // independent and the dependent outputs run as two launches, each ordered
  // longest contraction first, which keeps the long tiles out of the tail.
  // Causal score outputs count the tiles that hold work (about half, plus the
  // diagonal), as in the kernel choice: the attention core's P with P V then
  // stays one launch (measured 77.5 -> 72.2 us on 8 heads of 512, s = 2048).
  // Outputs whose tiles wait only on row blocks of others (the MLP forward's
  // row-parallel tiles) keep one launch up to 2.5 times as many tiles: their
  // long tiles start as their rows complete and fill the column-parallel
  // tiles' last rounds (the H = 4096 layer's MLP forward, 1280 tiles on 152
  // SMs: 376 -> 338 us as one launch); a tile that waits on a column block
  // (dW, dK) waits for the producers' last row blocks, so those plans split
  // at the base threshold (the attention backward as one launch: 95 -> 118 us).
  int total = 0;
  bool has_dep = false, col_dep = false;
  for (int i = 0; i < ng; ++i) {
    const int rb = (groups[i].M + 127) / 128, t = rb * ((groups[i].N + 255) / 256);
    total += groups[i].kr_mode == KR_TRI ? (t + rb) / 2 : t;
    has_dep = has_dep || groups[i].dep_kind != DEP_NONE;
    col_dep = col_dep || groups[i].dep_kind == DEP_COL;
  }
  const int split_tiles = col_dep ? g_split_tiles_per_sm : g_split_tiles_per_sm * 5 / 2;
  if (has_dep && total > split_tiles * dev->num_sms) {
    GemmGroup first[kMaxGroups], second[kMaxGroups];
    int n1 = 0, n2 = 0;
    for (int i = 0; i < ng; ++i) {
      GemmGroup g = groups[i];
      const bool dependent = g.dep_kind != DEP_NONE;
      g.dep_kind = DEP_NONE;
      g.prod_row = -1;
      g.prod_col = -1;
      if (dependent) second[n2++] = g;
      else first[n1++] = g;
    }
    st = launch_tc_groups(pl, used, first, n1, 0, 0, dev, name, s, true);
    if (st != TP_OK) return st;
    return launch_tc_groups(pl, used, second, n2, 0, 0, dev, name, s, true);
  }
  return launch_tc_groups(pl, used, groups, ng, interleave, pl.ncounters, dev, name, s, false);
}

tp_status run_plan(Plan& pl, tp_dtype dt, const char* name, cudaStream_t s) {
  return timed(name, s, [&] { return run_plan_impl(pl, dt, name, s); });
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

  Plan p;
  const int rows = p.counters((M + 255) / 256 * 2);  // 128-row blocks, pair tiles rounded up
  // Column-parallel linear + bias + GELU: one output block per shard, tiles
  // enumerated row block by row block across the shards.
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(kmajor(X, M, h, h), kmajor(W[i], ns, h, h), h);
    GemmGroup& g = p.add_group(M, ns, si, si + 1, EPI_BIAS_GELU, ot, bb(Z) + i * ns * es, hp);
    g.out2 = bb(Y) + i * ns * es;
    g.bias = a ? a[i] : nullptr;
    g.prod_row = rows;
  }
  p.interleave = N;
  // Row-parallel linear: the shards are the segments of one output (g = sum);
  // a row block starts once all shards of its Y rows are stored.
  const int s0 = p.ns;
  for (int i = 0; i < N; ++i)
    p.add_seg(kmajor(cb(Y) + i * ns * es, M, ns, hp), kmajor(U[i], h, ns, ns), ns);
  GemmGroup& g = p.add_group(M, h, s0, s0 + N, EPI_STORE, ot, Out, h);
  g.bias = b;
  g.dep_kind = DEP_ROW;
  g.dep_base = rows;
  return run_plan(p, dt, "gemm_mlp_fwd", s);
}

extern "C" tp_status tp_mlp_bwd(tp_dtype dt, int64_t M, int64_t h, int64_t hp, int N,
                                const void* dOut, const void* X, const void* const* W,
                                const void* const* U, const void* Z, const void* Y, void* dZ,
                                void* dX, void* const* dW, void* const* da, void* const* dU,
                                void* db, int accumulate, void* stream) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (M < 0 || h <= 0 || hp <= 0 || N < 1 || N > 8 || hp % N != 0) return TP_ERR_INVALID;
  if (M > INT32_MAX || h > INT32_MAX || hp > INT32_MAX) return TP_ERR_INVALID;
  if (!shards_ok(W, N) || !shards_ok(U, N) || !shards_ok(dW, N) || !shards_ok(dU, N) ||
      !opt_shards_ok(da, N))
    return TP_ERR_INVALID;
  if (M > 0 && (!dOut || !X || !Z || !Y || !dZ || !dX)) return TP_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t ns = hp / N;
  const size_t es = esize(dt);
  const int ot = dt == TP_F32 ? OUT_F32 : OUT_BF16;

  Plan p;
  const int rows = p.counters((M + 255) / 256 * 2);  // 128-row blocks, pair tiles rounded up
  int cols[8];
  for (int i = 0; i < N; ++i) cols[i] = p.counters((ns + 255) / 256);
  // dZ_i = (dOut U_i) * GELU'(Z_i): g backward is the identity, every shard
  // sees dOut.  Counted per row block (for dX) and per column block (for dW, da).
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(kmajor(dOut, M, h, h), mnmajor(U[i], h, ns, ns), h);
    GemmGroup& g = p.add_group(M, ns, si, si + 1, EPI_DGELU, ot, bb(dZ) + i * ns * es, hp);
    g.aux = cb(Z) + i * ns * es;
    g.ld_aux = hp;
    g.prod_row = rows;
    g.prod_col = cols[i];
  }
  p.interleave = N;
  // Independent of dZ: dU_i = dOut^T Y_i and db = colsum(dOut).
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(mnmajor(dOut, M, h, h), mnmajor(cb(Y) + i * ns * es, M, ns, hp), M);
    GemmGroup& g = p.add_group(h, ns, si, si + 1, EPI_F32, OUT_F32, dU[i], ns);
    g.accumulate = accumulate;
  }
  if (db) p.add_colsum(dOut, M, h, h, db, accumulate);
  // dX = sum_i dZ_i W_i (f backward = sum over shards, fused), per row block.
  const int s0 = p.ns;
  for (int i = 0; i < N; ++i)
    p.add_seg(kmajor(cb(dZ) + i * ns * es, M, ns, hp), mnmajor(W[i], ns, h, h), ns);
  GemmGroup& gx = p.add_group(M, h, s0, s0 + N, EPI_STORE, ot, dX, h);
  gx.dep_kind = DEP_ROW;
  gx.dep_base = rows;
  // dW_i = dZ_i^T X and da_i = colsum(dZ_i), per column block of dZ_i.
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(mnmajor(cb(dZ) + i * ns * es, M, ns, hp), mnmajor(X, M, h, h), M);
    GemmGroup& g = p.add_group(ns, h, si, si + 1, EPI_F32, OUT_F32, dW[i], h);
    g.accumulate = accumulate;
    g.dep_kind = DEP_COL;
    g.dep_base = cols[i];
  }
  if (da) {
    for (int i = 0; i < N; ++i) {
      GemmGroup& g = p.add_colsum(cb(dZ) + i * ns * es, M, ns, hp, da[i], accumulate);
      g.dep_kind = DEP_COL;
      g.dep_base = cols[i];
    }
  }
  return run_plan(p, dt, "gemm_mlp_bwd", s);
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
  // Output projection: O = sum_i C_i Wo_i^T + bo (the shards are segments).
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

extern "C" tp_status tp_attn_proj_bwd(tp_dtype dt, int64_t M, int64_t h, int n_heads, int N,
                                      const void* dQKV, const void* dO, const void* X,
                                      const void* C, const void* const* Wqkv,
                                      const void* const* Wo, void* dX, void* dC,
                                      void* const* dWqkv, void* const* dbqkv, void* const* dWo,
                                      void* dbo, int accumulate, void* stream) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (M < 0 || h <= 0 || N < 1 || N > 8 || n_heads < 1 || n_heads % N != 0 || h % n_heads != 0)
    return TP_ERR_INVALID;
  if (M > INT32_MAX || 3 * h > INT32_MAX) return TP_ERR_INVALID;
  if (!shards_ok(Wqkv, N) || !shards_ok(Wo, N) || !shards_ok(dWqkv, N) || !shards_ok(dWo, N) ||
      !opt_shards_ok(dbqkv, N))
    return TP_ERR_INVALID;
  if (M > 0 && (!dQKV || !dO || !X || !C || !dX || !dC)) return TP_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t d = h / N;
  const int64_t w = 3 * d;
  const size_t es = esize(dt);
  const int ot = dt == TP_F32 ? OUT_F32 : OUT_BF16;

  // One launch, longest contractions first; every input is given, so no tile waits.
  Plan p;
  // dX = sum_i dQKV_i Wqkv_i (f backward: sum over shards, fused).
  for (int i = 0; i < N; ++i)
    p.add_seg(kmajor(cb(dQKV) + i * w * es, M, w, 3 * h), mnmajor(Wqkv[i], w, h, h), w);
  p.add_group(M, h, 0, N, EPI_STORE, ot, dX, h);
  // dC_i = dO Wo_i (g backward: identity).
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(kmajor(dO, M, h, h), mnmajor(Wo[i], h, d, d), h);
    p.add_group(M, d, si, si + 1, EPI_STORE, ot, bb(dC) + i * d * es, h);
  }
  // Weight gradients: contractions over tokens.
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(mnmajor(cb(dQKV) + i * w * es, M, w, 3 * h), mnmajor(X, M, h, h), M);
    GemmGroup& g = p.add_group(w, h, si, si + 1, EPI_F32, OUT_F32, dWqkv[i], h);
    g.accumulate = accumulate;
  }
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(mnmajor(dO, M, h, h), mnmajor(cb(C) + i * d * es, M, d, h), M);
    GemmGroup& g = p.add_group(h, d, si, si + 1, EPI_F32, OUT_F32, dWo[i], d);
    g.accumulate = accumulate;
  }
  // Bias gradients: column sums as GEMMs against the ones block.
  if (dbqkv)
    for (int i = 0; i < N; ++i) p.add_colsum(cb(dQKV) + i * w * es, M, w, 3 * h, dbqkv[i], accumulate);
  if (dbo) p.add_colsum(dO, M, h, h, dbo, accumulate);
  return run_plan(p, dt, "gemm_attn_bwd", s);
}

// ===========================================================================
// Attention core
// ===========================================================================
namespace {

// Pointers of (sequence bi, global head j) in the shard-major QKV layout:
// shard i = j / (heads per shard) holds [Q_i K_i V_i], each h/N columns, its
// heads in order inside each.
struct HeadPtrs {
  const uint8_t *q, *k, *v;
  size_t qc, kc, vc, cc;  // element columns of Q, K, V in QKV and of the head in C
};
HeadPtrs head_ptrs(const void* QKV, int64_t bi, int64_t s, int64_t h, int n_heads, int N, int j) {
  const int64_t d = h / n_heads, per = n_heads / N, i = j / per, jl = j % per;
  const int64_t base = i * 3 * (h / N);
  HeadPtrs r;
  r.qc = static_cast<size_t>(base + jl * d);
  r.kc = static_cast<size_t>(base + h / N + jl * d);
  r.vc = static_cast<size_t>(base + 2 * (h / N) + jl * d);
  r.cc = static_cast<size_t>(j * d);
  const uint8_t* row0 = cb(QKV) + static_cast<size_t>(bi * s) * static_cast<size_t>(3 * h) * 2;
  r.q = row0 + r.qc * 2;
  r.k = row0 + r.kc * 2;
  r.v = row0 + r.vc * 2;
  return r;
}

struct AttnDims {
  int64_t b, d, P;  // sequences, head width, 64-key parts per score row
  int64_t pairs;    // b * n_heads
};

tp_status attn_args(tp_dtype dt, int64_t T, int64_t s, int64_t h, int n_heads, int N, AttnDims* out) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (T < 0 || s <= 0 || h <= 0 || n_heads < 1 || N < 1 || N > 8 || n_heads % N != 0 ||
      h % n_heads != 0 || T % s != 0)
    return TP_ERR_INVALID;
  if (T > INT32_MAX || s > INT32_MAX || 3 * h > INT32_MAX) return TP_ERR_INVALID;
  if (dt != TP_BF16) return TP_ERR_UNSUPPORTED;  // the fused epilogues live in the tensor-core engine
  const int64_t d = h / n_heads;
  // TMA: every head's column offset and the probabilities' row pitch s are
  // whole 16-byte units
  if (d % 8 != 0 || s % 8 != 0) return TP_ERR_ALIGN;
  out->b = T / s;
  out->d = d;
  out->P = (s + 63) / 64;
  out->pairs = out->b * n_heads;
  return TP_OK;
}

// Attention-dropout keep words: 32 keys per uint32, per (pair, query row).
size_t attn_keep_bytes(const AttnDims& a, int64_t s) {
  return round256(static_cast<size_t>(a.pairs * s * ((s + 31) / 32)) * 4);
}
size_t attn_fwd_ws(const AttnDims& a, int64_t s) {
  return round256(static_cast<size_t>(a.pairs * a.P * s) * 8) + round256(static_cast<size_t>(a.pairs * s) * 4) +
         attn_keep_bytes(a, s);
}
size_t attn_bwd_ws(const AttnDims& a, int64_t s) {
  return round256(static_cast<size_t>(a.pairs * s) * 4) + round256(static_cast<size_t>(a.pairs * s * s) * 2) +
         attn_keep_bytes(a, s);
}

// Attention dropout needs whole 16-key generator blocks per row and fits its keep
// kernel's grid (s and the (sequence, head) pairs below 65536).
bool drop_ok(float p, int64_t s) {
  return p >= 0.f && p < 1.f && (p == 0.f || (s % 16 == 0 && s <= 65535));
}

// (sequence, head) pairs per GEMM launch: within the engine's group and
// counter limits (groups_per_pair outputs and counters_per_pair counters each).
int64_t pairs_per_launch(int groups_per_pair, int64_t counters_per_pair) {
  int64_t n = kMaxGroups / groups_per_pair;
  if (counters_per_pair > 0) n = std::min<int64_t>(n, kMaxCounters / counters_per_pair);
  return n;
}

}  // namespace

extern "C" size_t tp_attn_core_workspace_size(int64_t T, int64_t s, int64_t h, int n_heads) {
  AttnDims a;
  if (attn_args(TP_BF16, T, s, h, n_heads, 1, &a) != TP_OK || T == 0) return 0;
  return std::max(attn_fwd_ws(a, s), attn_bwd_ws(a, s));
}

namespace {
// keep_out (optional): where the forward leaves the attention-dropout keep
// words (else the workspace); keep_in (optional): the backward reads them
// there instead of drawing them again.
tp_status attn_core_fwd_impl(tp_dtype dt, int64_t T, int64_t s, int64_t h, int n_heads, int N, int causal,
                             float p_drop, uint64_t seed, uint64_t stream0, const void* QKV, void* P,
                             void* Pd, void* C, float* lse, void* workspace, size_t ws_bytes,
                             void* stream, uint32_t* keep_out = nullptr) {
  AttnDims a;
  tp_status st = attn_args(dt, T, s, h, n_heads, N, &a);
  if (st != TP_OK) return st;
  if (!drop_ok(p_drop, s) || (p_drop > 0.f && a.pairs > 65535)) return TP_ERR_INVALID;
  if (T == 0) return TP_OK;
  if (!QKV || !P || !C || (p_drop > 0.f && !Pd)) return TP_ERR_INVALID;
  if (workspace == nullptr || ws_bytes < attn_fwd_ws(a, s)) return TP_ERR_WORKSPACE;
  if (!al256(workspace)) return TP_ERR_ALIGN;
  if (!al16(P) || (p_drop > 0.f && !al16(Pd))) return TP_ERR_ALIGN;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  float* parts = static_cast<float*>(workspace);
  float* row_lse = lse ? lse
                       : reinterpret_cast<float*>(bb(workspace) +
                                                  round256(static_cast<size_t>(a.pairs * a.P * s) * 8));
  uint32_t* keep = keep_out ? keep_out
                            : reinterpret_cast<uint32_t*>(bb(workspace) +
                                                          round256(static_cast<size_t>(a.pairs * a.P * s) * 8) +
                                                          round256(static_cast<size_t>(a.pairs * s) * 4));
  const float alpha = static_cast<float>(1.0 / sqrt(static_cast<double>(a.d)));
  const int kr_s = causal ? KR_TRI : KR_NONE;
  // 1. scores alpha q k^T per (sequence, head), causal tiles only: per row and
  //    64-key part the max m and e = exp(alpha q k^T - m), e stored where P goes
  //    and (m, sum e) to the part statistics
  const int64_t per1 = pairs_per_launch(1, 0);
  for (int64_t g0 = 0; g0 < a.pairs; g0 += per1) {
    Plan p;
    for (int64_t g = g0; g < std::min(a.pairs, g0 + per1); ++g) {
      const HeadPtrs hp = head_ptrs(QKV, g / n_heads, s, h, n_heads, N, static_cast<int>(g % n_heads));
      const int si = p.add_seg(kmajor(hp.q, s, a.d, 3 * h), kmajor(hp.k, s, a.d, 3 * h), a.d);
      GemmGroup& gr = p.add_group(s, s, si, si + 1, EPI_SMAX_PARTS, OUT_BF16,
                                  bb(P) + static_cast<size_t>(g * s * s) * 2, s);
      gr.alpha = alpha;
      gr.causal = causal != 0;
      gr.kr_mode = kr_s;
      gr.ce_part = parts;
      gr.ce_part0 = static_cast<int>(g * a.P);
      gr.ce_rows = static_cast<int>(s);
      gr.tri_ok = 1;  // tiles after a row block's last key: zeros written by step 2
    }
    st = run_plan(p, dt, "gemm_attn_scores", strm);
    if (st != TP_OK) return st;
  }
  // 2. log-sum-exp per row (parts merged in a fixed order), then in place
  //    P = e exp(m - lse) (zero where masked); with attention dropout also the
  //    keep words (drawn here) and P keep / (1 - p) to Pd
  const cudaError_t e = timed("attn_norm", strm, [&] {
    return launch_attn_norm(parts, static_cast<int>(a.P), s, a.pairs, causal != 0, row_lse, P,
                            p_drop > 0.f ? Pd : nullptr, keep, p_drop, seed, stream0, n_heads, n_heads / N,
                            strm);
  });
  if (e != cudaSuccess) return TP_ERR_CUDA;
  // 3. C_j = P V_j (with dropout Pd V_j), the contraction stopped at the
  //    tile's last query when causal (the keys after it have P = 0)
  const int64_t per3 = pairs_per_launch(1, 0);
  for (int64_t g0 = 0; g0 < a.pairs; g0 += per3) {
    Plan p;
    for (int64_t g = g0; g < std::min(a.pairs, g0 + per3); ++g) {
      const int64_t bi = g / n_heads;
      const HeadPtrs hp = head_ptrs(QKV, bi, s, h, n_heads, N, static_cast<int>(g % n_heads));
      const void* Pg = bb(p_drop > 0.f ? Pd : P) + static_cast<size_t>(g * s * s) * 2;
      const int si = p.add_seg(kmajor(Pg, s, s, s), mnmajor(hp.v, s, a.d, 3 * h), s);
      GemmGroup& gr = p.add_group(s, a.d, si, si + 1, EPI_STORE, OUT_BF16,
                                  bb(C) + (static_cast<size_t>(bi * s) * h + hp.cc) * 2, h);
      gr.kr_mode = causal ? KR_END : KR_NONE;
    }
    st = run_plan(p, dt, "gemm_attn_pv", strm);
    if (st != TP_OK) return st;
  }
  return TP_OK;
}

tp_status attn_core_bwd_impl(tp_dtype dt, int64_t T, int64_t s, int64_t h, int n_heads, int N, int causal,
                             float p_drop, uint64_t seed, uint64_t stream0, const void* QKV, const void* P,
                             const void* Pd, const void* C, const void* dC, void* dQKV, void* workspace,
                             size_t ws_bytes, void* stream, const uint32_t* keep_in = nullptr) {
  AttnDims a;
  tp_status st = attn_args(dt, T, s, h, n_heads, N, &a);
  if (st != TP_OK) return st;
  if (!drop_ok(p_drop, s) || (p_drop > 0.f && a.pairs > 65535)) return TP_ERR_INVALID;
  if (T == 0) return TP_OK;
  if (!QKV || !P || !C || !dC || !dQKV || (p_drop > 0.f && !Pd)) return TP_ERR_INVALID;
  if (workspace == nullptr || ws_bytes < attn_bwd_ws(a, s)) return TP_ERR_WORKSPACE;
  if (!al256(workspace)) return TP_ERR_ALIGN;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  float* D = static_cast<float*>(workspace);
  uint8_t* dS = bb(workspace) + round256(static_cast<size_t>(a.pairs * s) * 4);
  uint32_t* keep_ws = reinterpret_cast<uint32_t*>(dS + round256(static_cast<size_t>(a.pairs * s * s) * 2));
  const uint32_t* keep = keep_in ? keep_in : keep_ws;
  const int wpr = static_cast<int>((s + 31) / 32);
  const float alpha = static_cast<float>(1.0 / sqrt(static_cast<double>(a.d)));
  // 1. D = rowsum(dC * C) per head and token (= sum over keys of P dP)
  cudaError_t e = timed("attn_rowdot", strm, [&] {
    return launch_attn_rowdot(C, dC, h, s, n_heads, static_cast<int>(a.d), a.pairs, D, strm);
  });
  if (e != cudaSuccess) return TP_ERR_CUDA;
  if (p_drop > 0.f && keep_in == nullptr) {  // the forward's keep bits, drawn again
    e = timed("attn_keep", strm, [&] {
      return launch_attn_keep(a.pairs, s, n_heads, n_heads / N, causal != 0, seed, stream0, p_drop, keep_ws,
                              strm);
    });
    if (e != cudaSuccess) return TP_ERR_CUDA;
  }
  // 2. per pair: dS = P (dC V^T - D) alpha and dV = P^T dC; then dQ = dS K per
  //    row block of dS, dK = dS^T Q per column block of dS
  const int64_t rows_per_pair = (s + 255) / 256 * 2;
  const int64_t cols_per_pair = (s + 255) / 256;
  const int64_t per = pairs_per_launch(4, rows_per_pair + cols_per_pair);
  if (per < 1) return TP_ERR_INVALID;
  for (int64_t g0 = 0; g0 < a.pairs; g0 += per) {
    Plan p;
    const int64_t g1 = std::min(a.pairs, g0 + per);
    int rows[kMaxGroups], cols[kMaxGroups];
    auto dS_of = [&](int64_t g) { return dS + static_cast<size_t>(g * s * s) * 2; };
    auto dC_of = [&](int64_t g, const HeadPtrs& hp) {
      return cb(dC) + (static_cast<size_t>((g / n_heads) * s) * h + hp.cc) * 2;
    };
    auto dqkv_of = [&](int64_t g, size_t col) {
      return bb(dQKV) + (static_cast<size_t>((g / n_heads) * s) * 3 * h + col) * 2;
    };
    for (int64_t g = g0; g < g1; ++g) {
      const HeadPtrs hp = head_ptrs(QKV, g / n_heads, s, h, n_heads, N, static_cast<int>(g % n_heads));
      rows[g - g0] = p.counters(rows_per_pair);
      cols[g - g0] = p.counters(cols_per_pair);
      const int si = p.add_seg(kmajor(dC_of(g, hp), s, a.d, h), kmajor(hp.v, s, a.d, 3 * h), a.d);
      GemmGroup& gr = p.add_group(s, s, si, si + 1, EPI_SMAX_BWD, OUT_BF16, dS_of(g), s);
      gr.aux = cb(P) + static_cast<size_t>(g * s * s) * 2;
      gr.ld_aux = s;
      gr.row_lse = D + g * s;
      gr.alpha = alpha;
      gr.kr_mode = causal ? KR_TRI : KR_NONE;
      gr.tri_ok = 1;  // dQ and dK read only the causal tiles of dS
      gr.prod_row = rows[g - g0];
      gr.prod_col = cols[g - g0];
      if (p_drop > 0.f) {
        gr.drop_mask = keep + g * s * wpr;
        gr.drop_wpr = wpr;
        gr.drop_scale = 1.f / (1.f - p_drop);
      }
    }
    for (int64_t g = g0; g < g1; ++g) {
      const HeadPtrs hp = head_ptrs(QKV, g / n_heads, s, h, n_heads, N, static_cast<int>(g % n_heads));
      const void* Pg = cb(p_drop > 0.f ? Pd : P) + static_cast<size_t>(g * s * s) * 2;
      const int si = p.add_seg(mnmajor(Pg, s, s, s), mnmajor(dC_of(g, hp), s, a.d, h), s);
      GemmGroup& gr = p.add_group(s, a.d, si, si + 1, EPI_STORE, OUT_BF16, dqkv_of(g, hp.vc), 3 * h);
      gr.kr_mode = causal ? KR_BEGIN : KR_NONE;
    }
    for (int64_t g = g0; g < g1; ++g) {
      const HeadPtrs hp = head_ptrs(QKV, g / n_heads, s, h, n_heads, N, static_cast<int>(g % n_heads));
      const int si = p.add_seg(kmajor(dS_of(g), s, s, s), mnmajor(hp.k, s, a.d, 3 * h), s);
      GemmGroup& gr = p.add_group(s, a.d, si, si + 1, EPI_STORE, OUT_BF16, dqkv_of(g, hp.qc), 3 * h);
      gr.kr_mode = causal ? KR_END : KR_NONE;
      gr.dep_kind = DEP_ROW;
      gr.dep_base = rows[g - g0];
    }
    for (int64_t g = g0; g < g1; ++g) {
      const HeadPtrs hp = head_ptrs(QKV, g / n_heads, s, h, n_heads, N, static_cast<int>(g % n_heads));
      const int si = p.add_seg(mnmajor(dS_of(g), s, s, s), mnmajor(hp.q, s, a.d, 3 * h), s);
      GemmGroup& gr = p.add_group(s, a.d, si, si + 1, EPI_STORE, OUT_BF16, dqkv_of(g, hp.kc), 3 * h);
      gr.kr_mode = causal ? KR_BEGIN : KR_NONE;
      gr.dep_kind = DEP_COL;
      gr.dep_base = cols[g - g0];
    }
    st = run_plan(p, dt, "gemm_attn_bwd", strm);
    if (st != TP_OK) return st;
  }
  return TP_OK;
}
}  // namespace

extern "C" tp_status tp_attn_core_fwd(tp_dtype dt, int64_t T, int64_t s, int64_t h, int n_heads, int N,
                                      int causal, const void* QKV, void* P, void* C, float* lse,
                                      void* workspace, size_t ws_bytes, void* stream) {
  return attn_core_fwd_impl(dt, T, s, h, n_heads, N, causal, 0.f, 0, 0, QKV, P, nullptr, C, lse, workspace,
                            ws_bytes, stream);
}

extern "C" tp_status tp_attn_core_bwd(tp_dtype dt, int64_t T, int64_t s, int64_t h, int n_heads, int N,
                                      int causal, const void* QKV, const void* P, const void* C,
                                      const void* dC, void* dQKV, void* workspace, size_t ws_bytes,
                                      void* stream) {
  return attn_core_bwd_impl(dt, T, s, h, n_heads, N, causal, 0.f, 0, 0, QKV, P, nullptr, C, dC, dQKV,
                            workspace, ws_bytes, stream);
}

extern "C" tp_status tp_attn_core_dropout_fwd(tp_dtype dt, int64_t T, int64_t s, int64_t h, int n_heads,
                                              int N, int causal, float p_attn, uint64_t seed,
                                              uint64_t stream0, const void* QKV, void* P, void* Pd, void* C,
                                              float* lse, void* workspace, size_t ws_bytes, void* stream) {
  return attn_core_fwd_impl(dt, T, s, h, n_heads, N, causal, p_attn, seed, stream0, QKV, P, Pd, C, lse,
                            workspace, ws_bytes, stream);
}

extern "C" tp_status tp_attn_core_dropout_bwd(tp_dtype dt, int64_t T, int64_t s, int64_t h, int n_heads,
                                              int N, int causal, float p_attn, uint64_t seed,
                                              uint64_t stream0, const void* QKV, const void* P,
                                              const void* Pd, const void* C, const void* dC, void* dQKV,
                                              void* workspace, size_t ws_bytes, void* stream) {
  return attn_core_bwd_impl(dt, T, s, h, n_heads, N, causal, p_attn, seed, stream0, QKV, P, Pd, C, dC, dQKV,
                            workspace, ws_bytes, stream);
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

// ===========================================================================
// Vocab-parallel cross-entropy
// ===========================================================================
namespace {
int64_t ce_parts(const int64_t* rs, int N) {
  int64_t P = 0;
  for (int r = 0; r < N; ++r) P += (rs[r + 1] - rs[r] + 63) / 64;
  return P;
}

bool ce_args_ok(int64_t T, int64_t h, int64_t V, int N, const void* X, const void* const* E,
                const int64_t* rs, const int64_t* targets) {
  if (T < 0 || h <= 0 || V <= 0 || N > kMaxGroups || !ranges_ok(rs, N, V) || !shards_ok(E, N))
    return false;
  if (T > INT32_MAX || V > INT32_MAX || h > INT32_MAX) return false;
  return T == 0 || (X != nullptr && targets != nullptr);
}
}  // namespace

extern "C" size_t tp_vocab_cross_entropy_workspace_size(int64_t T, int64_t V, int N,
                                                        const int64_t* range_starts) {
  if (T <= 0 || V <= 0 || N < 1 || N > kMaxGroups || !ranges_ok(range_starts, N, V)) return 0;
  return round256(static_cast<size_t>(ce_parts(range_starts, N)) * static_cast<size_t>(T) * 8) +
         round256(static_cast<size_t>(T) * 4);
}

extern "C" tp_status tp_vocab_cross_entropy_fwd(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                                                const void* X, const void* const* E,
                                                const int64_t* range_starts, const int64_t* targets,
                                                float* loss, float* lse, void* workspace,
                                                size_t workspace_bytes, void* stream) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (!ce_args_ok(T, h, V, N, X, E, range_starts, targets)) return TP_ERR_INVALID;
  if (T > 0 && (loss == nullptr || lse == nullptr)) return TP_ERR_INVALID;
  if (T == 0) return TP_OK;
  if (dt != TP_BF16) return TP_ERR_UNSUPPORTED;  // the fused epilogue lives in the tensor-core engine
  const size_t need = tp_vocab_cross_entropy_workspace_size(T, V, N, range_starts);
  if (workspace == nullptr || workspace_bytes < need) return TP_ERR_WORKSPACE;
  if (!al256(workspace)) return TP_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t P = ce_parts(range_starts, N);
  float* part = static_cast<float*>(workspace);
  float* tlogit = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                           round256(static_cast<size_t>(P) * T * 8));
  // Logits per range with the cross-entropy epilogue: no logits are stored.
  Plan p;
  int64_t part0 = 0;
  for (int r = 0; r < N; ++r) {
    const int64_t nr = range_starts[r + 1] - range_starts[r];
    const int si = p.add_seg(kmajor(X, T, h, h), kmajor(E[r], nr, h, h), h);
    GemmGroup& g = p.add_group(T, nr, si, si + 1, EPI_CE_FWD, OUT_F32, nullptr, 0);
    g.col0 = range_starts[r];
    g.row_target = targets;
    g.ce_part = part;
    g.ce_target = tlogit;
    g.ce_part0 = static_cast<int>(part0);
    g.ce_rows = static_cast<int>(T);
    part0 += (nr + 63) / 64;
  }
  tp_status st = run_plan(p, dt, "gemm_ce_fwd", s);
  if (st != TP_OK) return st;
  const cudaError_t e = timed("ce_reduce", s, [&] {
    return launch_ce_reduce(part, static_cast<int>(P), T, targets, V, tlogit, loss, lse, s);
  });
  return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

extern "C" tp_status tp_vocab_cross_entropy_bwd(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                                                const void* X, const void* const* E,
                                                const int64_t* range_starts, const int64_t* targets,
                                                const float* lse, const float* dloss,
                                                void* const* dLogits, const int64_t* ld_dlogits,
                                                void* dX, void* stream) {
  if (!dtype_ok(dt)) return TP_ERR_UNSUPPORTED;
  if (!ce_args_ok(T, h, V, N, X, E, range_starts, targets) || ld_dlogits == nullptr)
    return TP_ERR_INVALID;
  if (T > 0 && (lse == nullptr || dloss == nullptr || !shards_ok(dLogits, N))) return TP_ERR_INVALID;
  for (int r = 0; r < N; ++r)
    if (ld_dlogits[r] < range_starts[r + 1] - range_starts[r]) return TP_ERR_INVALID;
  if (T == 0) return TP_OK;
  if (dt != TP_BF16) return TP_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Plan p;
  const int rows = p.counters((T + 255) / 256 * 2);  // 128-row blocks, pair tiles rounded up
  // dLogits_r = (softmax - onehot) * dloss, the logits recomputed per range.
  for (int r = 0; r < N; ++r) {
    const int64_t nr = range_starts[r + 1] - range_starts[r];
    const int si = p.add_seg(kmajor(X, T, h, h), kmajor(E[r], nr, h, h), h);
    GemmGroup& g = p.add_group(T, nr, si, si + 1, EPI_CE_BWD, OUT_BF16, dLogits[r], ld_dlogits[r]);
    g.col0 = range_starts[r];
    g.row_target = targets;
    g.row_lse = lse;
    g.row_dloss = dloss;
    g.prod_row = dX ? rows : -1;
  }
  p.interleave = N;
  // dX = sum_r dLogits_r E_r: the output layer's input gradient, summed over
  // ranges; a row block starts once its dLogits rows are stored.
  if (dX) {
    const int s0 = p.ns;
    for (int r = 0; r < N; ++r) {
      const int64_t nr = range_starts[r + 1] - range_starts[r];
      p.add_seg(kmajor(dLogits[r], T, nr, ld_dlogits[r]), mnmajor(E[r], nr, h, h), nr);
    }
    GemmGroup& gx = p.add_group(T, h, s0, s0 + N, EPI_STORE, OUT_BF16, dX, h);
    gx.dep_kind = DEP_ROW;
    gx.dep_base = rows;
  }
  return run_plan(p, dt, "gemm_ce_bwd", s);
}

extern "C" size_t tied_embed_grad_workspace_size(int64_t T, int64_t V) {
  if (T < 0 || V <= 0) return 0;
  return sort_workspace_bytes(T, V);
}

tp_status tp::tied_embed_grad_check(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                                    const int64_t* ids, const void* dEmb, const void* X,
                                    const void* const* dLogits, const int64_t* ld_dlogits,
                                    const int64_t* range_starts, void* const* dE) {
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
  return TP_OK;
}

extern "C" tp_status tied_embed_grad(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                                     const int64_t* ids, const void* dEmb, const void* X,
                                     const void* const* dLogits, const int64_t* ld_dlogits,
                                     const int64_t* range_starts, void* const* dE, int accumulate,
                                     void* workspace, size_t ws_bytes, void* stream) {
  const tp_status chk =
      tied_embed_grad_check(dt, T, h, V, N, ids, dEmb, X, dLogits, ld_dlogits, range_starts, dE);
  if (chk != TP_OK) return chk;
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
// Transformer layer
// ===========================================================================
namespace {

// Workspace carve-up of the layer (each piece 256-byte aligned).
struct LayerWs {
  uint8_t* base;
  size_t off;
  template <class T>
  T* take(size_t bytes) {
    T* p = reinterpret_cast<T*>(base + off);
    off += round256(bytes);
    return p;
  }
};

size_t layer_ws_bytes(const tp_layer_config& c) {
  const size_t th = static_cast<size_t>(c.T * c.h) * 2;
  size_t b = 0;
  b += 8 * round256(th);                                          // O, M, dM, dln2, dh1, dO, dC, dln1
  b += round256(static_cast<size_t>(c.T * c.hp) * 2);             // dZ
  b += round256(static_cast<size_t>(c.T * 3 * c.h) * 2);          // dQKV
  b += round256(ln_bwd_scratch_floats(c.T, c.h) * 4);             // LayerNorm partials
  b += tp_attn_core_workspace_size(c.T, c.s, c.h, c.n_heads);     // core
  return b;
}

tp_status layer_check(const tp_layer_config* c, const tp_layer_params* w) {
  if (!c || !w) return TP_ERR_INVALID;
  if (c->T < 0 || c->s <= 0 || c->h <= 0 || c->hp <= 0 || c->N < 1 || c->N > 8 || c->n_heads < 1 ||
      c->n_heads % c->N != 0 || c->h % c->n_heads != 0 || c->hp % c->N != 0 || c->T % c->s != 0)
    return TP_ERR_INVALID;
  if (c->h % 16 != 0 || c->h > 8192) return TP_ERR_INVALID;
  if (!(c->p_hidden >= 0.f && c->p_hidden < 1.f) || !drop_ok(c->p_attn, c->s) || !(c->eps > 0.f))
    return TP_ERR_INVALID;
  // Bulk tensor copies need whole 16-byte units: the probabilities' row pitch
  // s, every head's column offset (d) and every MLP shard's column offset
  // (h'/N).  Checked here so that nothing is launched before the attention
  // core or the MLP would refuse them.
  if (c->s % 8 != 0 || (c->h / c->n_heads) % 8 != 0 || (c->hp / c->N) % 8 != 0) return TP_ERR_ALIGN;
  if (!w->g1 || !w->b1 || !w->g2 || !w->b2 || !shards_ok(w->Wqkv, c->N) || !shards_ok(w->Wo, c->N) ||
      !shards_ok(w->W, c->N) || !shards_ok(w->U, c->N) || !opt_shards_ok(w->bqkv, c->N) ||
      !opt_shards_ok(w->a, c->N))
    return TP_ERR_INVALID;
  return TP_OK;
}

// QKV_i = X Wqkv_i^T + bqkv_i and, separately, O = sum_i C_i Wo_i^T + bo.
tp_status qkv_proj(int64_t M, int64_t h, int N, const void* X, const void* const* Wqkv,
                   const void* const* bqkv, void* QKV, cudaStream_t s) {
  const int64_t d = h / N;
  Plan p;
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(kmajor(X, M, h, h), kmajor(Wqkv[i], 3 * d, h, h), h);
    GemmGroup& g = p.add_group(M, 3 * d, si, si + 1, EPI_STORE, OUT_BF16, bb(QKV) + i * 3 * d * 2, 3 * h);
    g.bias = bqkv ? bqkv[i] : nullptr;
  }
  return run_plan(p, TP_BF16, "gemm_layer_qkv", s);
}
tp_status out_proj(int64_t M, int64_t h, int N, const void* C, const void* const* Wo, const void* bo,
                   void* O, cudaStream_t s) {
  const int64_t d = h / N;
  Plan p;
  for (int i = 0; i < N; ++i) p.add_seg(kmajor(cb(C) + i * d * 2, M, d, h), kmajor(Wo[i], h, d, d), d);
  GemmGroup& go = p.add_group(M, h, 0, N, EPI_STORE, OUT_BF16, O, h);
  go.bias = bo;
  return run_plan(p, TP_BF16, "gemm_layer_oproj", s);
}
// dC_i = dO Wo_i, dWo_i = dO^T C_i, dbo = colsum(dO).
tp_status out_proj_bwd(int64_t M, int64_t h, int N, const void* dO, const void* C, const void* const* Wo,
                       void* dC, void* const* dWo, void* dbo, int accumulate, cudaStream_t s) {
  const int64_t d = h / N;
  Plan p;
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(kmajor(dO, M, h, h), mnmajor(Wo[i], h, d, d), h);
    p.add_group(M, d, si, si + 1, EPI_STORE, OUT_BF16, bb(dC) + i * d * 2, h);
  }
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(mnmajor(dO, M, h, h), mnmajor(cb(C) + i * d * 2, M, d, h), M);
    GemmGroup& g = p.add_group(h, d, si, si + 1, EPI_F32, OUT_F32, dWo[i], d);
    g.accumulate = accumulate;
  }
  if (dbo) p.add_colsum(dO, M, h, h, dbo, accumulate);
  return run_plan(p, TP_BF16, "gemm_layer_oproj_bwd", s);
}
// dX = sum_i dQKV_i Wqkv_i, dWqkv_i = dQKV_i^T X, dbqkv_i = colsum(dQKV_i).
tp_status qkv_proj_bwd(int64_t M, int64_t h, int N, const void* dQKV, const void* X,
                       const void* const* Wqkv, void* dX, void* const* dWqkv, void* const* dbqkv,
                       int accumulate, cudaStream_t s) {
  const int64_t w = 3 * (h / N);
  Plan p;
  for (int i = 0; i < N; ++i) p.add_seg(kmajor(cb(dQKV) + i * w * 2, M, w, 3 * h), mnmajor(Wqkv[i], w, h, h), w);
  p.add_group(M, h, 0, N, EPI_STORE, OUT_BF16, dX, h);
  for (int i = 0; i < N; ++i) {
    const int si = p.add_seg(mnmajor(cb(dQKV) + i * w * 2, M, w, 3 * h), mnmajor(X, M, h, h), M);
    GemmGroup& g = p.add_group(w, h, si, si + 1, EPI_F32, OUT_F32, dWqkv[i], h);
    g.accumulate = accumulate;
  }
  if (dbqkv)
    for (int i = 0; i < N; ++i) p.add_colsum(cb(dQKV) + i * w * 2, M, w, 3 * h, dbqkv[i], accumulate);
  return run_plan(p, TP_BF16, "gemm_layer_qkv_bwd", s);
}

uint64_t layer_stream(uint64_t layer, int kind) { return layer * 256 + static_cast<uint64_t>(kind) * 64; }

}  // namespace

extern "C" tp_status tp_position_embed_dropout(int64_t T, int64_t h, int64_t max_pos, const void* words,
                                               const void* pos_table, const int64_t* positions, float p,
                                               uint64_t seed, uint64_t stream_id, void* out, void* stream) {
  if (T < 0 || h <= 0 || max_pos <= 0 || h % 16 != 0 || !(p >= 0.f && p < 1.f)) return TP_ERR_INVALID;
  if (T == 0) return TP_OK;
  if (!words || !pos_table || !positions || !out) return TP_ERR_INVALID;
  if (!al16(words) || !al16(pos_table) || !al16(out)) return TP_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = timed("pos_embed_dropout", s, [&] {
    return launch_pos_embed_dropout(words, pos_table, positions, T, h, max_pos, seed, stream_id, p, out, s);
  });
  return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

extern "C" size_t tp_transformer_layer_workspace_size(const tp_layer_config* cfg) {
  if (!cfg || cfg->T <= 0 || cfg->s <= 0 || cfg->T % cfg->s != 0 || cfg->n_heads < 1 || cfg->h <= 0 ||
      cfg->hp <= 0)
    return 0;
  return layer_ws_bytes(*cfg);
}

extern "C" tp_status tp_transformer_layer_fwd(const tp_layer_config* cfg, const tp_layer_params* w,
                                              const void* x, void* out, const tp_layer_saved* sv,
                                              void* workspace, size_t ws_bytes, void* stream) {
  tp_status st = layer_check(cfg, w);
  if (st != TP_OK) return st;
  const tp_layer_config& c = *cfg;
  if (c.T == 0) return TP_OK;
  if (!x || !out || !sv || !sv->ln1 || !sv->mean1 || !sv->rstd1 || !sv->QKV || !sv->P || !sv->C ||
      !sv->h1 || !sv->ln2 || !sv->mean2 || !sv->rstd2 || !sv->Z || !sv->Y || (c.p_attn > 0.f && !sv->Pd))
    return TP_ERR_INVALID;
  if (!workspace || ws_bytes < layer_ws_bytes(c)) return TP_ERR_WORKSPACE;
  if (!al256(workspace)) return TP_ERR_ALIGN;
  if (!al16(x) || !al16(out) || !al16(sv->h1)) return TP_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LayerWs ws{bb(workspace), 0};
  const size_t th = static_cast<size_t>(c.T * c.h) * 2;
  void* O = ws.take<uint8_t>(th);
  void* M = ws.take<uint8_t>(th);
  ws.off += 6 * round256(th) + round256(static_cast<size_t>(c.T * c.hp) * 2) +
            round256(static_cast<size_t>(c.T * 3 * c.h) * 2) +
            round256(ln_bwd_scratch_floats(c.T, c.h) * 4);
  void* core_ws = ws.take<uint8_t>(0);
  const size_t core_bytes = tp_attn_core_workspace_size(c.T, c.s, c.h, c.n_heads);

  cudaError_t e = timed("layer_ln", s, [&] {
    return launch_ln_fwd(x, w->g1, w->b1, c.T, c.h, c.eps, sv->ln1, sv->mean1, sv->rstd1, s);
  });
  if (e != cudaSuccess) return TP_ERR_CUDA;
  if ((st = qkv_proj(c.T, c.h, c.N, sv->ln1, w->Wqkv, w->bqkv, sv->QKV, s)) != TP_OK) return st;
  st = attn_core_fwd_impl(TP_BF16, c.T, c.s, c.h, c.n_heads, c.N, c.causal, c.p_attn, c.seed,
                          layer_stream(c.layer, 0), sv->QKV, sv->P, sv->Pd, sv->C, nullptr, core_ws,
                          core_bytes, stream, sv->attn_keep);
  if (st != TP_OK) return st;
  if ((st = out_proj(c.T, c.h, c.N, sv->C, w->Wo, w->bo, O, s)) != TP_OK) return st;
  e = timed("layer_dropout_add", s, [&] {
    return launch_dropout_add(O, x, c.T * c.h, c.seed, layer_stream(c.layer, 1), c.p_hidden, sv->h1, s);
  });
  if (e != cudaSuccess) return TP_ERR_CUDA;
  e = timed("layer_ln", s, [&] {
    return launch_ln_fwd(sv->h1, w->g2, w->b2, c.T, c.h, c.eps, sv->ln2, sv->mean2, sv->rstd2, s);
  });
  if (e != cudaSuccess) return TP_ERR_CUDA;
  st = tp_mlp_fwd(TP_BF16, c.T, c.h, c.hp, c.N, sv->ln2, w->W, w->a, w->U, w->b, sv->Z, sv->Y, M, stream);
  if (st != TP_OK) return st;
  e = timed("layer_dropout_add", s, [&] {
    return launch_dropout_add(M, sv->h1, c.T * c.h, c.seed, layer_stream(c.layer, 2), c.p_hidden, out, s);
  });
  return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

extern "C" tp_status tp_transformer_layer_bwd(const tp_layer_config* cfg, const tp_layer_params* w,
                                              const void* x, const tp_layer_saved* sv, const void* dout,
                                              void* dx, const tp_layer_grads* g, int accumulate,
                                              void* workspace, size_t ws_bytes, void* stream) {
  tp_status st = layer_check(cfg, w);
  if (st != TP_OK) return st;
  const tp_layer_config& c = *cfg;
  if (c.T == 0) return TP_OK;
  if (!x || !dout || !dx || !sv || !g || !g->dg1 || !g->db1 || !g->dg2 || !g->db2 ||
      !shards_ok(g->dWqkv, c.N) || !shards_ok(g->dWo, c.N) || !shards_ok(g->dW, c.N) ||
      !shards_ok(g->dU, c.N) || !opt_shards_ok(g->dbqkv, c.N) || !opt_shards_ok(g->da, c.N))
    return TP_ERR_INVALID;
  if (!sv->ln1 || !sv->QKV || !sv->P || !sv->C || !sv->h1 || !sv->ln2 || !sv->Z || !sv->Y ||
      (c.p_attn > 0.f && !sv->Pd))
    return TP_ERR_INVALID;
  if (!workspace || ws_bytes < layer_ws_bytes(c)) return TP_ERR_WORKSPACE;
  if (!al256(workspace)) return TP_ERR_ALIGN;
  if (!al16(dout) || !al16(dx)) return TP_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LayerWs ws{bb(workspace), 0};
  const size_t th = static_cast<size_t>(c.T * c.h) * 2;
  ws.take<uint8_t>(th);  // O (forward)
  ws.take<uint8_t>(th);  // M (forward)
  void* dM = ws.take<uint8_t>(th);
  void* dln2 = ws.take<uint8_t>(th);
  void* dh1 = ws.take<uint8_t>(th);
  void* dO = ws.take<uint8_t>(th);
  void* dC = ws.take<uint8_t>(th);
  void* dln1 = ws.take<uint8_t>(th);
  void* dZ = ws.take<uint8_t>(static_cast<size_t>(c.T * c.hp) * 2);
  void* dQKV = ws.take<uint8_t>(static_cast<size_t>(c.T * 3 * c.h) * 2);
  float* partial = ws.take<float>(ln_bwd_scratch_floats(c.T, c.h) * 4);
  void* core_ws = ws.take<uint8_t>(0);
  const size_t core_bytes = tp_attn_core_workspace_size(c.T, c.s, c.h, c.n_heads);

  // MLP output dropout, then the MLP
  cudaError_t e = timed("layer_dropout_add", s, [&] {
    return launch_dropout_add(dout, nullptr, c.T * c.h, c.seed, layer_stream(c.layer, 2), c.p_hidden, dM, s);
  });
  if (e != cudaSuccess) return TP_ERR_CUDA;
  st = tp_mlp_bwd(TP_BF16, c.T, c.h, c.hp, c.N, dM, sv->ln2, w->W, w->U, sv->Z, sv->Y, dZ, dln2, g->dW,
                  g->da, g->dU, g->db, accumulate, stream);
  if (st != TP_OK) return st;
  // LayerNorm 2, plus the residual path: dh1 = dout + LN2'(dln2)
  e = timed("layer_ln_bwd", s, [&] {
    return launch_ln_bwd(dln2, sv->h1, w->g2, sv->mean2, sv->rstd2, dout, c.T, c.h, dh1, g->dg2, g->db2,
                         accumulate, partial, s);
  });
  if (e != cudaSuccess) return TP_ERR_CUDA;
  // attention output dropout, output projection, attention core, QKV projection
  e = timed("layer_dropout_add", s, [&] {
    return launch_dropout_add(dh1, nullptr, c.T * c.h, c.seed, layer_stream(c.layer, 1), c.p_hidden, dO, s);
  });
  if (e != cudaSuccess) return TP_ERR_CUDA;
  if ((st = out_proj_bwd(c.T, c.h, c.N, dO, sv->C, w->Wo, dC, g->dWo, g->dbo, accumulate, s)) != TP_OK)
    return st;
  st = attn_core_bwd_impl(TP_BF16, c.T, c.s, c.h, c.n_heads, c.N, c.causal, c.p_attn, c.seed,
                          layer_stream(c.layer, 0), sv->QKV, sv->P, sv->Pd, sv->C, dC, dQKV, core_ws,
                          core_bytes, stream, sv->attn_keep);
  if (st != TP_OK) return st;
  if ((st = qkv_proj_bwd(c.T, c.h, c.N, dQKV, sv->ln1, w->Wqkv, dln1, g->dWqkv, g->dbqkv, accumulate, s)) !=
      TP_OK)
    return st;
  // LayerNorm 1, plus the residual path: dx = dh1 + LN1'(dln1)
  e = timed("layer_ln_bwd", s, [&] {
    return launch_ln_bwd(dln1, x, w->g1, sv->mean1, sv->rstd1, dh1, c.T, c.h, dx, g->dg1, g->db1, accumulate,
                         partial, s);
  });
  return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

// ===========================================================================
// Mixed-precision Adam step
// ===========================================================================
extern "C" size_t tp_adam_step_workspace_size(void) { return opt_workspace_bytes(); }

extern "C" tp_status tp_adam_step(const tp_param_group* groups, int ngroups, const tp_adam_config* cfg,
                                  tp_optimizer_state* state, void* workspace, size_t ws_bytes,
                                  void* stream) {
  if (cfg == nullptr || state == nullptr || ngroups < 0 || ngroups > kMaxOptGroups) return TP_ERR_INVALID;
  if (ngroups > 0 && groups == nullptr) return TP_ERR_INVALID;
  if (!(cfg->beta1 >= 0.0 && cfg->beta1 < 1.0 && cfg->beta2 >= 0.0 && cfg->beta2 < 1.0))
    return TP_ERR_INVALID;
  if (cfg->use_scaler && cfg->growth_interval < 1) return TP_ERR_INVALID;
  auto al = [](const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; };
  OptParams P;
  memset(&P, 0, sizeof(P));
  const int64_t chunk = opt_chunk_elems();
  int64_t c = 0;
  for (int i = 0; i < ngroups; ++i) {
    const tp_param_group& g = groups[i];
    if (g.n < 0) return TP_ERR_INVALID;
    if (g.n > 0) {
      if (!g.param || !g.grad || !g.exp_avg || !g.exp_avg_sq) return TP_ERR_INVALID;
      if (!al(g.param, 16) || !al(g.grad, 16) || !al(g.exp_avg, 16) || !al(g.exp_avg_sq, 16) ||
          !al(g.model_param, 8))
        return TP_ERR_ALIGN;
    }
    OptGroup& o = P.group[i];
    o.param = g.param;
    o.grad = g.grad;
    o.exp_avg = g.exp_avg;
    o.exp_avg_sq = g.exp_avg_sq;
    o.model_param = g.model_param;
    o.n = g.n;
    o.chunk_begin = c;
    o.weight_decay = static_cast<float>(g.weight_decay);
    c += (g.n + chunk - 1) / chunk;
  }
  if (!al(state, 4)) return TP_ERR_ALIGN;
  if (workspace == nullptr || ws_bytes < opt_workspace_bytes()) return TP_ERR_WORKSPACE;
  if (!al(workspace, 16)) return TP_ERR_ALIGN;
  P.state = state;
  P.nchunks = c;
  P.ngroups = ngroups;
  P.use_scaler = cfg->use_scaler != 0;
  P.growth_interval = cfg->growth_interval;
  P.hysteresis = cfg->hysteresis;
  P.beta1 = static_cast<float>(cfg->beta1);
  P.one_minus_beta1 = static_cast<float>(1.0 - cfg->beta1);
  P.beta2 = static_cast<float>(cfg->beta2);
  P.one_minus_beta2 = static_cast<float>(1.0 - cfg->beta2);
  P.eps = static_cast<float>(cfg->eps);
  P.min_scale = cfg->min_scale;
  P.growth_factor = cfg->growth_factor;
  P.backoff_factor = cfg->backoff_factor;
  P.lr = cfg->lr;
  P.beta1_d = cfg->beta1;
  P.beta2_d = cfg->beta2;
  P.max_norm = cfg->max_norm;
  DeviceState* dev = nullptr;
  if (device_state(&dev) != TP_OK) return TP_ERR_CUDA;
  const int sms = dev->num_sms;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = timed("adam_norm", s, [&] { return launch_adam_norm(P, sms, workspace, s); });
  if (e != cudaSuccess) return TP_ERR_CUDA;
  e = timed("adam_update", s, [&] { return launch_adam_update(P, sms, workspace, s); });
  return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
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
  std::lock_guard<std::mutex> lk(g_prof_mu);
  prof_flush_locked();
  g_prof_agg.clear();
}

extern "C" int tp_profile_read(const char** names, int64_t* calls, int64_t* kernel_launches,
                               double* total_ms, int cap) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  prof_flush_locked();
  const int n = static_cast<int>(g_prof_agg.size());
  for (int i = 0; i < n && i < cap; ++i) {
    if (names) names[i] = g_prof_agg[i].name;
    if (calls) calls[i] = g_prof_agg[i].calls;
    if (kernel_launches) kernel_launches[i] = g_prof_agg[i].kernels;
    if (total_ms) total_ms[i] = g_prof_agg[i].ms;
  }
  return n;
}

extern "C" tp_status tp_gelu_eval(const float* z, float* y, float* dy, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (z == nullptr || (y == nullptr && dy == nullptr)))) return TP_ERR_INVALID;
  const cudaError_t e = launch_gelu_eval(z, y, dy, n, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

extern "C" void tp_debug_inject_fault(int kind) { g_fault_kind = kind; }

extern "C" void tp_debug_set_gemm_kernel(int mode) { g_gemm_mode = (mode >= 0 && mode <= 2) ? mode : 2; }

extern "C" void tp_debug_set_split_threshold(int tiles_per_sm) {
  g_split_tiles_per_sm = tiles_per_sm > 0 ? tiles_per_sm : 8;
}

extern "C" void tp_debug_set_pdl(int on) { g_pdl = on != 0; }

extern "C" void tp_debug_set_wait_limit_ms(int ms) {
  g_wait_limit_ns = static_cast<unsigned long long>(ms > 0 ? ms : 1000) * 1000000ull;
}
