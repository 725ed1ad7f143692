// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "tp.h"

namespace tp {

constexpr int kMaxGroups = 40;    // output matrices in one GEMM launch
constexpr int kMaxSegs = 48;      // (A, B) operand pairs summed into the outputs
constexpr int kEpiWarps = 16;     // epilogue warps of the tensor-core engine
constexpr int kMaxCounters = 512; // tile-completion counters of one launch
constexpr int kMaxRanges = 64;    // vocabulary ranges

// Error bits of the device error word.
constexpr unsigned kErrTimeout = 1u;

// Epilogue kinds of the GEMM engines.
enum Epi : int {
  EPI_STORE = 0,      // out = acc (+ bias[n]); bf16 or f32
  EPI_BIAS_GELU = 1,  // z = acc + bias[n]; out = z, out2 = GELU(z)
  EPI_DGELU = 2,      // out = acc * GELU'(aux[m, n])
  EPI_F32 = 3,        // out (f32) = acc (+ out if accumulate)
  EPI_SEGSUM = 4,     // out (f32) = acc + sum_{j in seg(row)} seg_src[perm[j], n] (+ out)
  EPI_CE_FWD = 5,     // cross-entropy partials: per row and 64-column part, (max, sum exp(acc - max))
                      // to ce_part; the logit at the row's target column to ce_target; no output
  EPI_CE_BWD = 6,     // out (bf16) = (exp(acc - row_lse[m]) - [col0 + n == row_target[m]]) * row_dloss[m]
  EPI_SMAX_BWD = 8,   // out (bf16) = aux[m, n] * (acc - row_lse[m]) * alpha  (softmax backward)
  EPI_SMAX_PARTS = 9  // attention scores: per row and 64-column part, m = max of alpha acc over the
                      // columns causal keeps and (m, sum e) to ce_part; out (bf16) = e =
                      // exp(alpha acc - m), 0 where causal masks (n > m)
};

// Per-tile k-block ranges of causal attention (rows and columns of the output
// are query / key positions of one sequence, or the contraction runs over them):
//   KR_TRI    a tile whose every column lies after its every row has no
//             k-blocks (its epilogue still runs, on zeros);
//   KR_END    the contraction runs over keys <= the tile's last row;
//   KR_BEGIN  the contraction runs over queries >= the tile's first row.
enum KRange : int { KR_NONE = 0, KR_TRI = 1, KR_END = 2, KR_BEGIN = 3 };

enum OutType : int { OUT_BF16 = 0, OUT_F32 = 1 };

// Tile dependencies inside one launch.  A producing group counts finished
// tiles per row block (prod_row + m-tile) and/or per column block (prod_col +
// n-tile); a consuming group's tile waits until its counter reaches
// dep_target: DEP_ROW uses counter dep_base + m-tile (same row tiling as the
// producer), DEP_COL uses dep_base + m0 / 256 (its rows are the producer's
// columns, as for a contraction over tokens of the producer's output).
enum Dep : int { DEP_NONE = 0, DEP_ROW = 1, DEP_COL = 2 };

// One output matrix D (M x N) = sum over its segments of A_s B_s^T.
struct GemmGroup {
  int M, N;
  int seg_begin, seg_end;
  int epi, out_type, accumulate, vec_ok;
  int tiles_m, tiles_n, tile_begin, k_empty;  // k_empty: no k-blocks, D = 0
  int dep_kind, dep_base, dep_target;
  int prod_row, prod_col;                     // counter bases, -1 = none
  int bn;                                     // tile width: 256, or 128 (one-SM kernel)
  void* out;            // D, row pitch ldo (elements)
  void* out2;           // second output (GELU: Y), same pitch as out
  const void* aux;      // DGELU: Z, row pitch ld_aux
  const void* bias;     // column bias (length N) or null; same dtype as inputs
  int64_t ldo, ld_aux;
  // EPI_SEGSUM: row r of D is vocabulary id seg_row0 + r; its tokens are
  // perm[offsets[id] .. offsets[id+1]); seg_src rows have pitch ld_seg.
  const int* seg_offsets;
  const int* seg_perm;
  const void* seg_src;
  int64_t ld_seg;
  int64_t seg_row0;
  // EPI_CE_FWD / EPI_CE_BWD: global column of the group's column 0 (its
  // vocabulary range start), per-row target ids; the forward writes part
  // (ce_part0 + n / 64) of row m at ce_part[2 * (part * ce_rows + m)] (max,
  // sum); the backward reads row_lse and row_dloss.  EPI_SMAX_PARTS writes
  // its parts the same way.
  int64_t col0;
  const int64_t* row_target;
  const float* row_lse;
  const float* row_dloss;
  float* ce_part;
  float* ce_target;
  int ce_part0, ce_rows;
  // Attention: the accumulator is scaled by alpha in the CE_FWD, SMAX_PARTS
  // and SMAX_BWD epilogues (CE_FWD: 1 outside attention); causal masks
  // columns n > m in CE_FWD and SMAX_PARTS; kr_mode selects the tile's
  // k-block range (KRange).
  float alpha;
  int causal, kr_mode;
  int tri_ok;  // KR_TRI tiles with no k-blocks need not run (their outputs are never read)
  int tri;     // set by the launcher: only the causal tiles are enumerated
  // Attention dropout: keep bits of row m, keys 32 w .. 32 w + 31, at
  // drop_mask[m * drop_wpr + w]; kept values are scaled by drop_scale.
  // SMAX_BWD scales its accumulator (dP) by the mask.
  const uint32_t* drop_mask;
  int drop_wpr;
  float drop_scale;
  // Bulk tensor-store maps of out / out2 and the bulk-load map of aux in
  // TcGemmParams::mapO, or -1 (set by the launcher).
  int out_map, out2_map, aux_map;
  // Tile order (set by the launcher): column tiles fastest instead of row
  // blocks, so consecutive tiles share the A operand's row block.
  int n_fastest;
  // Stripe (set by the launcher; attention instance): stripe_n > 1 identical
  // groups starting at group stripe_first whose tiles are enumerated cycling
  // through the groups.
  int stripe_first, stripe_n;
};

// One operand pair of the tensor-core engine.  Operands are bf16.
// A "K-major" operand is stored (rows = M or N, cols = K); "MN-major" is
// stored (rows = K, cols = M or N).
struct TcSeg {
  int K;
  int a_mn, b_mn;
  int n_mma;    // MMA N: 256, or 16 for a column sum against the ones block
  int b_fixed;  // B is the ones block: every k-block loads the same box
  int a_3d, b_3d;  // MN-major operand mapped in 3D: one box covers all its 64-wide blocks
  int pad;
};

constexpr int kMaxStoreMaps = 48;  // output maps of one launch (more outputs store without the TMA)

struct TcGemmParams {
  CUtensorMap mapA[kMaxSegs];
  CUtensorMap mapB[kMaxSegs];
  CUtensorMap mapO[kMaxStoreMaps];
  TcSeg seg[kMaxSegs];
  GemmGroup grp[kMaxGroups];
  int num_groups, num_segs, total_tiles;
  int fault_skip;        // fault injection: producer skips its first stage
  int sched_slot;        // dynamic tile counter slot (set by the launcher)
  int interleave_groups; // leading groups sharing one row tiling, enumerated in
  int interleave_tiles;  // super-rows of interleave_gm row blocks: (super-row,
  int interleave_nt;     // column tile across the groups, row block)
  int interleave_gm;
  int num_counters;
  int pair;              // 1: two-SM kernel (256-row pair tiles), 0: one-SM kernel
  int attn;              // 1: the kernels' attention instance (causal ranges, softmax epilogues)
  int has_dep;           // 1: some tile waits on others (tile claims are not made ahead)
  unsigned* err;         // device error word
  unsigned long long wait_limit_ns;
};

// One operand pair of the fp32 SIMT engine: element (m, k) of A at
// A[m*sam + k*sak], element (n, k) of B at B[n*sbn + k*sbk].
struct SimtSeg {
  const float* A;
  const float* B;
  int64_t sam, sak, sbn, sbk;
  int K, pad;
};

struct SimtGemmParams {
  SimtSeg seg[kMaxSegs];
  GemmGroup grp[kMaxGroups];
  int num_groups, num_segs, total_tiles, pad;
};

// Vocabulary range table.
struct RangeTable {
  int64_t start[kMaxRanges + 1];
  const void* ptr[kMaxRanges];
  int n;
};

// Attention core row kernels: the probabilities from the scores launch's
// stored e = exp(alpha s - m_part) and per-part (m_part, sum e) (their
// log-sum-exp merged in a fixed order, then P = e exp(m_part - lse) in place;
// when Pd is given also the attention-dropout keep words, drawn as
// launch_attn_keep draws them, and Pd = P keep / (1 - p)), and the
// per-(pair, token) dot product of dC and C over a head's columns.  P and Pd
// are (pairs, s, s) bf16 with 16-byte aligned rows (s % 8 == 0; s % 16 == 0
// with dropout).
cudaError_t launch_attn_norm(const void* part, int P, int64_t s, int64_t pairs, int causal, float* lse,
                             void* Pm, void* Pd, uint32_t* keep, float p_drop, uint64_t seed,
                             uint64_t stream0, int n_heads, int heads_per_shard, cudaStream_t st);
cudaError_t launch_attn_rowdot(const void* C, const void* dC, int64_t h, int64_t s, int n_heads, int d,
                               int64_t pairs, float* D, cudaStream_t st);

// Transformer-layer row kernels (LayerNorm, dropout + residual, attention
// dropout bits).  Dropout keeps element e iff its 16-bit Philox4x32-10 field is >=
// dropout_threshold(p).
uint32_t dropout_threshold(float p);
cudaError_t launch_ln_fwd(const void* x, const float* g, const float* b, int64_t T, int64_t h, float eps,
                          void* y, float* mean, float* rstd, cudaStream_t st);
int ln_bwd_blocks(int64_t T);
size_t ln_bwd_scratch_floats(int64_t T, int64_t h);  // the backward's partial sums
cudaError_t launch_ln_bwd(const void* dy, const void* x, const float* g, const float* mean,
                          const float* rstd, const void* dres, int64_t T, int64_t h, void* dx,
                          float* dg, float* db, int accumulate, float* partial, cudaStream_t st);
cudaError_t launch_dropout_add(const void* x, const void* res, int64_t n, uint64_t seed, uint64_t stream,
                               float p, void* out, cudaStream_t st);
cudaError_t launch_pos_embed_dropout(const void* words, const void* pos_table, const int64_t* positions,
                                     int64_t T, int64_t h, int64_t max_pos, uint64_t seed, uint64_t stream,
                                     float p, void* out, cudaStream_t st);
cudaError_t launch_attn_keep(int64_t pairs, int64_t s, int n_heads, int heads_per_shard, int causal,
                             uint64_t seed, uint64_t stream0, float p, uint32_t* words, cudaStream_t st);

// Mixed-precision Adam step.  Parameter groups are cut into chunks of
// opt_chunk_elems() elements; chunk c belongs to the last group whose
// chunk_begin <= c.
constexpr int kMaxOptGroups = 64;
constexpr int kMaxOptGrid = 4096;

struct OptGroup {
  float* param;
  const float* grad;
  float* exp_avg;
  float* exp_avg_sq;
  void* model_param;  // bf16 or null
  int64_t n, chunk_begin;
  float weight_decay;
  int pad;
};

struct OptParams {
  OptGroup group[kMaxOptGroups];
  tp_optimizer_state* state;
  int64_t nchunks;
  int ngroups;
  int use_scaler, growth_interval, hysteresis;
  float beta1, one_minus_beta1, beta2, one_minus_beta2, eps;
  float min_scale, growth_factor, backoff_factor;
  double lr, beta1_d, beta2_d, max_norm;
};

int64_t opt_chunk_elems();
size_t opt_workspace_bytes();
// Norm partials, then the one-block finalize (scaler, clip, bias corrections).
cudaError_t launch_adam_norm(const OptParams& p, int num_sms, void* ws, cudaStream_t s);
// The per-element update (skips itself when the finalize found an overflow).
cudaError_t launch_adam_update(const OptParams& p, int num_sms, void* ws, cudaStream_t s);

// Every kernel launch the library makes is counted (reported by the profiler).
void count_launches(int n);

// Programmatic dependent launch.  A kernel launched through launch_k may begin
// while the previous kernel on its stream is still running, once every block
// of that kernel has called pdl_trigger() or exited.  Before it touches global
// memory every thread of it calls pdl_wait(), which returns once the previous
// kernel has completed and its writes are visible (that kernel did the same,
// so every earlier kernel has completed too).  Row kernels trigger at entry
// (the gather only by exiting); the persistent GEMMs when a CTA finds no tile
// left: the next kernel's launch and block set-up then overlap their tail.  pdl_on() is the host switch
// (tp_debug_set_pdl); off, launch_k launches plainly and pdl_wait returns at
// once.
bool pdl_on();
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_on() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launchers (each returns the launch error).
cudaError_t launch_tc_gemm(const TcGemmParams& p, int num_sms, cudaStream_t s);
cudaError_t launch_simt_gemm(const SimtGemmParams& p, cudaStream_t s);
cudaError_t launch_gelu_eval(const float* z, float* y, float* dy, int64_t n, cudaStream_t s);
cudaError_t launch_embed_gather(const int64_t* ids, int64_t T, int64_t row_bytes,
                                const RangeTable& rt, void* out, cudaStream_t s);
// Grouping of tokens by id.  ws holds offsets[V+1], perm[T], counts[V].
size_t sort_workspace_bytes(int64_t T, int64_t V);
// Every host-side argument check of tied_embed_grad except the workspace's,
// in its order; TP_OK when the arguments are valid.
tp_status tied_embed_grad_check(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                                const int64_t* ids, const void* dEmb, const void* X,
                                const void* const* dLogits, const int64_t* ld_dlogits,
                                const int64_t* range_starts, void* const* dE);
cudaError_t launch_embed_sort(const int64_t* ids, int64_t T, int64_t V, void* ws, cudaStream_t s);
cudaError_t launch_ce_reduce(const void* part, int P, int64_t T, const int64_t* targets, int64_t V,
                             const float* target_logit, float* loss, float* lse, cudaStream_t s);
int* sort_offsets(void* ws);
int* sort_perm(void* ws, int64_t V);
// Input-side embedding gradient alone: dE_r rows = segment sums (+ old).
cudaError_t launch_segment_sum(const void* ws, int64_t V, int64_t T, const void* dEmb, int in_f32,
                               int64_t h, const RangeTable& dE, int accumulate, cudaStream_t s);

}  // namespace tp
