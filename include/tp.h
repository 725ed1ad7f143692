/*
 * tp.h -- C ABI of the GB300 (sm_103a) tensor-parallel block library (libtp.so).
 *
 * One GPU computes the tensor-parallel transformer block with its N shards laid
 * out logically in device memory: the column -> GELU -> row MLP, the head-split
 * attention projections, the vocab-parallel word embedding and the gradient of
 * the tied input/output embedding.  The all-reduces of the multi-GPU method
 * become on-chip sums over shards in a fixed shard order.
 *
 * Pages cited:
 *   [Walkthrough] "Megatron" distributed-training walkthrough
 *                 (formulaic.cloudchewie.com, docs/.../5-megatron)
 *   [TP notes]    "Megatron tensor / model parallelism" notes
 *                 (amentiraz.github.io, posts/Megtron张量/模型并行)
 *   [Core DDP]    megatron.core.distributed overview (zwxr.cn news 246059)
 *   [Study notes] Megatron / ZeRO study notes (baty7811.com blog)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Matrices are row-major with a row pitch equal to their column count
 *    unless a pitch argument says otherwise.  M = b*s tokens, h hidden size,
 *    hp = h' the FFN width, N the number of shards (1 <= N <= 8; vocabulary
 *    ranges 1 <= N <= 64).
 *  - "Shard arrays" (const void* const* X_shards) are HOST arrays of N DEVICE
 *    pointers; shard i is its own contiguous buffer.  Every other pointer is a
 *    device pointer unless marked (host).
 *  - dtype TP_BF16: bf16 inputs and activations, fp32 accumulation, fp32 weight
 *    and embedding gradients.  dtype TP_F32: everything fp32 (fp32 FMA, no
 *    tensor-core rounding).  Weight-gradient outputs are fp32 in both cases
 *    (the fp32 main_grad of [Core DDP] §3.2, grad_reduce_in_fp32).
 *  - bf16 operands of the tensor-core path must start on 16-byte boundaries and
 *    have row pitches that are multiples of 8 elements (TMA); violations return
 *    TP_ERR_ALIGN before anything is launched.  M (and T) may be any value >= 0.
 *  - Ownership: the caller allocates and owns every buffer, including the
 *    workspace.  The library allocates nothing: its state is static device
 *    memory (an error word, tile-scheduler and tile-completion counters, the
 *    optimizer's completion counters, a 16 x 64 block of ones) and it never
 *    frees caller memory.  Tensor-core GEMM launches and optimizer norm passes
 *    each rotate over 64 counter slots, so at most 64 launches of each may be
 *    in flight at the same time across all streams of a device.  A call captured into a
 *    CUDA graph keeps the slot it was given at capture: replay such a graph
 *    on one stream at a time (replays in sequence reuse the slot safely, since
 *    every launch resets its counters as it ends).
 *  - Execution: work is enqueued asynchronously on `stream` (a cudaStream_t
 *    passed as void*; NULL = legacy default stream).  Argument errors return
 *    synchronously before any launch.  Device-side errors (a bounded wait that
 *    expired) are reported by tp_get_status().
 *  - First call on a device: the first call of any entry point with a device
 *    current does one-time set-up (looks up the library's static device
 *    symbols, writes its block of ones, sets kernel attributes), which may
 *    load the module and synchronise the device.  It runs once per device,
 *    also when several host threads make their first calls together.  Make
 *    one call per device during set-up, before any stream capture and before
 *    latency-sensitive stream work.
 *  - accumulate: 0 = overwrite the gradient outputs, 1 = add into them.
 */
#ifndef TP_H_
#define TP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TP_API __attribute__((visibility("default")))
#else
#define TP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TP_OK = 0,
  TP_ERR_INVALID = 1,     /* bad size, null pointer, N out of range, bad vocab ranges */
  TP_ERR_UNSUPPORTED = 2, /* dtype/op combination not provided */
  TP_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  TP_ERR_TIMEOUT = 4,     /* a bounded device wait expired; the kernel exited early */
  TP_ERR_WORKSPACE = 5,   /* workspace null or smaller than the *_workspace_size query */
  TP_ERR_ALIGN = 6        /* pointer or pitch violates the 16-byte / 8-element TMA rule */
} tp_status;

typedef enum { TP_F32 = 0, TP_BF16 = 1 } tp_dtype;

/* ------------------------------------------------------------------------ */
/* MLP block: ColumnParallelLinear -> GELU -> RowParallelLinear              */
/* ------------------------------------------------------------------------ */

/*
 * tp_mlp_fwd -- forward of the tensor-parallel MLP.
 * [TP notes] §MLP层 (A split by columns, B by rows); [Walkthrough]
 * §ColumnParallelLinear (f = identity, F.linear(X, W_i, a_i), no gather) and
 * §RowParallelLinear (F.linear(Y_i, U_i), g = sum over shards, then + b).
 *   Z[:, i] = X W_i^T + a_i ;  Y = GELU(Z) (erf form) ;  Out = sum_i Y_i U_i^T + b
 * One launch: a row block of Out starts once all shards of its Y rows are stored.
 * Arguments:
 *   X   (M, h)                 input
 *   W   shard array, W_i (hp/N, h)   column-parallel weight (torch layout)
 *   a   shard array or NULL, a_i (hp/N)  column bias
 *   U   shard array, U_i (h, hp/N)   row-parallel weight
 *   b   (h) or NULL            row bias, added once after the shard sum
 *   Z, Y (M, hp) out           pre-activation and activation, shard i in
 *                              columns [i hp/N, (i+1) hp/N); saved for backward
 *   Out (M, h) out
 * hp % N == 0 (TP_ERR_INVALID otherwise).
 */
TP_API tp_status tp_mlp_fwd(tp_dtype dt, int64_t M, int64_t h, int64_t hp, int N,
                     const void* X, const void* const* W, const void* const* a,
                     const void* const* U, const void* b,
                     void* Z, void* Y, void* Out, void* stream);

/*
 * tp_mlp_bwd -- backward of the tensor-parallel MLP.
 * [Walkthrough] §RowParallelLinear (g backward = identity: every shard sees
 * dOut) and §ColumnParallelLinear (f backward = all-reduce: dX sums shards).
 *   dZ_i = (dOut U_i) * GELU'(Z_i)      dU_i = dOut^T Y_i    dW_i = dZ_i^T X
 *   da_i = colsum(dZ_i)   db = colsum(dOut)   dX = sum_i dZ_i W_i
 * All of it is one launch: a tile of dX, dW_i or da_i starts as soon as the
 * dZ tiles it reads are stored.  The bias gradients are column sums computed
 * on the tensor cores (A^T times a ones block), deterministic, no workspace.
 * Arguments:
 *   dOut (M, h), X (M, h), W, U as in tp_mlp_fwd, Z, Y (M, hp) from tp_mlp_fwd
 *   dZ  (M, hp) out            activation-gradient buffer (bf16/f32 like Z);
 *                              holds dZ on return
 *   dX  (M, h) out
 *   dW  shard array, dW_i (hp/N, h) fp32 out
 *   da  shard array or NULL, da_i (hp/N) fp32 out
 *   dU  shard array, dU_i (h, hp/N) fp32 out
 *   db  (h) fp32 out or NULL
 */
TP_API tp_status tp_mlp_bwd(tp_dtype dt, int64_t M, int64_t h, int64_t hp, int N,
                     const void* dOut, const void* X, const void* const* W,
                     const void* const* U, const void* Z, const void* Y,
                     void* dZ, void* dX, void* const* dW, void* const* da,
                     void* const* dU, void* db, int accumulate, void* stream);

/* ------------------------------------------------------------------------ */
/* Head-split attention projections                                          */
/* ------------------------------------------------------------------------ */

/*
 * tp_attn_proj_fwd -- QKV projection split by heads, output projection split
 * by rows with the sum over shards.
 * [TP notes] §Self-Attention层 (Q, K, V split by columns, one or more heads
 * per shard, n_heads % N == 0; the output linear split by rows like the MLP's
 * B); [Walkthrough] §ParallelSelfAttention (QKV outputs not reduced, the output
 * projection all-reduced).
 *   QKV[:, i*3h/N : (i+1)*3h/N] = X Wqkv_i^T + bqkv_i       (= [Q_i K_i V_i])
 *   O = sum_i C_i Wo_i^T + bo,   C_i = C[:, i h/N : (i+1) h/N]
 * Arguments:
 *   X (M, h); Wqkv shard array, Wqkv_i (3h/N, h) = rows [Q_i; K_i; V_i];
 *   bqkv shard array or NULL, (3h/N); C (M, h) attention context;
 *   Wo shard array, Wo_i (h, h/N); bo (h) or NULL;
 *   QKV (M, 3h) out (shard-major); O (M, h) out.
 */
TP_API tp_status tp_attn_proj_fwd(tp_dtype dt, int64_t M, int64_t h, int n_heads, int N,
                           const void* X, const void* const* Wqkv, const void* const* bqkv,
                           const void* C, const void* const* Wo, const void* bo,
                           void* QKV, void* O, void* stream);

/*
 * tp_attn_proj_bwd -- backward of tp_attn_proj_fwd ([TP notes] §Self-Attention层:
 * forward/backward as for the MLP).  One launch.
 *   dWqkv_i = dQKV_i^T X   dbqkv_i = colsum(dQKV_i)   dX = sum_i dQKV_i Wqkv_i
 *   dWo_i = dO^T C_i       dbo = colsum(dO)           dC_i = dO Wo_i
 * Arguments: dQKV (M, 3h) shard-major as QKV; dO (M, h); X, C (M, h);
 *   Wqkv, Wo shard arrays; dX (M, h) out; dC (M, h) out;
 *   dWqkv shard array (3h/N, h) fp32 out; dbqkv shard array (3h/N) fp32 or NULL;
 *   dWo shard array (h, h/N) fp32 out; dbo (h) fp32 or NULL.
 */
TP_API tp_status tp_attn_proj_bwd(tp_dtype dt, int64_t M, int64_t h, int n_heads, int N,
                           const void* dQKV, const void* dO, const void* X, const void* C,
                           const void* const* Wqkv, const void* const* Wo,
                           void* dX, void* dC, void* const* dWqkv, void* const* dbqkv,
                           void* const* dWo, void* dbo, int accumulate, void* stream);

/* ------------------------------------------------------------------------ */
/* Attention core (per head, between the QKV and output projections)        */
/* ------------------------------------------------------------------------ */

/*
 * tp_attn_core_fwd -- softmax attention of every head of every sequence
 * ([TP notes] §Self-Attention层: each head computed on its own, heads split
 * across shards by columns; [Walkthrough] §ParallelSelfAttention).  The
 * pages draw the per-head formula as a figure; it is read as
 *   S = Q_j K_j^T / sqrt(d),  P = softmax over keys (row max subtracted),
 *   C[:, j d:(j+1) d] = P V_j,
 * with GPT's causal mask (key position > query position excluded) when
 * causal != 0.  No attention dropout.
 * Layout (bf16 only; TP_ERR_UNSUPPORTED for TP_F32):
 *   T = b s tokens, b sequences of s tokens each in consecutive rows;
 *   d = h / n_heads; N shards, n_heads % N == 0, heads per shard in order.
 *   QKV (T, 3h)   the shard-major output of tp_attn_proj_fwd: shard i holds
 *                 columns [i 3h/N, (i+1) 3h/N) = [Q_i K_i V_i], each h/N wide
 *                 and holding its heads in order.
 *   P   out (b, n_heads, s, s) bf16 probabilities (row = query, col = key;
 *                 zero where masked), saved for the backward.
 *   C   out (T, h) context, head j in columns [j d, (j+1) d) (the C input of
 *                 tp_attn_proj_fwd).
 *   lse out (b, n_heads, s) fp32 log-sum-exp of every score row, or NULL.
 *   workspace of tp_attn_core_workspace_size bytes, 256-byte aligned.
 * Constraints: T % s == 0 (TP_ERR_INVALID); d and s multiples of 8 and P
 * 16-byte aligned (TP_ERR_ALIGN, TMA's 16-byte rule for head offsets and P's
 * rows).
 * Three steps: the scores launch stores, per row and 64-key part,
 * e = exp(S - m) with m the part's max into P, and (m, sum e) into the
 * workspace; a row kernel merges the parts into lse and rescales P in place
 * to e exp(m - lse); then C = P V.  No (s x s) fp32 score matrix is stored,
 * and the scores are computed once.
 */
TP_API tp_status tp_attn_core_fwd(tp_dtype dt, int64_t T, int64_t s, int64_t h, int n_heads, int N,
                                  int causal, const void* QKV, void* P, void* C, float* lse,
                                  void* workspace, size_t ws_bytes, void* stream);

/*
 * tp_attn_core_bwd -- gradient of tp_attn_core_fwd with respect to QKV,
 * given its P and C and the context gradient dC (T, h):
 *   D = rowsum(dC_j * C_j),  dS = P * (dC_j V_j^T - D) / sqrt(d),
 *   dQ_j = dS K_j,  dK_j = dS^T Q_j,  dV_j = P^T dC_j,
 * written to dQKV (T, 3h) in the QKV layout (every column written).
 * workspace as for the forward (it holds dS, (b, n_heads, s, s) bf16).
 */
TP_API tp_status tp_attn_core_bwd(tp_dtype dt, int64_t T, int64_t s, int64_t h, int n_heads, int N,
                                  int causal, const void* QKV, const void* P, const void* C,
                                  const void* dC, void* dQKV, void* workspace, size_t ws_bytes,
                                  void* stream);

/* Workspace bytes of tp_attn_core_fwd and _bwd (0 for invalid sizes or T = 0). */
TP_API size_t tp_attn_core_workspace_size(int64_t T, int64_t s, int64_t h, int n_heads);

/*
 * tp_attn_core_dropout_fwd / _bwd -- the attention core with attention
 * dropout on the probabilities (rate p_attn, 0 <= p_attn < 1), the dropout
 * that sits inside the tensor-parallel region and therefore draws from one
 * random stream per shard ([Walkthrough] §模型并行, the dropout figure:
 * different seeds inside the parallel region, the same seed after the shard
 * sum; §ParallelSelfAttention: attention dropout through the model-parallel
 * RNG tracker).
 *   C = (P * keep / (1 - p_attn)) V per head; P is stored before dropout, and
 *   Pd (same layout as P, bf16) receives P * keep / (1 - p_attn).
 * keep: element ((sequence * n_heads + head) * s + query) * s + key of the
 * stream stream0 + shard(head) under seed, drawn from Philox4x32-10
 * (Salmon et al., SC 2011): the 16-bit field 16 (e mod 2) of output word
 * (e mod 8) / 2 at counter (e / 8 as two 32-bit words, low first, then the
 * stream as two words) under key (seed as two words), kept iff it is >=
 * floor(p_attn * 65536) computed from the fp32 p_attn.  The backward draws the
 * same bits again.  p_attn > 0 needs s % 16 == 0, s <= 65535 and at most 65535
 * (sequence, head) pairs (TP_ERR_INVALID otherwise) and a non-NULL, 16-byte
 * aligned Pd (TP_ERR_ALIGN).
 * Other arguments as tp_attn_core_fwd / _bwd; the backward's dV is Pd^T dC
 * and its dP is (dC V^T) * keep / (1 - p_attn).
 */
TP_API tp_status tp_attn_core_dropout_fwd(tp_dtype dt, int64_t T, int64_t s, int64_t h, int n_heads,
                                          int N, int causal, float p_attn, uint64_t seed,
                                          uint64_t stream0, const void* QKV, void* P, void* Pd, void* C,
                                          float* lse, void* workspace, size_t ws_bytes, void* stream);
TP_API tp_status tp_attn_core_dropout_bwd(tp_dtype dt, int64_t T, int64_t s, int64_t h, int n_heads,
                                          int N, int causal, float p_attn, uint64_t seed,
                                          uint64_t stream0, const void* QKV, const void* P,
                                          const void* Pd, const void* C, const void* dC, void* dQKV,
                                          void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* One tensor-parallel transformer layer                                     */
/* ------------------------------------------------------------------------ */

/* Sizes and rates of a layer (host struct). */
typedef struct {
  int64_t T, s, h, hp; /* tokens (b sequences of s), hidden size, FFN width */
  int32_t n_heads, N;  /* heads, shards (heads % N == 0, hp % N == 0, 1 <= N <= 8) */
  int32_t causal;      /* GPT causal attention mask */
  float eps;           /* LayerNorm epsilon */
  float p_attn;        /* attention-probability dropout rate */
  float p_hidden;      /* dropout rate after each row-parallel linear */
  uint64_t seed;       /* dropout key */
  uint64_t layer;      /* layer index: the layer's streams are 256 * layer + {0..63 attention
                          (one per shard), 64 attention output, 128 MLP output} */
} tp_layer_config;

/* Weights (host struct of device pointers; shard arrays are host arrays of N
 * device pointers as elsewhere).  LayerNorm parameters fp32, the rest bf16. */
typedef struct {
  const float* g1;
  const float* b1;          /* LayerNorm 1 (h) */
  const void* const* Wqkv;  /* (3h/N, h) per shard, rows [Q_i; K_i; V_i] */
  const void* const* bqkv;  /* (3h/N) per shard or NULL */
  const void* const* Wo;    /* (h, h/N) per shard */
  const void* bo;           /* (h) or NULL */
  const float* g2;
  const float* b2;          /* LayerNorm 2 (h) */
  const void* const* W;     /* MLP column-parallel (hp/N, h) per shard */
  const void* const* a;     /* (hp/N) per shard or NULL */
  const void* const* U;     /* MLP row-parallel (h, hp/N) per shard */
  const void* b;            /* (h) or NULL */
} tp_layer_params;

/* Activations the forward writes and the backward reads (caller-owned device
 * buffers, bf16 unless marked). */
typedef struct {
  void* ln1;    /* (T, h) LayerNorm 1 output */
  float* mean1;
  float* rstd1; /* (T) fp32 */
  void* QKV;    /* (T, 3h) shard-major */
  void* P;      /* (b, n_heads, s, s) probabilities before dropout */
  void* Pd;     /* same shape after dropout; may be NULL when p_attn == 0 */
  void* C;      /* (T, h) attention context */
  void* h1;     /* (T, h) residual stream after the attention block */
  void* ln2;    /* (T, h) LayerNorm 2 output */
  float* mean2;
  float* rstd2; /* (T) fp32 */
  void* Z;
  void* Y;      /* (T, hp) MLP pre-activation and activation */
  uint32_t* attn_keep; /* optional (may be NULL): b * n_heads * s * ceil(s / 32) uint32 words; the
                          forward leaves the attention-dropout keep bits there and the backward reads
                          them instead of drawing them again */
} tp_layer_saved;

/* Parameter gradients (fp32 device buffers; shard arrays as the weights). */
typedef struct {
  float* dg1;
  float* db1;
  void* const* dWqkv;
  void* const* dbqkv; /* or NULL */
  void* const* dWo;
  float* dbo;         /* or NULL */
  float* dg2;
  float* db2;
  void* const* dW;
  void* const* da;    /* or NULL */
  void* const* dU;
  float* db;          /* or NULL */
} tp_layer_grads;

/*
 * tp_transformer_layer_fwd -- [Walkthrough] §ParallelTransformerLayer
 * (attention + MLP, with the dropout after each row-parallel linear defined in
 * the layer), LayerNorm before each block as in GPT:
 *   ln1 = LN(x; g1, b1);  QKV_i = ln1 Wqkv_i^T + bqkv_i;  C = attention core
 *   (causal, attention dropout per shard);  O = sum_i C_i Wo_i^T + bo;
 *   h1 = x + dropout(O);  ln2 = LN(h1; g2, b2);  Z, Y, M = MLP(ln2);
 *   out = h1 + dropout(M).
 * LayerNorm: biased variance, fp32 statistics and parameters, bf16 output.
 * x, out (T, h) bf16; saved as above.  Needs h % 16 == 0, h <= 8192, and the
 * constraints of the attention core and MLP entry points; s, d = h / n_heads
 * and h' / N multiples of 8 (16-byte units for the bulk tensor copies), else
 * TP_ERR_ALIGN before anything is launched.
 * tp_transformer_layer_bwd -- the gradient: dx (T, h) bf16 and the parameter
 * gradients (accumulate: add into them).  Both draw the dropout bits from the
 * config's streams; the backward draws the hidden-dropout bits again, and the
 * attention-dropout bits too unless saved->attn_keep holds the forward's.
 */
/*
 * tp_position_embed_dropout -- the first layer's input ([Walkthrough]
 * §Embedding.forward: word embeddings plus position embeddings, then the
 * embedding dropout):  out = (words + pos_table[positions]) * keep / (1 - p).
 *   words (T, h) bf16 (the vocab-parallel lookup), pos_table (max_pos, h)
 *   bf16, positions (T) int64 (a position outside [0, max_pos) adds a zero
 *   row), out (T, h) bf16.
 *   keep: element row * h + col of stream stream_id under key seed, drawn as
 *   for tp_attn_core_dropout_fwd.  h % 16 == 0; 16-byte aligned rows.
 */
TP_API tp_status tp_position_embed_dropout(int64_t T, int64_t h, int64_t max_pos, const void* words,
                                           const void* pos_table, const int64_t* positions, float p,
                                           uint64_t seed, uint64_t stream_id, void* out, void* stream);

TP_API size_t tp_transformer_layer_workspace_size(const tp_layer_config* cfg);
TP_API tp_status tp_transformer_layer_fwd(const tp_layer_config* cfg, const tp_layer_params* w,
                                          const void* x, void* out, const tp_layer_saved* sv,
                                          void* workspace, size_t ws_bytes, void* stream);
TP_API tp_status tp_transformer_layer_bwd(const tp_layer_config* cfg, const tp_layer_params* w,
                                          const void* x, const tp_layer_saved* sv, const void* dout,
                                          void* dx, const tp_layer_grads* g, int accumulate,
                                          void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Vocab-parallel word embedding and tied output layer                       */
/* ------------------------------------------------------------------------ */

/*
 * vocab_parallel_embed -- masked lookup in every vocabulary range plus the
 * sum over ranges.
 * [Walkthrough] §VocabParallelEmbedding (mask ids outside [start, end), shift
 * by start, F.embedding, zero the masked rows, all-reduce); [TP notes]
 * §输入层Embedding (300-word, two-range example).
 *   out[t] = sum_r [s_r <= id_t < s_{r+1}] E_r[id_t - s_r]
 * Exactly one range owns an id in [0, V), so the sum is a select; an id outside
 * [0, V) gives a zero row (status TP_OK).  Bit-exact copy of the owning row.
 * Arguments:
 *   ids (T) int64; E shard array, E_r (s_{r+1} - s_r, h);
 *   range_starts (host) int64[N+1], range_starts[0] = 0, strictly increasing,
 *   range_starts[N] = V; out (T, h).
 */
TP_API tp_status vocab_parallel_embed(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                               const int64_t* ids, const void* const* E,
                               const int64_t* range_starts, void* out, void* stream);

/*
 * tp_vocab_logits -- logits of the tied output layer per vocabulary range.
 * [Walkthrough] §_VocabParallelCrossEntropy (the output layer uses WE^T; each
 * range yields its own column block); [TP notes] §输出层Embedding.
 *   L_r = X E_r^T      (T, s_{r+1} - s_r), stored with row pitch ld_logits[r]
 * Arguments: X (T, h); E shard array; range_starts (host) as above;
 *   logits shard array, L_r with pitch ld_logits[r] (host int64[N],
 *   >= s_{r+1} - s_r; a multiple of 8 for bf16).
 */
TP_API tp_status tp_vocab_logits(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                          const void* X, const void* const* E, const int64_t* range_starts,
                          void* const* logits, const int64_t* ld_logits, void* stream);

/*
 * tp_vocab_cross_entropy_fwd -- per-token loss of the vocab-parallel
 * cross-entropy without storing the logits.
 * [Walkthrough] §_VocabParallelCrossEntropy forward; [Study notes]
 * §交叉熵张量并行 stages 1-4; [TP notes] §Cross-entropy层 (no all-gather of
 * the (b, s, v) logits).  The logits GEMM per range runs with an epilogue that
 * keeps each 64-column part of a row on chip and writes only its (max, sum of
 * exp(logit - max)) and, where the row's target falls in it, the target logit;
 * a reduction kernel then merges the parts in fixed order (the all-reduce MAX
 * and SUM of the pages) and computes
 *   lse[t]  = max_t + log(sum_t)
 *   loss[t] = log(sum_t) - (logit[t, target_t] - max_t)   (0 <= target_t < V)
 *   loss[t] = log(sum_t)                                  (target in no range,
 *                                                          the pages' masking)
 * Logits are fp32 accumulations of bf16 inputs and never rounded to bf16.
 * Arguments: X (T, h) bf16; E shard array (|r|, h) bf16; range_starts host
 *   int64[N+1]; targets (T) int64 device; loss, lse (T) fp32 device out;
 *   workspace of tp_vocab_cross_entropy_workspace_size bytes, 256-byte aligned
 *   (TP_ERR_WORKSPACE if smaller or NULL, TP_ERR_ALIGN if misaligned).
 * bf16 only (TP_ERR_UNSUPPORTED for fp32).  Deterministic.
 */
TP_API tp_status tp_vocab_cross_entropy_fwd(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                                     const void* X, const void* const* E,
                                     const int64_t* range_starts, const int64_t* targets,
                                     float* loss, float* lse, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* Bytes of the forward's workspace: (max, sum) fp32 pairs for every row and
 * 64-column part of every range, plus one fp32 target logit per row, each
 * block rounded up to 256 bytes.  0 for invalid sizes or ranges. */
TP_API size_t tp_vocab_cross_entropy_workspace_size(int64_t T, int64_t V, int N,
                                                    const int64_t* range_starts);

/*
 * tp_vocab_cross_entropy_bwd -- gradient of the per-token losses.
 * [Walkthrough] §_VocabParallelCrossEntropy backward (softmax, minus 1 at the
 * target in the range that owns it, times the upstream gradient); the
 * logits-side input gradient sums the ranges' products ([Walkthrough]
 * §ColumnParallelLinear backward all-reduce).  One launch (two for large
 * sizes): the logits are recomputed per range with the epilogue
 *   dLogits_r[t, v] = (exp(logit - lse[t]) - [s_r + v == target_t]) * dloss[t]
 * and, if dX is given, dX = sum_r dLogits_r E_r with each row block starting
 * once its dLogits rows are stored.  dLogits feed tied_embed_grad for dE.
 * Arguments: X, E, range_starts, targets as in the forward; lse (T) fp32 from
 *   the forward; dloss (T) fp32; dLogits shard array, block r (T, |r|) bf16
 *   out with pitch ld_dlogits[r] (host int64[N], >= |r|, a multiple of 8);
 *   dX (T, h) bf16 out or NULL.  bf16 only.
 */
TP_API tp_status tp_vocab_cross_entropy_bwd(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                                     const void* X, const void* const* E,
                                     const int64_t* range_starts, const int64_t* targets,
                                     const float* lse, const float* dloss,
                                     void* const* dLogits, const int64_t* ld_dlogits, void* dX,
                                     void* stream);

/*
 * tied_embed_grad -- gradient of the word embedding shared by the input and
 * output layers: the sum of both contributions ([TP notes] §输出层Embedding).
 *   dE[v] = sum_{t : id_t = v} dEmb[t]  +  sum_t dLogits[t, v] X[t, :]
 * The scatter part is deterministic: tokens are grouped by id with a counting
 * sort that is stable in token order, and each row sums its tokens in that
 * order in fp32 before it is added to the GEMM part.
 * Arguments:
 *   ids (T) int64 (ids outside [0, V) contribute nothing); dEmb (T, h);
 *   X (T, h); dLogits shard array, (T, s_{r+1} - s_r) with pitch ld_dlogits[r]
 *   (host int64[N]), or NULL for the input-side part alone;
 *   range_starts (host) as above; dE shard array, dE_r (s_{r+1} - s_r, h) fp32 out;
 *   workspace >= tied_embed_grad_workspace_size(T, V).  On return the
 *   workspace starts with the grouping: int32 offsets[V + 1] (segment of id v
 *   is offsets[v] .. offsets[v+1]) followed by int32 perm[T] (token positions
 *   sorted by (id, position); entries past offsets[V] are unspecified).
 */
TP_API tp_status tied_embed_grad(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                          const int64_t* ids, const void* dEmb, const void* X,
                          const void* const* dLogits, const int64_t* ld_dlogits,
                          const int64_t* range_starts, void* const* dE, int accumulate,
                          void* workspace, size_t ws_bytes, void* stream);

TP_API size_t tied_embed_grad_workspace_size(int64_t T, int64_t V);

/*
 * tied_embed_grad_noalloc -- tied_embed_grad without a caller workspace.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory for the workspace, such as code running under
 * a memory manager that owns every device allocation (a serving runtime that
 * reserves HBM up front) or code that must not call cudaMalloc because it
 * would synchronise the device.  It allocates nothing: the grouping scratch
 * lives in a fixed 1.5 MiB static device array inside the library, which every
 * GPU that loads the library holds until the process exits.
 * Arguments, layouts and results are those of tied_embed_grad, minus the
 * workspace.
 * Limits and behaviour:
 *  - tied_embed_grad_workspace_size(T, V) must not exceed 1.5 MiB (for
 *    example V <= 131072 with T <= 65536); larger sizes return
 *    TP_ERR_WORKSPACE before anything is launched.
 *  - The first call on a device also looks up the array's device address with
 *    that device current, which may synchronise the device: make that first
 *    call during set-up, before any stream capture.
 *  - Argument errors are those of tied_embed_grad and come first, then the
 *    size limit, and only then anything that touches the device.
 *  - All calls share the one array, which keeps the last call's contents: calls
 *    that overlap on the GPU (different streams, no ordering between them) race
 *    and give wrong results.  Order them on one stream or with events.
 */
TP_API tp_status tied_embed_grad_noalloc(tp_dtype dt, int64_t T, int64_t h, int64_t V, int N,
                                         const int64_t* ids, const void* dEmb, const void* X,
                                         const void* const* dLogits, const int64_t* ld_dlogits,
                                         const int64_t* range_starts, void* const* dE,
                                         int accumulate, void* stream);

/* ------------------------------------------------------------------------ */
/* Mixed-precision Adam step                                                 */
/* ------------------------------------------------------------------------ */

/* Optimizer state that lives on the device between steps (24 bytes, 4-byte
 * aligned, caller-owned device memory).  scale, growth_tracker,
 * hysteresis_tracker and step are read and updated by every tp_adam_step;
 * found_inf and grad_norm are outputs of the last step. */
typedef struct {
  float scale;                /* loss scale the gradients carry (unused without the scaler) */
  int32_t growth_tracker;     /* overflow-free steps since the last growth or overflow */
  int32_t hysteresis_tracker; /* overflows left before the scale backs off */
  int32_t step;               /* number of updates applied so far (Adam's t) */
  int32_t found_inf;          /* out: 1 if the last step saw inf/nan and was skipped */
  float grad_norm;            /* out: L2 norm of all unscaled gradients of the last step
                                 (inf or nan when found_inf) */
} tp_optimizer_state;

/* Hyper-parameters of the step (host struct, read during the call). */
typedef struct {
  double lr, beta1, beta2, eps; /* Adam; 0 <= beta1, beta2 < 1 */
  double max_norm;              /* global-norm clip threshold; <= 0 disables clipping */
  int32_t use_scaler;           /* 1: dynamic loss scaling, 0: gradients are unscaled */
  float min_scale;              /* the scale never backs off below this */
  float growth_factor;          /* scale *= growth_factor after growth_interval clean steps */
  float backoff_factor;         /* scale *= backoff_factor once hysteresis overflows are used up */
  int32_t growth_interval;      /* >= 1 */
  int32_t hysteresis;           /* value the hysteresis tracker is reset to on growth */
} tp_adam_config;

/* One parameter group: n elements in flat fp32 device buffers (host struct). */
typedef struct {
  float* param;        /* fp32 main parameters, updated in place */
  const float* grad;   /* fp32 main gradients (times the loss scale when the scaler is on) */
  float* exp_avg;      /* Adam first moment m, updated in place */
  float* exp_avg_sq;   /* Adam second moment v, updated in place */
  void* model_param;   /* bf16 model parameters written from the updated main ones, or NULL */
  int64_t n;           /* >= 0 */
  double weight_decay; /* L2 term added to the gradient: g + weight_decay * param */
} tp_param_group;

/*
 * tp_adam_step -- one step of the mixed-precision optimizer over all groups
 * ([Walkthrough] §MixedPrecisionOptimizer.step and §DynamicGradScaler;
 * [Study notes] §梯度裁剪 and §Adam优化器中的Momentum和Variance), in the
 * pages' order:
 *   1. g = grad / scale (scale = state->scale with the scaler, else 1) and a
 *      check of every g for inf/nan, across all groups;
 *   2. with the scaler, the scale update: an overflow resets growth_tracker,
 *      decrements hysteresis_tracker and, once that is <= 0, sets scale =
 *      max(scale * backoff_factor, min_scale); a clean step increments
 *      growth_tracker and, when it reaches growth_interval, resets it, resets
 *      hysteresis_tracker to hysteresis and multiplies scale by growth_factor;
 *   3. on overflow nothing else changes (params, moments and step stay);
 *   4. ||g|| over all groups; if max_norm > 0 and ||g|| > max_norm,
 *      g *= max_norm / ||g||;
 *   5. t = step + 1; per element g += weight_decay * p; m = b1 m + (1-b1) g;
 *      v = b2 v + (1-b2) g^2; p -= lr / (1 - b1^t) * m / (sqrt(v / (1 - b2^t)) + eps);
 *   6. model_param = bf16(p) (round to nearest even) where given.
 * The fp32 main gradients are the DDP buffer's main_grad ([Core DDP] §3.2),
 * so "copy gradients to the main parameters" is the identity here.
 * Arguments:
 *   groups      HOST array of ngroups descriptors (NULL allowed when ngroups is 0);
 *               0 <= ngroups <= 64.  param, grad, exp_avg and exp_avg_sq of a
 *               group with n > 0 are non-NULL and 16-byte aligned; model_param
 *               is NULL or 8-byte aligned.  No two buffers overlap.
 *   cfg         HOST pointer.
 *   state       DEVICE pointer to the tp_optimizer_state, 4-byte aligned.
 *   workspace   device scratch of tp_adam_step_workspace_size() bytes, 16-byte
 *               aligned (TP_ERR_WORKSPACE if smaller or NULL, TP_ERR_ALIGN if
 *               misaligned).
 * Precision: per-element arithmetic in fp32; the norm sums fp32 squares of up
 * to 32 elements and adds those partial sums in fp64, in an order fixed for a
 * given GPU model (bit-identical results run to run).  An unscaled gradient
 * whose fp32 square overflows (|g| > ~1.8e19) counts as an overflow.
 * Errors: TP_ERR_INVALID for NULL cfg/state, ngroups out of range, n < 0, a
 * NULL buffer, betas outside [0, 1) or growth_interval < 1 with the scaler;
 * TP_ERR_ALIGN for misaligned buffers; all before anything is launched.
 * Launches two kernels: the norm pass (whose last block sums the partials in
 * a fixed order and makes the scaler, skip and clip decisions) and the update.
 */
TP_API tp_status tp_adam_step(const tp_param_group* groups, int ngroups, const tp_adam_config* cfg,
                              tp_optimizer_state* state, void* workspace, size_t ws_bytes,
                              void* stream);

TP_API size_t tp_adam_step_workspace_size(void);

/* ------------------------------------------------------------------------ */
/* Status, profiling and debugging                                           */
/* ------------------------------------------------------------------------ */

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device: TP_OK, TP_ERR_TIMEOUT (a bounded wait expired), or
 * TP_ERR_CUDA (a CUDA error, sticky or not). */
TP_API tp_status tp_get_status(void* stream);

/* Human-readable name of a status code (static string). */
TP_API const char* tp_status_string(tp_status s);

/* Number of SMs the persistent kernels size their grids for (current device). */
TP_API int tp_num_sms(void);

/* Timing of the library's device work.  When enabled, the device work of every
 * library call is bracketed by CUDA events on its stream; tp_profile_read()
 * synchronises the device and returns, per kind of work (the names the calls
 * give it, e.g. "gemm_mlp_fwd", "embed_gather"), the number of calls, the
 * number of kernels they launched and the total device milliseconds since the
 * last reset.  Disabled by default (no events). */
TP_API void tp_profile_enable(int on);
TP_API void tp_profile_reset(void);
/* Fills up to `cap` entries; returns the number of kinds recorded.
 * names[i] points at a static string.  Any output array may be NULL. */
TP_API int tp_profile_read(const char** names, int64_t* calls, int64_t* kernel_launches,
                           double* total_ms, int cap);

/* Evaluates, on the device, the GELU and GELU' that the GEMM epilogues use
 * (GELU(z) = z Phi(z) with erf from Abramowitz & Stegun 7.1.26, |erf error|
 * <= 1.5e-7).  z, y, dy: n fp32 device values; y or dy may be NULL.  A test
 * hook for the device math ([TP notes] §MLP层). */
TP_API tp_status tp_gelu_eval(const float* z, float* y, float* dy, int64_t n, void* stream);

/* Fault injection for testing the bounded waits (host-controlled; never
 * faults the GPU).  kind 1: the TMA producer of the next tensor-core GEMM
 * launch skips its first stage, so the consumer's bounded wait expires and
 * the kernel returns early with TP_ERR_TIMEOUT recorded.  kind 0: off.
 * wait_limit_ms sets the bounded-wait limit (default 1000 ms). */
TP_API void tp_debug_inject_fault(int kind);
/* Selects the tensor-core GEMM kernel for bf16 work: 0 the one-SM kernel
 * (128 x 256 tiles), 1 the two-SM kernel (CTA pairs computing 256 x 256 tiles
 * with tcgen05 cta_group::2), 2 (default) per launch: the two-SM kernel for
 * launches of more than 5 one-SM tiles per SM (6 with causal contraction
 * ranges, 8 when tiles wait on other tiles of the launch), of very long
 * contractions (over 500 k-blocks of tiles per SM with at least 2 tiles per
 * SM) or of long tiles (at least 1 tile per SM averaging 48 k-blocks or more,
 * no causal ranges); the one-SM kernel otherwise.  All give the same results
 * up to fp32 summation order; tests run each. */
TP_API void tp_debug_set_gemm_kernel(int mode);
/* Plans whose outputs depend on each other run as one launch (dependent tiles
 * wait for the tiles they read) unless they have more than `tiles_per_sm`
 * 128 x 256 tiles per SM (5/2 times that, rounded down, when no tile waits on
 * a column block of another output); larger plans run as two launches,
 * independent outputs first.  Default 8; values <= 0 restore it. */
TP_API void tp_debug_set_split_threshold(int tiles_per_sm);
TP_API void tp_debug_set_wait_limit_ms(int ms);
/* Programmatic dependent launch of the library's kernels: on (default), a
 * kernel may start while the previous kernel on its stream finishes, waiting
 * on the device for that kernel's completion before it touches memory (its
 * set-up overlaps the previous kernel's tail); off (0), every kernel starts
 * after the previous one has completed.  Results are identical either way. */
TP_API void tp_debug_set_pdl(int on);

#ifdef __cplusplus
}
#endif

#endif /* TP_H_ */
