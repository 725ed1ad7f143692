"""fp64 CPU oracle of the tensor-parallel transformer block (TEST INFRASTRUCTURE).

This module is test infrastructure.  Only the tests, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / reference leg of ``bench.py`` may import it; the
product path (the CUDA library and its binding) never does, and shares no code
with it.  It is plain numpy in float64: every function writes out the
definition the pages give, in their order and notation, with a library matmul
as the only primitive.  No blocking, fusion or reordering beyond the pages'.

Pages cited (titles as used throughout this repository):
  [Walkthrough]  "Megatron" distributed-training walkthrough
                 (formulaic.cloudchewie.com, docs/.../5-megatron)
  [TP notes]     "Megatron tensor / model parallelism" notes
                 (amentiraz.github.io, posts/Megtron张量/模型并行)
  [Study notes]  Megatron / ZeRO study notes (baty7811.com blog)
  [Core DDP]     megatron.core.distributed overview (zwxr.cn news 246059)

Notation: M = b*s tokens, h hidden size, h' = FFN width, N shards.  Column
shard i holds W_i (h'/N, h) (torch ``weight`` layout, so A_i = W_i^T); row
shard i holds U_i (h, h'/N) (B_i = U_i^T).  Every matrix is row-major.

Readings where the pages are silent or garbled:
  * GELU is the exact erf form (the pages' formula is an image).
  * The row-parallel bias is added once, after the shard sum.
  * The second vocabulary range of the 300-word example is [150, 300).
  * An id that falls in no range yields a zero row (masked sum), not an error.
  * The oracle keeps every intermediate in fp64; it does not mimic bf16
    rounding of saved activations (the tolerance absorbs it).
  * Attention per head is softmax(Q K^T / sqrt(d)) V (the pages draw it as a
    figure), with GPT's causal mask when asked; no attention dropout.

Parity status per function is stated in its docstring: "pinned by ..." names
the tests that tie it to something other than itself.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

_SQRT2 = math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


# --------------------------------------------------------------------------
# GELU
# --------------------------------------------------------------------------
def gelu(z):
    """GELU(z) = z * Phi(z) = z/2 * (1 + erf(z / sqrt 2)), exact erf form.

    [TP notes] §MLP层: GELU is the non-linear activation between A and B (its
    formula is an image on the page; the erf form is taken).
    Pinned by: special values (gelu(0)=0, gelu(x)-gelu(-x)=x, gelu(x)/x->1),
    math.erf on sample points, torch float64 F.gelu(approximate='none').
    """
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1.0 + _erf(z / _SQRT2))


def gelu_prime(z):
    """dGELU/dz = Phi(z) + z * phi(z), phi the standard normal density.

    Derivative of the form above.  Pinned by: gelu_prime(0)=1/2 and central
    finite differences of ``gelu``.
    """
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * (1.0 + _erf(z / _SQRT2)) + z * np.exp(-0.5 * z * z) * _INV_SQRT_2PI


# --------------------------------------------------------------------------
# Column-parallel linear (A split by columns) and row-parallel linear
# --------------------------------------------------------------------------
def column_parallel_fwd(X, W_shards, a_shards=None):
    """Y_i = GELU(X A_i + a_i) per shard, with A_i = W_i^T.

    [Walkthrough] §ColumnParallelLinear: f is the identity in forward, each
    shard computes F.linear(X, W_i, a_i) = X W_i^T + a_i, and the output stays
    split (no gather) because [TP notes] §MLP层 feeds Y_i straight into the
    row-split B.  Returns (Z_i list, Y_i list).
    Pinned by: unsharded equality, N=1 vs torch float64, finite differences.
    """
    Z, Y = [], []
    for i, W in enumerate(W_shards):
        Zi = X @ W.T
        if a_shards is not None:
            Zi = Zi + a_shards[i][None, :]
        Z.append(Zi)
        Y.append(gelu(Zi))
    return Z, Y


def row_parallel_fwd(Y_shards, U_shards, b=None):
    """Out = sum_i Y_i B_i + b with B_i = U_i^T.

    [Walkthrough] §RowParallelLinear: each shard computes F.linear(Y_i, U_i)
    without bias; g is the all-reduce (sum) over shards in forward; the bias,
    which is not split, is added once after the reduction.
    Pinned by: unsharded equality (sharded sum == XA->GELU->B), bias-once test.
    """
    Out = None
    for Yi, Ui in zip(Y_shards, U_shards):
        Pi = Yi @ Ui.T
        Out = Pi if Out is None else Out + Pi
    if b is not None:
        Out = Out + b[None, :]
    return Out


def mlp_fwd(X, W_shards, a_shards, U_shards, b):
    """Tensor-parallel MLP forward: A column-split -> GELU -> B row-split.

    [TP notes] §MLP层 (A by columns, B by rows, one all-reduce in forward).
    Returns Z (M,h') and Y (M,h') with shard i in columns [i h'/N, (i+1) h'/N),
    and Out (M,h).  Pinned through its two halves (unsharded equality, torch
    float64 at N = 1) and the whole-block torch autograd check.
    """
    Z, Y = column_parallel_fwd(X, W_shards, a_shards)
    Out = row_parallel_fwd(Y, U_shards, b)
    return np.concatenate(Z, axis=1), np.concatenate(Y, axis=1), Out


def mlp_bwd(dOut, X, W_shards, a_shards, U_shards):
    """Tensor-parallel MLP backward.

    [Walkthrough] §RowParallelLinear: g backward is the identity, so every
    shard sees the whole dOut;  §ColumnParallelLinear: f backward is an
    all-reduce, so dX is the sum over shards.  Per shard i:
        dY_i = dOut U_i,  dZ_i = dY_i * GELU'(Z_i)
        dU_i = dOut^T Y_i,  dW_i = dZ_i^T X
        da_i = column sums of dZ_i,  db = column sums of dOut
        dX   = sum_i dZ_i W_i
    Z_i, Y_i are recomputed here in fp64 from X (the oracle never takes values
    from the device).  Returns a dict of fp64 arrays (dW, dU, da are lists;
    dZ is (M, h') with shard i in columns [i h'/N, (i+1) h'/N), the layout of
    Z).
    Pinned by: central finite differences on tiny shapes (of X, W, U, a, b
    and of the saved pre-activation Z itself), torch float64 autograd of the
    unsharded block (including the gradient at the first linear's output),
    unsharded dX.
    """
    Z, Y = column_parallel_fwd(X, W_shards, a_shards)
    dW, dU, da, dZ = [], [], [], []
    dX = None
    for i in range(len(W_shards)):
        dYi = dOut @ U_shards[i]
        dZi = dYi * gelu_prime(Z[i])
        dZ.append(dZi)
        dU.append(dOut.T @ Y[i])
        dW.append(dZi.T @ X)
        da.append(dZi.sum(axis=0))
        part = dZi @ W_shards[i]
        dX = part if dX is None else dX + part
    out = dict(dX=dX, dW=dW, dU=dU, da=da, db=dOut.sum(axis=0), dZ=np.concatenate(dZ, axis=1))
    return out


def mlp_bwd_sampled(dOut, X, W_shards, a_shards, U_shards, rows, units):
    """The same definitions as ``mlp_bwd``, evaluated only where asked.

    ``rows``: token indices r for which dZ[r] and dX[r] are formed (both are
    row-local).
    ``units``: per shard, the FFN units j for which column j of dZ_i is formed
    over all tokens, giving row j of dW_i, column j of dU_i and da_i[j].
    Used at full workload sizes where the whole fp64 backward is too slow.
    """
    # dZ and dX rows: dZ_i[r] needs only X[r] and dOut[r]
    Xr, dOr = X[rows], dOut[rows]
    Zr, _ = column_parallel_fwd(Xr, W_shards, a_shards)
    dXr = None
    dZrows = []
    for i in range(len(W_shards)):
        dZr = (dOr @ U_shards[i]) * gelu_prime(Zr[i])
        dZrows.append(dZr)
        part = dZr @ W_shards[i]
        dXr = part if dXr is None else dXr + part
    dW, dU, da = [], [], []
    for i, J in enumerate(units):
        Wj = W_shards[i][J]
        Zj = X @ Wj.T
        if a_shards is not None:
            Zj = Zj + a_shards[i][J][None, :]
        dZj = (dOut @ U_shards[i][:, J]) * gelu_prime(Zj)
        dW.append(dZj.T @ X)
        dU.append(dOut.T @ gelu(Zj))
        da.append(dZj.sum(axis=0))
    return dict(dX_rows=dXr, dZ_rows=np.concatenate(dZrows, axis=1), dW_rows=dW, dU_cols=dU, da=da,
                db=dOut.sum(axis=0))


# --------------------------------------------------------------------------
# Head-split attention projections
# --------------------------------------------------------------------------
def attn_proj_fwd(X, Wqkv_shards, bqkv_shards, C, Wo_shards, bo):
    """QKV projection split by heads (column split) and output projection
    split by rows, with the sum over shards.

    [TP notes] §Self-Attention层: Q, K, V are split by columns, one or more
    heads per shard; the output linear B is split by rows exactly like the MLP.
    [Walkthrough] §ParallelSelfAttention: QKV outputs are not reduced; the
    output projection's result is all-reduced.
        QKV_i = X Wqkv_i^T + bqkv_i   (shard-major [Q_i K_i V_i] columns)
        O     = sum_i C_i Wo_i^T + bo,  C_i = C[:, i h/N:(i+1) h/N]
    C is the attention context (the attention core is not part of the block).
    Pinned by: unsharded equality with a single (3h,h)/(h,h) projection.
    """
    N = len(Wqkv_shards)
    d = C.shape[1] // N
    QKV = []
    for i in range(N):
        q = X @ Wqkv_shards[i].T
        if bqkv_shards is not None:
            q = q + bqkv_shards[i][None, :]
        QKV.append(q)
    O = None
    for i in range(N):
        part = C[:, i * d:(i + 1) * d] @ Wo_shards[i].T
        O = part if O is None else O + part
    if bo is not None:
        O = O + bo[None, :]
    return np.concatenate(QKV, axis=1), O


def attn_proj_bwd(dQKV, dO, X, C, Wqkv_shards, Wo_shards):
    """Backward of ``attn_proj_fwd`` ([TP notes] §Self-Attention层: same
    forward/backward principle as the MLP).
        dWqkv_i = dQKV_i^T X,  dbqkv_i = column sums of dQKV_i
        dX      = sum_i dQKV_i Wqkv_i            (f backward: sum over shards)
        dWo_i   = dO^T C_i,    dbo = column sums of dO
        dC_i    = dO Wo_i                        (g backward: identity)
    Pinned by: central finite differences on tiny shapes.
    """
    N = len(Wqkv_shards)
    w = dQKV.shape[1] // N
    d = C.shape[1] // N
    dWqkv, dbqkv, dWo, dC = [], [], [], []
    dX = None
    for i in range(N):
        g = dQKV[:, i * w:(i + 1) * w]
        dWqkv.append(g.T @ X)
        dbqkv.append(g.sum(axis=0))
        part = g @ Wqkv_shards[i]
        dX = part if dX is None else dX + part
        dWo.append(dO.T @ C[:, i * d:(i + 1) * d])
        dC.append(dO @ Wo_shards[i])
    return dict(dX=dX, dWqkv=dWqkv, dbqkv=dbqkv, dWo=dWo, dbo=dO.sum(axis=0),
                dC=np.concatenate(dC, axis=1))


def attn_proj_bwd_weight_rows(dQKV, dO, X, C, N, qkv_rows, o_rows):
    """Rows of the weight gradients of ``attn_proj_bwd`` (same definitions,
    evaluated only where asked, for full-size workloads):
    dWqkv_i[j] = dQKV_i[:, j]^T X for j in qkv_rows[i];
    dWo_i[k]   = dO[:, k]^T C_i   for k in o_rows[i];
    and the bias gradients in full (column sums of dQKV_i and of dO).
    Pinned by: equality with the rows of ``attn_proj_bwd``."""
    w = dQKV.shape[1] // N
    d = C.shape[1] // N
    dWqkv, dWo, dbqkv = [], [], []
    for i in range(N):
        g = dQKV[:, i * w:(i + 1) * w]
        dWqkv.append(g[:, qkv_rows[i]].T @ X)
        dWo.append(dO[:, o_rows[i]].T @ C[:, i * d:(i + 1) * d])
        dbqkv.append(g.sum(axis=0))
    return dWqkv, dWo, dbqkv, dO.sum(axis=0)


# --------------------------------------------------------------------------
# Vocab-parallel embedding
# --------------------------------------------------------------------------
def attention_head_columns(h, n_heads, N, j):
    """Column offsets of global head j in the shard-major QKV (T, 3h) and in
    the context C (T, h).  Shard i owns heads [i n_heads/N, (i+1) n_heads/N)
    and its QKV columns [i 3h/N, (i+1) 3h/N) = [Q_i K_i V_i], each h/N wide,
    its heads in order inside each ([TP notes] §Self-Attention层: Q, K, V
    split by columns with whole heads per shard).  Returns (q, k, v, c)."""
    d = h // n_heads
    per = n_heads // N
    i, jl = divmod(j, per)
    base = i * 3 * (h // N)
    return base + jl * d, base + h // N + jl * d, base + 2 * (h // N) + jl * d, j * d


def attention_head(q, k, v, causal, keep=None, p=0.0):
    """One head of one sequence: S = q k^T / sqrt(d), keys after the query
    masked to -inf when causal, P = softmax over keys with the row max
    subtracted ([Walkthrough] §_VocabParallelCrossEntropy's stable softmax),
    out = P v; with attention dropout, out = (P * keep / (1 - p)) v.  The
    pages draw the single-head formula as a figure; the scaled dot product
    with the 1/sqrt(d) factor is the plain reading, and the causal mask is
    GPT's.  Returns (P (s, s), out (s, d)), P before dropout.  Pinned through
    ``attention_core``: torch scaled_dot_product_attention in float64."""
    s, d = q.shape
    S = (q @ k.T) / math.sqrt(d)
    if causal:
        S = np.where(np.tril(np.ones((s, s), dtype=bool)), S, -np.inf)
    E = np.exp(S - S.max(axis=1, keepdims=True))
    P = E / E.sum(axis=1, keepdims=True)
    Pd = P if keep is None else P * keep / (1.0 - p)
    return P, Pd @ v


def attention_head_grad(q, k, v, P, g, keep=None, p=0.0):
    """Gradient of ``attention_head`` given its P and the output gradient g
    (the chain rule through out = Pd v, the dropout, the softmax and
    S = q k^T / sqrt(d)):
        dv = Pd^T g,  dP = (g v^T) * keep / (1 - p),
        dS = P * (dP - sum_keys(P * dP)) / sqrt(d),  dq = dS k,  dk = dS^T q.
    Masked entries have P = 0 and carry no gradient.  Returns (dq, dk, dv).
    Pinned through ``attention_core_grad``: torch autograd in float64."""
    d = q.shape[1]
    Pd = P if keep is None else P * keep / (1.0 - p)
    dP = g @ v.T
    if keep is not None:
        dP = dP * keep / (1.0 - p)
    dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True)) / math.sqrt(d)
    return dS @ k, dS.T @ q, Pd.T @ g


def attention_keep(bi, j, s, n_heads, N, p, seed, layer):
    """Attention-dropout keep flags (s, s) of sequence bi, head j: elements
    ((bi n_heads + j) s + query) s + key of the stream of head j's shard.
    Pinned through ``dropout_keep`` (the generator's known-answer vectors)
    and the planted shared-stream test (the shards' masks must differ)."""
    if p <= 0.0:
        return None
    shard = j // (n_heads // N)
    e0 = ((bi * n_heads + j) * s) * s
    return dropout_keep(seed, dropout_stream(layer, 0, shard), e0, s * s, p).reshape(s, s)


def attention_core(QKV, s, n_heads, N, causal, p_attn=0.0, seed=0, layer=0):
    """Per-head attention between the QKV projection and the output
    projection for b = T / s sequences of s tokens: every (sequence, head)
    pair runs ``attention_head`` on its columns of the shard-major QKV and
    writes head j's output to context columns [j d, (j+1) d).  Heads are
    independent ([TP notes] §Self-Attention层; [Walkthrough]
    §ParallelSelfAttention: every rank computes its own heads, and its
    attention dropout draws from its own stream).
    Returns (C (T, h), P (b, n_heads, s, s)), P before dropout.
    Pinned by: torch scaled_dot_product_attention in float64 per head, torch
    multi_head_attention_forward through the sharded projections, a closed
    form (q = 0: the running or full mean of v), brute force on a tiny case,
    and torch autograd of a whole layer with dropout."""
    T, h3 = QKV.shape
    h = h3 // 3
    d = h // n_heads
    b = T // s
    C = np.zeros((T, h))
    P = np.zeros((b, n_heads, s, s))
    for bi in range(b):
        rows = slice(bi * s, (bi + 1) * s)
        for j in range(n_heads):
            qc, kc, vc, cc = attention_head_columns(h, n_heads, N, j)
            keep = attention_keep(bi, j, s, n_heads, N, p_attn, seed, layer)
            P[bi, j], C[rows, cc:cc + d] = attention_head(
                QKV[rows, qc:qc + d], QKV[rows, kc:kc + d], QKV[rows, vc:vc + d], causal,
                keep=keep, p=p_attn)
    return C, P


def attention_core_grad(QKV, P, dC, s, n_heads, N, p_attn=0.0, seed=0, layer=0):
    """Gradient of ``attention_core`` with respect to QKV, given its
    probabilities P and the context gradient dC: ``attention_head_grad`` per
    (sequence, head), written back in the QKV layout.
    Pinned by: torch autograd through scaled_dot_product_attention in
    float64, through multi_head_attention_forward, and through a whole layer."""
    T, h3 = QKV.shape
    h = h3 // 3
    d = h // n_heads
    b = T // s
    dQKV = np.zeros((T, h3))
    for bi in range(b):
        rows = slice(bi * s, (bi + 1) * s)
        for j in range(n_heads):
            qc, kc, vc, cc = attention_head_columns(h, n_heads, N, j)
            keep = attention_keep(bi, j, s, n_heads, N, p_attn, seed, layer)
            dq, dk, dv = attention_head_grad(QKV[rows, qc:qc + d], QKV[rows, kc:kc + d],
                                             QKV[rows, vc:vc + d], P[bi, j], dC[rows, cc:cc + d],
                                             keep=keep, p=p_attn)
            dQKV[rows, qc:qc + d], dQKV[rows, kc:kc + d], dQKV[rows, vc:vc + d] = dq, dk, dv
    return dQKV


def vocab_mask(ids, start, end):
    """Mask and shift of one vocabulary range.

    [Walkthrough] §VocabParallelEmbedding: input_mask = (id < start) | (id >= end);
    masked_input = id - start, with masked positions set to 0.
    Returns (masked_input, input_mask).
    Pinned by: the page's own example ids [2,7,1,5], range [0,3) -> [2,0,1,0].
    """
    ids = np.asarray(ids, dtype=np.int64)
    mask = (ids < start) | (ids >= end)
    masked = ids - start
    masked[mask] = 0
    return masked, mask


def vocab_parallel_embed_partials(ids, E_shards, range_starts):
    """Per-range partial lookups: each range looks up the ids it owns and
    writes zero rows elsewhere ([Walkthrough] §VocabParallelEmbedding;
    [TP notes] §输入层Embedding).  Returns a list of (T,h) fp64 partials.
    Pinned through ``vocab_parallel_embed`` (the page's example, brute force)
    and the planted wrong-range partial test."""
    parts = []
    for r, Er in enumerate(E_shards):
        masked, mask = vocab_mask(ids, range_starts[r], range_starts[r + 1])
        out = np.asarray(Er)[masked].astype(np.float64)
        out[mask, :] = 0.0
        parts.append(out)
    return parts


def vocab_parallel_embed(ids, E_shards, range_starts):
    """out[t] = sum_r partial_r[t]: the all-reduce (sum) over ranges of the
    masked lookups.  Pinned by: the 300-word two-range example, brute force
    over every id on small vocabularies, equality with the full lookup."""
    parts = vocab_parallel_embed_partials(ids, E_shards, range_starts)
    out = parts[0].copy()
    for p in parts[1:]:
        out += p
    return out


def vocab_logits(X, E_shards):
    """Per-range logits L_r = X E_r^T ([Walkthrough] §_VocabParallelCrossEntropy:
    the output layer uses the transpose of the input word embedding; each
    range holds its own block of columns).  Pinned by: equality with the
    unsharded X E^T."""
    return [X @ np.asarray(Er, dtype=np.float64).T for Er in E_shards]


def embed_sort(ids, V):
    """Tokens grouped by id, stable in token order: (offsets (V+1), perm).

    perm lists the token positions t with 0 <= id_t < V sorted by (id_t, t);
    offsets[v]..offsets[v+1] is the segment of id v.  This is the grouping the
    scatter-add of the embedding gradient runs over.  Pinned by: brute force
    (every segment is exactly the increasing list of positions holding v).
    """
    ids = np.asarray(ids, dtype=np.int64)
    valid = np.nonzero((ids >= 0) & (ids < V))[0]
    order = valid[np.argsort(ids[valid], kind="stable")]
    counts = np.bincount(ids[valid], minlength=V) if len(valid) else np.zeros(V, np.int64)
    offsets = np.zeros(V + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    return offsets, order


def embed_scatter_grad(ids, dEmb, V):
    """Input-side gradient of the word embedding: dE_in[v] = sum over tokens
    t with id_t = v of dEmb[t] (backward of the lookup; an id outside [0,V)
    contributes nothing, as its forward row was masked to zero).  A brute
    force loop over tokens.  Pinned by: column sums equal sum_t dEmb[t] over
    valid tokens; per-id brute force on small vocabularies."""
    ids = np.asarray(ids, dtype=np.int64)
    out = np.zeros((V, dEmb.shape[1]), dtype=np.float64)
    for t in range(len(ids)):
        v = int(ids[t])
        if 0 <= v < V:
            out[v] += dEmb[t]
    return out


def tied_embed_grad(ids, dEmb, X, dLogits_shards, range_starts, V):
    """Gradient of the tied word embedding = input-side scatter-add + output
    side dLogits^T X, kept separately and then summed.

    [TP notes] §输出层Embedding: the input and output layers share one word
    embedding, and the update must use the sum of both gradients.
    Returns a list of per-range (|r|, h) fp64 blocks.
    Pinned by: the decomposition, the dLogits=0 and dEmb=0 reductions.
    """
    scatter = embed_scatter_grad(ids, dEmb, V)
    out = []
    for r, dL in enumerate(dLogits_shards):
        s, e = range_starts[r], range_starts[r + 1]
        gemm = dL.T @ X
        out.append(scatter[s:e] + gemm)
    return out


def tied_embed_grad_rows(ids, dEmb, X, dLogits_full, vocab_rows):
    """``tied_embed_grad`` for a subset of vocabulary rows (global ids),
    dLogits given unsharded (T, V).  Row v = sum_{t: id_t = v} dEmb[t] +
    dLogits[:, v]^T X."""
    ids = np.asarray(ids, dtype=np.int64)
    rows = []
    for v in vocab_rows:
        acc = dLogits_full[:, v] @ X
        sel = np.nonzero(ids == v)[0]
        for t in sel:
            acc = acc + dEmb[t]
        rows.append(acc)
    return np.stack(rows) if rows else np.zeros((0, X.shape[1]))


# --------------------------------------------------------------------------
# Vocab-parallel cross-entropy
# --------------------------------------------------------------------------
def vocab_parallel_cross_entropy(X, E_shards, range_starts, targets):
    """Per-token loss of the vocab-parallel cross-entropy, and its log-sum-exp.

    Follows the forward of [Walkthrough] §_VocabParallelCrossEntropy and the
    four stages of [Study notes] §交叉熵张量并行 ([TP notes] §Cross-entropy层
    states why: no all-gather of the (b, s, v) logits):
      1. each range's logits L_r = X E_r^T;
      2. the row maximum over all ranges (all-reduce MAX) is subtracted;
      3a. predicted logit: each range picks its shifted logit at the target
          when the target lies in its range and 0 otherwise; the ranges' values
          are summed (all-reduce SUM);
      3b. the sum of exp of the shifted logits, per range then over ranges;
      4. loss = log(sum) - predicted.
    A target in no range gets predicted = 0 (every range masks it), so its loss
    is log(sum) of the shifted logits, as the pages' masking gives.
    Returns (loss, lse) with lse = max + log(sum) per token.
    Pinned by: torch cross_entropy on the unsharded logits (valid targets),
    invariance to the vocabulary split, the all-zero-logits closed form
    log V, and stability at logits of order 1e3.
    """
    targets = np.asarray(targets, dtype=np.int64)
    logits = [np.asarray(X, dtype=np.float64) @ np.asarray(Er, dtype=np.float64).T for Er in E_shards]
    T = logits[0].shape[0]
    logits_max = np.max(np.stack([L.max(axis=1) for L in logits]), axis=0)  # all-reduce MAX
    shifted = [L - logits_max[:, None] for L in logits]
    predicted = np.zeros(T)
    rows = np.arange(T)
    for r, L in enumerate(shifted):
        start, end = range_starts[r], range_starts[r + 1]
        target_mask = (targets < start) | (targets >= end)
        masked_target = np.where(target_mask, 0, targets - start)
        pred_r = L[rows, masked_target]
        pred_r[target_mask] = 0.0
        predicted += pred_r  # all-reduce SUM
    sum_exp = np.zeros(T)
    for L in shifted:
        sum_exp += np.exp(L).sum(axis=1)  # all-reduce SUM
    loss = np.log(sum_exp) - predicted
    return loss, logits_max + np.log(sum_exp)


def vocab_parallel_cross_entropy_grad(X, E_shards, range_starts, targets, dloss):
    """Gradient of the per-token losses w.r.t. each range's logits.

    [Walkthrough] §_VocabParallelCrossEntropy backward: every logit gets its
    softmax probability; the target position in the range that owns it gets
    1 subtracted (a target in no range subtracts nothing); the result is
    scaled by the upstream gradient of its token.  Returns the per-range
    (T, |r|) blocks.
    Pinned by: torch autograd of cross_entropy on the unsharded logits, and
    the all-zero-logits closed form 1/V - onehot.
    """
    targets = np.asarray(targets, dtype=np.int64)
    dloss = np.asarray(dloss, dtype=np.float64)
    logits = [np.asarray(X, dtype=np.float64) @ np.asarray(Er, dtype=np.float64).T for Er in E_shards]
    T = logits[0].shape[0]
    logits_max = np.max(np.stack([L.max(axis=1) for L in logits]), axis=0)
    exp_logits = [np.exp(L - logits_max[:, None]) for L in logits]
    sum_exp = sum(e.sum(axis=1) for e in exp_logits)
    rows = np.arange(T)
    grads = []
    for r, e in enumerate(exp_logits):
        start, end = range_starts[r], range_starts[r + 1]
        target_mask = (targets < start) | (targets >= end)
        masked_target = np.where(target_mask, 0, targets - start)
        g = e / sum_exp[:, None]  # softmax
        g[rows, masked_target] -= 1.0 - target_mask.astype(np.float64)
        grads.append(g * dloss[:, None])
    return grads


def logits_side_dx(dLogits_shards, E_shards):
    """Input gradient of the tied output layer: dX = sum_r dLogits_r E_r.
    The logits are a column-parallel linear over the vocabulary ([Study
    notes] §交叉熵张量并行 stage 1, parallel_lm_logits), so its input gradient
    is the sum over ranges of the per-range products (the f operator's
    backward all-reduce, [Walkthrough] §ColumnParallelLinear).
    Pinned by: equality with the unsharded dLogits E."""
    return sum(np.asarray(dL, dtype=np.float64) @ np.asarray(Er, dtype=np.float64)
               for dL, Er in zip(dLogits_shards, E_shards))


# --------------------------------------------------------------------------
# Mixed-precision optimizer step
# --------------------------------------------------------------------------
def grad_scaler_update(state, found_inf, cfg):
    """Dynamic loss-scale update ([Walkthrough] §DynamicGradScaler.update).

    On an overflow the growth tracker resets and the hysteresis tracker counts
    down; once it is <= 0 the scale backs off (times backoff_factor, not below
    min_scale), and keeps backing off on further overflows until a growth
    resets the tracker.  growth_interval overflow-free steps in a row multiply
    the scale by growth_factor and reset both trackers.  Returns a new dict.
    Pinned by: the growth, hysteresis, back-off and floor behaviours the page
    states, step by step.
    """
    s = dict(state)
    if found_inf:
        s["growth_tracker"] = 0
        s["hysteresis_tracker"] -= 1
        if s["hysteresis_tracker"] <= 0:
            s["scale"] = max(s["scale"] * cfg["backoff_factor"], cfg["min_scale"])
    else:
        s["growth_tracker"] += 1
        if s["growth_tracker"] == cfg["growth_interval"]:
            s["growth_tracker"] = 0
            s["hysteresis_tracker"] = cfg["hysteresis"]
            s["scale"] = s["scale"] * cfg["growth_factor"]
    return s


def unscale_and_check(grads, scale):
    """Main gradients divided by the loss scale, and whether any is inf/nan
    across all groups ([Walkthrough] §MixedPrecisionOptimizer.step, step 2).
    Pinned through the optimizer-step tests (overflow skip, unscale before
    the norm clip)."""
    out = [np.asarray(g, dtype=np.float64) / scale for g in grads]
    found_inf = any(not np.all(np.isfinite(g)) for g in out)
    return out, found_inf


def clip_by_global_norm(grads, max_norm):
    """Gradient clipping by the L2 norm of all gradients as one vector
    ([Study notes] §梯度裁剪: if ||g|| > max_norm, g <- g * max_norm / ||g||;
    otherwise unchanged; max_norm <= 0 disables).  Returns (grads, ||g||).
    Pinned by: a closed form (||g|| = 5 scaled to 1) and torch
    clip_grad_norm_ (which adds 1e-6 to the norm: 2e-7 relative here)."""
    total = math.sqrt(sum(float(np.sum(np.asarray(g, dtype=np.float64) ** 2)) for g in grads))
    if max_norm > 0 and total > max_norm:
        grads = [np.asarray(g, dtype=np.float64) * (max_norm / total) for g in grads]
    return grads, total


def adam_update(param, grad, m, v, step, cfg, weight_decay):
    """One Adam update of one tensor ([Study notes] §Adam优化器中的Momentum和
    Variance: m_t = b1 m + (1-b1) g, v_t = b2 v + (1-b2) g^2, theta -= lr *
    m_hat / (sqrt(v_hat) + eps), with the hats the usual bias corrections
    1 - b^t; weight decay as torch Adam's, added to the gradient, since
    [Walkthrough] builds Adam(param_groups, lr, weight_decay, betas, eps)).
    step is the 1-based count of applied updates.  Returns (param, m, v).
    Pinned by: torch.optim.Adam in float64 over several steps."""
    g = np.asarray(grad, dtype=np.float64) + weight_decay * np.asarray(param, dtype=np.float64)
    m = cfg["beta1"] * np.asarray(m, dtype=np.float64) + (1 - cfg["beta1"]) * g
    v = cfg["beta2"] * np.asarray(v, dtype=np.float64) + (1 - cfg["beta2"]) * g * g
    m_hat = m / (1 - cfg["beta1"] ** step)
    v_hat = v / (1 - cfg["beta2"] ** step)
    param = np.asarray(param, dtype=np.float64) - cfg["lr"] * m_hat / (np.sqrt(v_hat) + cfg["eps"])
    return param, m, v


def mixed_precision_adam_step(groups, state, cfg):
    """One step of the mixed-precision optimizer ([Walkthrough]
    §MixedPrecisionOptimizer.step, in its order):
      1. the gradients are the fp32 main gradients (copy to main: identity);
      2. unscale by the loss scale and check for inf/nan (if the scaler is on);
      3. update the loss scale;
      4. on inf/nan skip the update (parameters, moments and the step count
         stay; the scale has already changed);
      5. clip by the global L2 norm;
      6. Adam on the fp32 main parameters;
      7. copy the main parameters to the bf16 model parameters.
    groups: list of dicts param, grad, m, v, weight_decay (fp64 arrays).
    state: scale, growth_tracker, hysteresis_tracker, step.
    Returns (updated, grad_norm, new groups with param/m/v/model, new state);
    grad_norm is the norm of the unscaled gradients (inf/nan on overflow).
    Pinned through its parts and by the skip test."""
    scale = state["scale"] if cfg["use_scaler"] else 1.0
    grads, found_inf = unscale_and_check([g["grad"] for g in groups], scale)
    new_state = dict(state)
    if cfg["use_scaler"]:
        new_state = grad_scaler_update(state, found_inf, cfg)
    norm_sq = sum(float(np.sum(g * g)) for g in grads)
    grad_norm = math.sqrt(norm_sq) if math.isfinite(norm_sq) else norm_sq
    if found_inf:
        return False, grad_norm, [dict(g) for g in groups], new_state
    grads, _ = clip_by_global_norm(grads, cfg["max_norm"])
    step = state["step"] + 1
    new_state["step"] = step
    out = []
    for grp, g in zip(groups, grads):
        p, m, v = adam_update(grp["param"], g, grp["m"], grp["v"], step, cfg, grp["weight_decay"])
        out.append(dict(grp, param=p, m=m, v=v))
    return True, grad_norm, out, new_state


# --------------------------------------------------------------------------
# Transformer layer: counter-based dropout, LayerNorm, residuals
# --------------------------------------------------------------------------
# Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
# easy as 1, 2, 3", SC 2011): ten rounds of two 32 x 32 -> 64-bit products
# with a Weyl-sequence key schedule.  The pages fix only where the random
# streams differ (dropout inside the tensor-parallel region draws per shard,
# outside it all shards draw the same numbers: [Walkthrough] §模型并行, the
# dropout figure); the generator and the mask layout below are this build's.
_PH_M0, _PH_M1 = 0xD2511F53, 0xCD9E8D57
_PH_W0, _PH_W1 = 0x9E3779B9, 0xBB67AE85
_U32 = np.uint64(0xFFFFFFFF)


def philox4x32(c0, c1, c2, c3, k0, k1):
    """Philox4x32-10 of counters (c0, c1, c2, c3) under key (k0, k1), 32-bit
    words held in uint64 arrays (every product of two 32-bit words is exact
    in 64 bits); c0 .. c3 may be arrays.  Returns the four output words.
    Pinned by: the known-answer vectors published with the generator
    (tests/golden/philox4x32_kat.json)."""
    s32 = np.uint64(32)
    x0, x1, x2, x3 = np.broadcast_arrays(*(np.asarray(c, dtype=np.uint64) & _U32 for c in (c0, c1, c2, c3)))
    x0, x1, x2, x3 = x0.copy(), x1.copy(), x2.copy(), x3.copy()
    key0, key1 = np.uint64(k0) & _U32, np.uint64(k1) & _U32
    for r in range(10):
        if r > 0:
            key0 = (key0 + np.uint64(_PH_W0)) & _U32
            key1 = (key1 + np.uint64(_PH_W1)) & _U32
        p0 = np.uint64(_PH_M0) * x0
        p1 = np.uint64(_PH_M1) * x2
        x0, x1, x2, x3 = (p1 >> s32) ^ x1 ^ key0, p1 & _U32, (p0 >> s32) ^ x3 ^ key1, p0 & _U32
    return x0, x1, x2, x3


def dropout_keep(seed, stream, e0, n, p):
    """Keep flags of elements e0 .. e0+n-1 of one dropout site.  Element e
    takes the 16-bit field 16 (e mod 2) of output word (e mod 8) / 2 of
    Philox4x32-10 at counter (b mod 2^32, b / 2^32, stream mod 2^32,
    stream / 2^32), b = e / 8, under key (seed mod 2^32, seed / 2^32), and is
    kept iff that field is >= floor(p 2^16) (keep probability
    1 - floor(p 2^16) / 2^16).  Pinned by: the generator's known-answer
    vectors, the keep rate, distinct streams and seeds."""
    e = np.arange(e0, e0 + n, dtype=np.uint64)
    b = e // np.uint64(8)
    st = np.uint64(stream)
    sd = np.uint64(seed)
    words = philox4x32(b & _U32, b >> np.uint64(32), st & _U32, st >> np.uint64(32),
                       sd & _U32, sd >> np.uint64(32))
    W = np.stack(words, axis=0)  # (4, n)
    w = ((e % np.uint64(8)) // np.uint64(2)).astype(np.int64)
    shift = np.uint64(16) * (e % np.uint64(2))
    field = (W[w, np.arange(n)] >> shift) & np.uint64(0xFFFF)
    return field >= np.uint64(int(math.floor(p * 65536.0)))


def dropout_stream(layer, kind, shard=0):
    """Stream id of a dropout site: kind 0 = attention probabilities (one
    stream per shard: inside the tensor-parallel region), 1 = attention
    output, 2 = MLP output (one stream shared by all shards: after the
    shard sum).  Layers are 256 streams apart."""
    return layer * 256 + kind * 64 + (shard if kind == 0 else 0)


def layernorm(x, g, b, eps):
    """LayerNorm over the last axis with biased variance, fp64 (the fp32
    gain and bias of [Study notes]' mixed-precision notes):
        y = (x - mean) / sqrt(var + eps) * g + b.
    Returns (y, mean, rstd).  Pinned by: torch layer_norm in float64."""
    x = np.asarray(x, dtype=np.float64)
    mean = x.mean(axis=-1)
    var = ((x - mean[..., None]) ** 2).mean(axis=-1)
    rstd = 1.0 / np.sqrt(var + eps)
    return (x - mean[..., None]) * rstd[..., None] * g + b, mean, rstd


def layernorm_grad(dy, x, g, mean, rstd):
    """Gradient of ``layernorm``: with xhat = (x - mean) rstd and n features,
        dxhat = dy g,  dx = rstd (dxhat - mean(dxhat) - xhat mean(dxhat xhat)),
        dg = sum over rows of dy xhat,  db = sum over rows of dy.
    Pinned by: torch autograd through layer_norm in float64."""
    xhat = (np.asarray(x, dtype=np.float64) - mean[..., None]) * rstd[..., None]
    dxhat = dy * g
    dx = rstd[..., None] * (dxhat - dxhat.mean(axis=-1, keepdims=True) -
                            xhat * (dxhat * xhat).mean(axis=-1, keepdims=True))
    return dx, (dy * xhat).sum(axis=0), dy.sum(axis=0)


def dropout_residual(res, x, keep, p):
    """out = res + x * keep / (1 - p): the dropout after a row-parallel
    linear and the residual add of [Walkthrough] §ParallelTransformerLayer.
    Pinned through the layer's torch autograd check and its planted unscaled
    dropout."""
    return res + x * keep / (1.0 - p)


def transformer_layer_fwd(x, P, cfg):
    """One tensor-parallel transformer layer ([Walkthrough]
    §ParallelTransformerLayer = attention + MLP, with the dropout after each
    row-parallel linear defined in the layer; LayerNorm before each block, as
    in Megatron's GPT):
        ln1 = LN(x; g1, b1)
        QKV = [ln1 Wqkv_i^T + bqkv_i]_i            (column-parallel, per shard)
        C   = attention core of QKV (attention dropout per shard stream)
        O   = sum_i C_i Wo_i^T + bo                 (row-parallel + shard sum)
        h1  = x + dropout(O)                        (one stream for all shards)
        ln2 = LN(h1; g2, b2)
        Z, Y, M = MLP(ln2)                          (column -> GELU -> row)
        out = h1 + dropout(M)
    P: g1, b1, Wqkv, bqkv, Wo, bo, g2, b2, W, a, U, b (lists for shards).
    cfg: s, n_heads, N, causal, eps, p_attn, p_hidden, seed, layer.
    Returns (out, saved) with every intermediate the backward needs.
    Pinned by: torch autograd of the same layer in float64."""
    T, h = x.shape
    ln1, m1, r1 = layernorm(x, P["g1"], P["b1"], cfg["eps"])
    QKV, _ = attn_proj_fwd(ln1, P["Wqkv"], P["bqkv"], np.zeros((T, h)), P["Wo"], None)
    C, Pr = attention_core(QKV, cfg["s"], cfg["n_heads"], cfg["N"], cfg["causal"],
                           cfg["p_attn"], cfg["seed"], cfg["layer"])
    _, O = attn_proj_fwd(ln1, P["Wqkv"], P["bqkv"], C, P["Wo"], P["bo"])
    keep1 = dropout_keep(cfg["seed"], dropout_stream(cfg["layer"], 1), 0, T * h,
                         cfg["p_hidden"]).reshape(T, h)
    h1 = dropout_residual(x, O, keep1, cfg["p_hidden"])
    ln2, m2, r2 = layernorm(h1, P["g2"], P["b2"], cfg["eps"])
    Z, Y, M = mlp_fwd(ln2, P["W"], P["a"], P["U"], P["b"])
    keep2 = dropout_keep(cfg["seed"], dropout_stream(cfg["layer"], 2), 0, T * h,
                         cfg["p_hidden"]).reshape(T, h)
    out = dropout_residual(h1, M, keep2, cfg["p_hidden"])
    saved = dict(x=x, ln1=ln1, m1=m1, r1=r1, QKV=QKV, C=C, P=Pr, O=O, keep1=keep1, h1=h1,
                 ln2=ln2, m2=m2, r2=r2, Z=Z, Y=Y, M=M, keep2=keep2)
    return out, saved


def transformer_layer_bwd(dout, saved, P, cfg):
    """Backward of ``transformer_layer_fwd`` by the chain rule through its
    steps in reverse: the residual passes dout to h1 unchanged, the dropout
    scales by keep / (1 - p), then MLP, LayerNorm 2, attention output
    projection, attention core, QKV projection, LayerNorm 1.
    Returns dx and the parameter gradients (same keys as P, prefixed d).
    Pinned by: torch autograd through the same layer in float64."""
    p = cfg["p_hidden"]
    dM = dout * saved["keep2"] / (1.0 - p)
    g = mlp_bwd(dM, saved["ln2"], P["W"], P["a"], P["U"])
    dln2 = g["dX"]
    dh1_ln, dg2, db2 = layernorm_grad(dln2, saved["h1"], P["g2"], saved["m2"], saved["r2"])
    dh1 = dout + dh1_ln
    dO = dh1 * saved["keep1"] / (1.0 - p)
    T, h = dO.shape
    zero_qkv = np.zeros_like(saved["QKV"])
    dC = attn_proj_bwd(zero_qkv, dO, saved["ln1"], saved["C"], P["Wqkv"], P["Wo"])["dC"]
    dQKV = attention_core_grad(saved["QKV"], saved["P"], dC, cfg["s"], cfg["n_heads"], cfg["N"],
                               cfg["p_attn"], cfg["seed"], cfg["layer"])
    ga = attn_proj_bwd(dQKV, dO, saved["ln1"], saved["C"], P["Wqkv"], P["Wo"])
    dx_ln, dg1, db1 = layernorm_grad(ga["dX"], saved["x"], P["g1"], saved["m1"], saved["r1"])
    return dict(dx=dh1 + dx_ln, dg1=dg1, db1=db1, dWqkv=ga["dWqkv"], dbqkv=ga["dbqkv"],
                dWo=ga["dWo"], dbo=ga["dbo"], dg2=dg2, db2=db2, dW=g["dW"], da=g["da"],
                dU=g["dU"], db=g["db"], dQKV=dQKV, dC=dC, dO=dO)


def embed_position_dropout(words, pos_table, positions, keep, p):
    """Input of the first layer ([Walkthrough] §Embedding.forward): word
    embeddings (the vocab-parallel lookup, summed over ranges) plus position
    embeddings, then dropout: (words + pos_table[positions]) * keep / (1 - p).
    A position outside the table adds a zero row (this build's reading: the
    pages index in range only).  Pinned by: torch's embedding lookup (no
    dropout), zero dropped entries and 1/(1 - p) survivors."""
    pos = np.asarray(positions)
    ok = (pos >= 0) & (pos < len(pos_table))
    pe = np.where(ok[:, None], np.asarray(pos_table, dtype=np.float64)[np.where(ok, pos, 0)], 0.0)
    return (np.asarray(words, dtype=np.float64) + pe) * keep / (1.0 - p)


# --------------------------------------------------------------------------
# Closed forms the pages state
# --------------------------------------------------------------------------
def param_count(H, L, V):
    """(12 H^2 + 4 H) L + 2 H V: per layer 3H^2 (QKV) + H^2 (attention output)
    + 4H^2 + 4H^2 (MLP up/down) + 2*(2H) (two LayerNorms), plus the input
    embedding and output projection, 2 H V ([Walkthrough], model set-up
    paragraph after model_provider).  Pinned by: the page's 2,827,821,056."""
    return (12 * H * H + 4 * H) * L + 2 * H * V


def tp_block_comm_volume(b, s, h):
    """Communication of one MLP (or attention) block under tensor parallelism:
    one all-reduce in forward and one in backward, each a reduce-scatter plus
    an all-gather of phi = b*s*h elements, so 2*phi each and 4*phi in all
    ([TP notes] §MLP层的通讯量分析, §Self-Attention层的通讯量分析).
    Returns (phi, number of shard sums, total volume)."""
    phi = b * s * h
    n_sums = 2
    return phi, n_sums, n_sums * 2 * phi
