"""Seeded synthetic inputs for the tensor-parallel block.

This module is shared by the tests, ``bench.py`` and ``smoke()``: it holds the
workload shapes, the seeds and the random draws, and nothing of the block's
arithmetic (no GEMM, no activation, no masking, no reduction).  The same bytes
feed both the CUDA path and the fp64 oracle.

Recipe (one rule for every tensor):
  * every tensor is drawn in full (unsharded) from its own PCG64 stream,
    ``numpy.random.Generator(PCG64([seed, stream_id]))``, as float32 normals
    scaled by the tensor's standard deviation, then rounded once to the
    workload's dtype (bf16 by round-to-nearest-even through torch);
  * the full tensor is then split into its shards, so a sharded and an
    unsharded computation see identical values (init-then-split);
  * weights ~ N(0, 0.02), activations and upstream gradients ~ N(0, 1),
    biases are zero unless a test asks for N(0, bias_std);
  * token ids are uniform integers in [0, V) drawn from their own stream.

No public dataset is involved: the pages name none for this path.
"""
from __future__ import annotations

import numpy as np
import torch

__all__ = ["WORKLOADS", "normal", "uniform_ids", "mlp_inputs", "attn_inputs",
           "embed_inputs", "ce_inputs", "adam_inputs", "attn_core_inputs", "layer_inputs", "split_rows", "split_cols"]

# Workloads: shapes and seeds only.  Names state the sizes.
WORKLOADS = {
    # tiny fp32 MLP: b=1, s=8, h=64, h'=4h=256, N=2
    "mlp_tiny_f32": dict(kind="mlp", dtype="f32", b=1, s=8, h=64, hp=256, N=2, seed=1000),
    # tiny fp32 vocab-parallel embedding: V=300, h=16, two ranges, ids [0,212,7,9]
    "embed_tiny_f32": dict(kind="embed", dtype="f32", V=300, h=16, b=1, s=4,
                           ranges=[0, 150, 300], ids=[0, 212, 7, 9], seed=1000),
    # bf16 MLP: b=4, s=1024, h=1024, h'=4096, N=4
    "mlp_b4_s1024_h1024_hp4096_N4": dict(kind="mlp", dtype="bf16", b=4, s=1024, h=1024,
                                         hp=4096, N=4, seed=1001),
    # bf16 MLP at model width: b=2, s=2048, h=4096, h'=16384, N=2
    "mlp_b2_s2048_h4096_hp16384_N2": dict(kind="mlp", dtype="bf16", b=2, s=2048, h=4096,
                                          hp=16384, N=2, seed=1002),
    # bf16 head-split attention projections: b=1, s=2048, h=4096, 8 heads of 512, N=8
    "attn_b1_s2048_h4096_heads8_N8": dict(kind="attn", dtype="bf16", b=1, s=2048, h=4096,
                                          n_heads=8, N=8, seed=1003),
    # bf16 vocab-parallel tied embedding: V=50257, h=4096, b=4, s=2048, two ranges
    "embed_tied_V50257_h4096_T8192": dict(kind="embed", dtype="bf16", V=50257, h=4096, b=4,
                                          s=2048, ranges=[0, 25129, 50257], seed=1004),
    # bf16 vocab-parallel cross-entropy on the same output layer: T=8192 tokens, two ranges
    "ce_V50257_h4096_T8192": dict(kind="ce", dtype="bf16", V=50257, h=4096, b=4, s=2048,
                                  ranges=[0, 25129, 50257], seed=1005),
    # bf16 causal attention core between the projections: b=1, s=2048, 8 heads of 512, N=8
    "attn_core_b1_s2048_heads8_d512_causal": dict(kind="attn_core", dtype="bf16", b=1, s=2048,
                                                  h=4096, n_heads=8, N=8, causal=True, seed=1007),
    # bf16 transformer layer of the H=4096 model: b=1, s=2048, 8 heads of 512, h'=16384, N=8,
    # causal, attention and hidden dropout 0.1
    "layer_b1_s2048_h4096_heads8_hp16384_N8": dict(kind="layer", dtype="bf16", b=1, s=2048, h=4096,
                                                   hp=16384, n_heads=8, N=8, causal=True, eps=1e-5,
                                                   p_attn=0.1, p_hidden=0.1, layer=0, seed=1008),
    # fp32 mixed-precision Adam step over one transformer layer of the H=4096 model:
    # QKV (3H, H), attention output (H, H), MLP up (4H, H), MLP down (H, 4H) with
    # weight decay; two LayerNorms' gain and bias (H each) without; 201,342,976 values
    "adam_layer_H4096": dict(kind="adam", dtype="f32", H=4096, seed=1006,
                             sizes=[3 * 4096 * 4096, 4096 * 4096, 4 * 4096 * 4096,
                                    4 * 4096 * 4096, 4096, 4096, 4096, 4096],
                             weight_decay=[0.1, 0.1, 0.1, 0.1, 0.0, 0.0, 0.0, 0.0],
                             state=dict(scale=4096.0, growth_tracker=0, hysteresis_tracker=2,
                                        step=100),
                             hyper=dict(lr=1e-4, beta1=0.9, beta2=0.95, eps=1e-8, max_norm=1.0,
                                        use_scaler=1, min_scale=1.0, growth_factor=2.0,
                                        backoff_factor=0.5, growth_interval=1000, hysteresis=2)),
}

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def normal(seed: int, stream: int, shape, std: float, dtype: str) -> torch.Tensor:
    """N(0, std^2) draw, float32 then rounded once to ``dtype``; CPU tensor."""
    g = _gen(seed, stream)
    a = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return torch.from_numpy(a).to(_TORCH_DTYPE[dtype])


def uniform_ids(seed: int, stream: int, T: int, V: int) -> torch.Tensor:
    """T token ids uniform in [0, V) as int64; CPU tensor."""
    g = _gen(seed, stream)
    return torch.from_numpy(g.integers(0, V, size=T, dtype=np.int64))


def split_rows(t: torch.Tensor, N: int):
    """Contiguous copies of N equal row blocks of ``t``."""
    n = t.shape[0] // N
    return [t[i * n:(i + 1) * n].contiguous() for i in range(N)]


def split_cols(t: torch.Tensor, N: int):
    """Contiguous copies of N equal column blocks of ``t``."""
    n = t.shape[1] // N
    return [t[:, i * n:(i + 1) * n].contiguous() for i in range(N)]


def mlp_inputs(cfg: dict, bias_std: float = 0.0, M: int | None = None) -> dict:
    """Inputs of the column->GELU->row MLP block.

    Returns full tensors and their shards:
      X (M,h), dOut (M,h) ~ N(0,1);
      W (h',h) ~ N(0,0.02), split by rows into W_i (h'/N,h)  [column-parallel A];
      U (h,h') ~ N(0,0.02), split by columns into U_i (h,h'/N) [row-parallel B];
      a (h') and b (h) biases (zero unless ``bias_std`` > 0).
    """
    dt, seed, N = cfg["dtype"], cfg["seed"], cfg["N"]
    h, hp = cfg["h"], cfg["hp"]
    M = cfg["b"] * cfg["s"] if M is None else M
    X = normal(seed, 1, (M, h), 1.0, dt)
    W = normal(seed, 2, (hp, h), 0.02, dt)
    U = normal(seed, 3, (h, hp), 0.02, dt)
    dOut = normal(seed, 4, (M, h), 1.0, dt)
    if bias_std > 0:
        a = normal(seed, 5, (hp,), bias_std, dt)
        b = normal(seed, 6, (h,), bias_std, dt)
    else:
        a = torch.zeros(hp, dtype=_TORCH_DTYPE[dt])
        b = torch.zeros(h, dtype=_TORCH_DTYPE[dt])
    return dict(M=M, h=h, hp=hp, N=N, dtype=dt, X=X, W=W, U=U, a=a, b=b, dOut=dOut,
                W_shards=split_rows(W, N), U_shards=split_cols(U, N),
                a_shards=[x.contiguous() for x in a.chunk(N)])


def attn_inputs(cfg: dict, bias_std: float = 0.0, M: int | None = None) -> dict:
    """Inputs of the head-split attention projections.

    Wqkv (3h,h) is stored in the global [Q; K; V] order; shard i gathers the rows
    of its heads from each of Q, K and V, giving (3h/N, h) = [Q_i; K_i; V_i].
    Wo (h,h) is split by columns into Wo_i (h, h/N).  C is the attention context
    that feeds the output projection (the attention core is not part of the
    block), ~N(0,1), as are X and the upstream gradients dQKV, dO.
    """
    dt, seed, N = cfg["dtype"], cfg["seed"], cfg["N"]
    h = cfg["h"]
    M = cfg["b"] * cfg["s"] if M is None else M
    X = normal(seed, 11, (M, h), 1.0, dt)
    Wqkv = normal(seed, 12, (3 * h, h), 0.02, dt)
    Wo = normal(seed, 13, (h, h), 0.02, dt)
    C = normal(seed, 14, (M, h), 1.0, dt)
    dQKV = normal(seed, 15, (M, 3 * h), 1.0, dt)
    dO = normal(seed, 16, (M, h), 1.0, dt)
    if bias_std > 0:
        bqkv = normal(seed, 17, (3 * h,), bias_std, dt)
        bo = normal(seed, 18, (h,), bias_std, dt)
    else:
        bqkv = torch.zeros(3 * h, dtype=_TORCH_DTYPE[dt])
        bo = torch.zeros(h, dtype=_TORCH_DTYPE[dt])
    d = h // N
    Wqkv_shards, bqkv_shards = [], []
    for i in range(N):
        rows = [Wqkv[j * h + i * d: j * h + (i + 1) * d] for j in range(3)]
        Wqkv_shards.append(torch.cat(rows, 0).contiguous())
        bqkv_shards.append(torch.cat([bqkv[j * h + i * d: j * h + (i + 1) * d] for j in range(3)]).contiguous())
    return dict(M=M, h=h, N=N, n_heads=cfg["n_heads"], dtype=dt, X=X, Wqkv=Wqkv, Wo=Wo, C=C,
                dQKV=dQKV, dO=dO, bqkv=bqkv, bo=bo, Wqkv_shards=Wqkv_shards,
                bqkv_shards=bqkv_shards, Wo_shards=split_cols(Wo, N))


def embed_inputs(cfg: dict, T: int | None = None) -> dict:
    """Inputs of the vocab-parallel embedding and its tied output layer.

    E (V,h) ~ N(0,0.02) for bf16 workloads (N(0,1) for the tiny fp32 one),
    split by the vocabulary ranges into E_r (|r|, h).  ids uniform in [0,V)
    unless the workload fixes them.  X (the last hidden state feeding the
    output layer), dEmb (gradient reaching the embedding output) and dLogits
    (gradient of the logits) ~ N(0,1).  dLogits is stored per range, (T, |r|).
    """
    dt, seed, V, h = cfg["dtype"], cfg["seed"], cfg["V"], cfg["h"]
    ranges = list(cfg["ranges"])
    if "ids" in cfg and T is None:
        ids = torch.tensor(cfg["ids"], dtype=torch.int64)
    else:
        T = cfg["b"] * cfg["s"] if T is None else T
        ids = uniform_ids(seed, 21, T, V)
    T = ids.numel()
    E = normal(seed, 22, (V, h), 1.0 if dt == "f32" else 0.02, dt)
    X = normal(seed, 23, (T, h), 1.0, dt)
    dEmb = normal(seed, 24, (T, h), 1.0, dt)
    dLogits = normal(seed, 25, (T, V), 1.0, dt)
    E_shards = [E[ranges[r]:ranges[r + 1]].contiguous() for r in range(len(ranges) - 1)]
    dL_shards = [dLogits[:, ranges[r]:ranges[r + 1]].contiguous() for r in range(len(ranges) - 1)]
    return dict(T=T, V=V, h=h, N=len(ranges) - 1, dtype=dt, ranges=ranges, ids=ids, E=E,
                E_shards=E_shards, X=X, dEmb=dEmb, dLogits=dLogits, dLogits_shards=dL_shards)


def ce_inputs(cfg: dict) -> dict:
    """Inputs of the vocab-parallel cross-entropy: the last hidden state X
    (T, h) ~ N(0, 1), the tied embedding E (V, h) ~ N(0, 0.02) split into its
    vocabulary ranges, targets uniform in [0, V), and the upstream gradient of
    the mean loss, dloss = 1/T per token (fp32)."""
    dt, seed = cfg["dtype"], cfg["seed"]
    T, h, V, ranges = cfg["b"] * cfg["s"], cfg["h"], cfg["V"], list(cfg["ranges"])
    X = normal(seed, 31, (T, h), 1.0, dt)
    E = normal(seed, 32, (V, h), 0.02, dt)
    targets = uniform_ids(seed, 33, T, V)
    dloss = torch.full((T,), 1.0 / T, dtype=torch.float32)
    E_shards = [E[ranges[r]:ranges[r + 1]].contiguous() for r in range(len(ranges) - 1)]
    return dict(T=T, h=h, V=V, N=len(ranges) - 1, ranges=ranges, X=X, E=E, E_shards=E_shards,
                targets=targets, dloss=dloss)


def adam_inputs(cfg: dict, sizes=None) -> dict:
    """Inputs of one mixed-precision Adam step (fp32, flat groups): main
    parameters ~ N(0, 0.02), unscaled gradients ~ N(0, 1e-3) stored times the
    loss scale (what a scaled backward leaves in the fp32 main gradients),
    first moments ~ N(0, 1e-4), second moments the square of an N(0, 1e-3)
    draw, all mid-training (state step 100).  ``sizes`` overrides the group
    sizes (weight decay then alternates 0.1, 0.0)."""
    seed = cfg["seed"]
    sizes = list(cfg["sizes"]) if sizes is None else list(sizes)
    wds = list(cfg["weight_decay"]) if len(sizes) == len(cfg["sizes"]) else \
        [0.1 if i % 2 == 0 else 0.0 for i in range(len(sizes))]
    scale = float(cfg["state"]["scale"])
    groups = []
    for i, n in enumerate(sizes):
        groups.append(dict(
            param=normal(seed, 100 + 4 * i, (n,), 0.02, "f32"),
            grad=normal(seed, 101 + 4 * i, (n,), 1e-3 * scale, "f32"),
            m=normal(seed, 102 + 4 * i, (n,), 1e-4, "f32"),
            v=normal(seed, 103 + 4 * i, (n,), 1e-3, "f32").square_(),
            weight_decay=wds[i]))
    return dict(groups=groups, state=dict(cfg["state"]), hyper=dict(cfg["hyper"]))


def attn_core_inputs(cfg: dict) -> dict:
    """Inputs of the attention core on an attention workload: the shard-major
    QKV (T, 3h) and the context gradient dC (T, h), both ~ N(0, 1) bf16, for
    b sequences of s tokens."""
    seed, b, s, h = cfg["seed"], cfg["b"], cfg["s"], cfg["h"]
    T = b * s
    return dict(T=T, s=s, h=h, n_heads=cfg["n_heads"], N=cfg["N"],
                QKV=normal(seed, 41, (T, 3 * h), 1.0, "bf16"),
                dC=normal(seed, 42, (T, h), 1.0, "bf16"))


def layer_inputs(cfg: dict, T: int | None = None) -> dict:
    """Inputs of one transformer layer: x and dout ~ N(0, 1) bf16 (T, h);
    unsharded weights ~ N(0, 0.02) bf16 split into shards as the layer uses
    them (Wqkv rows [Q; K; V] with shard i taking its h/N rows of each,
    Wo / U by columns, W by rows), biases ~ N(0, 0.02), LayerNorm gains
    1 + N(0, 0.1) and biases N(0, 0.1) in fp32.  T defaults to b s."""
    seed, h, hp, N = cfg["seed"], cfg["h"], cfg["hp"], cfg["N"]
    T = cfg["b"] * cfg["s"] if T is None else T
    d = h // N
    Wqkv = normal(seed, 51, (3 * h, h), 0.02, "bf16")
    bqkv = normal(seed, 52, (3 * h,), 0.02, "bf16")
    Wo = normal(seed, 53, (h, h), 0.02, "bf16")
    W = normal(seed, 54, (hp, h), 0.02, "bf16")
    U = normal(seed, 55, (h, hp), 0.02, "bf16")
    n = hp // N
    return dict(
        T=T, x=normal(seed, 56, (T, h), 1.0, "bf16"), dout=normal(seed, 57, (T, h), 1.0, "bf16"),
        g1=1.0 + normal(seed, 58, (h,), 0.1, "f32"), b1=normal(seed, 59, (h,), 0.1, "f32"),
        g2=1.0 + normal(seed, 60, (h,), 0.1, "f32"), b2=normal(seed, 61, (h,), 0.1, "f32"),
        Wqkv=[torch.cat([Wqkv[j * h + i * d: j * h + (i + 1) * d] for j in range(3)]).contiguous()
              for i in range(N)],
        bqkv=[torch.cat([bqkv[j * h + i * d: j * h + (i + 1) * d] for j in range(3)]).contiguous()
              for i in range(N)],
        Wo=split_cols(Wo, N), bo=normal(seed, 62, (h,), 0.02, "bf16"),
        W=[W[i * n:(i + 1) * n].contiguous() for i in range(N)],
        a=[t.contiguous() for t in normal(seed, 63, (hp,), 0.02, "bf16").split(n)],
        U=split_cols(U, N), b=normal(seed, 64, (h,), 0.02, "bf16"))
