"""GPU parity of the transformer layer and its pieces (dropout bits, position
embedding, attention dropout, the whole layer forward and backward) against
the fp64 oracle, through the C ABI.

Dropout keep bits are integer decisions: they must match the oracle bit for
bit.  Activations and gradients are bf16 (or fp32 from bf16 products): held to
the bf16 bar (2e-2 max relative error).
"""
import numpy as np
import pytest
import torch

import oracle.tp_oracle as O
import synthetic_inputs as SI
from tests.gpu_util import assert_close, f64, f64_list

pytestmark = pytest.mark.gpu


def _tp():
    import megatron_tensor_transformer_tp_gb300 as tp
    return tp


def f32p(p):
    """The dropout rate as the library receives it (fp32)."""
    return float(np.float32(p))


@pytest.mark.parametrize("p,seed,stream", [(0.1, 7, 3), (0.5, 2**40 + 1, 64), (0.9, 0, 0)])
def test_dropout_bits_match_oracle(p, seed, stream):
    tp = _tp()
    T, h = 96, 272
    words = torch.ones(T, h, dtype=torch.bfloat16, device="cuda")
    table = torch.zeros(4, h, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(T, dtype=torch.int64, device="cuda")
    out = torch.empty_like(words)
    tp.tp_position_embed_dropout(words, table, pos, p, seed, stream, out)
    got = (out.float() != 0).cpu().numpy().reshape(-1)
    want = O.dropout_keep(seed, stream, 0, T * h, f32p(p))
    assert np.array_equal(got, want)


def test_position_embed_dropout_parity():
    tp = _tp()
    T, h, P = 200, 128, 50
    g = np.random.default_rng(3)
    words = SI.normal(3, 1, (T, h), 1.0, "bf16")
    table = SI.normal(3, 2, (P, h), 0.02, "bf16")
    pos = torch.from_numpy(g.integers(0, P, T).astype(np.int64))
    pos[5], pos[6] = -1, P  # outside the table: zero rows
    out = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    tp.tp_position_embed_dropout(words.cuda(), table.cuda(), pos.cuda(), 0.2, 9, 5, out)
    keep = O.dropout_keep(9, 5, 0, T * h, f32p(0.2)).reshape(T, h)
    ref = O.embed_position_dropout(f64(words), f64(table), pos.numpy(), keep, f32p(0.2))
    assert_close(out, ref, "bf16", "embedding output")


@pytest.mark.parametrize("causal", [True, False])
def test_attn_core_dropout_parity(causal):
    tp = _tp()
    b, s, h, H, N, p, seed, layer = 2, 160, 256, 4, 2, 0.25, 11, 3
    T = b * s
    QKV = SI.normal(21, 1, (T, 3 * h), 1.0, "bf16")
    dC = SI.normal(21, 2, (T, h), 1.0, "bf16")
    Q = QKV.cuda()
    P = torch.empty(b, H, s, s, dtype=torch.bfloat16, device="cuda")
    Pd = torch.empty_like(P)
    C = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    dQKV = torch.empty(T, 3 * h, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(tp.tp_attn_core_workspace_size(T, s, h, H), dtype=torch.uint8, device="cuda")
    stream0 = tp.layer_stream(layer, 0)
    tp.tp_attn_core_dropout_fwd(Q, s, H, N, causal, p, seed, stream0, P, Pd, C, None, ws)
    tp.tp_attn_core_dropout_bwd(Q, P, Pd, C, dC.cuda(), s, H, N, causal, p, seed, stream0, dQKV, ws)
    assert tp.tp_get_status() == tp.TP_OK
    Qn = f64(QKV)
    rC, rP = O.attention_core(Qn, s, H, N, causal, f32p(p), seed, layer)
    assert_close(C, rC, "bf16", "C", elementwise=False)  # sums products of the bf16 P
    assert_close(P, rP, "bf16", "P")
    lower = np.tril(np.ones((s, s), dtype=bool)) if causal else np.ones((s, s), dtype=bool)
    Pdn = Pd.float().cpu().numpy()
    for bi in range(b):
        for j in range(H):
            keep = O.attention_keep(bi, j, s, H, N, f32p(p), seed, layer)
            assert np.array_equal((Pdn[bi, j] != 0) & lower, keep & lower), (bi, j)
    rd = O.attention_core_grad(Qn, rP, f64(dC), s, H, N, f32p(p), seed, layer)
    assert_close(dQKV, rd, "bf16", "dQKV", elementwise=False)  # from the bf16 dS and P


def alloc_layer(cfg, T):
    bf = torch.bfloat16
    h, hp, H, s = cfg["h"], cfg["hp"], cfg["n_heads"], cfg["s"]
    b = T // s
    e = lambda *shape, dt=bf: torch.empty(*shape, dtype=dt, device="cuda")
    saved = dict(ln1=e(T, h), mean1=e(T, dt=torch.float32), rstd1=e(T, dt=torch.float32),
                 QKV=e(T, 3 * h), P=e(b, H, s, s), Pd=e(b, H, s, s), C=e(T, h), h1=e(T, h),
                 ln2=e(T, h), mean2=e(T, dt=torch.float32), rstd2=e(T, dt=torch.float32),
                 Z=e(T, hp), Y=e(T, hp))
    return saved


def run_layer(cfg, inp, keep_buffer=False):
    tp = _tp()
    T, h, hp, N = inp["T"], cfg["h"], cfg["hp"], cfg["N"]
    c = dict(cfg, T=T)
    d = lambda t: t.cuda().contiguous()
    params = dict(g1=d(inp["g1"]), b1=d(inp["b1"]), g2=d(inp["g2"]), b2=d(inp["b2"]),
                  Wqkv=[d(t) for t in inp["Wqkv"]], bqkv=[d(t) for t in inp["bqkv"]],
                  Wo=[d(t) for t in inp["Wo"]], bo=d(inp["bo"]), W=[d(t) for t in inp["W"]],
                  a=[d(t) for t in inp["a"]], U=[d(t) for t in inp["U"]], b=d(inp["b"]))
    saved = alloc_layer(cfg, T)
    if keep_buffer:
        s = cfg["s"]
        saved["attn_keep"] = torch.empty((T // s) * cfg["n_heads"] * s * ((s + 31) // 32),
                                         dtype=torch.int32, device="cuda")
    x, dout = d(inp["x"]), d(inp["dout"])
    out = torch.empty_like(x)
    ws = torch.empty(tp.tp_transformer_layer_workspace_size(c), dtype=torch.uint8, device="cuda")
    tp.tp_transformer_layer_fwd(c, params, x, out, saved, ws)
    z = lambda *shape: torch.full(shape, float("nan"), device="cuda")
    d3, n = h // N, hp // N
    grads = dict(dg1=z(h), db1=z(h), dg2=z(h), db2=z(h), dbo=z(h), db=z(h),
                 dWqkv=[z(3 * d3, h) for _ in range(N)], dbqkv=[z(3 * d3) for _ in range(N)],
                 dWo=[z(h, d3) for _ in range(N)], dW=[z(n, h) for _ in range(N)],
                 da=[z(n) for _ in range(N)], dU=[z(h, n) for _ in range(N)])
    dx = torch.empty_like(x)
    tp.tp_transformer_layer_bwd(c, params, x, saved, dout, dx, grads, ws)
    assert tp.tp_get_status() == tp.TP_OK
    return out, saved, dx, grads


def oracle_layer(cfg, inp):
    P = dict(g1=f64(inp["g1"]), b1=f64(inp["b1"]), g2=f64(inp["g2"]), b2=f64(inp["b2"]),
             Wqkv=f64_list(inp["Wqkv"]), bqkv=f64_list(inp["bqkv"]), Wo=f64_list(inp["Wo"]),
             bo=f64(inp["bo"]), W=f64_list(inp["W"]), a=f64_list(inp["a"]), U=f64_list(inp["U"]),
             b=f64(inp["b"]))
    oc = dict(s=cfg["s"], n_heads=cfg["n_heads"], N=cfg["N"], causal=cfg["causal"], eps=cfg["eps"],
              p_attn=f32p(cfg["p_attn"]), p_hidden=f32p(cfg["p_hidden"]), seed=cfg["seed"],
              layer=cfg["layer"])
    out, sv = O.transformer_layer_fwd(f64(inp["x"]), P, oc)
    g = O.transformer_layer_bwd(f64(inp["dout"]), sv, P, oc)
    return out, sv, g


def check_layer(cfg, inp):
    # Only ln1 is computed from the layer's input alone; every later tensor is
    # computed from saved bf16 activations (ln1, QKV, P, C, h1, ln2, Z, Y, dZ),
    # so for those the element-wise measure is reported, not asserted.
    out, saved, dx, grads = run_layer(cfg, inp)
    rout, rsv, rg = oracle_layer(cfg, inp)
    for k in ("ln1", "QKV", "C", "h1", "ln2"):
        assert_close(saved[k], rsv[k], "bf16", k, elementwise=(k == "ln1"))
    assert_close(out, rout, "bf16", "out", elementwise=False)
    assert_close(dx, rg["dx"], "bf16", "dx", elementwise=False)
    for k in ("dg1", "db1", "dg2", "db2", "dbo", "db"):
        assert_close(grads[k], rg[k], "bf16", k, elementwise=False)
    for k in ("dWqkv", "dbqkv", "dWo", "dW", "da", "dU"):
        for i, (a, r) in enumerate(zip(grads[k], rg[k])):
            assert_close(a, r, "bf16", f"{k}[{i}]", elementwise=False)


SMALL = dict(s=128, h=256, hp=1024, n_heads=4, N=2, causal=True, eps=1e-5, p_attn=0.1, p_hidden=0.1,
             layer=2, seed=1008)


def test_layer_parity_small_with_dropout():
    cfg = dict(SMALL)
    check_layer(cfg, SI.layer_inputs(dict(cfg, b=2)))


def test_layer_parity_no_dropout_one_shard():
    cfg = dict(SMALL, p_attn=0.0, p_hidden=0.0, N=1, n_heads=2, s=96, layer=0)
    check_layer(cfg, SI.layer_inputs(dict(cfg, b=2)))


def test_layer_parity_s40_hidden_dropout_only():
    """Three sequences of 40 tokens: every sequence ends inside a tile;
    attention dropout off (it needs s % 16 == 0), hidden dropout on."""
    cfg = dict(SMALL, s=40, p_attn=0.0, p_hidden=0.1, layer=3)
    check_layer(cfg, SI.layer_inputs(dict(cfg, b=3)))


def test_layer_parity_rows_wider_than_4096():
    """LayerNorm's widest layout (32 values per thread) on a ragged width:
    h = 4608 leaves the last column group partly past the row; 9 heads of 512
    over 3 shards, one sequence of 64 tokens, both dropouts on."""
    cfg = dict(SMALL, s=64, h=4608, hp=4608, n_heads=9, N=3, layer=4)
    check_layer(cfg, SI.layer_inputs(dict(cfg, b=1)))


def test_layer_parity_widest_rows_8192():
    """The widest rows the layer accepts (h = 8192, 16 heads of 512 over 2
    shards), one sequence of 32 tokens."""
    cfg = dict(SMALL, s=32, h=8192, hp=8192, n_heads=16, N=2, layer=5)
    check_layer(cfg, SI.layer_inputs(dict(cfg, b=1)))


def test_layer_deterministic():
    cfg = dict(SMALL)
    inp = SI.layer_inputs(dict(cfg, b=1))
    a, b = run_layer(cfg, inp), run_layer(cfg, inp)
    assert torch.equal(a[0], b[0]) and torch.equal(a[2], b[2])
    for k in a[3]:
        x, y = a[3][k], b[3][k]
        if isinstance(x, list):
            assert all(torch.equal(u, v) for u, v in zip(x, y))
        else:
            assert torch.equal(x, y)


def test_layer_b1_s2048_h4096_heads8_hp16384_N8_full():
    """The layer at the H=4096 model's shapes (one sequence of 2048 tokens),
    every output and gradient against the oracle."""
    cfg = SI.WORKLOADS["layer_b1_s2048_h4096_heads8_hp16384_N8"]
    check_layer(cfg, SI.layer_inputs(cfg))


@pytest.mark.parametrize("mode", [0, 1])
def test_attn_core_dropout_non_causal_both_kernels(mode):
    tp = _tp()
    b, s, h, H, N, p, seed, layer = 1, 512, 512, 4, 4, 0.3, 5, 1
    T = b * s
    QKV = SI.normal(23, 1, (T, 3 * h), 1.0, "bf16")
    dC = SI.normal(23, 2, (T, h), 1.0, "bf16")
    P = torch.empty(b, H, s, s, dtype=torch.bfloat16, device="cuda")
    Pd, C = torch.empty_like(P), torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    dQKV = torch.empty(T, 3 * h, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(tp.tp_attn_core_workspace_size(T, s, h, H), dtype=torch.uint8, device="cuda")
    tp.tp_debug_set_gemm_kernel(mode)
    try:
        tp.tp_attn_core_dropout_fwd(QKV.cuda(), s, H, N, False, p, seed, tp.layer_stream(layer, 0), P, Pd, C,
                                    None, ws)
        tp.tp_attn_core_dropout_bwd(QKV.cuda(), P, Pd, C, dC.cuda(), s, H, N, False, p, seed,
                                    tp.layer_stream(layer, 0), dQKV, ws)
        assert tp.tp_get_status() == tp.TP_OK
    finally:
        tp.tp_debug_set_gemm_kernel(2)
    Qn = f64(QKV)
    rC, rP = O.attention_core(Qn, s, H, N, False, f32p(p), seed, layer)
    assert_close(C, rC, "bf16", "C", elementwise=False)  # sums products of the bf16 P
    rd = O.attention_core_grad(Qn, rP, f64(dC), s, H, N, f32p(p), seed, layer)
    assert_close(dQKV, rd, "bf16", "dQKV", elementwise=False)
    Pdn = Pd.float().cpu().numpy()
    for j in range(H):
        assert np.array_equal(Pdn[0, j] != 0, O.attention_keep(0, j, s, H, N, f32p(p), seed, layer))


def test_layer_one_head_per_shard_three_sequences():
    cfg = dict(SMALL, n_heads=8, N=8, s=64, h=512, hp=1024, layer=5)
    check_layer(cfg, SI.layer_inputs(dict(cfg, b=3)))


def test_layer_gradients_accumulate():
    tp = _tp()
    cfg = dict(SMALL, s=64)
    inp = SI.layer_inputs(dict(cfg, b=1))
    out, saved, dx, grads = run_layer(cfg, inp)
    # run the backward again adding into the same gradient buffers: every gradient doubles
    c = dict(cfg, T=inp["T"])
    d = lambda t: t.cuda().contiguous()
    params = dict(g1=d(inp["g1"]), b1=d(inp["b1"]), g2=d(inp["g2"]), b2=d(inp["b2"]),
                  Wqkv=[d(t) for t in inp["Wqkv"]], bqkv=[d(t) for t in inp["bqkv"]],
                  Wo=[d(t) for t in inp["Wo"]], bo=d(inp["bo"]), W=[d(t) for t in inp["W"]],
                  a=[d(t) for t in inp["a"]], U=[d(t) for t in inp["U"]], b=d(inp["b"]))
    before = {k: ([t.clone() for t in v] if isinstance(v, list) else v.clone()) for k, v in grads.items()}
    ws = torch.empty(tp.tp_transformer_layer_workspace_size(c), dtype=torch.uint8, device="cuda")
    dx2 = torch.empty_like(dx)
    tp.tp_transformer_layer_bwd(c, params, d(inp["x"]), saved, d(inp["dout"]), dx2, grads, ws, accumulate=True)
    assert tp.tp_get_status() == tp.TP_OK
    assert torch.equal(dx, dx2)
    for k, v in grads.items():
        pairs = zip(v, before[k]) if isinstance(v, list) else [(v, before[k])]
        for a, b in pairs:
            assert torch.allclose(a, 2 * b, rtol=1e-5, atol=1e-6), k


def test_layer_saved_keep_words_bit_exact():
    """The keep words the forward saves are the oracle's attention-dropout
    flags bit for bit: 32 keys per word, every word whose first key is at or
    before the query drawn in full, the later words zero, and the keys past s
    of a row's last word zero (s = 48: a half-filled last word)."""
    cfg = dict(SMALL, s=48)
    inp = SI.layer_inputs(dict(cfg, b=2))
    _, saved, _, _ = run_layer(cfg, inp, keep_buffer=True)
    s, H, N, p, seed, layer = cfg["s"], cfg["n_heads"], cfg["N"], cfg["p_attn"], cfg["seed"], cfg["layer"]
    wpr = (s + 31) // 32
    words = saved["attn_keep"].cpu().numpy().view(np.uint32).reshape(-1, H, s, wpr)
    for bi in range(words.shape[0]):
        for j in range(H):
            keep = O.attention_keep(bi, j, s, H, N, f32p(p), seed, layer)
            want = np.zeros((s, wpr), dtype=np.uint32)
            for q in range(s):
                for w in range(wpr):
                    if 32 * w > q:
                        continue
                    for k in range(min(32, s - 32 * w)):
                        want[q, w] |= np.uint32(int(keep[q, 32 * w + k]) << k)
            assert np.array_equal(words[bi, j], want), (bi, j)


def test_layer_saved_keep_words_match_redrawn():
    """Keeping the attention-dropout bits from the forward gives the same
    results as drawing them again in the backward."""
    cfg = dict(SMALL)
    inp = SI.layer_inputs(dict(cfg, b=2))
    a, b = run_layer(cfg, inp), run_layer(cfg, inp, keep_buffer=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[2], b[2])
    for k in a[3]:
        x, y = a[3][k], b[3][k]
        if isinstance(x, list):
            assert all(torch.equal(u, v) for u, v in zip(x, y))
        else:
            assert torch.equal(x, y)
