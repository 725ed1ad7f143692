"""The library's calls are CUDA-graph capturable: a captured and replayed
MLP step and transformer-layer step give bit-identical results to the same
calls made eagerly (every reduction has a fixed order, and the per-launch
scheduler counters reset themselves at the end of each launch)."""
import pytest
import torch

import synthetic_inputs as SI

pytestmark = pytest.mark.gpu


def _tp():
    import megatron_tensor_transformer_tp_gb300 as tp
    return tp


def graph_equals_eager(step, outputs):
    step()  # eager (also does the one-time device setup outside the capture)
    torch.cuda.synchronize()
    ref = [t.clone() for t in outputs]
    for t in outputs:
        t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        for t in outputs:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(outputs, ref):
            assert torch.equal(a, b)
    tp = _tp()
    assert tp.tp_get_status() == tp.TP_OK


def test_mlp_step_in_cuda_graph():
    tp = _tp()
    cfg = dict(SI.WORKLOADS["mlp_b4_s1024_h1024_hp4096_N4"], b=1, s=512)
    inp = SI.mlp_inputs(cfg)
    d = lambda t: t.cuda().contiguous()
    M, h, hp, N = inp["M"], inp["h"], inp["hp"], inp["N"]
    X, dOut = d(inp["X"]), d(inp["dOut"])
    W, U, a = [d(t) for t in inp["W_shards"]], [d(t) for t in inp["U_shards"]], [d(t) for t in inp["a_shards"]]
    bias = d(inp["b"])
    bf, f = torch.bfloat16, torch.float32
    Z, Y = torch.empty(M, hp, dtype=bf, device="cuda"), torch.empty(M, hp, dtype=bf, device="cuda")
    Out, dZ = torch.empty(M, h, dtype=bf, device="cuda"), torch.empty(M, hp, dtype=bf, device="cuda")
    dX = torch.empty(M, h, dtype=bf, device="cuda")
    dW = [torch.empty(hp // N, h, dtype=f, device="cuda") for _ in range(N)]
    dU = [torch.empty(h, hp // N, dtype=f, device="cuda") for _ in range(N)]
    da = [torch.empty(hp // N, dtype=f, device="cuda") for _ in range(N)]
    db = torch.empty(h, dtype=f, device="cuda")

    def step():
        tp.tp_mlp_fwd(X, W, a, U, bias, Z, Y, Out)
        tp.tp_mlp_bwd(dOut, X, W, U, Z, Y, dZ, dX, dW, da, dU, db)

    graph_equals_eager(step, [Out, dX, db] + dW + dU)


def test_layer_step_in_cuda_graph():
    tp = _tp()
    cfg = dict(s=128, h=256, hp=1024, n_heads=4, N=2, causal=True, eps=1e-5, p_attn=0.1, p_hidden=0.1,
               layer=1, seed=3, b=2)
    inp = SI.layer_inputs(cfg)
    T, h, hp, N, H, s = inp["T"], cfg["h"], cfg["hp"], cfg["N"], cfg["n_heads"], cfg["s"]
    c = dict(cfg, T=T)
    d = lambda t: t.cuda().contiguous()
    params = dict(g1=d(inp["g1"]), b1=d(inp["b1"]), g2=d(inp["g2"]), b2=d(inp["b2"]),
                  Wqkv=[d(t) for t in inp["Wqkv"]], bqkv=[d(t) for t in inp["bqkv"]],
                  Wo=[d(t) for t in inp["Wo"]], bo=d(inp["bo"]), W=[d(t) for t in inp["W"]],
                  a=[d(t) for t in inp["a"]], U=[d(t) for t in inp["U"]], b=d(inp["b"]))
    bf, f32 = torch.bfloat16, torch.float32
    e = lambda *shape, dt=bf: torch.empty(*shape, dtype=dt, device="cuda")
    b = T // s
    saved = dict(ln1=e(T, h), mean1=e(T, dt=f32), rstd1=e(T, dt=f32), QKV=e(T, 3 * h), P=e(b, H, s, s),
                 Pd=e(b, H, s, s), C=e(T, h), h1=e(T, h), ln2=e(T, h), mean2=e(T, dt=f32),
                 rstd2=e(T, dt=f32), Z=e(T, hp), Y=e(T, hp))
    d3, n = h // N, hp // N
    grads = dict(dg1=e(h, dt=f32), db1=e(h, dt=f32), dg2=e(h, dt=f32), db2=e(h, dt=f32), dbo=e(h, dt=f32),
                 db=e(h, dt=f32), dWqkv=[e(3 * d3, h, dt=f32) for _ in range(N)],
                 dbqkv=[e(3 * d3, dt=f32) for _ in range(N)], dWo=[e(h, d3, dt=f32) for _ in range(N)],
                 dW=[e(n, h, dt=f32) for _ in range(N)], da=[e(n, dt=f32) for _ in range(N)],
                 dU=[e(h, n, dt=f32) for _ in range(N)])
    x, dout = d(inp["x"]), d(inp["dout"])
    out, dx = torch.empty_like(x), torch.empty_like(x)
    ws = torch.empty(tp.tp_transformer_layer_workspace_size(c), dtype=torch.uint8, device="cuda")

    def step():
        tp.tp_transformer_layer_fwd(c, params, x, out, saved, ws)
        tp.tp_transformer_layer_bwd(c, params, x, saved, dout, dx, grads, ws)

    graph_equals_eager(step, [out, dx, grads["dg1"], grads["db2"]] + grads["dWqkv"] + grads["dW"])
