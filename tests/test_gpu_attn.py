"""GPU parity of the head-split attention projections against the fp64
oracle, through the C ABI (tp_attn_proj_fwd / tp_attn_proj_bwd)."""
import numpy as np
import pytest
import torch

import oracle.tp_oracle as O
import synthetic_inputs as SI
from tests.gpu_util import assert_close, dev, dev_list, f64, f64_list

pytestmark = pytest.mark.gpu


def run_attn(inp, bias=True):
    import megatron_tensor_transformer_tp_gb300 as tp
    M, h, N, nh = inp["M"], inp["h"], inp["N"], inp["n_heads"]
    dt = torch.bfloat16 if inp["dtype"] == "bf16" else torch.float32
    X, C, dQKV, dO = dev(inp["X"]), dev(inp["C"]), dev(inp["dQKV"]), dev(inp["dO"])
    Wq, Wo = dev_list(inp["Wqkv_shards"]), dev_list(inp["Wo_shards"])
    bq = dev_list(inp["bqkv_shards"]) if bias else None
    bo = dev(inp["bo"]) if bias else None
    QKV = torch.empty(M, 3 * h, dtype=dt, device="cuda")
    Oo = torch.empty(M, h, dtype=dt, device="cuda")
    tp.tp_attn_proj_fwd(X, Wq, bq, C, Wo, bo, QKV, Oo, nh)
    d = h // N
    f = torch.float32
    dX = torch.empty(M, h, dtype=dt, device="cuda")
    dC = torch.empty(M, h, dtype=dt, device="cuda")
    dWq = [torch.full((3 * d, h), float("nan"), dtype=f, device="cuda") for _ in range(N)]
    dWo = [torch.full((h, d), float("nan"), dtype=f, device="cuda") for _ in range(N)]
    dbq = [torch.full((3 * d,), float("nan"), dtype=f, device="cuda") for _ in range(N)] if bias else None
    dbo = torch.full((h,), float("nan"), dtype=f, device="cuda") if bias else None
    tp.tp_attn_proj_bwd(dQKV, dO, X, C, Wq, Wo, dX, dC, dWq, dbq, dWo, dbo, nh)
    assert tp.tp_get_status() == tp.TP_OK
    return dict(QKV=QKV, O=Oo, dX=dX, dC=dC, dWqkv=dWq, dbqkv=dbq, dWo=dWo, dbo=dbo)


@pytest.mark.parametrize("dtype,M,h,nh,N", [("f32", 37, 64, 4, 2), ("bf16", 300, 512, 8, 4),
                                            ("bf16", 129, 256, 4, 1), ("bf16", 64, 1024, 8, 8)])
def test_attn_small_full_parity(dtype, M, h, nh, N):
    cfg = dict(kind="attn", dtype=dtype, b=1, s=M, h=h, n_heads=nh, N=N, seed=90)
    inp = SI.attn_inputs(cfg, bias_std=0.3)
    res = run_attn(inp)
    X, C, dQKV, dO = f64(inp["X"]), f64(inp["C"]), f64(inp["dQKV"]), f64(inp["dO"])
    Ws, Wos, bs = f64_list(inp["Wqkv_shards"]), f64_list(inp["Wo_shards"]), f64_list(inp["bqkv_shards"])
    QKV, Oo = O.attn_proj_fwd(X, Ws, bs, C, Wos, f64(inp["bo"]))
    assert_close(res["QKV"], QKV, dtype, "QKV")
    assert_close(res["O"], Oo, dtype, "O")
    g = O.attn_proj_bwd(dQKV, dO, X, C, Ws, Wos)
    assert_close(res["dX"], g["dX"], dtype, "dX")
    assert_close(res["dC"], g["dC"], dtype, "dC")
    assert_close(res["dbo"], g["dbo"], dtype, "dbo")
    for i in range(N):
        assert_close(res["dWqkv"][i], g["dWqkv"][i], dtype, f"dWqkv[{i}]")
        assert_close(res["dWo"][i], g["dWo"][i], dtype, f"dWo[{i}]")
        assert_close(res["dbqkv"][i], g["dbqkv"][i], dtype, f"dbqkv[{i}]")


def test_attn_b1_s2048_h4096_heads8_N8_sampled():
    inp = SI.attn_inputs(SI.WORKLOADS["attn_b1_s2048_h4096_heads8_N8"])
    res = run_attn(inp)
    M, h, N = inp["M"], inp["h"], inp["N"]
    d = h // N
    rng = np.random.default_rng(6)
    rows = np.sort(rng.choice(M, 40, replace=False)).tolist() + [M - 1]
    X, C, dQKV, dO = f64(inp["X"]), f64(inp["C"]), f64(inp["dQKV"]), f64(inp["dO"])
    Ws, Wos, bs = f64_list(inp["Wqkv_shards"]), f64_list(inp["Wo_shards"]), f64_list(inp["bqkv_shards"])
    QKV, Oo = O.attn_proj_fwd(X[rows], Ws, bs, C[rows], Wos, f64(inp["bo"]))
    assert_close(res["QKV"][rows], QKV, "bf16", "QKV rows")
    assert_close(res["O"][rows], Oo, "bf16", "O rows")
    g = O.attn_proj_bwd(dQKV[rows], dO[rows], X[rows], C[rows], Ws, Wos)
    assert_close(res["dX"][rows], g["dX"], "bf16", "dX rows")
    assert_close(res["dC"][rows], g["dC"], "bf16", "dC rows")
    # weight gradients contract over all tokens: sample output rows
    qrows = [rng.choice(3 * d, 5, replace=False).tolist() for _ in range(N)]
    orows = [rng.choice(h, 5, replace=False).tolist() for _ in range(N)]
    gwq, gwo, gbq, gbo = O.attn_proj_bwd_weight_rows(dQKV, dO, X, C, N, qrows, orows)
    for i in range(N):
        assert_close(res["dWqkv"][i][qrows[i]], gwq[i], "bf16", f"dWqkv[{i}] rows")
        assert_close(res["dWo"][i][orows[i]], gwo[i], "bf16", f"dWo[{i}] rows")
        assert_close(res["dbqkv"][i], gbq[i], "bf16", f"dbqkv[{i}]")
    assert_close(res["dbo"], gbo, "bf16", "dbo")
