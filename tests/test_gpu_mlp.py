"""GPU parity of the tensor-parallel MLP block against the fp64 oracle,
through the C ABI (tp_mlp_fwd / tp_mlp_bwd)."""
import numpy as np
import pytest
import torch

import oracle.tp_oracle as O
import synthetic_inputs as SI
from tests.gpu_util import assert_close, dev, dev_list, f64, f64_list

pytestmark = pytest.mark.gpu


def _tp():
    import megatron_tensor_transformer_tp_gb300 as tp
    return tp


def run_mlp(inp, bias=True, accumulate=False, grads_init=None):
    tp = _tp()
    M, h, hp, N = inp["M"], inp["h"], inp["hp"], inp["N"]
    dt = torch.bfloat16 if inp["dtype"] == "bf16" else torch.float32
    X, dOut = dev(inp["X"]), dev(inp["dOut"])
    W, U = dev_list(inp["W_shards"]), dev_list(inp["U_shards"])
    a = dev_list(inp["a_shards"]) if bias else None
    b = dev(inp["b"]) if bias else None
    Z = torch.empty(M, hp, dtype=dt, device="cuda")
    Y = torch.empty_like(Z)
    Out = torch.empty(M, h, dtype=dt, device="cuda")
    tp.tp_mlp_fwd(X, W, a, U, b, Z, Y, Out)
    dZ = torch.empty_like(Z)
    dX = torch.empty(M, h, dtype=dt, device="cuda")
    f = torch.float32
    if grads_init is None:
        dW = [torch.full((hp // N, h), float("nan"), dtype=f, device="cuda") for _ in range(N)]
        dU = [torch.full((h, hp // N), float("nan"), dtype=f, device="cuda") for _ in range(N)]
        da = [torch.full((hp // N,), float("nan"), dtype=f, device="cuda") for _ in range(N)] if bias else None
        db = torch.full((h,), float("nan"), dtype=f, device="cuda") if bias else None
    else:
        dW, dU, da, db = grads_init
    tp.tp_mlp_bwd(dOut, X, W, U, Z, Y, dZ, dX, dW, da, dU, db, accumulate=accumulate)
    assert tp.tp_get_status() == tp.TP_OK
    return dict(Z=Z, Y=Y, Out=Out, dZ=dZ, dX=dX, dW=dW, dU=dU, da=da, db=db)


def oracle_full(inp):
    X, dOut = f64(inp["X"]), f64(inp["dOut"])
    W, U, a = f64_list(inp["W_shards"]), f64_list(inp["U_shards"]), f64_list(inp["a_shards"])
    Z, Y, Out = O.mlp_fwd(X, W, a, U, f64(inp["b"]))
    g = O.mlp_bwd(dOut, X, W, a, U)
    return Z, Y, Out, g


# Element-wise bar: Z, Y and db are computed from the inputs alone and are held
# to it.  Out and dU sum products of the saved Y; dZ applies GELU' to the saved
# Z; dX, dW and da sum products of the saved dZ.  The oracle keeps those
# intermediates in fp64: in bf16 the saved values differ from them by up to
# 2^-9 per element, in fp32 by up to 2^-24, and near-zero elements of the sums
# see that as a large relative error (in fp32 the element-wise bar's absolute
# allowance, 1e-4 x 1e-3 max |r|, is about two rounding steps of the largest
# value).  For them the element-wise measure is reported, not asserted.
def check_full(inp, res, dtype):
    Z, Y, Out, g = oracle_full(inp)
    ex = False
    assert_close(res["Z"], Z, dtype, "Z")
    assert_close(res["Y"], Y, dtype, "Y")
    assert_close(res["Out"], Out, dtype, "Out", elementwise=ex)
    assert_close(res["dZ"], g["dZ"], dtype, "dZ", elementwise=ex)
    assert_close(res["dX"], g["dX"], dtype, "dX", elementwise=ex)
    for i in range(inp["N"]):
        assert_close(res["dW"][i], g["dW"][i], dtype, f"dW[{i}]", elementwise=ex)
        assert_close(res["dU"][i], g["dU"][i], dtype, f"dU[{i}]", elementwise=ex)
        if res["da"] is not None:
            assert_close(res["da"][i], g["da"][i], dtype, f"da[{i}]", elementwise=ex)
    if res["db"] is not None:
        assert_close(res["db"], g["db"], dtype, "db")


def test_mlp_tiny_fp32_workload():
    """b=1, s=8, h=64, h'=256, N=2, fp32 (1e-4)."""
    inp = SI.mlp_inputs(SI.WORKLOADS["mlp_tiny_f32"])
    check_full(inp, run_mlp(inp), "f32")


def test_mlp_fp32_nonzero_bias_ragged():
    cfg = dict(SI.WORKLOADS["mlp_tiny_f32"], s=77, h=72, hp=264, N=3)
    inp = SI.mlp_inputs(cfg, bias_std=0.5)
    check_full(inp, run_mlp(inp), "f32")


@pytest.mark.parametrize("M,h,hp,N", [(300, 320, 1536, 3), (128, 256, 512, 1), (1, 64, 128, 2),
                                      (513, 1024, 2048, 8)])
def test_mlp_bf16_tiles_and_ragged_tails(M, h, hp, N):
    cfg = dict(kind="mlp", dtype="bf16", b=1, s=M, h=h, hp=hp, N=N, seed=77)
    inp = SI.mlp_inputs(cfg, bias_std=0.2)
    check_full(inp, run_mlp(inp), "bf16")


def test_mlp_bf16_no_bias_and_accumulate():
    cfg = dict(kind="mlp", dtype="bf16", b=1, s=200, h=256, hp=1024, N=4, seed=78)
    inp = SI.mlp_inputs(cfg)
    res = run_mlp(inp, bias=False)
    Z, Y, Out, g = oracle_full(inp)
    assert_close(res["Out"], Out, "bf16", "Out", elementwise=False)
    # accumulate: start from ones, expect ones + grad
    N, h, hp = inp["N"], inp["h"], inp["hp"]
    f = torch.float32
    init = ([torch.ones(hp // N, h, dtype=f, device="cuda") for _ in range(N)],
            [torch.ones(h, hp // N, dtype=f, device="cuda") for _ in range(N)],
            [torch.ones(hp // N, dtype=f, device="cuda") for _ in range(N)],
            torch.ones(h, dtype=f, device="cuda"))
    res2 = run_mlp(inp, bias=True, accumulate=True, grads_init=init)
    for i in range(N):
        assert_close(res2["dW"][i], g["dW"][i] + 1.0, "bf16", "dW acc", elementwise=False)
        assert_close(res2["dU"][i], g["dU"][i] + 1.0, "bf16", "dU acc", elementwise=False)
        assert_close(res2["da"][i], g["da"][i] + 1.0, "bf16", "da acc", elementwise=False)
    assert_close(res2["db"], g["db"] + 1.0, "bf16", "db acc")


def test_mlp_empty_tokens_zeroes_weight_grads():
    tp = _tp()
    cfg = dict(kind="mlp", dtype="bf16", b=1, s=0, h=64, hp=128, N=2, seed=79)
    inp = SI.mlp_inputs(cfg)
    res = run_mlp(inp)
    for i in range(2):
        assert torch.count_nonzero(res["dW"][i]) == 0 and torch.count_nonzero(res["dU"][i]) == 0
        assert torch.count_nonzero(res["da"][i]) == 0
    assert torch.count_nonzero(res["db"]) == 0
    assert tp.tp_get_status() == tp.TP_OK


def test_mlp_bwd_deterministic():
    cfg = dict(kind="mlp", dtype="bf16", b=1, s=384, h=512, hp=2048, N=4, seed=80)
    inp = SI.mlp_inputs(cfg, bias_std=0.1)
    r1, r2 = run_mlp(inp), run_mlp(inp)
    for k in ("Out", "dX", "db"):
        assert torch.equal(r1[k], r2[k]), k
    for i in range(4):
        assert torch.equal(r1["dW"][i], r2["dW"][i]) and torch.equal(r1["da"][i], r2["da"][i])


def _sampled_check(name):
    cfg = SI.WORKLOADS[name]
    inp = SI.mlp_inputs(cfg)
    res = run_mlp(inp)
    N, hp, M = inp["N"], inp["hp"], inp["M"]
    ns = hp // N
    g = np.random.default_rng(5)
    rows = np.sort(g.choice(M, 48, replace=False)).tolist() + [0, M - 1]
    units = [np.sort(g.choice(ns, 6, replace=False)).tolist() + [ns - 1] for _ in range(N)]
    X, dOut = f64(inp["X"]), f64(inp["dOut"])
    W, U, a = f64_list(inp["W_shards"]), f64_list(inp["U_shards"]), f64_list(inp["a_shards"])
    Zr, Yr, Outr = O.mlp_fwd(X[rows], W, a, U, f64(inp["b"]))
    assert_close(res["Z"][rows], Zr, "bf16", "Z rows")
    assert_close(res["Y"][rows], Yr, "bf16", "Y rows")
    assert_close(res["Out"][rows], Outr, "bf16", "Out rows", elementwise=False)
    s = O.mlp_bwd_sampled(dOut, X, W, a, U, rows, units)
    assert_close(res["dZ"][rows], s["dZ_rows"], "bf16", "dZ rows", elementwise=False)
    assert_close(res["dX"][rows], s["dX_rows"], "bf16", "dX rows", elementwise=False)
    for i, J in enumerate(units):
        assert_close(res["dW"][i][J], s["dW_rows"][i], "bf16", f"dW[{i}] rows", elementwise=False)
        assert_close(res["dU"][i][:, J], s["dU_cols"][i], "bf16", f"dU[{i}] cols", elementwise=False)
        assert_close(res["da"][i][J], s["da"][i], "bf16", f"da[{i}]", elementwise=False)
    assert_close(res["db"], s["db"], "bf16", "db")
    # properties at full size: every output finite
    for k in ("Z", "Y", "Out", "dZ", "dX"):
        assert torch.isfinite(res[k]).all(), k


def test_mlp_b4_s1024_h1024_hp4096_N4_sampled():
    _sampled_check("mlp_b4_s1024_h1024_hp4096_N4")


def test_mlp_b2_s2048_h4096_hp16384_N2_sampled():
    _sampled_check("mlp_b2_s2048_h4096_hp16384_N2")
