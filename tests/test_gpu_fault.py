"""Failure detection on the GPU without a GPU fault.

Every wait inside the tensor-core GEMM is bounded.  The host can make one
wait run out on purpose: with fault kind 1 the TMA producer of the next GEMM
launch never fills its first pipeline stage, so the consumer's bounded wait
expires, the CTAs wind down (in-flight copies drained, TMEM freed) and the
timeout is recorded in the device error word.  The test checks that the
status reads TP_ERR_TIMEOUT, that the context stays usable, and that the next
call is correct again.
"""
import numpy as np
import pytest
import torch

import oracle.tp_oracle as O
import synthetic_inputs as SI
from tests.gpu_util import assert_close, dev, dev_list, f64, f64_list

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_reports_timeout_and_recovers():
    import megatron_tensor_transformer_tp_gb300 as tp
    cfg = dict(kind="mlp", dtype="bf16", b=1, s=256, h=256, hp=512, N=2, seed=31)
    inp = SI.mlp_inputs(cfg)
    M, h, hp = inp["M"], inp["h"], inp["hp"]
    X = dev(inp["X"])
    W, U = dev_list(inp["W_shards"]), dev_list(inp["U_shards"])
    Z = torch.empty(M, hp, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty_like(Z)
    Out = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    assert tp.tp_get_status() == tp.TP_OK
    try:
        tp.tp_debug_set_wait_limit_ms(100)
        tp.tp_debug_inject_fault(1)
        tp.tp_mlp_fwd(X, W, None, U, None, Z, Y, Out)
        assert tp.tp_get_status() == tp.TP_ERR_TIMEOUT
    finally:
        tp.tp_debug_inject_fault(0)
        tp.tp_debug_set_wait_limit_ms(1000)
    # the status word was cleared and the context still works
    assert tp.tp_get_status() == tp.TP_OK
    x = torch.ones(4, device="cuda") * 2
    assert float(x.sum()) == 8.0
    tp.tp_mlp_fwd(X, W, None, U, None, Z, Y, Out)
    assert tp.tp_get_status() == tp.TP_OK
    _, _, ref = O.mlp_fwd(f64(inp["X"]), f64_list(inp["W_shards"]), None, f64_list(inp["U_shards"]), None)
    assert_close(Out, ref, "bf16", "Out after recovery", elementwise=False)  # sums the bf16 Y
