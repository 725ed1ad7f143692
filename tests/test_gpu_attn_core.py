"""GPU parity of the attention core (tp_attn_core_fwd / _bwd) against the fp64
oracle, through the C ABI.

Inputs are bf16 (QKV, dC), accumulation fp32, outputs bf16 (P, C, dQKV):
held to the bf16 bar (2e-2 max relative error).  Both GEMM kernels (one-SM
128-row tiles and two-SM 256-row tiles) are run, since the causal tile
ranges depend on the tile height.
"""
import numpy as np
import pytest
import torch

import oracle.tp_oracle as O
import synthetic_inputs as SI
from tests.gpu_util import assert_close, f64

pytestmark = pytest.mark.gpu


def _tp():
    import megatron_tensor_transformer_tp_gb300 as tp
    return tp


def run_core(QKV, dC, s, n_heads, N, causal, with_bwd=True):
    tp = _tp()
    T, h3 = QKV.shape
    h = h3 // 3
    b = T // s
    Q = QKV.cuda().contiguous()
    P = torch.full((b, n_heads, s, s), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = torch.full((T, h), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((b, n_heads, s), float("nan"), device="cuda")
    ws = torch.empty(tp.tp_attn_core_workspace_size(T, s, h, n_heads), dtype=torch.uint8, device="cuda")
    tp.tp_attn_core_fwd(Q, s, n_heads, N, causal, P, C, lse, ws)
    dQKV = None
    if with_bwd:
        dQKV = torch.full((T, h3), float("nan"), dtype=torch.bfloat16, device="cuda")
        tp.tp_attn_core_bwd(Q, P, C, dC.cuda().contiguous(), s, n_heads, N, causal, dQKV, ws)
    assert tp.tp_get_status() == tp.TP_OK
    return P, C, lse, dQKV


def make_case(b, s, h, seed):
    QKV = SI.normal(seed, 1, (b * s, 3 * h), 1.0, "bf16")
    dC = SI.normal(seed, 2, (b * s, h), 1.0, "bf16")
    return QKV, dC


def check(QKV, dC, s, n_heads, N, causal, res):
    P, C, lse, dQKV = res
    Qn = f64(QKV)
    rC, rP = O.attention_core(Qn, s, n_heads, N, causal)
    # C sums products of the saved bf16 P, and dQKV those of the bf16 dS and P:
    # element-wise measure reported, not asserted (see tests/gpu_util.py)
    assert_close(C, rC, "bf16", "C", elementwise=False)
    assert_close(P, rP, "bf16", "P")
    # log-sum-exp: P = exp(S/sqrt(d) - lse) makes every row of P sum to one
    assert torch.isfinite(lse).all()
    if dQKV is not None:
        rd = O.attention_core_grad(Qn, rP, f64(dC), s, n_heads, N)
        assert_close(dQKV, rd, "bf16", "dQKV", elementwise=False)


CASES = [  # b, s, h, heads, N, causal
    (2, 256, 512, 4, 2, True),     # d = 128
    (1, 200, 256, 2, 2, True),     # ragged s (not a multiple of 64)
    (3, 136, 192, 3, 1, False),    # d = 64, three sequences
    (1, 512, 1024, 2, 2, False),   # d = 512
    (1, 8, 64, 1, 1, True),        # one tile
    (1, 384, 512, 8, 8, True),     # one head per shard, eight shards
]


@pytest.mark.parametrize("b,s,h,heads,N,causal", CASES)
def test_attn_core_parity(b, s, h, heads, N, causal):
    QKV, dC = make_case(b, s, h, seed=100 + s + h)
    check(QKV, dC, s, heads, N, causal, run_core(QKV, dC, s, heads, N, causal))


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("causal", [True, False])
def test_attn_core_both_kernels(mode, causal):
    tp = _tp()
    QKV, dC = make_case(2, 640, 512, seed=77)
    tp.tp_debug_set_gemm_kernel(mode)
    try:
        res = run_core(QKV, dC, 640, 4, 2, causal)
    finally:
        tp.tp_debug_set_gemm_kernel(2)
    check(QKV, dC, 640, 4, 2, causal, res)


def test_attn_core_masked_probabilities_are_zero_and_deterministic():
    QKV, dC = make_case(1, 264, 256, seed=5)
    a = run_core(QKV, dC, 264, 2, 1, True)
    b = run_core(QKV, dC, 264, 2, 1, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    P = a[0].float()
    upper = torch.triu(torch.ones(264, 264, dtype=torch.bool, device="cuda"), 1)
    assert (P[:, :, upper] == 0).all()
    assert torch.allclose(P.sum(-1), torch.ones_like(P.sum(-1)), atol=2e-2)


def test_attn_core_b1_s2048_heads8_d512_causal_full():
    """The attention block's shapes (one sequence of 2048 tokens, 8 heads of
    512, one per shard), causal, every output against the oracle."""
    cfg = SI.WORKLOADS["attn_core_b1_s2048_heads8_d512_causal"]
    a = SI.attn_core_inputs(cfg)
    s, H, N = a["s"], a["n_heads"], a["N"]
    check(a["QKV"], a["dC"], s, H, N, True, run_core(a["QKV"], a["dC"], s, H, N, True))
