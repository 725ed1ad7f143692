"""The one-SM tensor-core kernel (128 x 256 tiles), selected explicitly.

The library uses the two-SM kernel (CTA pairs, 256 x 256 tiles) by default;
every other GPU test runs on it.  These cases run the MLP, attention and
tied-gradient paths once more on the one-SM kernel.
"""
import pytest

import synthetic_inputs as SI
from tests import test_gpu_attn as A
from tests import test_gpu_embed as E
from tests import test_gpu_mlp as Mt

pytestmark = pytest.mark.gpu


@pytest.fixture
def one_sm():
    import megatron_tensor_transformer_tp_gb300 as tp
    tp.tp_debug_set_gemm_kernel(0)
    yield
    tp.tp_debug_set_gemm_kernel(1)


def test_mlp_one_sm(one_sm):
    cfg = dict(kind="mlp", dtype="bf16", b=1, s=300, h=320, hp=1536, N=3, seed=77)
    inp = SI.mlp_inputs(cfg, bias_std=0.2)
    Mt.check_full(inp, Mt.run_mlp(inp), "bf16")


def test_mlp_b4_s1024_one_sm(one_sm):
    Mt._sampled_check("mlp_b4_s1024_h1024_hp4096_N4")


def test_attn_one_sm(one_sm):
    A.test_attn_small_full_parity("bf16", 300, 512, 8, 4)


def test_tied_grad_one_sm(one_sm):
    E.test_tied_grad_small_full("bf16", 1000, 136, 777, [0, 333, 1000])
