"""Both tensor-core GEMM kernels, each selected explicitly.

By default the library picks, per launch, the one-SM kernel (128 x 256 tiles)
or the two-SM kernel (CTA pairs, 256 x 256 tiles with tcgen05 cta_group::2);
at the test suite's small sizes it mostly picks the one-SM kernel.  These
cases run the MLP, attention and tied-gradient paths on each kernel, forced.
"""
import pytest

import synthetic_inputs as SI
from tests import test_gpu_attn as A
from tests import test_gpu_embed as E
from tests import test_gpu_mlp as Mt

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[0, 1], ids=["one_sm", "two_sm"])
def kernel(request):
    import megatron_tensor_transformer_tp_gb300 as tp
    tp.tp_debug_set_gemm_kernel(request.param)
    yield request.param
    tp.tp_debug_set_gemm_kernel(2)


@pytest.mark.parametrize("M,h,hp,N", [(300, 320, 1536, 3), (513, 1024, 2048, 8), (1, 64, 128, 2)])
def test_mlp(kernel, M, h, hp, N):
    cfg = dict(kind="mlp", dtype="bf16", b=1, s=M, h=h, hp=hp, N=N, seed=77)
    inp = SI.mlp_inputs(cfg, bias_std=0.2)
    Mt.check_full(inp, Mt.run_mlp(inp), "bf16")


def test_mlp_b4_s1024_sampled(kernel):
    Mt._sampled_check("mlp_b4_s1024_h1024_hp4096_N4")


def test_mlp_empty_tokens(kernel):
    Mt.test_mlp_empty_tokens_zeroes_weight_grads()


def test_attn(kernel):
    A.test_attn_small_full_parity("bf16", 300, 512, 8, 4)


def test_tied_grad(kernel):
    E.test_tied_grad_small_full("bf16", 1000, 136, 777, [0, 333, 1000])


def test_logits(kernel):
    E.test_logits_small_full("bf16", 777, 256, 129, [0, 1, 300, 777])
