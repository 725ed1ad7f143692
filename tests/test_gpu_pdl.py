"""Programmatic dependent launch changes when kernels start, not what they
compute: with it on (the default) every kernel still waits on the device for
the previous kernel's completion before it touches memory.  Each case runs a
multi-launch path with it on and off and compares the results bit for bit
(every kernel of the library is deterministic)."""
import pytest
import torch

import synthetic_inputs as SI
from tests import test_gpu_attn_core as AC
from tests import test_gpu_layer as L
from tests import test_gpu_mlp as Mt

pytestmark = pytest.mark.gpu


def _tp():
    import megatron_tensor_transformer_tp_gb300 as tp
    return tp


def _both(fn):
    tp = _tp()
    try:
        tp.tp_debug_set_pdl(False)
        off = fn()
        tp.tp_debug_set_pdl(True)
        on = fn()
    finally:
        tp.tp_debug_set_pdl(True)
    return on, off


def _flat(x):
    if isinstance(x, torch.Tensor):
        return [x]
    if isinstance(x, dict):
        return [t for k in sorted(x) for t in _flat(x[k])]
    if isinstance(x, (list, tuple)):
        return [t for v in x for t in _flat(v)]
    return []


def _assert_equal(on, off):
    a, b = _flat(on), _flat(off)
    assert len(a) == len(b) and a
    for i, (x, y) in enumerate(zip(a, b)):
        assert torch.equal(x, y), f"tensor {i} differs with programmatic dependent launch"


def test_layer_with_dropout_identical_with_and_without_pdl():
    cfg = dict(L.SMALL)
    inp = SI.layer_inputs(dict(cfg, b=2))
    _assert_equal(*_both(lambda: L.run_layer(cfg, inp, keep_buffer=True)))


def test_mlp_identical_with_and_without_pdl():
    """Split into independent and dependent launches (a split threshold of one
    tile per SM), so that GEMM launches follow each other."""
    tp = _tp()
    cfg = dict(kind="mlp", dtype="bf16", b=1, s=2048, h=1024, hp=4096, N=4, seed=78)
    inp = SI.mlp_inputs(cfg, bias_std=0.2)
    tp.tp_debug_set_split_threshold(1)
    try:
        _assert_equal(*_both(lambda: Mt.run_mlp(inp)))
    finally:
        tp.tp_debug_set_split_threshold(0)


def test_attention_core_identical_with_and_without_pdl():
    QKV, dC = AC.make_case(2, 256, 512, 31)
    _assert_equal(*_both(lambda: AC.run_core(QKV, dC, 256, 4, 2, True)))


def test_tied_gradient_identical_with_and_without_pdl():
    """The token grouping's four kernels, then the GEMM with the segment sums."""
    from tests import test_gpu_embed as E
    cfg = dict(kind="embed", dtype="bf16", V=5003, h=256, b=1, s=3001, ranges=[0, 1700, 5003], seed=22)
    inp = SI.embed_inputs(cfg)

    def run():
        dE, ws = E.run_tied(inp)
        offs, perm = E.sort_view(ws, inp["ids"].numel(), inp["V"])  # the grouping's results, not its scratch
        return dE, torch.from_numpy(offs), torch.from_numpy(perm)

    _assert_equal(*_both(run))


def test_cross_entropy_identical_with_and_without_pdl():
    """Statistics GEMM, the reduction kernel, then the gradient GEMM."""
    from tests import test_gpu_ce as C
    X, _, Es, targets, dloss = C.make_case(300, 256, [0, 700, 2048], seed=23)
    _assert_equal(*_both(lambda: C.run_ce(X, Es, [0, 700, 2048], targets, dloss)))


def test_adam_identical_with_and_without_pdl():
    """The norm pass (finalized in its last block), then the update."""
    from tests import test_gpu_opt as Op
    groups = Op.make_groups([70001, 33, 4096])

    def run():
        d = Op.DeviceOpt(groups, Op.STATE)
        st = d.step(Op.HYPER)
        assert st["found_inf"] == 0
        return [[g[k] for k in ("param", "m", "v", "model")] for g in d.g]

    _assert_equal(*_both(run))
