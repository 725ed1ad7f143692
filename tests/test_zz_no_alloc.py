"""The allocation-free tied-gradient entry point against the workspace one.

tied_embed_grad_noalloc serves callers that cannot allocate device memory for
a workspace: code running under a memory manager that owns every device
allocation (a serving runtime that reserves HBM up front), or code that must
not call cudaMalloc because it would synchronise the device in the middle of
its stream work.  It keeps its scratch in a fixed 1.5 MiB static device array
inside the library, shared by every call.

Both entry points run the same deterministic grouping and GEMM kernels, so
their results must be bit-identical: any difference means the static scratch
is laid out or reused wrongly.  Each case calls the allocation-free entry
point twice in a row through the C ABI and compares both results with
torch.equal against tied_embed_grad given a caller workspace; one comparison
per case is made against the fp64 oracle as well.  The largest case (a
grouping that fills the scratch up to its limit) runs first, so that a later,
smaller case would see its stale contents if a call failed to clear what must
start at zero.

Kept in a file of its own that pytest collects last, so a run that stops at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.tp_oracle as O
import synthetic_inputs as SI
from tests.gpu_util import assert_close, dev, f64

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 1536 * 1024


def _tp():
    import megatron_tensor_transformer_tp_gb300 as tp
    return tp


def _padded(t, tp):
    T, n = t.shape
    buf = torch.zeros(T, tp.logits_pitch(n, t.dtype), dtype=t.dtype, device="cuda")
    buf[:, :n] = t.cuda()
    return buf


def _grads(widths, h, init):
    if init is None:
        return [torch.full((w, h), float("nan"), device="cuda") for w in widths]
    return [t.clone() for t in init]


def _compare_twice(tp, ids, dEmb, X, dL, rs, h, accumulate=False, init=None):
    """Workspace entry point once, allocation-free entry point twice; every
    result bit-identical.  Returns the workspace result."""
    T, V = ids.numel(), rs[-1]
    widths = [rs[r + 1] - rs[r] for r in range(len(rs) - 1)]
    ref = _grads(widths, h, init)
    ws = torch.empty(tp.tied_embed_grad_workspace_size(T, V), dtype=torch.uint8, device="cuda")
    tp.tied_embed_grad(ids, dEmb, X, dL, rs, ref, accumulate=accumulate, workspace=ws)
    assert tp.tp_get_status() == tp.TP_OK
    for call in range(2):
        out = _grads(widths, h, init)
        tp.tied_embed_grad_noalloc(ids, dEmb, X, dL, rs, out, accumulate=accumulate)
        assert tp.tp_get_status() == tp.TP_OK
        for r in range(len(widths)):
            assert torch.equal(out[r], ref[r]), f"call {call}, range {r} differs from the workspace path"
    return ref


def test_noalloc_at_its_scratch_limit_input_side_only():
    """V = 131072, T = 131008: the grouping needs exactly 1.5 MiB.  dLogits is
    None, so only the input-side scatter runs (the segment-sum kernel)."""
    tp = _tp()
    V, T, h = 131072, 131008, 64
    assert tp.tied_embed_grad_workspace_size(T, V) == SCRATCH_BYTES
    rs = [0, 70001, V]
    ids_h = SI.uniform_ids(31, 1, T, V)
    ids_h[:9] = 5                      # a repeated id
    ids_h[9], ids_h[10] = -1, V        # ids in no range contribute nothing
    dEmb_h = SI.normal(31, 2, (T, h), 1.0, "bf16")
    ref = _compare_twice(tp, dev(ids_h), dev(dEmb_h), None, None, rs, h)
    sc = O.embed_scatter_grad(ids_h.numpy(), f64(dEmb_h), V)
    for r in range(2):
        assert_close(ref[r], sc[rs[r]:rs[r + 1]], "bf16", f"scatter[{r}]")


def test_noalloc_matches_workspace_entry_point_twice():
    """Both contributions (dLogits given), overwrite and accumulate."""
    tp = _tp()
    cfg = dict(kind="embed", dtype="bf16", V=5003, h=256, b=1, s=3001, ranges=[0, 1700, 5003],
               seed=21)
    inp = SI.embed_inputs(cfg)
    V, h, rs = inp["V"], inp["h"], inp["ranges"]
    ids, dEmb, X = dev(inp["ids"]), dev(inp["dEmb"]), dev(inp["X"])
    dL = [_padded(t, tp) for t in inp["dLogits_shards"]]
    ref = _compare_twice(tp, ids, dEmb, X, dL, rs, h)
    dLf = [f64(t) for t in inp["dLogits_shards"]]
    oracle = O.tied_embed_grad(inp["ids"].numpy(), f64(inp["dEmb"]), f64(inp["X"]), dLf, rs, V)
    for r in range(2):
        assert_close(ref[r], oracle[r], "bf16", f"dE[{r}]")
    # accumulate into an existing gradient
    g = torch.Generator().manual_seed(3)
    init = [torch.randn(rs[r + 1] - rs[r], h, generator=g).cuda() for r in range(2)]
    _compare_twice(tp, ids, dEmb, X, dL, rs, h, accumulate=True, init=init)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    tp = _tp()
    L = tp.lib()
    fake = (ctypes.c_void_p * 2)(0x100000, 0x200000)
    pp = ctypes.cast(fake, ctypes.POINTER(ctypes.c_void_p))
    rs = (ctypes.c_int64 * 3)(0, 1000000, 2000000)
    ld = (ctypes.c_int64 * 2)(1000000, 1000000)
    st = L.tied_embed_grad_noalloc(tp.TP_BF16, 1 << 20, 64, 2000000, 2, 0x300000, 0x400000,
                                   0x500000, pp, ld, rs, pp, 0, None)
    assert st == tp.TP_ERR_WORKSPACE
    # one token more than the limit case above
    assert tp.tied_embed_grad_workspace_size(131008 + 64, 131072) > SCRATCH_BYTES
