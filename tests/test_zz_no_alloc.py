"""The allocation-free tied-gradient entry point against the workspace one.

tied_embed_grad_noalloc serves callers that cannot allocate device memory for
a workspace (for example code running under a memory manager that owns every
device allocation, or code that must not call cudaMalloc because it would
synchronise the device).  It keeps its scratch in a fixed static device array
inside the library.  This test calls it through the C ABI twice in a row and
compares each result with tied_embed_grad given a caller workspace, at the
bf16 tolerance used by the other parity tests; it also checks that a size
whose grouping needs more than the fixed scratch is refused.

Kept in a file of its own that pytest collects last, so a run that stops at
the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import synthetic_inputs as SI
from tests.gpu_util import TOL, dev, dev_list, rel_err

pytestmark = pytest.mark.gpu


def _padded(t, tp):
    T, n = t.shape
    buf = torch.zeros(T, tp.logits_pitch(n, t.dtype), dtype=t.dtype, device="cuda")
    buf[:, :n] = t.cuda()
    return buf


def test_noalloc_matches_workspace_entry_point_twice():
    import megatron_tensor_transformer_tp_gb300 as tp
    cfg = dict(kind="embed", dtype="bf16", V=5003, h=256, b=1, s=3001, ranges=[0, 1700, 5003],
               seed=21)
    inp = SI.embed_inputs(cfg)
    T, V, h, rs = inp["T"], inp["V"], inp["h"], inp["ranges"]
    ids = dev(inp["ids"])
    dEmb, X = dev(inp["dEmb"]), dev(inp["X"])
    dL = [_padded(t, tp) for t in inp["dLogits_shards"]]
    widths = [rs[r + 1] - rs[r] for r in range(2)]

    ref = [torch.empty(w, h, device="cuda") for w in widths]
    ws = torch.empty(tp.tied_embed_grad_workspace_size(T, V), dtype=torch.uint8, device="cuda")
    tp.tied_embed_grad(ids, dEmb, X, dL, rs, ref, workspace=ws)
    assert tp.tp_get_status() == tp.TP_OK

    for call in range(2):
        out = [torch.full((w, h), float("nan"), device="cuda") for w in widths]
        tp.tied_embed_grad_noalloc(ids, dEmb, X, dL, rs, out)
        assert tp.tp_get_status() == tp.TP_OK
        for r in range(2):
            e = rel_err(out[r], ref[r].cpu().double().numpy())
            assert e <= TOL["bf16"], f"call {call}, range {r}: relative error {e:.3e}"


def test_noalloc_refuses_sizes_beyond_its_scratch():
    import megatron_tensor_transformer_tp_gb300 as tp
    L = tp.lib()
    fake = (ctypes.c_void_p * 2)(0x100000, 0x200000)
    pp = ctypes.cast(fake, ctypes.POINTER(ctypes.c_void_p))
    rs = (ctypes.c_int64 * 3)(0, 1000000, 2000000)
    ld = (ctypes.c_int64 * 2)(1000000, 1000000)
    st = L.tied_embed_grad_noalloc(tp.TP_BF16, 1 << 20, 64, 2000000, 2, 0x300000, 0x400000,
                                   0x500000, pp, ld, rs, pp, 0, None)
    assert st == tp.TP_ERR_WORKSPACE
