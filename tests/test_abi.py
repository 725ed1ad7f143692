"""Host-side tests of the C ABI (no GPU needed): the library loads, exports
every entry point include/tp.h declares, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import megatron_tensor_transformer_tp_gb300 as tp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "tp.h")).read()
    return re.findall(r"^TP_API\s+[\w\s\*]+?\b(\w+)\s*\(", src, flags=re.M)


def test_library_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 17
    L = ctypes.CDLL(tp.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    # and the binding exposes the same names
    assert all(hasattr(tp, n) for n in names)


def test_status_strings():
    for code, name in [(tp.TP_OK, "TP_OK"), (tp.TP_ERR_TIMEOUT, "TP_ERR_TIMEOUT"),
                       (tp.TP_ERR_ALIGN, "TP_ERR_ALIGN"), (tp.TP_ERR_WORKSPACE, "TP_ERR_WORKSPACE")]:
        assert tp.tp_status_string(code) == name


def test_workspace_sizes():
    ws = tp.tied_embed_grad_workspace_size(8192, 50257)
    assert ws >= 4 * (50257 + 1) + 4 * 8192 + 4 * 50257


L = tp.lib()
FAKE = 0x100000  # never dereferenced: every case below fails validation first


def ptrs(n, base=FAKE):
    arr = (ctypes.c_void_p * n)(*[base + 4096 * i for i in range(n)])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def mlp_fwd(dt=tp.TP_BF16, M=128, h=64, hp=256, N=2, X=FAKE, wbase=FAKE, null_w=False):
    w = ptrs(N, wbase)
    u = ptrs(N)
    return L.tp_mlp_fwd(dt, M, h, hp, N, X, None if null_w else w[0], None, u[0], None,
                        FAKE, FAKE, FAKE, None)


def test_mlp_fwd_validation():
    assert mlp_fwd(N=0) == tp.TP_ERR_INVALID
    assert mlp_fwd(N=9) == tp.TP_ERR_INVALID
    assert mlp_fwd(hp=255, N=2) == tp.TP_ERR_INVALID       # h' % N != 0
    assert mlp_fwd(M=-1) == tp.TP_ERR_INVALID
    assert mlp_fwd(dt=7) == tp.TP_ERR_UNSUPPORTED
    assert mlp_fwd(null_w=True) == tp.TP_ERR_INVALID
    assert mlp_fwd(X=FAKE + 2) == tp.TP_ERR_ALIGN           # bf16 TMA operand off 16 B
    assert mlp_fwd(h=60) == tp.TP_ERR_ALIGN                 # pitch not a multiple of 8
    assert mlp_fwd(M=0) == tp.TP_OK                         # nothing to do


def test_mlp_bwd_validation():
    w, u, dw, du, da = ptrs(2), ptrs(2), ptrs(2), ptrs(2), ptrs(2)
    # a null shard in dW
    bad = (ctypes.c_void_p * 2)(FAKE, None)
    badp = ctypes.cast(bad, ctypes.POINTER(ctypes.c_void_p))
    st = L.tp_mlp_bwd(tp.TP_BF16, 128, 64, 256, 2, FAKE, FAKE, w[0], u[0], FAKE, FAKE, FAKE, FAKE,
                      badp, da[0], du[0], FAKE, 0, None)
    assert st == tp.TP_ERR_INVALID
    # misaligned dOut
    st = L.tp_mlp_bwd(tp.TP_BF16, 128, 64, 256, 2, FAKE + 8, FAKE, w[0], u[0], FAKE, FAKE, FAKE, FAKE,
                      dw[0], da[0], du[0], FAKE, 0, None)
    assert st == tp.TP_ERR_ALIGN


def test_attn_validation():
    w, o = ptrs(8), ptrs(8)
    # heads not divisible by shards
    assert L.tp_attn_proj_fwd(tp.TP_BF16, 64, 4096, 6, 4, FAKE, w[0], None, FAKE, o[0], None, FAKE,
                              FAKE, None) == tp.TP_ERR_INVALID
    # hidden not divisible by heads
    assert L.tp_attn_proj_fwd(tp.TP_BF16, 64, 4100, 8, 8, FAKE, w[0], None, FAKE, o[0], None, FAKE,
                              FAKE, None) == tp.TP_ERR_INVALID


def rs_arr(vals):
    return (ctypes.c_int64 * len(vals))(*vals)


def test_vocab_ranges_validation():
    e = ptrs(2)
    bad = [[1, 150, 300], [0, 150, 299], [0, 150, 150, 300], [0, 200, 100]]
    for r in bad:
        n = len(r) - 1
        ee = ptrs(n)
        assert L.vocab_parallel_embed(tp.TP_F32, 4, 16, 300, n, FAKE, ee[0], rs_arr(r), FAKE,
                                      None) == tp.TP_ERR_INVALID
    assert L.vocab_parallel_embed(tp.TP_F32, 0, 16, 300, 2, None, e[0], rs_arr([0, 150, 300]), None,
                                  None) == tp.TP_OK


def test_tied_grad_workspace_and_pitch_checked():
    e, d = ptrs(2), ptrs(2)
    rs = rs_arr([0, 25129, 50257])
    ld = rs_arr([25136, 25128])
    assert L.tied_embed_grad(tp.TP_BF16, 8192, 4096, 50257, 2, FAKE, FAKE, FAKE, d[0], ld, rs, e[0],
                             0, None, 0, None) == tp.TP_ERR_WORKSPACE
    short = rs_arr([25128, 25128])  # pitch below the range width
    assert L.tied_embed_grad(tp.TP_BF16, 8192, 4096, 50257, 2, FAKE, FAKE, FAKE, d[0], short, rs, e[0],
                             0, FAKE, 1 << 30, None) == tp.TP_ERR_INVALID


def test_logits_pitch_rule():
    import torch
    assert tp.logits_pitch(25129, torch.bfloat16) == 25136
    assert tp.logits_pitch(25128, torch.bfloat16) == 25128
    assert tp.logits_pitch(150, torch.float32) == 152


def test_cross_entropy_validation_and_workspace_size():
    e = ptrs(2)
    rs = rs_arr([0, 100, 250])
    T, V = 64, 250
    need = tp.tp_vocab_cross_entropy_workspace_size(T, V, [0, 100, 250])
    # (max, sum) pairs for ceil(100/64) + ceil(150/64) = 5 parts per row, plus a
    # target logit per row, each block rounded up to 256 bytes
    assert need == (5 * T * 8 + 255) // 256 * 256 + (T * 4 + 255) // 256 * 256
    assert tp.tp_vocab_cross_entropy_workspace_size(T, V, [0, 100, 251]) == 0  # bad ranges

    def fwd(dt=tp.TP_BF16, ws=FAKE, nbytes=need, V=V, rs=rs):
        return L.tp_vocab_cross_entropy_fwd(dt, T, 64, V, 2, FAKE, e[0], rs, FAKE, FAKE, FAKE,
                                            ws, nbytes, None)
    assert fwd(dt=tp.TP_F32) == tp.TP_ERR_UNSUPPORTED
    assert fwd(ws=None) == tp.TP_ERR_WORKSPACE
    assert fwd(nbytes=need - 1) == tp.TP_ERR_WORKSPACE
    assert fwd(ws=FAKE + 16) == tp.TP_ERR_ALIGN
    assert fwd(V=251) == tp.TP_ERR_INVALID
    ld = rs_arr([104, 152])
    assert L.tp_vocab_cross_entropy_bwd(tp.TP_F32, T, 64, V, 2, FAKE, e[0], rs, FAKE, FAKE, FAKE,
                                        e[0], ld, None, None) == tp.TP_ERR_UNSUPPORTED
    short = rs_arr([104, 144])  # pitch below the second range's width
    assert L.tp_vocab_cross_entropy_bwd(tp.TP_BF16, T, 64, V, 2, FAKE, e[0], rs, FAKE, FAKE, FAKE,
                                        e[0], short, None, None) == tp.TP_ERR_INVALID
