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


ADAM_CFG = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, max_norm=1.0, use_scaler=1,
                min_scale=1.0, growth_factor=2.0, backoff_factor=0.5, growth_interval=1000,
                hysteresis=2)


def adam(groups, n, cfg=None, state=FAKE, ws=FAKE, ws_bytes=None):
    c = tp.tp_adam_config(*[(cfg or ADAM_CFG)[k] for k in tp._ADAM_KEYS])
    arr = (tp.tp_param_group * max(1, n))(*groups) if groups is not None else None
    if ws_bytes is None:
        ws_bytes = tp.tp_adam_step_workspace_size()
    return L.tp_adam_step(arr, n, ctypes.byref(c), state, ws, ws_bytes, None)


def group(n=1000, base=FAKE, model=None, **kw):
    g = dict(param=base, grad=base + 16 * 4096, exp_avg=base + 32 * 4096,
             exp_avg_sq=base + 48 * 4096, model_param=model, n=n, weight_decay=0.1)
    g.update(kw)
    return tp.tp_param_group(**g)


def test_adam_step_validation():
    assert tp.tp_adam_step_workspace_size() >= 256
    assert adam(None, 1) == tp.TP_ERR_INVALID                     # groups NULL
    assert adam([group()], -1) == tp.TP_ERR_INVALID
    assert adam([group()] * 65, 65) == tp.TP_ERR_INVALID          # more than 64 groups
    assert adam([group(n=-1)], 1) == tp.TP_ERR_INVALID
    assert adam([group(grad=None)], 1) == tp.TP_ERR_INVALID
    assert adam([group()], 1, state=None) == tp.TP_ERR_INVALID
    assert adam([group()], 1, cfg=dict(ADAM_CFG, beta2=1.0)) == tp.TP_ERR_INVALID
    assert adam([group()], 1, cfg=dict(ADAM_CFG, beta1=-0.1)) == tp.TP_ERR_INVALID
    assert adam([group()], 1, cfg=dict(ADAM_CFG, growth_interval=0)) == tp.TP_ERR_INVALID
    assert adam([group(base=FAKE + 4)], 1) == tp.TP_ERR_ALIGN     # fp32 buffers 16-byte aligned
    assert adam([group(model=FAKE + 2)], 1) == tp.TP_ERR_ALIGN    # bf16 copy 8-byte aligned
    assert adam([group()], 1, state=FAKE + 2) == tp.TP_ERR_ALIGN
    assert adam([group()], 1, ws=None) == tp.TP_ERR_WORKSPACE
    assert adam([group()], 1, ws_bytes=100) == tp.TP_ERR_WORKSPACE
    assert adam([group()], 1, ws=FAKE + 8) == tp.TP_ERR_ALIGN
    # an empty group needs no buffers
    assert adam([group(n=0, param=None, grad=None)], 1, ws=None) == tp.TP_ERR_WORKSPACE


def test_struct_layouts_match_header(tmp_path):
    """The binding's ctypes structures have the C header's sizes and offsets."""
    src = tmp_path / "layout.c"
    fields = {"tp_optimizer_state": tp.tp_optimizer_state, "tp_adam_config": tp.tp_adam_config,
              "tp_param_group": tp.tp_param_group, "tp_layer_config": tp.tp_layer_config,
              "tp_layer_params": tp.tp_layer_params, "tp_layer_saved": tp.tp_layer_saved,
              "tp_layer_grads": tp.tp_layer_grads}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "tp.h"', 'int main(void) {']
    for name, cls in fields.items():
        lines.append(f'printf("{name} %zu\\n", sizeof({name}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{name}.{f} %zu\\n", offsetof({name}, {f}));')
    lines.append("return 0; }")
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    import subprocess
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                  check=True).stdout.splitlines())
    for name, cls in fields.items():
        assert int(out[name]) == ctypes.sizeof(cls), name
        for f, _ in cls._fields_:
            assert int(out[f"{name}.{f}"]) == getattr(cls, f).offset, f"{name}.{f}"


def core(fn="fwd", dt=tp.TP_BF16, T=512, s=256, h=512, heads=4, N=2, ws_bytes=1 << 30, ws=FAKE * 256):
    if fn == "fwd":
        return L.tp_attn_core_fwd(dt, T, s, h, heads, N, 1, FAKE, FAKE, FAKE, None, ws, ws_bytes, None)
    return L.tp_attn_core_bwd(dt, T, s, h, heads, N, 1, FAKE, FAKE, FAKE, FAKE, FAKE, ws, ws_bytes, None)


def test_attn_core_validation_and_workspace_size():
    for fn in ("fwd", "bwd"):
        assert core(fn, dt=tp.TP_F32) == tp.TP_ERR_UNSUPPORTED
        assert core(fn, T=500) == tp.TP_ERR_INVALID             # T not a multiple of s
        assert core(fn, heads=3) == tp.TP_ERR_INVALID           # h % heads
        assert core(fn, heads=2, N=4) == tp.TP_ERR_INVALID      # heads % N
        assert core(fn, N=9, heads=9, h=576) == tp.TP_ERR_INVALID
        assert core(fn, s=252, T=504) == tp.TP_ERR_ALIGN        # s % 8
        assert core(fn, h=40, heads=8, N=2) == tp.TP_ERR_ALIGN  # d = 5
        assert core(fn, ws=None) == tp.TP_ERR_WORKSPACE
        assert core(fn, ws_bytes=1024) == tp.TP_ERR_WORKSPACE
        assert core(fn, ws=FAKE * 256 + 16) == tp.TP_ERR_ALIGN
        assert core(fn, T=0) == tp.TP_OK
    b, H, s = 2, 4, 256
    keep = b * H * s * (s // 32) * 4  # attention-dropout keep words
    fwd = b * H * (s // 64) * s * 8 + b * H * s * 4 + keep
    bwd = b * H * s * 4 + b * H * s * s * 2 + keep
    assert tp.tp_attn_core_workspace_size(512, 256, 512, 4) == max(fwd, bwd)
    assert tp.tp_attn_core_workspace_size(500, 256, 512, 4) == 0


def layer_cfg(**kw):
    c = dict(T=512, s=256, h=512, hp=2048, n_heads=4, N=2, causal=1, eps=1e-5, p_attn=0.1,
             p_hidden=0.1, seed=1, layer=0)
    c.update(kw)
    return tp._layer_cfg(c)


def layer_fwd(cfg, params=None, ws_bytes=None):
    import ctypes as C
    sh = ptrs(2)
    w = params or tp.tp_layer_params(FAKE, FAKE, C.cast(sh[0], C.c_void_p).value, None,
                                     C.cast(sh[0], C.c_void_p).value, None, FAKE, FAKE,
                                     C.cast(sh[0], C.c_void_p).value, None,
                                     C.cast(sh[0], C.c_void_p).value, None)
    sv = tp.tp_layer_saved(*([FAKE] * 14))
    if ws_bytes is None:
        ws_bytes = 1 << 34
    return L.tp_transformer_layer_fwd(C.byref(cfg), C.byref(w), FAKE, FAKE, C.byref(sv), FAKE * 256,
                                      ws_bytes, None), sh


def test_layer_validation():
    assert layer_fwd(layer_cfg(T=500))[0] == tp.TP_ERR_INVALID         # T % s
    assert layer_fwd(layer_cfg(h=520, n_heads=4))[0] == tp.TP_ERR_INVALID  # h % 16
    assert layer_fwd(layer_cfg(p_hidden=1.0))[0] == tp.TP_ERR_INVALID
    assert layer_fwd(layer_cfg(p_attn=0.1, s=200, T=400))[0] == tp.TP_ERR_INVALID  # s % 16 with dropout
    assert layer_fwd(layer_cfg(hp=2047))[0] == tp.TP_ERR_INVALID
    # 16-byte units for the bulk tensor copies, refused before any launch
    assert layer_fwd(layer_cfg(p_attn=0.0, s=45, T=90))[0] == tp.TP_ERR_ALIGN     # P row pitch
    assert layer_fwd(layer_cfg(h=192, n_heads=48, N=2))[0] == tp.TP_ERR_ALIGN    # head width 4
    assert layer_fwd(layer_cfg(hp=2056, N=2))[0] == tp.TP_ERR_ALIGN              # shard width 1028
    assert layer_fwd(layer_cfg(), ws_bytes=16)[0] == tp.TP_ERR_WORKSPACE
    assert layer_fwd(layer_cfg(T=0))[0] == tp.TP_OK
    c = layer_cfg()
    assert L.tp_transformer_layer_workspace_size(ctypes.byref(c)) > 0


def test_position_embed_dropout_validation():
    f = L.tp_position_embed_dropout
    assert f(8, 40, 16, FAKE, FAKE, FAKE, 0.1, 1, 2, FAKE, None) == tp.TP_ERR_INVALID   # h % 16
    assert f(8, 64, 16, FAKE, FAKE, FAKE, 1.5, 1, 2, FAKE, None) == tp.TP_ERR_INVALID
    assert f(8, 64, 16, FAKE + 2, FAKE, FAKE, 0.1, 1, 2, FAKE, None) == tp.TP_ERR_ALIGN
    assert f(0, 64, 16, None, None, None, 0.1, 1, 2, None, None) == tp.TP_OK


def layer_bwd(cfg, ws_bytes=1 << 34, grads_null_shard=False, dout=FAKE):
    """tp_transformer_layer_bwd with fake device pointers and real host shard arrays."""
    import ctypes as C
    sh = ptrs(2)
    vp = lambda a: C.cast(a[0], C.c_void_p).value
    w = tp.tp_layer_params(FAKE, FAKE, vp(sh), None, vp(sh), None, FAKE, FAKE, vp(sh), None, vp(sh), None)
    sv = tp.tp_layer_saved(*([FAKE] * 13 + [None]))
    dsh = ptrs(2)
    bad = (C.c_void_p * 2)(FAKE, None)
    dW = C.cast(bad, C.c_void_p).value if grads_null_shard else vp(dsh)
    g = tp.tp_layer_grads(FAKE, FAKE, vp(dsh), None, vp(dsh), FAKE, FAKE, FAKE, dW, None, vp(dsh), FAKE)
    return L.tp_transformer_layer_bwd(C.byref(cfg), C.byref(w), FAKE, C.byref(sv), dout, FAKE, C.byref(g),
                                      0, FAKE * 256, ws_bytes, None), (sh, dsh, bad)


def test_layer_backward_validation():
    assert layer_bwd(layer_cfg(T=500))[0] == tp.TP_ERR_INVALID                     # T % s
    assert layer_bwd(layer_cfg(p_attn=0.0, s=45, T=90))[0] == tp.TP_ERR_ALIGN       # P row pitch
    assert layer_bwd(layer_cfg(), grads_null_shard=True)[0] == tp.TP_ERR_INVALID    # a NULL dW shard
    assert layer_bwd(layer_cfg(), ws_bytes=16)[0] == tp.TP_ERR_WORKSPACE
    assert layer_bwd(layer_cfg(), dout=FAKE + 8)[0] == tp.TP_ERR_ALIGN
    assert layer_bwd(layer_cfg(T=0))[0] == tp.TP_OK


def test_attn_proj_backward_validation():
    w, o, dw, dwo = ptrs(4), ptrs(4), ptrs(4), ptrs(4)
    f = L.tp_attn_proj_bwd
    # heads not divisible by shards
    assert f(tp.TP_BF16, 64, 512, 6, 4, FAKE, FAKE, FAKE, FAKE, w[0], o[0], FAKE, FAKE, dw[0], None,
             dwo[0], None, 0, None) == tp.TP_ERR_INVALID
    # a NULL weight-gradient shard
    bad = (ctypes.c_void_p * 4)(FAKE, FAKE, None, FAKE)
    badp = ctypes.cast(bad, ctypes.POINTER(ctypes.c_void_p))
    assert f(tp.TP_BF16, 64, 512, 8, 4, FAKE, FAKE, FAKE, FAKE, w[0], o[0], FAKE, FAKE, badp, None,
             dwo[0], None, 0, None) == tp.TP_ERR_INVALID
    # dQKV off its 16-byte boundary: refused on the host
    assert f(tp.TP_BF16, 64, 512, 8, 4, FAKE + 2, FAKE, FAKE, FAKE, w[0], o[0], FAKE, FAKE, dw[0], None,
             dwo[0], None, 0, None) == tp.TP_ERR_ALIGN
    assert f(7, 64, 512, 8, 4, FAKE, FAKE, FAKE, FAKE, w[0], o[0], FAKE, FAKE, dw[0], None,
             dwo[0], None, 0, None) == tp.TP_ERR_UNSUPPORTED


def test_vocab_logits_validation():
    e, lg = ptrs(2), ptrs(2)
    rs = rs_arr([0, 100, 250])
    f = L.tp_vocab_logits
    assert f(tp.TP_BF16, 64, 64, 250, 2, FAKE, e[0], rs_arr([0, 100, 251]), lg[0], rs_arr([104, 152]),
             None) == tp.TP_ERR_INVALID                                    # ranges do not end at V
    assert f(tp.TP_BF16, 64, 64, 250, 2, FAKE, e[0], rs, lg[0], rs_arr([104, 144]),
             None) == tp.TP_ERR_INVALID                                    # pitch below the range width
    assert f(tp.TP_BF16, 64, 64, 250, 2, FAKE, e[0], rs, lg[0], None, None) == tp.TP_ERR_INVALID
    assert f(tp.TP_BF16, 64, 64, 250, 2, FAKE + 2, e[0], rs, lg[0], rs_arr([104, 152]),
             None) == tp.TP_ERR_ALIGN                                      # X off 16 bytes
    assert f(tp.TP_BF16, 0, 64, 250, 2, None, e[0], rs, None, rs_arr([104, 152]), None) == tp.TP_OK


def test_attn_core_dropout_validation():
    def fwd(p, s=256, T=512, Pd=FAKE):
        return L.tp_attn_core_dropout_fwd(tp.TP_BF16, T, s, 512, 4, 2, 1, p, 1, 0, FAKE, FAKE, Pd, FAKE,
                                          None, FAKE * 256, 1 << 30, None)
    assert fwd(1.0) == tp.TP_ERR_INVALID                  # p must be below 1
    assert fwd(-0.1) == tp.TP_ERR_INVALID
    assert fwd(0.1, s=200, T=400) == tp.TP_ERR_INVALID    # attention dropout needs s % 16 == 0
    assert fwd(0.1, Pd=None) == tp.TP_ERR_INVALID         # the dropped probabilities need a buffer
    bwd = L.tp_attn_core_dropout_bwd(tp.TP_BF16, 400, 200, 512, 4, 2, 1, 0.1, 1, 0, FAKE, FAKE, FAKE, FAKE,
                                     FAKE, FAKE, FAKE * 256, 1 << 30, None)
    assert bwd == tp.TP_ERR_INVALID


def test_tied_grad_noalloc_refuses_sizes_beyond_its_scratch():
    e, d = ptrs(2), ptrs(2)
    V = 1 << 20
    rs = rs_arr([0, V // 2, V])
    ld = rs_arr([V // 2, V // 2])
    assert tp.tied_embed_grad_workspace_size(1 << 16, V) > (3 << 19)     # beyond 1.5 MiB
    assert L.tied_embed_grad_noalloc(tp.TP_BF16, 1 << 16, 64, V, 2, FAKE, FAKE, FAKE, d[0], ld, rs, e[0],
                                     0, None) == tp.TP_ERR_WORKSPACE
    assert L.tied_embed_grad_noalloc(tp.TP_BF16, -1, 64, V, 2, FAKE, FAKE, FAKE, d[0], ld, rs, e[0],
                                     0, None) == tp.TP_ERR_INVALID


def test_tied_grad_noalloc_checks_arguments_before_size_and_device():
    """tied_embed_grad's argument checks come first, then the scratch limit,
    and only then the device (none here): each bad argument gives its own
    error, even with a size beyond the scratch."""
    e, d = ptrs(2), ptrs(2)
    f = L.tied_embed_grad_noalloc
    big_V = 1 << 20
    big_rs, big_ld = rs_arr([0, big_V // 2, big_V]), rs_arr([big_V // 2, big_V // 2])
    T = 1 << 16
    assert f(7, T, 64, big_V, 2, FAKE, FAKE, FAKE, d[0], big_ld, big_rs, e[0], 0, None) == \
        tp.TP_ERR_UNSUPPORTED                                              # dtype, oversized size
    assert f(tp.TP_BF16, T, 64, big_V, 2, FAKE, FAKE, FAKE, d[0], big_ld, rs_arr([0, 5, big_V - 1]),
             e[0], 0, None) == tp.TP_ERR_INVALID                           # ranges do not end at V
    assert f(tp.TP_BF16, T, 0, big_V, 2, FAKE, FAKE, FAKE, d[0], big_ld, big_rs, e[0], 0, None) == \
        tp.TP_ERR_INVALID                                                  # h = 0
    assert f(tp.TP_BF16, T, 64, big_V, 2, FAKE, FAKE, FAKE, d[0], rs_arr([8, 8]), big_rs, e[0], 0,
             None) == tp.TP_ERR_INVALID                                    # pitch below range width
    assert f(tp.TP_BF16, T, 64, big_V, 2, None, FAKE, FAKE, d[0], big_ld, big_rs, e[0], 0, None) == \
        tp.TP_ERR_INVALID                                                  # no ids
    assert f(tp.TP_BF16, T, 64, big_V, 2, FAKE, FAKE, None, d[0], big_ld, big_rs, e[0], 0, None) == \
        tp.TP_ERR_INVALID                                                  # dLogits without X
