"""Python binding of libtp.so, the GB300 tensor-parallel block library.

Argument marshalling only: every function here has the name of a C-ABI entry
point (include/tp.h), checks that the torch tensors it is given live on the
GPU and are contiguous, passes their device pointers and the current CUDA
stream to the library, and raises ``TPError`` on a non-OK status.  No step of
the computation runs in Python and there is no CPU path: if libtp.so is
missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

__all__ = [
    "TPError", "lib", "LIB_PATH", "TP_OK", "TP_ERR_INVALID", "TP_ERR_UNSUPPORTED", "TP_ERR_CUDA",
    "TP_ERR_TIMEOUT", "TP_ERR_WORKSPACE", "TP_ERR_ALIGN", "TP_F32", "TP_BF16",
    "tp_mlp_fwd", "tp_mlp_bwd", "tp_attn_proj_fwd", "tp_attn_proj_bwd", "vocab_parallel_embed",
    "tp_vocab_logits", "tied_embed_grad", "tied_embed_grad_workspace_size",
    "tp_vocab_cross_entropy_fwd", "tp_vocab_cross_entropy_bwd",
    "tp_vocab_cross_entropy_workspace_size",
    "tied_embed_grad_noalloc", "tp_get_status",
    "tp_status_string", "tp_num_sms", "tp_profile_enable", "tp_profile_reset", "tp_profile_read",
    "tp_debug_inject_fault", "tp_debug_set_wait_limit_ms", "tp_debug_set_gemm_kernel",
    "tp_debug_set_split_threshold", "tp_debug_set_pdl",
    "tp_gelu_eval", "logits_pitch", "tp_adam_step", "tp_adam_step_workspace_size",
    "tp_optimizer_state", "tp_adam_config", "tp_param_group", "make_optimizer_state",
    "read_optimizer_state", "tp_attn_core_fwd", "tp_attn_core_bwd", "tp_attn_core_workspace_size",
    "tp_attn_core_dropout_fwd", "tp_attn_core_dropout_bwd", "tp_position_embed_dropout",
    "tp_transformer_layer_workspace_size", "tp_transformer_layer_fwd", "tp_transformer_layer_bwd",
    "tp_layer_config", "layer_stream",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtp.so")

TP_OK, TP_ERR_INVALID, TP_ERR_UNSUPPORTED, TP_ERR_CUDA, TP_ERR_TIMEOUT, TP_ERR_WORKSPACE, TP_ERR_ALIGN = range(7)
TP_F32, TP_BF16 = 0, 1

_c_void_p, _i64, _int, _size_t = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_PP = ctypes.POINTER(ctypes.c_void_p)
_PI64 = ctypes.POINTER(ctypes.c_int64)



class tp_optimizer_state(ctypes.Structure):
    """Device-resident optimizer state (layout of the C struct)."""
    _fields_ = [("scale", ctypes.c_float), ("growth_tracker", ctypes.c_int32),
                ("hysteresis_tracker", ctypes.c_int32), ("step", ctypes.c_int32),
                ("found_inf", ctypes.c_int32), ("grad_norm", ctypes.c_float)]


class tp_adam_config(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("max_norm", ctypes.c_double),
                ("use_scaler", ctypes.c_int32), ("min_scale", ctypes.c_float),
                ("growth_factor", ctypes.c_float), ("backoff_factor", ctypes.c_float),
                ("growth_interval", ctypes.c_int32), ("hysteresis", ctypes.c_int32)]


class tp_param_group(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("grad", ctypes.c_void_p),
                ("exp_avg", ctypes.c_void_p), ("exp_avg_sq", ctypes.c_void_p),
                ("model_param", ctypes.c_void_p), ("n", ctypes.c_int64),
                ("weight_decay", ctypes.c_double)]


class tp_layer_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("s", ctypes.c_int64), ("h", ctypes.c_int64),
                ("hp", ctypes.c_int64), ("n_heads", ctypes.c_int32), ("N", ctypes.c_int32),
                ("causal", ctypes.c_int32), ("eps", ctypes.c_float), ("p_attn", ctypes.c_float),
                ("p_hidden", ctypes.c_float), ("seed", ctypes.c_uint64), ("layer", ctypes.c_uint64)]


class tp_layer_params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("g1", "b1", "Wqkv", "bqkv", "Wo", "bo", "g2", "b2",
                                                "W", "a", "U", "b")]


class tp_layer_saved(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("ln1", "mean1", "rstd1", "QKV", "P", "Pd", "C", "h1",
                                                "ln2", "mean2", "rstd2", "Z", "Y", "attn_keep")]


class tp_layer_grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("dg1", "db1", "dWqkv", "dbqkv", "dWo", "dbo", "dg2",
                                                "db2", "dW", "da", "dU", "db")]


_SIGNATURES = {
    "tp_mlp_fwd": (_int, [_int, _i64, _i64, _i64, _int, _c_void_p, _PP, _PP, _PP, _c_void_p,
                          _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "tp_mlp_bwd": (_int, [_int, _i64, _i64, _i64, _int, _c_void_p, _c_void_p, _PP, _PP, _c_void_p,
                          _c_void_p, _c_void_p, _c_void_p, _PP, _PP, _PP, _c_void_p, _int,
                          _c_void_p]),
    "tp_attn_proj_fwd": (_int, [_int, _i64, _i64, _int, _int, _c_void_p, _PP, _PP, _c_void_p, _PP,
                                _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "tp_attn_proj_bwd": (_int, [_int, _i64, _i64, _int, _int, _c_void_p, _c_void_p, _c_void_p,
                                _c_void_p, _PP, _PP, _c_void_p, _c_void_p, _PP, _PP, _PP,
                                _c_void_p, _int, _c_void_p]),
    "vocab_parallel_embed": (_int, [_int, _i64, _i64, _i64, _int, _c_void_p, _PP, _PI64,
                                    _c_void_p, _c_void_p]),
    "tp_vocab_logits": (_int, [_int, _i64, _i64, _i64, _int, _c_void_p, _PP, _PI64, _PP, _PI64,
                               _c_void_p]),
    "tied_embed_grad": (_int, [_int, _i64, _i64, _i64, _int, _c_void_p, _c_void_p, _c_void_p, _PP,
                               _PI64, _PI64, _PP, _int, _c_void_p, _size_t, _c_void_p]),
    "tied_embed_grad_workspace_size": (_size_t, [_i64, _i64]),
    "tp_vocab_cross_entropy_fwd": (_int, [_int, _i64, _i64, _i64, _int, _c_void_p, _PP, _PI64,
                                          _c_void_p, _c_void_p, _c_void_p, _c_void_p, _size_t,
                                          _c_void_p]),
    "tp_vocab_cross_entropy_workspace_size": (_size_t, [_i64, _i64, _int, _PI64]),
    "tp_vocab_cross_entropy_bwd": (_int, [_int, _i64, _i64, _i64, _int, _c_void_p, _PP, _PI64,
                                          _c_void_p, _c_void_p, _c_void_p, _PP, _PI64, _c_void_p,
                                          _c_void_p]),
    "tied_embed_grad_noalloc": (_int, [_int, _i64, _i64, _i64, _int, _c_void_p, _c_void_p,
                                       _c_void_p, _PP, _PI64, _PI64, _PP, _int, _c_void_p]),
    "tp_get_status": (_int, [_c_void_p]),
    "tp_status_string": (ctypes.c_char_p, [_int]),
    "tp_num_sms": (_int, []),
    "tp_profile_enable": (None, [_int]),
    "tp_profile_reset": (None, []),
    "tp_profile_read": (_int, [ctypes.POINTER(ctypes.c_char_p), _PI64, _PI64,
                               ctypes.POINTER(ctypes.c_double), _int]),
    "tp_debug_inject_fault": (None, [_int]),
    "tp_debug_set_gemm_kernel": (None, [_int]),
    "tp_debug_set_split_threshold": (None, [_int]),
    "tp_debug_set_pdl": (None, [_int]),
    "tp_gelu_eval": (_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p]),
    "tp_debug_set_wait_limit_ms": (None, [_int]),
    "tp_adam_step": (_int, [ctypes.POINTER(tp_param_group), _int, ctypes.POINTER(tp_adam_config),
                            _c_void_p, _c_void_p, _size_t, _c_void_p]),
    "tp_adam_step_workspace_size": (_size_t, []),
    "tp_attn_core_fwd": (_int, [_int, _i64, _i64, _i64, _int, _int, _int, _c_void_p, _c_void_p,
                                _c_void_p, _c_void_p, _c_void_p, _size_t, _c_void_p]),
    "tp_attn_core_bwd": (_int, [_int, _i64, _i64, _i64, _int, _int, _int, _c_void_p, _c_void_p,
                                _c_void_p, _c_void_p, _c_void_p, _c_void_p, _size_t, _c_void_p]),
    "tp_attn_core_workspace_size": (_size_t, [_i64, _i64, _i64, _int]),
    "tp_attn_core_dropout_fwd": (_int, [_int, _i64, _i64, _i64, _int, _int, _int, ctypes.c_float,
                                        ctypes.c_uint64, ctypes.c_uint64, _c_void_p, _c_void_p,
                                        _c_void_p, _c_void_p, _c_void_p, _c_void_p, _size_t, _c_void_p]),
    "tp_attn_core_dropout_bwd": (_int, [_int, _i64, _i64, _i64, _int, _int, _int, ctypes.c_float,
                                        ctypes.c_uint64, ctypes.c_uint64, _c_void_p, _c_void_p,
                                        _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _size_t,
                                        _c_void_p]),
    "tp_position_embed_dropout": (_int, [_i64, _i64, _i64, _c_void_p, _c_void_p, _c_void_p,
                                         ctypes.c_float, ctypes.c_uint64, ctypes.c_uint64, _c_void_p,
                                         _c_void_p]),
    "tp_transformer_layer_workspace_size": (_size_t, [ctypes.POINTER(tp_layer_config)]),
    "tp_transformer_layer_fwd": (_int, [ctypes.POINTER(tp_layer_config), ctypes.POINTER(tp_layer_params),
                                        _c_void_p, _c_void_p, ctypes.POINTER(tp_layer_saved), _c_void_p,
                                        _size_t, _c_void_p]),
    "tp_transformer_layer_bwd": (_int, [ctypes.POINTER(tp_layer_config), ctypes.POINTER(tp_layer_params),
                                        _c_void_p, ctypes.POINTER(tp_layer_saved), _c_void_p, _c_void_p,
                                        ctypes.POINTER(tp_layer_grads), _int, _c_void_p, _size_t,
                                        _c_void_p]),
}

_LIB: Optional[ctypes.CDLL] = None


class TPError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {_status_name(status)} ({status})")
        self.status = status


def _status_name(s: int) -> str:
    names = ["TP_OK", "TP_ERR_INVALID", "TP_ERR_UNSUPPORTED", "TP_ERR_CUDA", "TP_ERR_TIMEOUT",
             "TP_ERR_WORKSPACE", "TP_ERR_ALIGN"]
    return names[s] if 0 <= s < len(names) else f"status {s}"


def lib() -> ctypes.CDLL:
    """The loaded libtp.so (raises if it is missing: there is no fallback)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libtp.so not built ({LIB_PATH}); run "
                              "`python -m megatron_tensor_transformer_tp_gb300.build_lib`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


# ----------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------
def _check(status: int, where: str):
    if status != TP_OK:
        raise TPError(status, where)


def _dev(t: Optional[torch.Tensor], name: str) -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _ptrs(ts: Optional[Sequence[torch.Tensor]], name: str):
    if ts is None:
        return None
    arr = (ctypes.c_void_p * len(ts))(*[_dev(t, f"{name}[{i}]") for i, t in enumerate(ts)])
    return ctypes.cast(arr, _PP), arr  # keep arr alive with the cast


def _pp(x):
    return None if x is None else x[0]


def _i64s(vals):
    arr = (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])
    return arr


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return TP_BF16
    if t.dtype == torch.float32:
        return TP_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def logits_pitch(n_cols: int, dtype: torch.dtype) -> int:
    """Row pitch (elements) for a logits block of ``n_cols`` columns: a
    multiple of 16 bytes, as the tensor-core path needs for TMA."""
    per = 16 // (2 if dtype == torch.bfloat16 else 4)
    return (n_cols + per - 1) // per * per


# ----------------------------------------------------------------------------
# MLP block
# ----------------------------------------------------------------------------
def tp_mlp_fwd(X, W, a, U, b, Z, Y, Out, stream=None):
    """Z, Y, Out <- column-parallel linear + GELU + row-parallel linear (shard sum)."""
    M, h = X.shape
    N = len(W)
    hp = Z.shape[1]
    w, u = _ptrs(W, "W"), _ptrs(U, "U")
    av = _ptrs(a, "a")
    _check(lib().tp_mlp_fwd(_dtype(X), M, h, hp, N, _dev(X, "X"), w[0], _pp(av), u[0], _dev(b, "b"),
                            _dev(Z, "Z"), _dev(Y, "Y"), _dev(Out, "Out"), _stream(stream)),
           "tp_mlp_fwd")


def tp_mlp_bwd(dOut, X, W, U, Z, Y, dZ, dX, dW, da, dU, db, accumulate=False, stream=None):
    M, h = X.shape
    N = len(W)
    hp = Z.shape[1]
    w, u, dw, du = _ptrs(W, "W"), _ptrs(U, "U"), _ptrs(dW, "dW"), _ptrs(dU, "dU")
    dav = _ptrs(da, "da")
    _check(lib().tp_mlp_bwd(_dtype(X), M, h, hp, N, _dev(dOut, "dOut"), _dev(X, "X"), w[0], u[0],
                            _dev(Z, "Z"), _dev(Y, "Y"), _dev(dZ, "dZ"), _dev(dX, "dX"), dw[0],
                            _pp(dav), du[0], _dev(db, "db"), int(bool(accumulate)),
                            _stream(stream)),
           "tp_mlp_bwd")


# ----------------------------------------------------------------------------
# Attention projections
# ----------------------------------------------------------------------------
def tp_attn_proj_fwd(X, Wqkv, bqkv, C, Wo, bo, QKV, O, n_heads, stream=None):
    M, h = X.shape
    N = len(Wqkv)
    wq, wo = _ptrs(Wqkv, "Wqkv"), _ptrs(Wo, "Wo")
    bq = _ptrs(bqkv, "bqkv")
    _check(lib().tp_attn_proj_fwd(_dtype(X), M, h, n_heads, N, _dev(X, "X"), wq[0], _pp(bq),
                                  _dev(C, "C"), wo[0], _dev(bo, "bo"), _dev(QKV, "QKV"),
                                  _dev(O, "O"), _stream(stream)),
           "tp_attn_proj_fwd")


def tp_attn_proj_bwd(dQKV, dO, X, C, Wqkv, Wo, dX, dC, dWqkv, dbqkv, dWo, dbo, n_heads,
                     accumulate=False, stream=None):
    M, h = X.shape
    N = len(Wqkv)
    wq, wo, dwq, dwo = _ptrs(Wqkv, "Wqkv"), _ptrs(Wo, "Wo"), _ptrs(dWqkv, "dWqkv"), _ptrs(dWo, "dWo")
    dbq = _ptrs(dbqkv, "dbqkv")
    _check(lib().tp_attn_proj_bwd(_dtype(X), M, h, n_heads, N, _dev(dQKV, "dQKV"), _dev(dO, "dO"),
                                  _dev(X, "X"), _dev(C, "C"), wq[0], wo[0], _dev(dX, "dX"),
                                  _dev(dC, "dC"), dwq[0], _pp(dbq), dwo[0], _dev(dbo, "dbo"),
                                  int(bool(accumulate)), _stream(stream)),
           "tp_attn_proj_bwd")


# ----------------------------------------------------------------------------
# Vocab-parallel embedding, logits, tied gradient
# ----------------------------------------------------------------------------
def vocab_parallel_embed(ids, E, range_starts, out, stream=None):
    T = ids.numel()
    N = len(E)
    h = out.shape[1]
    V = int(range_starts[-1])
    if ids.dtype != torch.int64:
        raise TypeError("ids must be int64")
    e = _ptrs(E, "E")
    rs = _i64s(range_starts)
    _check(lib().vocab_parallel_embed(_dtype(out), T, h, V, N, _dev(ids, "ids"), e[0], rs,
                                      _dev(out, "out"), _stream(stream)),
           "vocab_parallel_embed")


def tp_vocab_logits(X, E, range_starts, logits, stream=None):
    """logits: per-range tensors (T, pitch_r); columns [0, |r|) are written."""
    T, h = X.shape
    N = len(E)
    V = int(range_starts[-1])
    e, lg = _ptrs(E, "E"), _ptrs(logits, "logits")
    rs = _i64s(range_starts)
    ld = _i64s([t.shape[1] for t in logits])
    _check(lib().tp_vocab_logits(_dtype(X), T, h, V, N, _dev(X, "X"), e[0], rs, lg[0], ld,
                                 _stream(stream)),
           "tp_vocab_logits")


def tp_vocab_cross_entropy_workspace_size(T: int, V: int, range_starts) -> int:
    rs = _i64s(range_starts)
    return int(lib().tp_vocab_cross_entropy_workspace_size(T, V, len(range_starts) - 1, rs))


def tp_vocab_cross_entropy_fwd(X, E, range_starts, targets, loss, lse, workspace, stream=None):
    """loss, lse (T,) fp32 <- vocab-parallel cross-entropy of the logits X E_r^T
    (never stored); workspace: CUDA uint8 tensor of
    tp_vocab_cross_entropy_workspace_size bytes."""
    T, h = X.shape
    N = len(E)
    V = int(range_starts[-1])
    if targets.dtype != torch.int64:
        raise TypeError("targets must be int64")
    if workspace.dtype != torch.uint8:
        raise TypeError("workspace must be a uint8 tensor")
    e = _ptrs(E, "E")
    rs = _i64s(range_starts)
    _check(lib().tp_vocab_cross_entropy_fwd(_dtype(X), T, h, V, N, _dev(X, "X"), e[0], rs,
                                            _dev(targets, "targets"), _dev(loss, "loss"),
                                            _dev(lse, "lse"), _dev(workspace, "workspace"),
                                            workspace.numel(), _stream(stream)),
           "tp_vocab_cross_entropy_fwd")


def tp_vocab_cross_entropy_bwd(X, E, range_starts, targets, lse, dloss, dLogits, dX=None,
                               stream=None):
    """dLogits (per-range (T, pitch_r) bf16; columns [0, |r|) written) and, if
    given, dX (T, h) <- gradient of the per-token losses scaled by dloss."""
    T, h = X.shape
    N = len(E)
    V = int(range_starts[-1])
    if targets.dtype != torch.int64:
        raise TypeError("targets must be int64")
    e, dl = _ptrs(E, "E"), _ptrs(dLogits, "dLogits")
    rs = _i64s(range_starts)
    ld = _i64s([t.shape[1] for t in dLogits])
    _check(lib().tp_vocab_cross_entropy_bwd(_dtype(X), T, h, V, N, _dev(X, "X"), e[0], rs,
                                            _dev(targets, "targets"), _dev(lse, "lse"),
                                            _dev(dloss, "dloss"), dl[0], ld, _dev(dX, "dX"),
                                            _stream(stream)),
           "tp_vocab_cross_entropy_bwd")


def tied_embed_grad_workspace_size(T, V) -> int:
    return int(lib().tied_embed_grad_workspace_size(T, V))


def tied_embed_grad(ids, dEmb, X, dLogits, range_starts, dE, accumulate=False, workspace=None,
                    stream=None):
    """dLogits: per-range tensors (T, pitch_r) or None (input-side part only)."""
    T = ids.numel()
    N = len(dE)
    h = dEmb.shape[1]
    V = int(range_starts[-1])
    if ids.dtype != torch.int64:
        raise TypeError("ids must be int64")
    dl = _ptrs(dLogits, "dLogits")
    ld = _i64s([t.shape[1] for t in dLogits]) if dLogits is not None else None
    de = _ptrs(dE, "dE")
    rs = _i64s(range_starts)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().tied_embed_grad(_dtype(dEmb), T, h, V, N, _dev(ids, "ids"), _dev(dEmb, "dEmb"),
                                 _dev(X, "X"), _pp(dl), ld, rs, de[0], int(bool(accumulate)),
                                 _dev(workspace, "workspace"), ws_bytes, _stream(stream)),
           "tied_embed_grad")


def tied_embed_grad_noalloc(ids, dEmb, X, dLogits, range_starts, dE, accumulate=False,
                            stream=None):
    """tied_embed_grad for callers that cannot allocate a device workspace: the
    library uses its own fixed 1.5 MiB static device scratch (shared by all
    calls; calls that overlap on the GPU race).  Sizes whose grouping needs
    more scratch raise TPError(TP_ERR_WORKSPACE)."""
    T = ids.numel()
    N = len(dE)
    h = dEmb.shape[1]
    V = int(range_starts[-1])
    if ids.dtype != torch.int64:
        raise TypeError("ids must be int64")
    dl = _ptrs(dLogits, "dLogits")
    ld = _i64s([t.shape[1] for t in dLogits]) if dLogits is not None else None
    de = _ptrs(dE, "dE")
    rs = _i64s(range_starts)
    _check(lib().tied_embed_grad_noalloc(_dtype(dEmb), T, h, V, N, _dev(ids, "ids"),
                                         _dev(dEmb, "dEmb"), _dev(X, "X"), _pp(dl), ld, rs, de[0],
                                         int(bool(accumulate)), _stream(stream)),
           "tied_embed_grad_noalloc")


# ----------------------------------------------------------------------------
# status, profiling, debugging
# ----------------------------------------------------------------------------
def tp_attn_core_workspace_size(T, s, h, n_heads) -> int:
    return int(lib().tp_attn_core_workspace_size(T, s, h, n_heads))


def _ws_bytes(workspace):
    return workspace.numel() * workspace.element_size() if workspace is not None else 0


def tp_attn_core_fwd(QKV, s, n_heads, N, causal, P, C, lse=None, workspace=None, stream=None):
    """P (b, n_heads, s, s) bf16 and C (T, h) <- per-head softmax attention of
    the shard-major QKV (T, 3h); lse (b, n_heads, s) fp32 or None."""
    T, h3 = QKV.shape
    _check(lib().tp_attn_core_fwd(_dtype(QKV), T, s, h3 // 3, n_heads, N, int(bool(causal)),
                                  _dev(QKV, "QKV"), _dev(P, "P"), _dev(C, "C"), _dev(lse, "lse"),
                                  _dev(workspace, "workspace"), _ws_bytes(workspace),
                                  _stream(stream)),
           "tp_attn_core_fwd")


def tp_attn_core_bwd(QKV, P, C, dC, s, n_heads, N, causal, dQKV, workspace=None, stream=None):
    """dQKV (T, 3h) <- gradient of tp_attn_core_fwd given P, C and dC."""
    T, h3 = QKV.shape
    _check(lib().tp_attn_core_bwd(_dtype(QKV), T, s, h3 // 3, n_heads, N, int(bool(causal)),
                                  _dev(QKV, "QKV"), _dev(P, "P"), _dev(C, "C"), _dev(dC, "dC"),
                                  _dev(dQKV, "dQKV"), _dev(workspace, "workspace"),
                                  _ws_bytes(workspace), _stream(stream)),
           "tp_attn_core_bwd")


def layer_stream(layer: int, kind: int, shard: int = 0) -> int:
    """Dropout stream of a layer's site (the library's numbering): kind 0 =
    attention probabilities (per shard), 1 = attention output, 2 = MLP output."""
    return layer * 256 + kind * 64 + (shard if kind == 0 else 0)


def tp_attn_core_dropout_fwd(QKV, s, n_heads, N, causal, p_attn, seed, stream0, P, Pd, C, lse=None,
                             workspace=None, stream=None):
    T, h3 = QKV.shape
    _check(lib().tp_attn_core_dropout_fwd(_dtype(QKV), T, s, h3 // 3, n_heads, N, int(bool(causal)),
                                          float(p_attn), int(seed), int(stream0), _dev(QKV, "QKV"),
                                          _dev(P, "P"), _dev(Pd, "Pd"), _dev(C, "C"), _dev(lse, "lse"),
                                          _dev(workspace, "workspace"), _ws_bytes(workspace),
                                          _stream(stream)),
           "tp_attn_core_dropout_fwd")


def tp_attn_core_dropout_bwd(QKV, P, Pd, C, dC, s, n_heads, N, causal, p_attn, seed, stream0, dQKV,
                             workspace=None, stream=None):
    T, h3 = QKV.shape
    _check(lib().tp_attn_core_dropout_bwd(_dtype(QKV), T, s, h3 // 3, n_heads, N, int(bool(causal)),
                                          float(p_attn), int(seed), int(stream0), _dev(QKV, "QKV"),
                                          _dev(P, "P"), _dev(Pd, "Pd"), _dev(C, "C"), _dev(dC, "dC"),
                                          _dev(dQKV, "dQKV"), _dev(workspace, "workspace"),
                                          _ws_bytes(workspace), _stream(stream)),
           "tp_attn_core_dropout_bwd")


def tp_position_embed_dropout(words, pos_table, positions, p, seed, stream_id, out, stream=None):
    T, h = words.shape
    if positions.dtype != torch.int64:
        raise TypeError("positions must be int64")
    _check(lib().tp_position_embed_dropout(T, h, pos_table.shape[0], _dev(words, "words"),
                                           _dev(pos_table, "pos_table"), _dev(positions, "positions"),
                                           float(p), int(seed), int(stream_id), _dev(out, "out"),
                                           _stream(stream)),
           "tp_position_embed_dropout")


def _layer_cfg(cfg: dict) -> tp_layer_config:
    return tp_layer_config(cfg["T"], cfg["s"], cfg["h"], cfg["hp"], cfg["n_heads"], cfg["N"],
                           int(bool(cfg["causal"])), cfg["eps"], cfg["p_attn"], cfg["p_hidden"],
                           cfg["seed"], cfg["layer"])


def tp_transformer_layer_workspace_size(cfg: dict) -> int:
    c = _layer_cfg(cfg)
    return int(lib().tp_transformer_layer_workspace_size(ctypes.byref(c)))


def _ptr_or_shards(v, name, keep):
    if v is None:
        return None
    if isinstance(v, (list, tuple)):
        arr = _ptrs(v, name)
        keep.append(arr)
        return ctypes.cast(arr[0], ctypes.c_void_p).value
    return _dev(v, name)


def _struct(cls, d, keep):
    return cls(*[_ptr_or_shards(d.get(n), n, keep) for n, _ in cls._fields_])


def tp_transformer_layer_fwd(cfg, params, x, out, saved, workspace, stream=None):
    """params / saved: dicts keyed by the C structs' field names (tensors, or
    lists of shard tensors for the shard arrays)."""
    keep = []
    c = _layer_cfg(cfg)
    w, sv = _struct(tp_layer_params, params, keep), _struct(tp_layer_saved, saved, keep)
    _check(lib().tp_transformer_layer_fwd(ctypes.byref(c), ctypes.byref(w), _dev(x, "x"), _dev(out, "out"),
                                          ctypes.byref(sv), _dev(workspace, "workspace"),
                                          _ws_bytes(workspace), _stream(stream)),
           "tp_transformer_layer_fwd")


def tp_transformer_layer_bwd(cfg, params, x, saved, dout, dx, grads, workspace, accumulate=False,
                             stream=None):
    keep = []
    c = _layer_cfg(cfg)
    w, sv = _struct(tp_layer_params, params, keep), _struct(tp_layer_saved, saved, keep)
    g = _struct(tp_layer_grads, grads, keep)
    _check(lib().tp_transformer_layer_bwd(ctypes.byref(c), ctypes.byref(w), _dev(x, "x"), ctypes.byref(sv),
                                          _dev(dout, "dout"), _dev(dx, "dx"), ctypes.byref(g),
                                          int(bool(accumulate)), _dev(workspace, "workspace"),
                                          _ws_bytes(workspace), _stream(stream)),
           "tp_transformer_layer_bwd")


def tp_adam_step_workspace_size() -> int:
    return int(lib().tp_adam_step_workspace_size())


def make_optimizer_state(scale=1.0, growth_tracker=0, hysteresis_tracker=0, step=0,
                         device="cuda") -> torch.Tensor:
    """The 24-byte tp_optimizer_state packed into a uint8 device tensor."""
    st = tp_optimizer_state(scale, growth_tracker, hysteresis_tracker, step, 0, 0.0)
    raw = torch.frombuffer(bytearray(bytes(st)), dtype=torch.uint8)
    return raw.to(device)


def read_optimizer_state(state: torch.Tensor) -> dict:
    """Copies the device state back and unpacks it (synchronous)."""
    st = tp_optimizer_state.from_buffer_copy(bytes(state.cpu().numpy().tobytes()))
    return {name: getattr(st, name) for name, _ in tp_optimizer_state._fields_}


_ADAM_KEYS = ("lr", "beta1", "beta2", "eps", "max_norm", "use_scaler", "min_scale",
              "growth_factor", "backoff_factor", "growth_interval", "hysteresis")


def tp_adam_step(groups, cfg: dict, state: torch.Tensor, workspace: torch.Tensor, stream=None):
    """groups: sequence of dicts with fp32 tensors param, grad, m, v, optional
    bf16 tensor model (or None) and float weight_decay; cfg: dict with the keys
    of tp_adam_config; state: the device tensor from make_optimizer_state."""
    arr = (tp_param_group * max(1, len(groups)))()
    for i, g in enumerate(groups):
        n = g["param"].numel()
        for k in ("param", "grad", "m", "v"):
            if g[k].dtype != torch.float32 or g[k].numel() != n:
                raise TypeError(f"groups[{i}][{k!r}] must be float32 with {n} elements")
        model = g.get("model")
        if model is not None and (model.dtype != torch.bfloat16 or model.numel() != n):
            raise TypeError(f"groups[{i}]['model'] must be bfloat16 with {n} elements")
        arr[i] = tp_param_group(_dev(g["param"], "param"), _dev(g["grad"], "grad"),
                                _dev(g["m"], "m"), _dev(g["v"], "v"), _dev(model, "model"),
                                n, float(g.get("weight_decay", 0.0)))
    c = tp_adam_config(*[cfg[k] for k in _ADAM_KEYS])
    if state.numel() * state.element_size() != ctypes.sizeof(tp_optimizer_state):
        raise ValueError("state must be the 24-byte tensor from make_optimizer_state")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().tp_adam_step(arr, len(groups), ctypes.byref(c), _dev(state, "state"),
                              _dev(workspace, "workspace"), ws_bytes, _stream(stream)),
           "tp_adam_step")


def tp_get_status(stream=None) -> int:
    return int(lib().tp_get_status(_stream(stream)))


def tp_status_string(s: int) -> str:
    return lib().tp_status_string(s).decode()


def tp_num_sms() -> int:
    return int(lib().tp_num_sms())


def tp_profile_enable(on: bool = True):
    lib().tp_profile_enable(int(bool(on)))


def tp_profile_reset():
    lib().tp_profile_reset()


def tp_profile_read(cap: int = 64) -> dict:
    """{kind: (calls, kernel launches, total device ms)} since the last reset."""
    names = (ctypes.c_char_p * cap)()
    calls = (ctypes.c_int64 * cap)()
    kernels = (ctypes.c_int64 * cap)()
    ms = (ctypes.c_double * cap)()
    n = lib().tp_profile_read(names, calls, kernels, ms, cap)
    return {names[i].decode(): (int(calls[i]), int(kernels[i]), float(ms[i]))
            for i in range(min(n, cap))}


def tp_gelu_eval(z, y=None, dy=None, stream=None):
    """y, dy <- the device GELU and GELU' of fp32 z (test hook)."""
    _check(lib().tp_gelu_eval(_dev(z, "z"), _dev(y, "y"), _dev(dy, "dy"), z.numel(), _stream(stream)),
           "tp_gelu_eval")


def tp_debug_inject_fault(kind: int):
    lib().tp_debug_inject_fault(int(kind))


def tp_debug_set_gemm_kernel(mode: int):
    """0: one-SM tensor-core kernel, 1: two-SM kernel, 2: per launch (default)."""
    lib().tp_debug_set_gemm_kernel(int(mode))


def tp_debug_set_split_threshold(tiles_per_sm: int):
    """Tiles per SM above which a plan with dependent outputs runs as two launches."""
    lib().tp_debug_set_split_threshold(int(tiles_per_sm))


def tp_debug_set_pdl(on: bool):
    """Programmatic dependent launch of the library's kernels (default on)."""
    lib().tp_debug_set_pdl(1 if on else 0)


def tp_debug_set_wait_limit_ms(ms: int):
    lib().tp_debug_set_wait_limit_ms(int(ms))
