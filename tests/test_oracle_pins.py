"""Pins of the fp64 oracle to what the pages and the mathematics fix.

Each check is written as a function of the oracle module so that the
planted-mistake tests at the bottom can re-run it against a deliberately
broken oracle (on the CPU) and show that the pin catches the mistake.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.tp_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def rng(seed=0):
    return np.random.default_rng(seed)


def tiny_mlp(seed=0, M=3, h=4, hp=8, N=2, bias=True):
    g = rng(seed)
    X = g.standard_normal((M, h))
    W = g.standard_normal((hp, h)) * 0.5
    U = g.standard_normal((h, hp)) * 0.5
    a = g.standard_normal(hp) * 0.3 if bias else np.zeros(hp)
    b = g.standard_normal(h) * 0.3 if bias else np.zeros(h)
    dOut = g.standard_normal((M, h))
    n = hp // N
    return dict(X=X, W=W, U=U, a=a, b=b, dOut=dOut, N=N,
                Ws=[W[i * n:(i + 1) * n] for i in range(N)],
                Us=[U[:, i * n:(i + 1) * n] for i in range(N)],
                As=[a[i * n:(i + 1) * n] for i in range(N)])


# ----------------------------------------------------------------------------
# GELU
# ----------------------------------------------------------------------------
def check_gelu(mod):
    xs = np.linspace(-6, 6, 97)
    errs = []
    # math.erf (C library) as an independent routine
    ref = np.array([0.5 * x * (1 + math.erf(x / math.sqrt(2))) for x in xs])
    errs.append(np.max(np.abs(mod.gelu(xs) - ref)))
    # torch float64 exact GELU, a third implementation
    t = F.gelu(torch.tensor(xs, dtype=torch.float64), approximate="none").numpy()
    errs.append(np.max(np.abs(mod.gelu(xs) - t)))
    # special values and the odd-part identity gelu(x) - gelu(-x) = x
    errs.append(abs(mod.gelu(0.0)))
    errs.append(np.max(np.abs(mod.gelu(xs) - mod.gelu(-xs) - xs)))
    errs.append(abs(mod.gelu(30.0) / 30.0 - 1.0))
    # textbook normal-table values: gelu(x) = x Phi(x)
    gd = golden("gelu_row_split.json")
    # (the table has 10 digits, so it is held to 1e-9, scaled into the 1e-12 gate)
    errs.append(abs(mod.gelu(1.0) - gd["Phi_1"]) * 1e-3)
    errs.append(abs(mod.gelu(2.0) - 2 * gd["Phi_2"]) * 1e-3)
    return max(errs)


def check_gelu_prime(mod):
    xs = np.linspace(-5, 5, 41)
    eps = 1e-6
    fd = (mod.gelu(xs + eps) - mod.gelu(xs - eps)) / (2 * eps)
    e1 = np.max(np.abs(mod.gelu_prime(xs) - fd))
    e2 = abs(mod.gelu_prime(0.0) - 0.5)
    # torch autograd of the exact GELU
    t = torch.tensor(xs, dtype=torch.float64, requires_grad=True)
    F.gelu(t, approximate="none").sum().backward()
    e3 = np.max(np.abs(mod.gelu_prime(xs) - t.grad.numpy()))
    return max(e1, e2, e3)


def test_gelu_pinned():
    assert check_gelu(O) < 1e-12


def test_gelu_prime_pinned():
    assert check_gelu_prime(O) < 1e-8


def test_gelu_row_split_differs_closed_form():
    gd = golden("gelu_row_split.json")
    assert round(float(O.gelu(2.0)), 4) == gd["gelu_2"]
    assert round(float(2 * O.gelu(1.0)), 4) == gd["two_gelu_1"]


# ----------------------------------------------------------------------------
# MLP forward: sharded == unsharded, row split differs, bias once
# ----------------------------------------------------------------------------
def torch_mlp(X, W, a, U, b):
    """Unsharded X A -> GELU -> B with torch float64 library routines."""
    t = lambda x: torch.tensor(x, dtype=torch.float64)
    Z = F.linear(t(X), t(W), t(a))
    return F.linear(F.gelu(Z, approximate="none"), t(U), t(b)).numpy()


def check_mlp_fwd_unsharded(mod):
    worst = 0.0
    g = rng(1)
    M, h, hp = 5, 16, 64
    X = g.standard_normal((M, h))
    W = g.standard_normal((hp, h)) * 0.3
    U = g.standard_normal((h, hp)) * 0.3
    a = g.standard_normal(hp) * 0.2
    b = g.standard_normal(h) * 0.2
    ref = torch_mlp(X, W, a, U, b)
    for N in (1, 2, 4, 8):
        n = hp // N
        Z, Y, Out = mod.mlp_fwd(X, [W[i * n:(i + 1) * n] for i in range(N)],
                                [a[i * n:(i + 1) * n] for i in range(N)],
                                [U[:, i * n:(i + 1) * n] for i in range(N)], b)
        worst = max(worst, np.max(np.abs(Out - ref)))
        Zref = X @ W.T + a
        worst = max(worst, np.max(np.abs(Z - Zref)))
    return worst


def test_mlp_sharded_equals_unsharded():
    assert check_mlp_fwd_unsharded(O) < 1e-12


def test_row_split_before_gelu_differs():
    """Splitting A by rows (X by columns) and applying GELU to the partials
    gives a different result; the difference is far above any tolerance."""
    g = rng(2)
    M, h, hp, N = 8, 32, 64, 2
    X = g.standard_normal((M, h))
    A = g.standard_normal((h, hp)) * 0.3
    k = h // N
    row_split = sum(O.gelu(X[:, i * k:(i + 1) * k] @ A[i * k:(i + 1) * k]) for i in range(N))
    correct = O.gelu(X @ A)
    rel = np.max(np.abs(row_split - correct)) / np.max(np.abs(correct))
    assert rel > 10 * 2e-2


def test_bias_added_once_after_shard_sum():
    d = tiny_mlp(3, M=4, h=8, hp=16, N=4)
    _, _, out_b = O.mlp_fwd(d["X"], d["Ws"], d["As"], d["Us"], d["b"])
    _, _, out_0 = O.mlp_fwd(d["X"], d["Ws"], d["As"], d["Us"], np.zeros_like(d["b"]))
    assert np.max(np.abs((out_b - out_0) - d["b"][None, :])) < 1e-12


# ----------------------------------------------------------------------------
# MLP backward: central finite differences in fp64, torch autograd
# ----------------------------------------------------------------------------
def mlp_loss(mod, d, X=None, Ws=None, As=None, Us=None, b=None):
    _, _, Out = mod.mlp_fwd(d["X"] if X is None else X, d["Ws"] if Ws is None else Ws,
                            d["As"] if As is None else As, d["Us"] if Us is None else Us,
                            d["b"] if b is None else b)
    return float(np.sum(Out * d["dOut"]))


def fd_grad(f, x, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = x[idx]
        x[idx] = old + eps
        fp = f()
        x[idx] = old - eps
        fm = f()
        x[idx] = old
        g[idx] = (fp - fm) / (2 * eps)
    return g


def check_mlp_bwd_fd(mod):
    d = tiny_mlp(4)
    grads = mod.mlp_bwd(d["dOut"], d["X"], d["Ws"], d["As"], d["Us"])
    worst = 0.0
    X = d["X"].copy()
    worst = max(worst, np.max(np.abs(grads["dX"] - fd_grad(lambda: mlp_loss(mod, d, X=X), X))))
    for i in range(d["N"]):
        Ws = [w.copy() for w in d["Ws"]]
        worst = max(worst, np.max(np.abs(grads["dW"][i] - fd_grad(lambda: mlp_loss(mod, d, Ws=Ws), Ws[i]))))
        Us = [u.copy() for u in d["Us"]]
        worst = max(worst, np.max(np.abs(grads["dU"][i] - fd_grad(lambda: mlp_loss(mod, d, Us=Us), Us[i]))))
        As = [a.copy() for a in d["As"]]
        worst = max(worst, np.max(np.abs(grads["da"][i] - fd_grad(lambda: mlp_loss(mod, d, As=As), As[i]))))
    b = d["b"].copy()
    worst = max(worst, np.max(np.abs(grads["db"] - fd_grad(lambda: mlp_loss(mod, d, b=b), b))))
    # the saved pre-activation: Out as a function of Z alone (Y = GELU(Z), then
    # the row-parallel sum), differentiated numerically at the forward's Z
    Z, _, _ = mod.mlp_fwd(d["X"], d["Ws"], d["As"], d["Us"], d["b"])
    n = Z.shape[1] // d["N"]

    def loss_of_z():
        Y = [mod.gelu(Z[:, i * n:(i + 1) * n]) for i in range(d["N"])]
        return float(np.sum(mod.row_parallel_fwd(Y, d["Us"], d["b"]) * d["dOut"]))
    worst = max(worst, np.max(np.abs(grads["dZ"] - fd_grad(loss_of_z, Z))))
    return worst


def test_mlp_bwd_finite_differences():
    assert check_mlp_bwd_fd(O) < 1e-7


def test_mlp_bwd_matches_torch_autograd_unsharded():
    d = tiny_mlp(5, M=6, h=8, hp=32, N=4)
    t = lambda x: torch.tensor(x, dtype=torch.float64, requires_grad=True)
    X, W, a, U, b = t(d["X"]), t(d["W"]), t(d["a"]), t(d["U"]), t(d["b"])
    z = F.linear(X, W, a)
    z.retain_grad()
    out = F.linear(F.gelu(z, approximate="none"), U, b)
    (out * torch.tensor(d["dOut"])).sum().backward()
    g = O.mlp_bwd(d["dOut"], d["X"], d["Ws"], d["As"], d["Us"])
    assert np.max(np.abs(g["dZ"] - z.grad.numpy())) < 1e-12
    assert np.max(np.abs(g["dX"] - X.grad.numpy())) < 1e-12
    assert np.max(np.abs(np.concatenate(g["dW"], 0) - W.grad.numpy())) < 1e-12
    assert np.max(np.abs(np.concatenate(g["dU"], 1) - U.grad.numpy())) < 1e-12
    assert np.max(np.abs(np.concatenate(g["da"]) - a.grad.numpy())) < 1e-12
    assert np.max(np.abs(g["db"] - b.grad.numpy())) < 1e-12


def test_mlp_bwd_sampled_equals_full():
    d = tiny_mlp(6, M=10, h=8, hp=32, N=4)
    full = O.mlp_bwd(d["dOut"], d["X"], d["Ws"], d["As"], d["Us"])
    rows = [0, 3, 9]
    units = [[0, 5], [1], [2, 3, 7], [6]]
    s = O.mlp_bwd_sampled(d["dOut"], d["X"], d["Ws"], d["As"], d["Us"], rows, units)
    assert np.max(np.abs(s["dX_rows"] - full["dX"][rows])) < 1e-12
    assert np.max(np.abs(s["dZ_rows"] - full["dZ"][rows])) < 1e-12
    for i, J in enumerate(units):
        assert np.max(np.abs(s["dW_rows"][i] - full["dW"][i][J])) < 1e-12
        assert np.max(np.abs(s["dU_cols"][i] - full["dU"][i][:, J])) < 1e-12
        assert np.max(np.abs(s["da"][i] - full["da"][i][J])) < 1e-12


def test_comm_volume_4phi():
    phi, n_sums, vol = O.tp_block_comm_volume(4, 1024, 1024)
    assert phi == 4 * 1024 * 1024 and n_sums == 2 and vol == 4 * phi


# ----------------------------------------------------------------------------
# Attention projections
# ----------------------------------------------------------------------------
def tiny_attn(seed=7, M=3, h=8, N=2):
    g = rng(seed)
    d = h // N
    X = g.standard_normal((M, h))
    Wqkv = g.standard_normal((3 * h, h)) * 0.5
    Wo = g.standard_normal((h, h)) * 0.5
    bqkv = g.standard_normal(3 * h) * 0.3
    bo = g.standard_normal(h) * 0.3
    C = g.standard_normal((M, h))
    Ws = [np.concatenate([Wqkv[j * h + i * d: j * h + (i + 1) * d] for j in range(3)]) for i in range(N)]
    Bs = [np.concatenate([bqkv[j * h + i * d: j * h + (i + 1) * d] for j in range(3)]) for i in range(N)]
    Wos = [Wo[:, i * d:(i + 1) * d] for i in range(N)]
    return dict(X=X, Wqkv=Wqkv, Wo=Wo, bqkv=bqkv, bo=bo, C=C, Ws=Ws, Bs=Bs, Wos=Wos, N=N, h=h, d=d,
                dQKV=g.standard_normal((M, 3 * h)), dO=g.standard_normal((M, h)))


def test_attn_proj_sharded_equals_unsharded():
    a = tiny_attn(M=5, h=16, N=4)
    QKV, Oo = O.attn_proj_fwd(a["X"], a["Ws"], a["Bs"], a["C"], a["Wos"], a["bo"])
    full = torch.nn.functional.linear(torch.tensor(a["X"]), torch.tensor(a["Wqkv"]), torch.tensor(a["bqkv"])).numpy()
    h, d, N = a["h"], a["d"], a["N"]
    for i in range(N):
        for j in range(3):
            got = QKV[:, i * 3 * d + j * d: i * 3 * d + (j + 1) * d]
            ref = full[:, j * h + i * d: j * h + (i + 1) * d]
            assert np.max(np.abs(got - ref)) < 1e-12
    Oref = F.linear(torch.tensor(a["C"]), torch.tensor(a["Wo"]), torch.tensor(a["bo"])).numpy()
    assert np.max(np.abs(Oo - Oref)) < 1e-12


def check_attn_bwd_fd(mod):
    a = tiny_attn()

    def loss(X=None, Ws=None, C=None, Wos=None):
        QKV, Oo = mod.attn_proj_fwd(a["X"] if X is None else X, a["Ws"] if Ws is None else Ws,
                                    a["Bs"], a["C"] if C is None else C,
                                    a["Wos"] if Wos is None else Wos, a["bo"])
        return float(np.sum(QKV * a["dQKV"]) + np.sum(Oo * a["dO"]))

    g = mod.attn_proj_bwd(a["dQKV"], a["dO"], a["X"], a["C"], a["Ws"], a["Wos"])
    worst = 0.0
    X = a["X"].copy()
    worst = max(worst, np.max(np.abs(g["dX"] - fd_grad(lambda: loss(X=X), X))))
    C = a["C"].copy()
    worst = max(worst, np.max(np.abs(g["dC"] - fd_grad(lambda: loss(C=C), C))))
    for i in range(a["N"]):
        Ws = [w.copy() for w in a["Ws"]]
        worst = max(worst, np.max(np.abs(g["dWqkv"][i] - fd_grad(lambda: loss(Ws=Ws), Ws[i]))))
        Wos = [w.copy() for w in a["Wos"]]
        worst = max(worst, np.max(np.abs(g["dWo"][i] - fd_grad(lambda: loss(Wos=Wos), Wos[i]))))
    worst = max(worst, np.max(np.abs(g["dbo"] - a["dO"].sum(0))))
    return worst


def test_attn_bwd_finite_differences():
    assert check_attn_bwd_fd(O) < 1e-7


def test_attn_proj_weight_rows_equal_the_full_gradients():
    """The sampled weight-gradient rows (used at full size) are the rows of the
    finite-difference-pinned full gradients, in the order asked for (up to the
    summation order of the library's matrix products: 1e-12 relative)."""
    a = tiny_attn(M=6, h=16, N=4)
    g = O.attn_proj_bwd(a["dQKV"], a["dO"], a["X"], a["C"], a["Ws"], a["Wos"])
    qkv_rows = [[0, 5, 11], [3], [11, 2], [7, 7]]
    o_rows = [[15, 0], [4], [9, 1, 2], [8]]
    dWqkv, dWo, dbqkv, dbo = O.attn_proj_bwd_weight_rows(a["dQKV"], a["dO"], a["X"], a["C"], a["N"],
                                                         qkv_rows, o_rows)
    for i in range(a["N"]):
        np.testing.assert_allclose(dWqkv[i], g["dWqkv"][i][qkv_rows[i]], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dWo[i], g["dWo"][i][o_rows[i]], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dbqkv[i], g["dbqkv"][i], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dbo, g["dbo"], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# Attention core (per head, between the projections)
# ----------------------------------------------------------------------------
def tiny_core(seed=3, b=2, s=5, n_heads=4, N=2, d=3, scale=1.0):
    """Per-head q, k, v (b, heads, s, d) and their shard-major QKV layout,
    assembled here by the layout's definition (shard i = [Q_i K_i V_i], its
    heads in order inside each)."""
    g = rng(seed)
    q, k, v = (g.standard_normal((b, n_heads, s, d)) * scale for _ in range(3))
    dC = g.standard_normal((b * s, n_heads * d))
    per = n_heads // N
    cols = []
    for i in range(N):
        for t in (q, k, v):
            for jl in range(per):
                cols.append(t[:, i * per + jl].reshape(b * s, d))
    QKV = np.concatenate(cols, axis=1)
    return dict(q=q, k=k, v=v, QKV=QKV, dC=dC, b=b, s=s, n_heads=n_heads, N=N, d=d)


def check_core_sdpa(mod, causal):
    """Largest difference to torch's scaled_dot_product_attention (float64)
    in the context and in dQKV (autograd)."""
    c = tiny_core()
    b, s, H, d = c["b"], c["s"], c["n_heads"], c["d"]
    C, P = mod.attention_core(c["QKV"], s, H, c["N"], causal)
    dQKV = mod.attention_core_grad(c["QKV"], P, c["dC"], s, H, c["N"])
    tq, tk, tv = (torch.tensor(c[x], requires_grad=True) for x in ("q", "k", "v"))
    out = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)  # (b, H, s, d)
    ref_C = out.permute(0, 2, 1, 3).reshape(b * s, H * d)
    ref_C.backward(torch.tensor(c["dC"]))
    err = np.abs(C - ref_C.detach().numpy()).max()
    # dQKV in the layout, compared through the same assembly as the inputs
    per = H // c["N"]
    k0 = 0
    for i in range(c["N"]):
        for t in (tq, tk, tv):
            for jl in range(per):
                ref = t.grad[:, i * per + jl].reshape(b * s, d).numpy()
                err = max(err, np.abs(dQKV[:, k0:k0 + d] - ref).max())
                k0 += d
    return err


@pytest.mark.parametrize("causal", [True, False])
def test_attention_core_matches_torch_sdpa(causal):
    assert check_core_sdpa(O, causal) < 1e-12


def check_core_mha(mod):
    """X -> sharded QKV projection -> attention core -> sharded output
    projection equals torch multi_head_attention_forward on the unsharded
    weights (causal), forward and input gradient."""
    a = tiny_attn(seed=9, M=12, h=16, N=2)
    s, H = 6, 4  # two sequences of 6 tokens, 2 heads per shard
    X = a["X"]
    QKV, _ = mod.attn_proj_fwd(X, a["Ws"], a["Bs"], a["C"], a["Wos"], a["bo"])
    C, P = mod.attention_core(QKV, s, H, a["N"], True)
    _, out = mod.attn_proj_fwd(X, a["Ws"], a["Bs"], C, a["Wos"], a["bo"])
    tX = torch.tensor(X.reshape(2, s, 16).transpose(1, 0, 2).copy())  # (s, b, h)
    mask = torch.triu(torch.ones(s, s, dtype=torch.bool), 1)
    ref, _ = F.multi_head_attention_forward(
        tX, tX, tX, 16, H, torch.tensor(a["Wqkv"]), torch.tensor(a["bqkv"]), None, None, False, 0.0,
        torch.tensor(a["Wo"]), torch.tensor(a["bo"]), training=False, need_weights=False,
        attn_mask=mask)
    ref = ref.numpy().transpose(1, 0, 2).reshape(12, 16)
    return np.abs(out - ref).max()


def test_attention_core_through_projections_matches_torch_mha():
    assert check_core_mha(O) < 1e-12


def check_core_uniform(mod):
    """q = 0 makes every allowed key equally likely: the causal context is the
    running mean of v, the full one the mean of all v."""
    c = tiny_core()
    QKV = c["QKV"].copy()
    b, s, H, N, d = c["b"], c["s"], c["n_heads"], c["N"], c["d"]
    per = H // N
    for i in range(N):  # zero the Q block of every shard
        QKV[:, i * 3 * per * d: i * 3 * per * d + per * d] = 0.0
    err = 0.0
    for causal in (True, False):
        C, _ = mod.attention_core(QKV, s, H, N, causal)
        for bi in range(b):
            for j in range(H):
                v = c["v"][bi, j]
                want = np.cumsum(v, axis=0) / np.arange(1, s + 1)[:, None] if causal else \
                    np.broadcast_to(v.mean(axis=0), (s, d))
                err = max(err, np.abs(C[bi * s:(bi + 1) * s, j * d:(j + 1) * d] - want).max())
    return err


def test_attention_core_uniform_closed_form():
    assert check_core_uniform(O) < 1e-14


def test_attention_head_brute_force():
    g = rng(4)
    q, k, v = (g.standard_normal((3, 2)) for _ in range(3))
    P, out = O.attention_head(q, k, v, True)
    for i in range(3):
        w = [math.exp(sum(q[i, c] * k[j, c] for c in range(2)) / math.sqrt(2)) for j in range(i + 1)]
        tot = sum(w)
        for c in range(2):
            assert abs(out[i, c] - sum(w[j] * v[j, c] for j in range(i + 1)) / tot) < 1e-14
        for j in range(3):
            assert abs(P[i, j] - (w[j] / tot if j <= i else 0.0)) < 1e-15


def test_planted_missing_attention_scale_is_caught(monkeypatch):
    real = O.attention_head

    def broken(q, k, v, causal, **kw):
        return real(q * math.sqrt(q.shape[1]), k, v, causal, **kw)  # the 1/sqrt(d) undone
    monkeypatch.setattr(O, "attention_head", broken)
    assert check_core_sdpa(O, True) > 1e-3


def test_planted_causal_mask_off_by_one_is_caught(monkeypatch):
    def broken(q, k, v, causal, **kw):
        s, d = q.shape
        S = (q @ k.T) / math.sqrt(d)
        if causal:  # the diagonal masked as well (a finite fill keeps row 0 defined)
            S = np.where(np.tril(np.ones((s, s), dtype=bool), -1), S, -1e300)
        E = np.exp(S - S.max(axis=1, keepdims=True))
        P = E / E.sum(axis=1, keepdims=True)
        return P, P @ v
    monkeypatch.setattr(O, "attention_head", broken)
    assert check_core_uniform(O) > 1e-3


def test_planted_softmax_over_queries_is_caught(monkeypatch):
    def broken(q, k, v, causal, **kw):
        s, d = q.shape
        S = (q @ k.T) / math.sqrt(d)
        if causal:
            S = np.where(np.tril(np.ones((s, s), dtype=bool)), S, -np.inf)
        E = np.exp(S - S.max(axis=0, keepdims=True))
        P = E / E.sum(axis=0, keepdims=True)
        return P, P @ v
    monkeypatch.setattr(O, "attention_head", broken)
    assert check_core_sdpa(O, False) > 1e-3


def test_planted_missing_softmax_correction_in_grad_is_caught(monkeypatch):
    def broken(q, k, v, P, g, **kw):
        dS = P * (g @ v.T) / math.sqrt(q.shape[1])  # the row-sum term dropped
        return dS @ k, dS.T @ q, P.T @ g
    monkeypatch.setattr(O, "attention_head_grad", broken)
    assert check_core_sdpa(O, True) > 1e-3


def test_planted_head_layout_swap_is_caught(monkeypatch):
    real = O.attention_head_columns

    def broken(h, n_heads, N, j):
        q, k, v, c = real(h, n_heads, N, j)
        return k, q, v, c  # Q and K blocks swapped
    monkeypatch.setattr(O, "attention_head_columns", broken)
    assert check_core_mha(O) > 1e-3


# ----------------------------------------------------------------------------
# Vocab-parallel embedding
# ----------------------------------------------------------------------------
def test_vocab_mask_page_example():
    gd = golden("vocab_mask_example.json")
    masked, mask = O.vocab_mask(gd["ids"], gd["start"], gd["end"])
    assert masked.tolist() == gd["masked_input"]
    assert mask.tolist() == gd["input_mask"]


def check_vocab300(mod):
    gd = golden("vocab300_two_ranges.json")
    V, rs, ids = gd["V"], gd["range_starts"], gd["ids"]
    E = rng(8).standard_normal((V, 16))
    Es = [E[rs[r]:rs[r + 1]] for r in range(2)]
    parts = mod.vocab_parallel_embed_partials(ids, Es, rs)
    ok = True
    for r in range(2):
        zero_rows = [t for t in range(len(ids)) if not np.any(parts[r][t])]
        ok &= zero_rows == gd["zero_rows_per_range"][r]
    out = mod.vocab_parallel_embed(ids, Es, rs)
    ok &= bool(np.array_equal(out, E[ids]))
    return ok


def test_vocab300_two_range_example():
    assert check_vocab300(O)


def test_vocab_embed_brute_force_small_vocab():
    g = rng(9)
    for V in (1, 7, 64):
        for N in (1, 2, 3):
            if N > V:
                continue
            cuts = sorted(g.choice(np.arange(1, V), size=N - 1, replace=False).tolist()) if N > 1 else []
            rs = [0] + cuts + [V]
            E = g.standard_normal((V, 5))
            Es = [E[rs[r]:rs[r + 1]] for r in range(N)]
            ids = list(range(V)) + [-1, V, V + 3, -7]
            out = O.vocab_parallel_embed(ids, Es, rs)
            for t, v in enumerate(ids):
                if 0 <= v < V:
                    assert np.array_equal(out[t], E[v])
                else:
                    assert not np.any(out[t])
            # torch F.embedding on the valid ids
            valid = [v for v in ids if 0 <= v < V]
            te = F.embedding(torch.tensor(valid), torch.tensor(E)).numpy()
            assert np.array_equal(out[:len(valid)], te)


def test_vocab_logits_equals_unsharded():
    g = rng(10)
    V, h, T = 37, 6, 5
    rs = [0, 11, 20, 37]
    E = g.standard_normal((V, h))
    X = g.standard_normal((T, h))
    Ls = O.vocab_logits(X, [E[rs[r]:rs[r + 1]] for r in range(3)])
    ref = F.linear(torch.tensor(X), torch.tensor(E)).numpy()
    assert np.max(np.abs(np.concatenate(Ls, 1) - ref)) < 1e-12


# ----------------------------------------------------------------------------
# Tied embedding gradient
# ----------------------------------------------------------------------------
def tied_case(seed=11, V=23, h=4, T=40, rs=(0, 9, 23)):
    g = rng(seed)
    ids = g.integers(-2, V + 2, size=T)
    ids[:6] = 5  # a repeated id
    return dict(ids=ids, V=V, rs=list(rs), dEmb=g.standard_normal((T, h)), X=g.standard_normal((T, h)),
                dL=g.standard_normal((T, V)))


def check_scatter(mod):
    c = tied_case()
    s = mod.embed_scatter_grad(c["ids"], c["dEmb"], c["V"])
    ref = np.zeros_like(s)
    valid = (c["ids"] >= 0) & (c["ids"] < c["V"])
    np.add.at(ref, c["ids"][valid], c["dEmb"][valid])
    e1 = np.max(np.abs(s - ref))
    e2 = np.max(np.abs(s.sum(0) - c["dEmb"][valid].sum(0)))
    # torch autograd of F.embedding on the valid tokens
    Et = torch.zeros((c["V"], c["dEmb"].shape[1]), dtype=torch.float64, requires_grad=True)
    out = F.embedding(torch.tensor(c["ids"][valid]), Et)
    (out * torch.tensor(c["dEmb"][valid])).sum().backward()
    e3 = np.max(np.abs(s - Et.grad.numpy()))
    return max(e1, e2, e3)


def test_scatter_grad_pinned():
    assert check_scatter(O) < 1e-12


def test_tied_grad_is_sum_of_both_contributions():
    c = tied_case()
    rs, V = c["rs"], c["V"]
    dLs = [c["dL"][:, rs[r]:rs[r + 1]] for r in range(2)]
    tg = np.concatenate(O.tied_embed_grad(c["ids"], c["dEmb"], c["X"], dLs, rs, V), 0)
    scatter = O.embed_scatter_grad(c["ids"], c["dEmb"], V)
    assert np.max(np.abs(tg - (scatter + c["dL"].T @ c["X"]))) < 1e-12
    # dLogits = 0 reduces to the embedding backward; dEmb = 0 to dLogits^T X
    z = [np.zeros_like(x) for x in dLs]
    t0 = np.concatenate(O.tied_embed_grad(c["ids"], c["dEmb"], c["X"], z, rs, V), 0)
    assert np.max(np.abs(t0 - scatter)) < 1e-12
    t1 = np.concatenate(O.tied_embed_grad(c["ids"], np.zeros_like(c["dEmb"]), c["X"], dLs, rs, V), 0)
    ref = F.linear(torch.tensor(c["dL"].T.copy()), torch.tensor(c["X"].T.copy())).numpy()
    assert np.max(np.abs(t1 - ref)) < 1e-12
    rows = [0, 5, 9, 22]
    tr = O.tied_embed_grad_rows(c["ids"], c["dEmb"], c["X"], c["dL"], rows)
    assert np.max(np.abs(tr - tg[rows])) < 1e-12


def test_embed_sort_brute_force():
    c = tied_case(12, V=17, T=60)
    offs, perm = O.embed_sort(c["ids"], c["V"])
    for v in range(c["V"]):
        seg = perm[offs[v]:offs[v + 1]].tolist()
        assert seg == [t for t in range(len(c["ids"])) if c["ids"][t] == v]
    assert offs[-1] == np.sum((c["ids"] >= 0) & (c["ids"] < c["V"]))


# ----------------------------------------------------------------------------
# Closed forms
# ----------------------------------------------------------------------------
def test_param_count_page_value():
    gd = golden("param_count.json")
    total = O.param_count(gd["H"], gd["L"], gd["V"])
    assert total == gd["total"]
    body = (12 * gd["H"] ** 2 + 4 * gd["H"]) * gd["L"]
    assert round(body / 1e9, 1) == gd["body_approx_billions"]


# ----------------------------------------------------------------------------
# Planted mistakes: each pin must catch a plausible error in the oracle
# ----------------------------------------------------------------------------
def _tanh_gelu(z):
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1 + np.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))


def test_planted_tanh_gelu_is_caught(monkeypatch):
    monkeypatch.setattr(O, "gelu", _tanh_gelu)
    assert check_gelu(O) > 1e-6


def test_planted_gelu_prime_dropped_term_is_caught(monkeypatch):
    monkeypatch.setattr(O, "gelu_prime", lambda z: 0.5 * (1 + O._erf(np.asarray(z) / math.sqrt(2))))
    assert check_gelu_prime(O) > 1e-3
    assert check_mlp_bwd_fd(O) > 1e-3


def test_planted_dz_from_wrong_shard_is_caught(monkeypatch):
    real = O.mlp_bwd

    def broken(*args, **kw):
        g = real(*args, **kw)
        n = g["dZ"].shape[1] // 2
        g["dZ"] = np.concatenate([g["dZ"][:, n:], g["dZ"][:, :n]], axis=1)  # shards swapped
        return g
    monkeypatch.setattr(O, "mlp_bwd", broken)
    assert check_mlp_bwd_fd(O) > 1e-3


def test_planted_sign_error_in_dx_is_caught(monkeypatch):
    real = O.mlp_bwd

    def broken(*args, **kw):
        g = real(*args, **kw)
        g["dX"] = -g["dX"]
        return g
    monkeypatch.setattr(O, "mlp_bwd", broken)
    assert check_mlp_bwd_fd(O) > 1e-3


def test_planted_transposed_operand_is_caught(monkeypatch):
    def broken_row(Y_shards, U_shards, b=None):
        out = sum(Yi @ Ui[:, ::-1].T for Yi, Ui in zip(Y_shards, U_shards))
        return out + b[None, :] if b is not None else out
    monkeypatch.setattr(O, "row_parallel_fwd", broken_row)
    assert check_mlp_fwd_unsharded(O) > 1e-3


def test_planted_bias_per_shard_is_caught(monkeypatch):
    def broken_row(Y_shards, U_shards, b=None):
        out = 0
        for Yi, Ui in zip(Y_shards, U_shards):
            out = out + Yi @ Ui.T + (b[None, :] if b is not None else 0)
        return out
    monkeypatch.setattr(O, "row_parallel_fwd", broken_row)
    assert check_mlp_fwd_unsharded(O) > 1e-3


def test_planted_unmasked_lookup_is_caught(monkeypatch):
    def broken_parts(ids, E_shards, range_starts):
        parts = []
        for r, Er in enumerate(E_shards):
            masked, mask = O.vocab_mask(ids, range_starts[r], range_starts[r + 1])
            parts.append(np.asarray(Er, dtype=np.float64)[masked])  # zeroing dropped
        return parts
    monkeypatch.setattr(O, "vocab_parallel_embed_partials", broken_parts)
    assert not check_vocab300(O)


def test_planted_scatter_off_by_one_is_caught(monkeypatch):
    def broken(ids, dEmb, V):
        out = np.zeros((V, dEmb.shape[1]))
        for t, v in enumerate(ids):
            if 0 <= v < V - 1:
                out[v + 1] += dEmb[t]
        return out
    monkeypatch.setattr(O, "embed_scatter_grad", broken)
    assert check_scatter(O) > 1e-3


# ----------------------------------------------------------------------------
# Vocab-parallel cross-entropy
# ----------------------------------------------------------------------------
def tiny_ce(seed=0, T=6, h=5, V=13, ranges=(0, 4, 9, 13), scale=1.0):
    g = rng(seed)
    X = g.standard_normal((T, h))
    E = g.standard_normal((V, h)) * scale
    t = g.integers(0, V, T)
    dl = g.standard_normal(T)
    Es = [E[ranges[r]:ranges[r + 1]] for r in range(len(ranges) - 1)]
    return X, E, Es, list(ranges), t, dl


def check_ce_torch(mod, scale=1.0):
    """Max |oracle - torch| of the loss and of its gradient (valid targets)."""
    X, E, Es, r, t, dl = tiny_ce(scale=scale)
    loss, lse = mod.vocab_parallel_cross_entropy(X, Es, r, t)
    L = torch.tensor(X @ E.T, dtype=torch.float64, requires_grad=True)
    ref = F.cross_entropy(L, torch.tensor(t), reduction="none")
    (ref * torch.tensor(dl)).sum().backward()
    g = np.concatenate(mod.vocab_parallel_cross_entropy_grad(X, Es, r, t, dl), axis=1)
    e_lse = np.abs(lse - torch.logsumexp(L.detach(), dim=1).numpy()).max()
    return max(np.abs(loss - ref.detach().numpy()).max(), np.abs(g - L.grad.numpy()).max(), e_lse)


def test_ce_matches_torch_cross_entropy():
    assert check_ce_torch(O) < 1e-12


def test_ce_stable_at_large_logits():
    # logits of order 1e3: exp without the max shift would overflow
    assert check_ce_torch(O, scale=300.0) < 1e-9


def test_ce_invariant_to_vocab_split():
    X, E, _, _, t, dl = tiny_ce(1)
    outs = []
    for r in ([0, 13], [0, 6, 13], [0, 1, 2, 12, 13]):
        Es = [E[r[i]:r[i + 1]] for i in range(len(r) - 1)]
        loss, lse = O.vocab_parallel_cross_entropy(X, Es, r, t)
        g = np.concatenate(O.vocab_parallel_cross_entropy_grad(X, Es, r, t, dl), axis=1)
        outs.append((loss, lse, g))
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert np.abs(a - b).max() < 1e-12


def test_ce_zero_logits_closed_form():
    # all logits 0: loss = log V for every token, grad = (1/V - onehot) * dloss;
    # a target in no range (the pages' masking): loss = log V, grad = dloss / V
    T, h, V = 5, 3, 11
    X = rng(2).standard_normal((T, h))
    E = np.zeros((V, h))
    t = np.array([0, 10, 5, -1, 11])
    dl = np.arange(1.0, T + 1)
    r = [0, 5, 11]
    Es = [E[0:5], E[5:11]]
    loss, lse = O.vocab_parallel_cross_entropy(X, Es, r, t)
    assert np.allclose(loss, math.log(V), atol=1e-15) and np.allclose(lse, math.log(V), atol=1e-15)
    g = np.concatenate(O.vocab_parallel_cross_entropy_grad(X, Es, r, t, dl), axis=1)
    want = np.full((T, V), 1.0 / V)
    for i, ti in enumerate(t):
        if 0 <= ti < V:
            want[i, ti] -= 1.0
    want *= dl[:, None]
    assert np.abs(g - want).max() < 1e-15


def test_logits_side_dx_equals_unsharded():
    X, E, Es, r, t, dl = tiny_ce(3)
    g = O.vocab_parallel_cross_entropy_grad(X, Es, r, t, dl)
    full = np.concatenate(g, axis=1) @ E
    assert np.abs(O.logits_side_dx(g, Es) - full).max() < 1e-12


def test_planted_unmasked_predicted_logit_is_caught(monkeypatch):
    real = O.vocab_parallel_cross_entropy

    def broken(X, E_shards, range_starts, targets):
        # every range contributes its logit at the clamped index (mask dropped)
        loss, lse = real(X, E_shards, range_starts, targets)
        targets = np.asarray(targets)
        extra = np.zeros(len(targets))
        for r, Er in enumerate(E_shards):
            s, e = range_starts[r], range_starts[r + 1]
            out = (targets < s) | (targets >= e)
            idx = np.clip(targets - s, 0, e - s - 1)
            L = X @ Er.T - (lse - 0)[:, None]
            extra += np.where(out, L[np.arange(len(targets)), idx], 0.0)
        return loss - extra, lse
    monkeypatch.setattr(O, "vocab_parallel_cross_entropy", broken)
    assert check_ce_torch(O) > 1e-3


def test_planted_missing_target_term_in_grad_is_caught(monkeypatch):
    def broken(X, E_shards, range_starts, targets, dloss):
        L = [X @ Er.T for Er in E_shards]
        m = np.max(np.stack([l.max(axis=1) for l in L]), axis=0)
        e = [np.exp(l - m[:, None]) for l in L]
        s = sum(x.sum(axis=1) for x in e)
        return [x / s[:, None] * np.asarray(dloss)[:, None] for x in e]  # softmax only
    monkeypatch.setattr(O, "vocab_parallel_cross_entropy_grad", broken)
    assert check_ce_torch(O) > 1e-3


def test_planted_per_range_max_is_caught(monkeypatch):
    def broken(X, E_shards, range_starts, targets):
        # each range shifts by its own maximum, then the sums are added as if shared
        targets = np.asarray(targets)
        T = X.shape[0]
        pred = np.zeros(T)
        sum_exp = np.zeros(T)
        for r, Er in enumerate(E_shards):
            L = X @ Er.T
            L = L - L.max(axis=1)[:, None]
            s, e = range_starts[r], range_starts[r + 1]
            inside = (targets >= s) & (targets < e)
            idx = np.where(inside, targets - s, 0)
            pred += np.where(inside, L[np.arange(T), idx], 0.0)
            sum_exp += np.exp(L).sum(axis=1)
        return np.log(sum_exp) - pred, np.log(sum_exp)
    monkeypatch.setattr(O, "vocab_parallel_cross_entropy", broken)
    assert check_ce_torch(O) > 1e-3


# ----------------------------------------------------------------------------
# Mixed-precision optimizer step
# ----------------------------------------------------------------------------
ADAM_CFG = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, max_norm=0.0, use_scaler=False,
                min_scale=1.0, growth_factor=2.0, backoff_factor=0.5, growth_interval=3, hysteresis=2)


def check_adam_torch(mod, steps=4):
    g = rng(11)
    shapes = [(7, 5), (9,)]
    wds = [0.1, 0.0]
    params = [g.standard_normal(s) for s in shapes]
    grads = [[g.standard_normal(s) for s in shapes] for _ in range(steps)]
    tparams = [torch.tensor(p, dtype=torch.float64, requires_grad=True) for p in params]
    opt = torch.optim.Adam([{"params": [tp], "weight_decay": wd} for tp, wd in zip(tparams, wds)],
                           lr=ADAM_CFG["lr"], betas=(ADAM_CFG["beta1"], ADAM_CFG["beta2"]),
                           eps=ADAM_CFG["eps"])
    groups = [dict(param=p.copy(), grad=None, m=np.zeros_like(p), v=np.zeros_like(p), weight_decay=wd)
              for p, wd in zip(params, wds)]
    state = dict(scale=1.0, growth_tracker=0, hysteresis_tracker=2, step=0)
    for k in range(steps):
        for tp, gr in zip(tparams, grads[k]):
            tp.grad = torch.tensor(gr, dtype=torch.float64)
        opt.step()
        for grp, gr in zip(groups, grads[k]):
            grp["grad"] = gr
        ok, _, groups, state = mod.mixed_precision_adam_step(groups, state, ADAM_CFG)
        assert ok
    return max(np.abs(grp["param"] - tp.detach().numpy()).max() for grp, tp in zip(groups, tparams))


def test_adam_matches_torch():
    assert check_adam_torch(O) < 1e-12


def check_clip(mod):
    """Error of the clip against the closed form: two groups whose joint norm is 5."""
    g = [np.array([3.0, 0.0]), np.array([[4.0]])]
    out, norm = mod.clip_by_global_norm(g, 1.0)
    return max(abs(norm - 5.0), abs(out[0][0] - 0.6), abs(out[0][1]), abs(out[1][0, 0] - 0.8))


def test_clip_closed_form_and_torch():
    assert check_clip(O) < 1e-15
    g = [np.array([3.0, 0.0]), np.array([[4.0]])]
    same, n2 = O.clip_by_global_norm(g, 10.0)
    assert n2 == 5.0 and same[0] is g[0]
    h = [rng(12).standard_normal((6, 4)) * 3, rng(13).standard_normal(5)]
    t = [torch.tensor(x, requires_grad=True) for x in h]
    for x, tt in zip(h, t):
        tt.grad = torch.tensor(x)
    torch.nn.utils.clip_grad_norm_(t, 2.0)
    out, _ = O.clip_by_global_norm(h, 2.0)
    for a, tt in zip(out, t):
        assert np.abs(a - tt.grad.numpy()).max() < 1e-6 * np.abs(a).max()


def test_grad_scaler_behaviour():
    cfg = dict(ADAM_CFG, use_scaler=True, min_scale=0.25)
    s = dict(scale=4.0, growth_tracker=0, hysteresis_tracker=2, step=0)
    # growth_interval (3) overflow-free steps grow the scale and reset the trackers
    for k in range(3):
        s = O.grad_scaler_update(s, False, cfg)
    assert s["scale"] == 8.0 and s["growth_tracker"] == 0 and s["hysteresis_tracker"] == 2
    # the first overflow only spends hysteresis; the second backs off
    s = O.grad_scaler_update(s, True, cfg)
    assert s["scale"] == 8.0 and s["hysteresis_tracker"] == 1
    s = O.grad_scaler_update(s, True, cfg)
    assert s["scale"] == 4.0
    # further overflows keep backing off (hysteresis is cumulative), down to min_scale
    for _ in range(6):
        s = O.grad_scaler_update(s, True, cfg)
    assert s["scale"] == 0.25
    # an overflow resets the run of clean steps
    s = O.grad_scaler_update(s, False, cfg)
    s = O.grad_scaler_update(s, True, cfg)
    assert s["growth_tracker"] == 0


def test_step_skipped_on_overflow_and_unscale_before_clip():
    cfg = dict(ADAM_CFG, use_scaler=True, max_norm=1.0)
    p = np.ones(4)
    grp = dict(param=p.copy(), grad=np.array([1.0, np.inf, 0.0, 0.0]), m=np.zeros(4), v=np.zeros(4),
               weight_decay=0.0)
    st = dict(scale=8.0, growth_tracker=1, hysteresis_tracker=1, step=5)
    ok, _, out, st2 = O.mixed_precision_adam_step([grp], st, cfg)
    assert not ok and np.array_equal(out[0]["param"], p) and st2["step"] == 5 and st2["scale"] == 4.0
    # scale 8 and grads (0, 0, 24, 32): unscaled norm 5 is clipped to 1, so the
    # clipped grads are (0, 0, 0.6, 0.8) and m = (1 - b1) * g after one step
    grp = dict(param=p.copy(), grad=np.array([0.0, 0.0, 24.0, 32.0]), m=np.zeros(4), v=np.zeros(4),
               weight_decay=0.0)
    ok, norm, out, st3 = O.mixed_precision_adam_step([grp], dict(st, hysteresis_tracker=2), cfg)
    assert ok and norm == 5.0 and st3["step"] == 6
    assert np.allclose(out[0]["m"], (1 - cfg["beta1"]) * np.array([0, 0, 0.6, 0.8]), atol=1e-15)


def test_planted_missing_bias_correction_is_caught(monkeypatch):
    def broken(param, grad, m, v, step, cfg, weight_decay):
        g = grad + weight_decay * param
        m = cfg["beta1"] * m + (1 - cfg["beta1"]) * g
        v = cfg["beta2"] * v + (1 - cfg["beta2"]) * g * g
        return param - cfg["lr"] * m / (np.sqrt(v) + cfg["eps"]), m, v
    monkeypatch.setattr(O, "adam_update", broken)
    assert check_adam_torch(O) > 1e-6


def test_planted_per_group_clip_is_caught(monkeypatch):
    real = O.clip_by_global_norm

    def broken(grads, max_norm):
        outs = [real([g], max_norm)[0][0] for g in grads]
        return outs, real(grads, max_norm)[1]
    monkeypatch.setattr(O, "clip_by_global_norm", broken)
    assert check_clip(O) > 1e-3


# ----------------------------------------------------------------------------
# Transformer layer: Philox dropout, LayerNorm, the whole layer
# ----------------------------------------------------------------------------
def check_philox(mod):
    """Largest number of mismatching output words over the published
    known-answer vectors (each vector also evaluated inside a batch)."""
    kat = golden("philox4x32_kat.json")["vectors"]
    bad = 0
    for v in kat:
        c = [int(x, 16) for x in v["ctr"]]
        k = [int(x, 16) for x in v["key"]]
        out = mod.philox4x32(*c, *k)
        bad += sum(int(out[j]) != int(v["out"][j], 16) for j in range(4))
        # the same counter as the middle element of an array of counters
        arr = mod.philox4x32(np.array([c[0] ^ 1, c[0], c[0] ^ 2], dtype=np.uint64), c[1], c[2], c[3], *k)
        bad += sum(int(arr[j][1]) != int(v["out"][j], 16) for j in range(4))
    return bad


def test_philox4x32_known_answers():
    assert check_philox(O) == 0


def test_planted_philox_key_schedule_off_by_one_round_is_caught(monkeypatch):
    real_w0 = O._PH_W0
    monkeypatch.setattr(O, "_PH_W0", (real_w0 + 1) & 0xFFFFFFFF)
    assert check_philox(O) > 0


def test_dropout_keep_layout_against_the_generator_directly():
    # element e: word (e mod 8) / 2, field 16 (e mod 2) at counter (e / 8, 0, stream, 0)
    seed, stream, p = (7 << 32) | 5, 3, 0.25
    k = O.dropout_keep(seed, stream, 40, 24, p)
    thr = math.floor(p * 65536)
    for i, e in enumerate(range(40, 64)):
        w = O.philox4x32(e // 8, 0, stream, 0, 5, 7)
        field = (int(w[(e % 8) // 2]) >> (16 * (e % 2))) & 0xFFFF
        assert bool(k[i]) == (field >= thr)


def test_dropout_keep_rate_and_streams():
    n, p = 200000, 0.1
    k = O.dropout_keep(11, 3, 0, n, p)
    keep = 1 - math.floor(p * 65536) / 65536
    assert abs(k.mean() - keep) < 5 * math.sqrt(keep * (1 - keep) / n)
    assert not np.array_equal(k, O.dropout_keep(11, 4, 0, n, p))      # another stream
    assert not np.array_equal(k, O.dropout_keep(11 + (1 << 32), 3, 0, n, p))  # the seed's upper word counts
    assert np.array_equal(k[1000:2000], O.dropout_keep(11, 3, 1000, 1000, p))  # offsets
    assert O.dropout_keep(11, 3, 0, 1000, 0.0).all()
    # the attention streams differ per shard, the hidden ones do not
    assert O.dropout_stream(2, 0, 0) != O.dropout_stream(2, 0, 1)
    assert O.dropout_stream(2, 1, 0) == O.dropout_stream(2, 1, 1)


def check_layernorm(mod):
    g = rng(21)
    x = g.standard_normal((7, 12)) * 3 + 1
    gam, bet = g.standard_normal(12), g.standard_normal(12)
    dy = g.standard_normal((7, 12))
    y, mean, rstd = mod.layernorm(x, gam, bet, 1e-5)
    tx = torch.tensor(x, requires_grad=True)
    tg, tb = torch.tensor(gam, requires_grad=True), torch.tensor(bet, requires_grad=True)
    ty = F.layer_norm(tx, (12,), tg, tb, 1e-5)
    ty.backward(torch.tensor(dy))
    dx, dg, db = mod.layernorm_grad(dy, x, gam, mean, rstd)
    return max(np.abs(y - ty.detach().numpy()).max(), np.abs(dx - tx.grad.numpy()).max(),
               np.abs(dg - tg.grad.numpy()).max(), np.abs(db - tb.grad.numpy()).max())


def test_layernorm_matches_torch():
    assert check_layernorm(O) < 1e-12


def tiny_layer(seed=31, s=6, b=2, h=16, H=4, N=2, hp=32, p_attn=0.2, p_hidden=0.25):
    g = rng(seed)
    T = b * s
    d = h // N
    Wqkv = g.standard_normal((3 * h, h)) * 0.3
    Wo = g.standard_normal((h, h)) * 0.3
    W = g.standard_normal((hp, h)) * 0.3
    U = g.standard_normal((h, hp)) * 0.3
    P = dict(g1=1 + 0.1 * g.standard_normal(h), b1=0.1 * g.standard_normal(h),
             bqkv_full=0.1 * g.standard_normal(3 * h), bo=0.1 * g.standard_normal(h),
             g2=1 + 0.1 * g.standard_normal(h), b2=0.1 * g.standard_normal(h),
             a_full=0.1 * g.standard_normal(hp), b=0.1 * g.standard_normal(h),
             Wqkv_full=Wqkv, Wo_full=Wo, W_full=W, U_full=U)
    P["Wqkv"] = [np.concatenate([Wqkv[j * h + i * d: j * h + (i + 1) * d] for j in range(3)]) for i in range(N)]
    P["bqkv"] = [np.concatenate([P["bqkv_full"][j * h + i * d: j * h + (i + 1) * d] for j in range(3)])
                 for i in range(N)]
    P["Wo"] = [Wo[:, i * d:(i + 1) * d] for i in range(N)]
    n = hp // N
    P["W"] = [W[i * n:(i + 1) * n] for i in range(N)]
    P["a"] = [P["a_full"][i * n:(i + 1) * n] for i in range(N)]
    P["U"] = [U[:, i * n:(i + 1) * n] for i in range(N)]
    cfg = dict(s=s, n_heads=H, N=N, causal=True, eps=1e-5, p_attn=p_attn, p_hidden=p_hidden,
               seed=77, layer=3)
    x = g.standard_normal((T, h))
    dout = g.standard_normal((T, h))
    return x, dout, P, cfg


def torch_layer(x, P, cfg, mod):
    """The same layer written with torch ops on the unsharded weights."""
    s, H, N = cfg["s"], cfg["n_heads"], cfg["N"]
    T, h = x.shape
    d = h // H
    b = T // s
    t = {k: torch.tensor(v, requires_grad=True) for k, v in P.items() if not isinstance(v, list)}
    tx = torch.tensor(x, requires_grad=True)
    ln1 = F.layer_norm(tx, (h,), t["g1"], t["b1"], cfg["eps"])
    qkv = F.linear(ln1, t["Wqkv_full"], t["bqkv_full"])
    q, k, v = qkv[:, :h], qkv[:, h:2 * h], qkv[:, 2 * h:]
    ctx = []
    for bi in range(b):
        heads = []
        for j in range(H):
            r, c = slice(bi * s, (bi + 1) * s), slice(j * d, (j + 1) * d)
            S = q[r, c] @ k[r, c].T / math.sqrt(d)
            S = S.masked_fill(torch.triu(torch.ones(s, s, dtype=torch.bool), 1), float("-inf"))
            Pj = torch.softmax(S, dim=1)
            keep = mod.attention_keep(bi, j, s, H, N, cfg["p_attn"], cfg["seed"], cfg["layer"])
            Pj = Pj * torch.tensor(keep) / (1 - cfg["p_attn"])
            heads.append(Pj @ v[r, c])
        ctx.append(torch.cat(heads, dim=1))
    C = torch.cat(ctx, dim=0)
    p = cfg["p_hidden"]
    k1 = torch.tensor(mod.dropout_keep(cfg["seed"], mod.dropout_stream(cfg["layer"], 1), 0, T * h, p).reshape(T, h))
    k2 = torch.tensor(mod.dropout_keep(cfg["seed"], mod.dropout_stream(cfg["layer"], 2), 0, T * h, p).reshape(T, h))
    h1 = tx + F.linear(C, t["Wo_full"], t["bo"]) * k1 / (1 - p)
    ln2 = F.layer_norm(h1, (h,), t["g2"], t["b2"], cfg["eps"])
    M = F.linear(F.gelu(F.linear(ln2, t["W_full"], t["a_full"])), t["U_full"], t["b"])
    return tx, t, h1 + M * k2 / (1 - p)


def check_layer(mod):
    x, dout, P, cfg = tiny_layer()
    out, saved = mod.transformer_layer_fwd(x, P, cfg)
    grads = mod.transformer_layer_bwd(dout, saved, P, cfg)
    tx, t, tout = torch_layer(x, P, cfg, mod)
    tout.backward(torch.tensor(dout))
    h = x.shape[1]
    N = cfg["N"]
    d = h // N
    err = np.abs(out - tout.detach().numpy()).max()
    err = max(err, np.abs(grads["dx"] - tx.grad.numpy()).max())
    for k in ("g1", "b1", "bo", "g2", "b2", "b"):
        err = max(err, np.abs(grads["d" + k] - t[k].grad.numpy()).max())
    gW, gU, gWqkv, gWo = t["W_full"].grad.numpy(), t["U_full"].grad.numpy(), t["Wqkv_full"].grad.numpy(), t["Wo_full"].grad.numpy()
    n = gW.shape[0] // N
    for i in range(N):
        err = max(err, np.abs(grads["dW"][i] - gW[i * n:(i + 1) * n]).max(),
                  np.abs(grads["dU"][i] - gU[:, i * n:(i + 1) * n]).max(),
                  np.abs(grads["da"][i] - t["a_full"].grad.numpy()[i * n:(i + 1) * n]).max(),
                  np.abs(grads["dWo"][i] - gWo[:, i * d:(i + 1) * d]).max())
        ref_qkv = np.concatenate([gWqkv[j * h + i * d: j * h + (i + 1) * d] for j in range(3)])
        ref_b = np.concatenate([t["bqkv_full"].grad.numpy()[j * h + i * d: j * h + (i + 1) * d] for j in range(3)])
        err = max(err, np.abs(grads["dWqkv"][i] - ref_qkv).max(), np.abs(grads["dbqkv"][i] - ref_b).max())
    return err


def test_transformer_layer_matches_torch_autograd():
    assert check_layer(O) < 1e-10


def test_position_embedding_input_against_torch_embedding():
    """The first layer's input: without dropout it is torch's embedding lookup
    of the positions plus the words; with a keep mask the dropped entries are
    exactly zero and the kept ones that sum divided by 1 - p (inverted
    dropout); a position outside the table adds nothing."""
    g = rng(31)
    T, h, P = 12, 8, 10
    words = g.standard_normal((T, h))
    table = g.standard_normal((P, h))
    pos = g.integers(0, P, T)
    ref = torch.nn.functional.embedding(torch.tensor(pos), torch.tensor(table)).numpy() + words
    out = O.embed_position_dropout(words, table, pos, np.ones((T, h)), 0.0)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-15)
    keep = g.random((T, h)) >= 0.25
    out = O.embed_position_dropout(words, table, pos, keep, 0.25)
    assert np.all(out[~keep] == 0.0)
    np.testing.assert_allclose(out[keep] * 0.75, ref[keep], rtol=1e-15, atol=1e-15)
    bad = pos.copy()
    bad[[0, 5]] = [-1, P]
    out = O.embed_position_dropout(words, table, bad, np.ones((T, h)), 0.0)
    np.testing.assert_array_equal(out[[0, 5]], words[[0, 5]])
    np.testing.assert_allclose(np.delete(out, [0, 5], 0), np.delete(ref, [0, 5], 0), rtol=0, atol=1e-15)


def test_planted_unbiased_layernorm_variance_is_caught(monkeypatch):
    def broken(x, g, b, eps):
        x = np.asarray(x, dtype=np.float64)
        mean = x.mean(axis=-1)
        var = x.var(axis=-1, ddof=1)
        rstd = 1.0 / np.sqrt(var + eps)
        return (x - mean[..., None]) * rstd[..., None] * g + b, mean, rstd
    monkeypatch.setattr(O, "layernorm", broken)
    assert check_layernorm(O) > 1e-3


def test_planted_unscaled_dropout_is_caught(monkeypatch):
    monkeypatch.setattr(O, "dropout_residual", lambda res, x, keep, p: res + x * keep)
    assert check_layer(O) > 1e-3


def test_planted_dropped_residual_gradient_is_caught(monkeypatch):
    real = O.layernorm_grad
    calls = []

    def broken(dy, x, g, mean, rstd):
        dx, dg, db = real(dy, x, g, mean, rstd)
        calls.append(1)
        return (dx - dy * 0.5 if len(calls) == 1 else dx), dg, db  # a wrong term in LN2's dx
    monkeypatch.setattr(O, "layernorm_grad", broken)
    assert check_layer(O) > 1e-3


def test_planted_shared_attention_dropout_stream_is_caught(monkeypatch):
    # every shard drawing from shard 0's stream is a plausible mistake: the
    # stream layout makes the shards' masks differ, which this detects
    real = O.dropout_stream
    monkeypatch.setattr(O, "dropout_stream", lambda layer, kind, shard=0: real(layer, kind, 0))
    x, dout, P, cfg = tiny_layer()
    k0 = O.attention_keep(0, 0, cfg["s"], cfg["n_heads"], cfg["N"], 0.5, 1, 0)
    k_other_shard = O.attention_keep(0, cfg["n_heads"] - 1, cfg["s"], cfg["n_heads"], cfg["N"], 0.5, 1, 0)
    monkeypatch.undo()
    r0 = O.attention_keep(0, 0, cfg["s"], cfg["n_heads"], cfg["N"], 0.5, 1, 0)
    r1 = O.attention_keep(0, cfg["n_heads"] - 1, cfg["s"], cfg["n_heads"], cfg["N"], 0.5, 1, 0)
    assert np.array_equal(k0, r0) and not np.array_equal(k_other_shard, r1)
