"""GPU parity of the vocab-parallel cross-entropy against the fp64 oracle,
through the C ABI (tp_vocab_cross_entropy_fwd / _bwd).

The forward never stores the logits: it keeps per-part (max, sum exp) pairs
and merges them in fixed order.  Its loss and log-sum-exp are fp32 results of
fp32-accumulated bf16 products (no bf16 rounding of logits), so they are held
to 1e-3 relative; dLogits and dX are bf16 outputs (2e-2).
"""
import numpy as np
import pytest
import torch

import oracle.tp_oracle as O
import synthetic_inputs as SI
from tests.gpu_util import assert_close, dev, f64, f64_list, rel_err

pytestmark = pytest.mark.gpu

LOSS_TOL = 1e-3


def _tp():
    import megatron_tensor_transformer_tp_gb300 as tp
    return tp


def run_ce(X, E_shards, ranges, targets, dloss, with_dx=True):
    tp = _tp()
    T, h = X.shape
    d = lambda t: t.cuda().contiguous()
    Xd, Es = d(X), [d(e) for e in E_shards]
    tg = d(targets)
    loss = torch.full((T,), float("nan"), device="cuda")
    lse = torch.full((T,), float("nan"), device="cuda")
    ws = torch.empty(tp.tp_vocab_cross_entropy_workspace_size(T, ranges[-1], ranges),
                     dtype=torch.uint8, device="cuda")
    tp.tp_vocab_cross_entropy_fwd(Xd, Es, ranges, tg, loss, lse, ws)
    dl = d(dloss)
    dLog = [torch.full((T, tp.logits_pitch(ranges[r + 1] - ranges[r], torch.bfloat16)), float("nan"),
                       dtype=torch.bfloat16, device="cuda") for r in range(len(E_shards))]
    dX = torch.full((T, h), float("nan"), dtype=torch.bfloat16, device="cuda") if with_dx else None
    tp.tp_vocab_cross_entropy_bwd(Xd, Es, ranges, tg, lse, dl, dLog, dX)
    assert tp.tp_get_status() == tp.TP_OK
    widths = [ranges[r + 1] - ranges[r] for r in range(len(E_shards))]
    return loss, lse, [g[:, :w] for g, w in zip(dLog, widths)], dX


def make_case(T, h, ranges, seed, invalid=()):
    g = np.random.default_rng(seed)
    V = ranges[-1]
    X = SI.normal(seed, 1, (T, h), 1.0, "bf16")
    E = SI.normal(seed, 2, (V, h), 0.05, "bf16")
    targets = torch.from_numpy(g.integers(0, V, T).astype(np.int64))
    for i, v in invalid:
        targets[i] = v
    dloss = torch.from_numpy(g.standard_normal(T).astype(np.float32))
    Es = [E[ranges[r]:ranges[r + 1]].contiguous() for r in range(len(ranges) - 1)]
    return X, E, Es, targets, dloss


def check_full(X, Es, ranges, targets, dloss, res):
    loss, lse, dLog, dX = res
    Xn, En = f64(X), f64_list(Es)
    t, dl = targets.numpy(), dloss.double().numpy()
    rl, rlse = O.vocab_parallel_cross_entropy(Xn, En, ranges, t)
    assert rel_err(loss, rl) <= LOSS_TOL, rel_err(loss, rl)
    assert rel_err(lse, rlse) <= LOSS_TOL, rel_err(lse, rlse)
    g = O.vocab_parallel_cross_entropy_grad(Xn, En, ranges, t, dl)
    for r, (a, b) in enumerate(zip(dLog, g)):
        assert_close(a, b, "bf16", f"dLogits[{r}]")
    if dX is not None:
        # dX sums products of the saved bf16 dLogits: element-wise measure reported
        assert_close(dX, O.logits_side_dx(g, En), "bf16", "dX", elementwise=False)


@pytest.mark.parametrize("T,h,ranges", [(200, 256, [0, 333, 1000]), (129, 128, [0, 64, 65, 300]),
                                        (300, 512, [0, 2048]), (1, 64, [0, 70, 140]),
                                        (150, 128, [0, 1, 9, 130, 131, 400, 512, 700, 1000])])
def test_ce_ragged_parity(T, h, ranges):
    X, E, Es, targets, dloss = make_case(T, h, ranges, seed=T + h)
    check_full(X, Es, ranges, targets, dloss, run_ce(X, Es, ranges, targets, dloss))


def test_ce_targets_in_no_range():
    # the pages' masking: predicted logit 0, so loss = log(sum of shifted exp)
    ranges = [0, 400, 900]
    X, E, Es, targets, dloss = make_case(160, 256, ranges, seed=5,
                                         invalid=[(0, -1), (7, 900), (100, 10**9)])
    check_full(X, Es, ranges, targets, dloss, run_ce(X, Es, ranges, targets, dloss))


def test_ce_deterministic_and_no_dx():
    ranges = [0, 777, 1500]
    X, E, Es, targets, dloss = make_case(257, 256, ranges, seed=6)
    a = run_ce(X, Es, ranges, targets, dloss)
    b = run_ce(X, Es, ranges, targets, dloss, with_dx=False)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for x, y in zip(a[2], b[2]):
        assert torch.equal(x, y)
    assert b[3] is None


def test_ce_embed_tied_V50257_h4096_T8192_sampled():
    """The tied-embedding workload: loss and log-sum-exp of every token are
    checked against the oracle on sampled rows (the oracle is per row), and
    dLogits / dX on the same rows."""
    cfg = SI.WORKLOADS["embed_tied_V50257_h4096_T8192"]
    e = SI.embed_inputs(cfg)
    T, h, ranges = e["ids"].numel(), e["h"], e["ranges"]
    g = np.random.default_rng(7)
    targets = torch.from_numpy(g.integers(0, ranges[-1], T).astype(np.int64))
    dloss = torch.full((T,), 1.0 / T)
    X, Es = e["X"], e["E_shards"]
    loss, lse, dLog, dX = run_ce(X, Es, ranges, targets, dloss)
    rows = np.sort(g.choice(T, 24, replace=False)).tolist() + [0, T - 1]
    Xn, En = f64(X)[rows], f64_list(Es)
    t, dl = targets.numpy()[rows], dloss.double().numpy()[rows]
    rl, rlse = O.vocab_parallel_cross_entropy(Xn, En, ranges, t)
    assert rel_err(loss[rows], rl) <= LOSS_TOL
    assert rel_err(lse[rows], rlse) <= LOSS_TOL
    gr = O.vocab_parallel_cross_entropy_grad(Xn, En, ranges, t, dl)
    for r in range(len(Es)):
        assert_close(dLog[r][rows], gr[r], "bf16", f"dLogits[{r}] rows")
    assert_close(dX[rows], O.logits_side_dx(gr, En), "bf16", "dX rows", elementwise=False)
    assert torch.isfinite(loss).all() and torch.isfinite(dX.float()).all()
