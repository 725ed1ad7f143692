"""GPU parity of the vocab-parallel embedding, the per-range logits and the
tied embedding gradient against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle.tp_oracle as O
import synthetic_inputs as SI
from tests.gpu_util import assert_close, dev, dev_list, f64, f64_list

pytestmark = pytest.mark.gpu


def _tp():
    import megatron_tensor_transformer_tp_gb300 as tp
    return tp


def padded(t, dtype):
    """Copy of a (T, n) shard into a device buffer with a TMA-friendly pitch."""
    tp = _tp()
    T, n = t.shape
    buf = torch.zeros(T, tp.logits_pitch(n, dtype), dtype=dtype, device="cuda")
    buf[:, :n] = t.cuda()
    return buf


def gather(inp, ids=None):
    tp = _tp()
    ids = inp["ids"] if ids is None else ids
    dt = torch.bfloat16 if inp["dtype"] == "bf16" else torch.float32
    out = torch.full((ids.numel(), inp["h"]), float("nan"), dtype=dt, device="cuda")
    tp.vocab_parallel_embed(dev(ids), dev_list(inp["E_shards"]), inp["ranges"], out)
    assert tp.tp_get_status() == tp.TP_OK
    return out


def test_embed_tiny_fp32_page_example_bit_exact():
    """V=300, ranges [0,150) / [150,300), ids [0,212,7,9]."""
    inp = SI.embed_inputs(SI.WORKLOADS["embed_tiny_f32"])
    out = gather(inp)
    ref = O.vocab_parallel_embed(inp["ids"].numpy(), f64_list(inp["E_shards"]), inp["ranges"])
    assert np.array_equal(f64(out), ref)


@pytest.mark.parametrize("dtype,h", [("f32", 16), ("bf16", 64), ("bf16", 20), ("f32", 3)])
def test_embed_brute_force_ids_and_out_of_range(dtype, h):
    V = 61
    cfg = dict(kind="embed", dtype=dtype, V=V, h=h, b=1, s=1, ranges=[0, 7, 30, 61], seed=5)
    inp = SI.embed_inputs(cfg, T=1)
    ids = torch.tensor(list(range(V)) + [-1, V, V + 100, -(2 ** 40), 2 ** 40, 3, 3], dtype=torch.int64)
    out = gather(inp, ids)
    ref = O.vocab_parallel_embed(ids.numpy(), f64_list(inp["E_shards"]), inp["ranges"])
    assert np.array_equal(f64(out), ref)


def test_embed_tied_V50257_h4096_T8192_gather_bit_exact():
    inp = SI.embed_inputs(SI.WORKLOADS["embed_tied_V50257_h4096_T8192"])
    out = gather(inp)
    ids = inp["ids"].numpy()
    Es = [e.float().numpy() for e in inp["E_shards"]]  # exact widening of bf16
    got = f64(out)
    for c in range(0, len(ids), 2048):
        ref = O.vocab_parallel_embed(ids[c:c + 2048], Es, inp["ranges"])
        assert np.array_equal(got[c:c + 2048], ref)


def test_embed_empty_tokens():
    inp = SI.embed_inputs(SI.WORKLOADS["embed_tiny_f32"])
    out = gather(inp, torch.zeros(0, dtype=torch.int64))
    assert out.numel() == 0


# ----------------------------------------------------------------------------
# logits per range
# ----------------------------------------------------------------------------
def run_logits(inp):
    tp = _tp()
    dt = torch.bfloat16 if inp["dtype"] == "bf16" else torch.float32
    T = inp["T"]
    rs = inp["ranges"]
    L = [torch.full((T, tp.logits_pitch(rs[r + 1] - rs[r], dt)), float("nan"), dtype=dt, device="cuda")
         for r in range(inp["N"])]
    tp.tp_vocab_logits(dev(inp["X"]), dev_list(inp["E_shards"]), rs, L)
    assert tp.tp_get_status() == tp.TP_OK
    return [L[r][:, :rs[r + 1] - rs[r]] for r in range(inp["N"])]


@pytest.mark.parametrize("dtype,V,h,T,ranges", [("bf16", 1000, 136, 333, [0, 333, 1000]),
                                                ("f32", 300, 16, 50, [0, 150, 300]),
                                                ("bf16", 777, 256, 129, [0, 1, 300, 777]),
                                                # eight ranges of uneven widths, one of a single word
                                                ("bf16", 1000, 128, 200, [0, 1, 9, 130, 131, 400, 512, 700, 1000])])
def test_logits_small_full(dtype, V, h, T, ranges):
    cfg = dict(kind="embed", dtype=dtype, V=V, h=h, b=1, s=T, ranges=ranges, seed=11)
    inp = SI.embed_inputs(cfg)
    L = run_logits(inp)
    ref = O.vocab_logits(f64(inp["X"]), f64_list(inp["E_shards"]))
    for r in range(inp["N"]):
        assert_close(L[r], ref[r], dtype, f"L[{r}]")


def test_logits_V50257_h4096_T8192_sampled():
    inp = SI.embed_inputs(SI.WORKLOADS["embed_tied_V50257_h4096_T8192"])
    L = run_logits(inp)
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(inp["T"], 24, replace=False)).tolist() + [inp["T"] - 1]
    ref = O.vocab_logits(f64(inp["X"][rows]), [e.float().numpy() for e in inp["E_shards"]])
    for r in range(inp["N"]):
        assert_close(L[r][rows], ref[r], "bf16", f"L[{r}] rows")
        assert torch.isfinite(L[r]).all()


# ----------------------------------------------------------------------------
# tied embedding gradient
# ----------------------------------------------------------------------------
def run_tied(inp, with_logits=True, accumulate=False, init=None, ids=None):
    tp = _tp()
    dt = torch.bfloat16 if inp["dtype"] == "bf16" else torch.float32
    ids = inp["ids"] if ids is None else ids
    T, V, h, rs = ids.numel(), inp["V"], inp["h"], inp["ranges"]
    dL = [padded(t, dt) for t in inp["dLogits_shards"]] if with_logits else None
    if init is None:
        dE = [torch.full((rs[r + 1] - rs[r], h), float("nan"), dtype=torch.float32, device="cuda")
              for r in range(inp["N"])]
    else:
        dE = [x.clone() for x in init]
    ws = torch.empty(tp.tied_embed_grad_workspace_size(T, V), dtype=torch.uint8, device="cuda")
    tp.tied_embed_grad(dev(ids), dev(inp["dEmb"][:T]), dev(inp["X"][:T]), dL, rs, dE,
                       accumulate=accumulate, workspace=ws)
    assert tp.tp_get_status() == tp.TP_OK
    return dE, ws


def sort_view(ws, T, V):
    w = ws.cpu().numpy()
    offs = w[:4 * (V + 1)].view(np.int32).astype(np.int64)
    start = (4 * (V + 1) + 255) // 256 * 256
    perm = w[start:start + 4 * T].view(np.int32).astype(np.int64)
    return offs, perm


@pytest.mark.parametrize("dtype,V,h,T,ranges", [("bf16", 1000, 136, 777, [0, 333, 1000]),
                                                ("f32", 300, 16, 40, [0, 150, 300]),
                                                ("bf16", 64, 256, 300, [0, 5, 64]),
                                                ("bf16", 1000, 128, 500, [0, 1, 9, 130, 131, 400, 512, 700, 1000])])
def test_tied_grad_small_full(dtype, V, h, T, ranges):
    cfg = dict(kind="embed", dtype=dtype, V=V, h=h, b=1, s=T, ranges=ranges, seed=12)
    inp = SI.embed_inputs(cfg)
    ids = inp["ids"].clone()
    ids[:5] = 7          # a repeated id
    ids[5] = -1          # masked ids contribute nothing
    ids[6] = V
    dE, ws = run_tied(inp, ids=ids)
    dLf = [f64(t) for t in inp["dLogits_shards"]]
    ref = O.tied_embed_grad(ids.numpy(), f64(inp["dEmb"]), f64(inp["X"]), dLf, ranges, V)
    for r in range(inp["N"]):
        assert_close(dE[r], ref[r], dtype, f"dE[{r}]")
    # index work: bit-exact against the oracle's grouping
    offs, perm = sort_view(ws, T, V)
    o_offs, o_perm = O.embed_sort(ids.numpy(), V)
    assert np.array_equal(offs, o_offs)
    assert np.array_equal(perm[:o_offs[-1]], o_perm)
    # input-side part alone (no output-layer gradient)
    dE0, _ = run_tied(inp, with_logits=False, ids=ids)
    sc = O.embed_scatter_grad(ids.numpy(), f64(inp["dEmb"]), V)
    for r in range(inp["N"]):
        assert_close(dE0[r], sc[ranges[r]:ranges[r + 1]], dtype, f"scatter[{r}]")
    # accumulate into ones
    ones = [torch.ones(ranges[r + 1] - ranges[r], h, device="cuda") for r in range(inp["N"])]
    dE1, _ = run_tied(inp, accumulate=True, init=ones, ids=ids)
    for r in range(inp["N"]):
        assert_close(dE1[r], ref[r] + 1.0, dtype, f"acc dE[{r}]")


def test_tied_grad_empty_tokens_zero():
    cfg = dict(kind="embed", dtype="bf16", V=100, h=64, b=1, s=1, ranges=[0, 50, 100], seed=13)
    inp = SI.embed_inputs(cfg)
    inp["dLogits_shards"] = [t[:0] for t in inp["dLogits_shards"]]
    dE, _ = run_tied(inp, ids=torch.zeros(0, dtype=torch.int64))
    for t in dE:
        assert torch.count_nonzero(t) == 0


def test_tied_grad_V50257_h4096_T8192_sampled_and_deterministic():
    inp = SI.embed_inputs(SI.WORKLOADS["embed_tied_V50257_h4096_T8192"])
    dE, ws = run_tied(inp)
    T, V, rs = inp["T"], inp["V"], inp["ranges"]
    ids = inp["ids"].numpy()
    offs, perm = sort_view(ws, T, V)
    o_offs, o_perm = O.embed_sort(ids, V)
    assert np.array_equal(offs, o_offs) and np.array_equal(perm[:T], o_perm)
    rng = np.random.default_rng(4)
    vocab_rows = sorted(set(rng.choice(V, 24, replace=False).tolist()
                            + ids[:8].tolist() + [0, rs[1] - 1, rs[1], V - 1]))
    dL_full = np.concatenate([t.float().numpy() for t in inp["dLogits_shards"]], axis=1)
    ref = O.tied_embed_grad_rows(ids, f64(inp["dEmb"]), f64(inp["X"]), dL_full, vocab_rows)
    for k, v in enumerate(vocab_rows):
        r = 0 if v < rs[1] else 1
        assert_close(dE[r][v - rs[r]][None, :], ref[k][None, :], "bf16", f"dE row {v}")
    dE2, _ = run_tied(inp)
    for r in range(2):
        assert torch.equal(dE[r], dE2[r])
