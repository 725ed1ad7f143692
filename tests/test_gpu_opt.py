"""GPU parity of the mixed-precision Adam step (tp_adam_step) against the fp64
oracle, through the C ABI.

Per-element arithmetic is fp32 on the device, so parameters, moments and the
parameter update itself are held to the fp32 bar (1e-4 max relative error);
the loss scale, trackers, step count and overflow flag must match exactly;
the bf16 model copy must equal the round-to-nearest-even bf16 of the device's
own fp32 parameters bit for bit, and the oracle's parameters within the bf16
bar.
"""
import math

import numpy as np
import pytest
import torch

import oracle.tp_oracle as O
import synthetic_inputs as SI
from tests.gpu_util import TOL, assert_close, rel_err

pytestmark = pytest.mark.gpu

HYPER = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, max_norm=0.1, use_scaler=1, min_scale=1.0,
             growth_factor=2.0, backoff_factor=0.5, growth_interval=1000, hysteresis=2)
STATE = dict(scale=1024.0, growth_tracker=0, hysteresis_tracker=2, step=7)
SEED = 1006


def _tp():
    import megatron_tensor_transformer_tp_gb300 as tp
    return tp


def make_groups(sizes, seed=SEED, scale=1024.0, grad_std=1e-3):
    """fp32 CPU groups from the shared generator (as adam_inputs, other sizes)."""
    cfg = dict(SI.WORKLOADS["adam_layer_H4096"], seed=seed,
               state=dict(STATE, scale=scale))
    gs = SI.adam_inputs(cfg, sizes=sizes)["groups"]
    if grad_std != 1e-3:
        for g in gs:
            g["grad"] *= grad_std / 1e-3
    return gs


class DeviceOpt:
    """Device copies of the groups, the state and the workspace."""

    def __init__(self, groups, state, with_model=True):
        tp = _tp()
        self.g = []
        for i, grp in enumerate(groups):
            d = {k: grp[k].cuda().contiguous() for k in ("param", "grad", "m", "v")}
            n = grp["param"].numel()
            use_model = with_model if isinstance(with_model, bool) else with_model[i]
            # sentinel: bf16 NaN, so an unwritten copy shows
            d["model"] = torch.full((n,), float("nan"), dtype=torch.bfloat16, device="cuda") \
                if use_model else None
            d["weight_decay"] = grp["weight_decay"]
            self.g.append(d)
        self.state = tp.make_optimizer_state(**state)
        self.ws = torch.empty(tp.tp_adam_step_workspace_size(), dtype=torch.uint8, device="cuda")

    def step(self, hyper):
        tp = _tp()
        tp.tp_adam_step(self.g, hyper, self.state, self.ws)
        assert tp.tp_get_status() == tp.TP_OK
        return tp.read_optimizer_state(self.state)

    def set_grads(self, groups):
        for d, grp in zip(self.g, groups):
            d["grad"].copy_(grp["grad"])


def oracle_groups(groups):
    return [dict(param=g["param"].double().numpy(), grad=g["grad"].double().numpy(),
                 m=g["m"].double().numpy(), v=g["v"].double().numpy(),
                 weight_decay=g["weight_decay"]) for g in groups]


def check_against(dev, before, ref_groups, ref_state, ref_norm, st, updated):
    """Device results vs the oracle's step; `before` are the inputs."""
    for k in ("scale", "growth_tracker", "hysteresis_tracker", "step"):
        assert st[k] == ref_state[k], (k, st[k], ref_state[k])
    assert st["found_inf"] == int(not updated)
    if math.isfinite(ref_norm):
        assert abs(st["grad_norm"] - ref_norm) <= TOL["f32"] * ref_norm, (st["grad_norm"], ref_norm)
    else:
        assert not math.isfinite(st["grad_norm"])
    for i, (d, b, r) in enumerate(zip(dev.g, before, ref_groups)):
        if b["param"].numel() == 0:
            continue
        p = d["param"].cpu()
        if not updated:
            # a skipped step leaves every buffer as it was
            for k in ("param", "m", "v"):
                assert torch.equal(d[k].cpu(), b[k]), (i, k)
            if d["model"] is not None:
                assert torch.isnan(d["model"].float()).all()
            continue
        assert_close(p, r["param"], "f32", f"param[{i}]")
        # the update itself, not only the parameter it is added to (recovered as a
        # difference of fp32 parameters, each element carries the parameter's 2^-24
        # relative rounding: element-wise measure reported, not asserted)
        assert_close(p.double() - b["param"].double(), r["param"] - b["param"].double().numpy(),
                     "f32", f"param update[{i}]", elementwise=False)
        assert_close(d["m"], r["m"], "f32", f"m[{i}]")
        assert_close(d["v"], r["v"], "f32", f"v[{i}]")
        if d["model"] is not None:
            assert torch.equal(d["model"].cpu(), p.to(torch.bfloat16)), f"model[{i}] != bf16(param)"
            assert_close(d["model"], r["param"], "bf16", f"model[{i}]")


def run_and_check(groups, state, hyper, with_model=True):
    dev = DeviceOpt(groups, state, with_model)
    st = dev.step(hyper)
    updated, norm, ref, ref_state = O.mixed_precision_adam_step(oracle_groups(groups), state, hyper)
    check_against(dev, groups, ref, ref_state, norm, st, updated)
    return dev, st


RAGGED = [1, 3, 8191, 8192, 8193, 100003, 0, 17, 4]


def test_adam_ragged_groups_clipped_with_scaler():
    groups = make_groups(RAGGED)
    _, st = run_and_check(groups, STATE, HYPER, with_model=[i % 3 != 1 for i in range(len(RAGGED))])
    assert st["grad_norm"] > HYPER["max_norm"]  # the clip was active


def test_adam_no_clip_no_scaler():
    groups = make_groups([5000, 12345], scale=1.0)
    hyper = dict(HYPER, max_norm=0.0, use_scaler=0)
    run_and_check(groups, dict(STATE, scale=1.0), hyper)


def test_adam_norm_below_threshold_leaves_gradients():
    # ||g|| < max_norm: no clipping
    groups = make_groups([20000], grad_std=1e-5)
    _, st = run_and_check(groups, STATE, dict(HYPER, max_norm=10.0))
    assert st["grad_norm"] < 10.0


def test_adam_first_step_bias_correction():
    groups = make_groups([3000, 4096])
    for g in groups:
        g["m"].zero_()
        g["v"].zero_()
    run_and_check(groups, dict(STATE, step=0), HYPER)


@pytest.mark.parametrize("bad", [float("inf"), float("-inf"), float("nan")])
def test_adam_overflow_skips_step(bad):
    groups = make_groups([9000, 700])
    groups[1]["grad"][123] = bad
    _, st = run_and_check(groups, STATE, HYPER)
    assert st["found_inf"] == 1 and st["step"] == STATE["step"]


def test_adam_overflow_after_unscale():
    # finite in fp32 as stored, but the unscaled value is inf only if the scale is < 1:
    # with scale 0.5 (min_scale below 1) 3e38 / 0.5 overflows fp32
    groups = make_groups([100], scale=1.0)
    groups[0]["grad"][5] = 3e38
    st0 = dict(STATE, scale=0.5)
    hyper = dict(HYPER, min_scale=0.25)
    dev = DeviceOpt(groups, st0)
    st = dev.step(hyper)
    assert st["found_inf"] == 1
    # the oracle divides in fp64, where 6e38 is finite: the device's overflow is
    # the fp32 one, so only the fp32 case is compared here
    assert st["hysteresis_tracker"] == 1 and st["scale"] == 0.5


def test_adam_scaler_sequence():
    """Six chained steps: two overflows (hysteresis 2 then back-off), then
    growth after growth_interval clean steps; each side chains its own state."""
    hyper = dict(HYPER, growth_interval=2, hysteresis=2)
    sizes = [4099, 8192 * 3 + 5]
    groups = make_groups(sizes)
    dev = DeviceOpt(groups, STATE)
    ref_groups, ref_state = oracle_groups(groups), dict(STATE)
    schedule = [False, True, True, False, False, False]  # overflow at steps 1 and 2
    for k, overflow in enumerate(schedule):
        gk = make_groups(sizes, seed=SEED + 1 + k)
        if overflow:
            gk[0]["grad"][k] = float("inf")
        dev.set_grads(gk)
        before = [dict(param=d["param"].cpu(), m=d["m"].cpu(), v=d["v"].cpu()) for d in dev.g]
        for d in dev.g:
            d["model"].fill_(float("nan"))
        for rg, g in zip(ref_groups, gk):
            rg["grad"] = g["grad"].double().numpy()
        st = dev.step(hyper)
        updated, norm, ref_groups, ref_state = O.mixed_precision_adam_step(ref_groups, ref_state, hyper)
        assert updated == (not overflow)
        check_against(dev, before, ref_groups, ref_state, norm, st, updated)
    assert ref_state["scale"] == STATE["scale"] * 0.5 * 2.0  # backed off once, grown once


def test_adam_no_groups_updates_state_only():
    tp = _tp()
    state = tp.make_optimizer_state(**STATE)
    ws = torch.empty(tp.tp_adam_step_workspace_size(), dtype=torch.uint8, device="cuda")
    tp.tp_adam_step([], HYPER, state, ws)
    st = tp.read_optimizer_state(state)
    _, norm, _, ref_state = O.mixed_precision_adam_step([], STATE, HYPER)
    for k in ("scale", "growth_tracker", "hysteresis_tracker", "step"):
        assert st[k] == ref_state[k]
    assert st["grad_norm"] == 0.0 == norm and st["found_inf"] == 0


def test_adam_deterministic():
    groups = make_groups([70001, 33])
    a, b = DeviceOpt(groups, STATE), DeviceOpt(groups, STATE)
    sa, sb = a.step(HYPER), b.step(HYPER)
    assert sa == sb
    for x, y in zip(a.g, b.g):
        for k in ("param", "m", "v", "model"):
            assert torch.equal(x[k], y[k])


def test_adam_layer_H4096_full():
    """The one-layer workload of the H=4096 model (201,342,976 values in 8
    groups), every element against the oracle."""
    cfg = SI.WORKLOADS["adam_layer_H4096"]
    inp = SI.adam_inputs(cfg)
    groups, state, hyper = inp["groups"], inp["state"], inp["hyper"]
    dev = DeviceOpt(groups, state)
    st = dev.step(hyper)
    updated, norm, ref, ref_state = O.mixed_precision_adam_step(oracle_groups(groups), state, hyper)
    assert updated and st["grad_norm"] > hyper["max_norm"]
    check_against(dev, groups, ref, ref_state, norm, st, updated)


def test_adam_sixty_four_groups():
    sizes = [(i * 997) % 5000 + 1 for i in range(64)]
    groups = make_groups(sizes)
    run_and_check(groups, STATE, HYPER, with_model=[i % 2 == 0 for i in range(64)])
