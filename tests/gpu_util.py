"""Helpers of the GPU parity tests: device copies, fp64 views for the oracle,
and the error measure.

The tolerance follows the required bar: max relative error (infinity-norm
relative: max |gpu - oracle| / max |oracle| over a tensor) 2e-2 for bf16 inputs
with fp32 accumulation, 1e-4 for fp32.
"""
import numpy as np
import torch

TOL = {"bf16": 2e-2, "f32": 1e-4}


def dev(t):
    return t.cuda().contiguous()


def dev_list(ts):
    return [dev(t) for t in ts]


def f64(t):
    """Exact fp64 numpy copy of a (CPU or GPU) tensor."""
    return t.detach().to("cpu", torch.float64).numpy()


def f64_list(ts):
    return [f64(t) for t in ts]


def rel_err(gpu, ref):
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    scale = np.max(np.abs(r)) if r.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(g))) if g.size else 0.0
    return float(np.max(np.abs(g - r)) / scale)


def assert_close(gpu, ref, dtype, what=""):
    e = rel_err(gpu, ref)
    assert e <= TOL[dtype], f"{what}: max relative error {e:.3e} > {TOL[dtype]:.0e}"
    return e
