"""Helpers of the GPU parity tests: device copies, fp64 views for the oracle,
and the error measures.

Two measures per compared tensor, both against the fp64 oracle:
  * infinity-norm relative error  max |g - r| / max |r|  (the reading of
    "max relative error"): 2e-2 for bf16 inputs with fp32 accumulation,
    1e-4 for fp32.  Asserted for every tensor.
  * element-wise relative error  max |g - r| / max(|r|, 1e-3 max |r|)  at the
    same bars.  Asserted by default.  A tensor that the method computes from
    a saved intermediate (Z, Y, dZ of the MLP; P, dS of the attention core;
    dLogits; the layer's saved activations) cannot meet it: the oracle keeps
    those intermediates in fp64, and the relative rounding of each saved
    element (2^-9 in bf16, 2^-24 in fp32) adds an absolute error of that
    order per summed term, which near-zero elements of a sum see as a large
    relative error.  Those call sites pass elementwise=False, and the measure
    is still computed and reported for them.

Every comparison is recorded in REPORT; the test session prints the worst
element-wise value per tensor at the end, and writes the records as JSON to
the file named by the TP_PARITY_REPORT environment variable when it is set.
"""
import numpy as np
import torch

TOL = {"bf16": 2e-2, "f32": 1e-4}
ELEM_FLOOR = 1e-3  # the element-wise measure's floor, as a fraction of max |r|

REPORT = []  # one dict per comparison: test, what, dtype, inf, elem, elem_asserted


def dev(t):
    return t.cuda().contiguous()


def dev_list(ts):
    return [dev(t) for t in ts]


def f64(t):
    """Exact fp64 numpy copy of a (CPU or GPU) tensor."""
    return t.detach().to("cpu", torch.float64).numpy()


def f64_list(ts):
    return [f64(t) for t in ts]


def _pair(gpu, ref):
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    return g, r


def rel_err(gpu, ref):
    """Infinity-norm relative error max |g - r| / max |r|."""
    g, r = _pair(gpu, ref)
    scale = np.max(np.abs(r)) if r.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(g))) if g.size else 0.0
    return float(np.max(np.abs(g - r)) / scale)


def elem_err(gpu, ref):
    """Element-wise relative error max |g - r| / max(|r|, 1e-3 max |r|)."""
    g, r = _pair(gpu, ref)
    if not r.size:
        return 0.0
    scale = np.max(np.abs(r))
    if scale == 0.0:
        return float(np.max(np.abs(g)))
    return float(np.max(np.abs(g - r) / np.maximum(np.abs(r), ELEM_FLOOR * scale)))


def _current_test():
    import os
    return os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]


def assert_close(gpu, ref, dtype, what="", elementwise=True):
    """Assert the infinity-norm bar and, unless `elementwise` is False, the
    element-wise bar; record both values.  Returns the infinity-norm error."""
    e, ee = rel_err(gpu, ref), elem_err(gpu, ref)
    REPORT.append({"test": _current_test(), "what": what, "dtype": dtype, "inf": e, "elem": ee,
                   "elem_asserted": bool(elementwise)})
    assert e <= TOL[dtype], f"{what}: max relative error {e:.3e} > {TOL[dtype]:.0e}"
    if elementwise:
        assert ee <= TOL[dtype], f"{what}: element-wise relative error {ee:.3e} > {TOL[dtype]:.0e}"
    return e
