"""The device GELU / GELU' of the GEMM epilogues against the fp64 oracle and
CUDA's own erf (through torch's exact GELU on the GPU).

The epilogues compute erf with Abramowitz & Stegun formula 7.1.26
(|error| <= 1.5e-7); with fp32 evaluation the values must stay within a few
1e-7 of the exact GELU, far inside the 1e-4 fp32 bar of the parity tests.
"""
import numpy as np
import pytest
import torch

import oracle.tp_oracle as O

pytestmark = pytest.mark.gpu


def test_device_gelu_matches_exact_and_cuda_erf():
    import megatron_tensor_transformer_tp_gb300 as tp
    z = torch.cat([torch.linspace(-12, 12, 200001), torch.tensor([0.0, -0.0, 1e-30, -1e-30, 40.0, -40.0])])
    zd = z.cuda()
    y = torch.empty_like(zd)
    dy = torch.empty_like(zd)
    tp.tp_gelu_eval(zd, y, dy)
    assert tp.tp_get_status() == tp.TP_OK
    z64 = z.double().numpy()
    # the exact values, in units scaled by max(1, |z|) for y (y ~ z for large z)
    ey = np.abs(y.cpu().double().numpy() - O.gelu(z64)) / np.maximum(1.0, np.abs(z64))
    edy = np.abs(dy.cpu().double().numpy() - O.gelu_prime(z64))
    assert ey.max() < 5e-7, ey.max()
    assert edy.max() < 5e-7, edy.max()
    # CUDA's erf-based GELU on the same device
    ref = torch.nn.functional.gelu(zd, approximate="none")
    assert float(((y - ref).abs() / zd.abs().clamp(min=1.0)).max()) < 5e-7
    assert float(y[-6:-4].abs().max()) == 0.0 and abs(float(dy[-6]) - 0.5) < 1e-7
