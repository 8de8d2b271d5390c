"""Device GELU / SiLU (both routes) against the exact functions in fp64.

The bar: |act_gpu - act_exact| <= 1e-3 + 4e-3 |act_exact| over x in [-16, 16],
and the same for the derivatives used by the backward pass.  GELU is exact
erf GELU x * Phi(x) (the form the oracle uses).
"""

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jg():
    import __graft_entry__
    __graft_entry__.build()
    import jagged_gdpa_gb300 as m
    return m


@pytest.mark.parametrize("act", ["gelu", "silu"])
@pytest.mark.parametrize("path", [0, 1, 2])
def test_activation_accuracy(jg, act, path):
    x = torch.linspace(-16.0, 16.0, 1 << 20, dtype=torch.float32)
    x = torch.cat([x, torch.tensor([0.0, -0.0, 1e-30, -1e-30, 1e-3, -1e-3])])
    y, dy = jg.jgdpa_eval_activation(act, x.cuda(), path=path)
    ref, dref = oracle.act(act, x.double().numpy())
    y = y.double().cpu().numpy()
    dy = dy.double().cpu().numpy()
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(dy))
    ey = np.abs(y - ref) / (1e-3 + 4e-3 * np.abs(ref))
    ed = np.abs(dy - dref) / (1e-3 + 4e-3 * np.abs(dref))
    assert ey.max() <= 1.0, f"value: worst at x={x[ey.argmax()].item()}: ratio {ey.max():.3f}"
    assert ed.max() <= 1.0, f"derivative: worst at x={x[ed.argmax()].item()}: ratio {ed.max():.3f}"
    assert y[-6] == 0.0  # act(0) = 0 exactly (masked elements rely on it)


def test_routes_agree(jg):
    x = torch.linspace(-12.0, 12.0, 1 << 18, dtype=torch.float32).cuda()
    for act in ("gelu", "silu"):
        y0, d0 = jg.jgdpa_eval_activation(act, x, path=0)
        y1, d1 = jg.jgdpa_eval_activation(act, x, path=1)
        assert torch.max(torch.abs(y0 - y1) / (2e-3 + 1e-3 * torch.abs(y1))).item() <= 1.0
        assert torch.max(torch.abs(d0 - d1) / (3e-3 + 1e-3 * torch.abs(d1))).item() <= 1.0
