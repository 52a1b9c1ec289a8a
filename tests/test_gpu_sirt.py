"""SIRT on the GPU (through ct_sirt_iterate) against the float64 oracle and SIRT's invariants.

The pages only name SIRT; the oracle's iterate is the textbook update with R = 1/(A 1) and
C = 1/(A^T 1).  Parity: GPU SIRT with GPU-made data vs oracle SIRT with oracle-made data, relative
L2 <= 1e-4 after 10 iterations (a proposed bound; float32 operator errors of ~1e-6 stay of that
order under the iteration, which is non-expansive in the R/C-weighted norms).
"""
import numpy as np
import pytest

import oracle
from fan_beam_projector_siddon_b300 import workloads as W
from tests._parity import rel_l2, torch_cuda

pytestmark = pytest.mark.gpu

SIRT_RTOL = 1e-4


@pytest.fixture(scope="module")
def ct():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fan_beam_projector_siddon_b300 import build
    build.build()
    import fan_beam_projector_siddon_b300 as ct
    return ct


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_sirt_matches_oracle_small(ct, n):
    import torch
    w = W.small_config(n)
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    x_true = w.phantom()
    y_or = go.project(x_true, threads=8)
    x_or, _ = go.sirt(y_or, 10)
    y = g.project(torch_cuda(x_true))
    x = torch.zeros(w.volume_shape, dtype=torch.float32, device="cuda")
    ws = g.new_workspace(sirt=True)
    # split into 4 + 6 iterations: the cached C is reused on the second call
    g.sirt(x, y, 4, ws, initialised=False)
    g.sirt(x, y, 6, ws, initialised=True)
    torch.cuda.synchronize()
    assert rel_l2(x.cpu().numpy(), x_or) <= SIRT_RTOL


def test_sirt_zero_iterations_and_argument_checks(ct):
    import torch
    w = W.small_config(5)
    g = ct.Geometry.from_workload(w)
    x = torch.ones(w.volume_shape, device="cuda")
    y = torch.ones(w.sino_shape, device="cuda")
    ws = g.new_workspace(sirt=True)
    g.sirt(x, y, 0, ws, initialised=False)
    torch.cuda.synchronize()
    assert torch.all(x == 1)
    with pytest.raises(ct.CtError):
        g.sirt(x, y, 1, ws, initialised=True, relaxation=2.5)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ct.CtError) as e:
        g.sirt(x, y, 1, small, initialised=False)
    assert e.value.status == 7


@pytest.mark.parametrize("n", [5, 3])
def test_sirt_full_size_fixed_point_and_descent(ct, n):
    """Full-size workload: consistent data from x_true is a fixed point, and from zero the
    R-weighted residual decreases over the 10 iterations."""
    import torch
    w = W.config(n)
    g = ct.Geometry.from_workload(w)
    x_true = torch_cuda(w.phantom())
    y = g.project(x_true)
    ws = g.new_workspace(sirt=True)
    x = x_true.clone()
    g.sirt(x, y, 2, ws, initialised=False)
    torch.cuda.synchronize()
    assert rel_l2(x.cpu().numpy(), x_true.cpu().numpy()) <= SIRT_RTOL
    L = g.project(torch.ones_like(x_true))            # A 1 = chord lengths -> R = 1 / L

    def weighted_residual(xx):
        r = (y - g.project(xx)).double()
        R = torch.where(L > 0, 1.0 / L.double(), torch.zeros_like(r))
        return float((R * r * r).sum())

    x = torch.zeros_like(x_true)
    r0 = weighted_residual(x)
    g.sirt(x, y, 5, ws, initialised=True)
    r5 = weighted_residual(x)
    g.sirt(x, y, 5, ws, initialised=True)
    r10 = weighted_residual(x)
    assert r10 < r5 < r0
    del ws, x, y, L
    torch.cuda.empty_cache()
