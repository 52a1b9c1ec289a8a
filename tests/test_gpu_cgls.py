"""CGLS on the GPU (through ct_cgls_iterate) against the float64 oracle's CGLS.

Parity: GPU CGLS with GPU-made data against oracle CGLS with oracle-made data, both from zero,
after k steps.  The GPU keeps its vectors (x, p, r, s) in float32 and its operator walks in
float32, so it is a perturbation of the float64 run whose size CGLS amplifies as its search
directions lose conjugacy.  The tolerance is fixed in advance and is not a function of the run:
the GPU iterate must lie within 1e-3 relative L2 of the oracle's, and its residual |y - A x|^2
within 1e-3 relative of the oracle's, on twins and step counts where float32 vector storage alone
moves the oracle's own iterate by at most 1e-5 (the test measures this with the oracle and
asserts it, so an ill-conditioned case fails instead of widening the bound).  That precondition
holds for the cone and tilt-series twins at 8 steps (about 1e-7) and for the 2D twins at 4 steps
(about 1e-6 and 1e-7); beyond that the 2D twins' 8-step sensitivity reaches 7e-4 (parallel) and
5e-5 (fan).
"""
import numpy as np
import pytest

import oracle
from fan_beam_projector_siddon_b300 import workloads as W
from tests._parity import rel_l2, torch_cuda

pytestmark = pytest.mark.gpu

CGLS_RTOL = 1e-3          # GPU iterate and residual against the float64 oracle's
CGLS_MAX_SENSITIVITY = 1e-5  # precondition: float32 storage moves the oracle's iterate <= this


def _float32_storage_sensitivity(go, y, x_ref, n_iter):
    """(relative change of the oracle's CGLS iterate, and |y - A x|^2 of that iterate) when the
    oracle's CGLS keeps its vectors in float32."""
    f = np.float32
    x = np.zeros(go.volume_shape, f)
    r = (y - go.project(x)).astype(f)
    s = go.backproject(r).astype(f)
    p = s.copy()
    gamma = float(np.sum(s.astype(np.float64) ** 2))
    for _ in range(n_iter):
        q = go.project(p).astype(f)
        alpha = gamma / float(np.sum(q.astype(np.float64) ** 2))
        x = (x + f(alpha) * p).astype(f)
        r = (r - f(alpha) * q).astype(f)
        s = go.backproject(r).astype(f)
        gamma_new = float(np.sum(s.astype(np.float64) ** 2))
        p = (s + f(gamma_new / gamma) * p).astype(f)
        gamma = gamma_new
    res = float(np.sum((y - go.project(x)) ** 2))
    return float(np.linalg.norm(x - x_ref) / np.linalg.norm(x_ref)), res


@pytest.fixture(scope="module")
def ct():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fan_beam_projector_siddon_b300 import build
    build.build()
    import fan_beam_projector_siddon_b300 as ct
    return ct


@pytest.mark.parametrize("n,steps", [(1, 4), (2, 4), (3, 8), (5, 8)])
def test_cgls_matches_oracle_small(ct, n, steps):
    import torch
    w = W.small_config(n)
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    x_true = w.phantom()
    y_or = go.project(x_true, threads=8)
    x_or, res_or = go.cgls(y_or, steps)
    sens, _ = _float32_storage_sensitivity(go, y_or, x_or, steps)
    assert sens <= CGLS_MAX_SENSITIVITY, sens
    y = g.project(torch_cuda(x_true))
    x = torch.zeros(w.volume_shape, dtype=torch.float32, device="cuda")
    ws = g.new_workspace(cgls=True)
    first = steps // 2 - 1                        # the state carries over between calls
    g.cgls(x, y, first, ws, initialised=False)
    g.cgls(x, y, steps - first, ws, initialised=True)
    torch.cuda.synchronize()
    assert rel_l2(x.cpu().numpy(), x_or) <= CGLS_RTOL
    r = (y - g.project(x)).double()
    res_gpu = float((r * r).sum())
    assert abs(res_gpu - res_or[-1]) <= CGLS_RTOL * res_or[-1], (res_gpu, res_or[-1])


def test_cgls_fixed_point_and_zero_iterations(ct):
    import torch
    w = W.small_config(3)
    g = ct.Geometry.from_workload(w)
    x_true = torch_cuda(w.phantom())
    y = g.project(x_true)
    ws = g.new_workspace(cgls=True)
    x = x_true.clone()
    g.cgls(x, y, 0, ws, initialised=False)
    torch.cuda.synchronize()
    assert torch.equal(x, x_true)
    g.cgls(x, y, 3, ws, initialised=True)
    torch.cuda.synchronize()
    assert rel_l2(x.cpu().numpy(), x_true.cpu().numpy()) <= 1e-5
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ct.CtError) as e:
        g.cgls(x, y, 1, small, initialised=False)
    assert e.value.status == 7


def test_cgls_full_size_residual_decreases(ct):
    """Full-size tilt-series workload: the residual |y - A x| decreases monotonically over 6
    CGLS steps from zero (CGLS minimises it over growing Krylov spaces)."""
    import torch
    w = W.config(5)
    g = ct.Geometry.from_workload(w)
    x_true = torch_cuda(w.phantom())
    y = g.project(x_true)
    ws = g.new_workspace(cgls=True)
    x = torch.zeros_like(x_true)
    res = []
    for k in range(6):
        g.cgls(x, y, 1, ws, initialised=k > 0)
        r = (y - g.project(x)).double()
        res.append(float((r * r).sum()))
    assert all(b < a for a, b in zip(res, res[1:]))
    assert res[-1] < 0.2 * float((y.double() ** 2).sum())
    del ws, x, y, x_true
    torch.cuda.empty_cache()
