"""Largest volumes the C ABI admits: nz * ny * nx just below 2^31 (the walk's 32-bit voxel
indices).  The volume is constant, so no host copy of it is needed: the forward projection of
ones is the chord length per ray (the oracle's float64 chords, from the geometry alone), and the
backprojection of ones sums to the total chord (<A^T 1, 1> = <1, A 1>)."""
import numpy as np
import pytest

import oracle
from fan_beam_projector_siddon_b300 import workloads as W

pytestmark = pytest.mark.gpu

N = 1290  # 1290^3 = 2,146,689,000 < 2^31 - 1


@pytest.fixture(scope="module")
def ct():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 40 * 2**30:
        pytest.skip("needs about 30 GB of free device memory")
    from fan_beam_projector_siddon_b300 import build
    build.build()
    import fan_beam_projector_siddon_b300 as ct
    return ct


def _geometries():
    cone = W.Workload("cone-max", W.CONE, W.circular_cone(4, 2000.0, 3000.0), (N, N, N), 1.0,
                      32, 32, 40.0, 40.0, 0, None)
    ang = np.array([0.0, 37.0, 90.0])
    par = W.Workload("parallel3d-max", W.PARALLEL3D, W.dual_axis_tilt(ang, ang), (N, N, N), 1.0,
                     32, 32, 40.0, 40.0, 0, None)
    return [cone, par]


@pytest.mark.parametrize("w", _geometries(), ids=lambda w: w.name)
def test_maximum_volume_forward_and_backward(ct, w):
    import torch
    assert w.n_voxels < 2**31
    g = ct.Geometry.from_workload(w)
    L, _ = oracle.Geometry.from_workload(w).ray_lengths()
    assert (L > 0).mean() > 0.5 and L.max() > N
    vol = torch.ones(w.volume_shape, dtype=torch.float32, device="cuda")
    ws = g.new_workspace()
    y = g.project(vol, workspace=ws).cpu().numpy().astype(np.float64)
    assert np.all(np.abs(y - L) <= 1e-4 * L), float(np.abs(y - L).max())
    assert np.all(y[L == 0] == 0)
    ones = torch.ones(w.sino_shape, dtype=torch.float32, device="cuda")
    back = g.backproject(ones, out=vol, workspace=ws)
    total = float(back.sum(dtype=torch.float64))
    assert abs(total - L.sum()) <= 1e-5 * L.sum(), (total, L.sum())
    del vol, ws, ones, back
    torch.cuda.empty_cache()
