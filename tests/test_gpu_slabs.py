"""Slab-tiled walks (volumes larger than L2): the forward projection and backprojection walk one
slab of the inner axis per launch, each ray restarting from its own crossing values.

* forced slabs on small cone and jittered-spiral twins: every ray of A against the oracle, the
  whole volume of A^T, the adjoint identity, and agreement with the untiled walk (the per-ray
  walks' segment weights are the same and the forward sums are added per slab; untiled
  shared-line walks are held to the oracle instead);
* tall volumes crossed by steep rays, so that rays cross several slabs;
* batched calls with slabs equal single calls;
* tiling is opt-in (measured slower on the 512^3 spiral, see include/ct.h).
"""
import numpy as np
import pytest

import oracle
from fan_beam_projector_siddon_b300 import workloads as W
from tests._parity import ADJ_RTOL, BP_RTOL, adjoint_gap, fp_violations, rel_l2, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ct():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fan_beam_projector_siddon_b300 import build
    build.build()
    import fan_beam_projector_siddon_b300 as ct
    return ct


def _cpu(t):
    import torch
    torch.cuda.synchronize()
    return t.cpu().numpy()


def _tall_cone():
    """A tall volume (nz = 150) seen from a source below it and a detector above it, so that the
    rays climb steeply through several 32-cell slabs."""
    views = W.circular_cone(17, 60.0, 150.0).copy()
    views[:, 2] -= 55.0           # source z
    views[:, 5] += 55.0           # detector centre z
    return W.Workload("cone-tall", W.CONE, views, (150, 77, 83), 1.0, 71, 97, 2.0, 3.0, 9,
                      lambda: W.ellipsoids_3d(10, 150, np.random.default_rng(9),
                                              axis_range=(4.0, 40.0))[:, :77, :83].copy())


CASES = [("cone", lambda: W.small_config(3)), ("spiral", lambda: W.small_config(4)),
         ("tall", _tall_cone)]


@pytest.mark.parametrize("name,make", CASES)
def test_slabs_match_the_oracle_and_the_untiled_walk(ct, name, make):
    w = make()
    g = ct.Geometry.from_workload(w)
    assert g.info.volume_layout == 1 and g.info.n_slabs == 1
    x = w.phantom()
    xs = torch_cuda(x)
    y_whole = _cpu(g.project(xs))
    yy = np.abs(W.random_sinogram(w, 8))
    b_whole = _cpu(g.backproject(torch_cuda(yy)))
    g.set_slabs(32)
    assert g.info.n_slabs == -(-w.vol_shape[0] // 32) and g.info.n_slabs >= 2
    assert g.info.slab_cells == 32
    go = oracle.Geometry.from_workload(w)
    y = _cpu(g.project(xs))
    y_or = go.project(x, threads=8)
    L, _ = go.ray_lengths()
    bad = fp_violations(y, y_or, L, float(np.abs(x).max()))
    assert bad.size == 0, (bad.size, bad[:5])
    assert np.all(y[L == 0] == 0)
    # Without shared lines the untiled walk takes the same segments, summed per slab: within
    # float32 rounding of the untiled sums.  With shared lines the untiled walks measure their
    # crossings along the line instead (other float32 roundings), so both are held to the oracle.
    same_segments = g.info.shared_lines == 0
    if same_segments:
        assert np.max(np.abs(y - y_whole)) <= 1e-5 * max(1.0, float(np.abs(y_whole).max()))
    else:
        assert fp_violations(y_whole, y_or, L, float(np.abs(x).max())).size == 0
    b = _cpu(g.backproject(torch_cuda(yy)))
    b_or = go.backproject(yy, threads=8)
    assert rel_l2(b, b_or) <= BP_RTOL
    if same_segments:
        assert rel_l2(b, b_whole) <= 1e-6
    else:
        assert rel_l2(b_whole, b_or) <= BP_RTOL
    rng = np.random.default_rng(3)
    xr = rng.uniform(-1, 1, size=w.volume_shape).astype(np.float32)
    yr = rng.uniform(-1, 1, size=w.sino_shape).astype(np.float32)
    gap, lhs, rhs = adjoint_gap(_cpu(g.project(torch_cuda(xr))), yr, xr,
                                _cpu(g.backproject(torch_cuda(yr))))
    assert gap <= ADJ_RTOL, (gap, lhs, rhs)
    # deterministic: the slabs are added in order
    assert np.array_equal(_cpu(g.project(xs)), y)
    g.set_slabs(0)
    assert g.info.n_slabs == 1
    assert np.array_equal(_cpu(g.project(xs)), y_whole)


def test_rays_cross_several_slabs(ct):
    """Precondition of the tall case: many rays span three or more 32-cell slabs."""
    w = _tall_cone()
    go = oracle.Geometry.from_workload(w)
    spans = []
    for k in range(0, w.n_views, 4):
        for iu in range(0, w.n_u, 7):
            for iv in range(0, w.n_v, 5):
                idx, _ = go.ray_segments(k, iu, iv)
                if idx.size:
                    z = idx // (w.vol_shape[1] * w.vol_shape[2])
                    spans.append(len(set((z // 32).tolist())))
    spans = np.array(spans)
    assert (spans >= 3).mean() > 0.2, np.bincount(spans)


def test_batched_calls_with_slabs(ct):
    import torch
    w = _tall_cone()
    g = ct.Geometry.from_workload(w)
    g.set_slabs(64)
    assert g.info.n_slabs == 3
    rng = np.random.default_rng(5)
    vols = torch_cuda(rng.uniform(0, 1, size=(5,) + tuple(w.volume_shape)))
    sinos = g.project(vols)
    for b in range(5):
        assert torch.equal(sinos[b], g.project(vols[b].contiguous()))
    ys = torch_cuda(rng.uniform(-1, 1, size=(5,) + tuple(w.sino_shape)))
    backs = g.backproject(ys)
    for b in range(5):
        assert rel_l2(_cpu(backs[b]), _cpu(g.backproject(ys[b].contiguous()))) <= 1e-6


def test_default_plan(ct):
    """Tiling is opt-in: no handle tiles by default; handles with the caller's order refuse it."""
    g4 = ct.Geometry.from_workload(W.config(4))
    assert g4.info.volume_layout == 1 and g4.info.n_slabs == 1
    g4.set_slabs(64)
    assert g4.info.n_slabs == 8 and g4.info.slab_cells == 64
    g4.set_slabs(600)                                # one slab or more cells: no tiling
    assert g4.info.n_slabs == 1
    g5 = ct.Geometry.from_workload(W.config(5))
    assert g5.info.n_slabs == 1                      # caller's order: no slabs
    with pytest.raises(ct.CtError):
        g5.set_slabs(32)
    with pytest.raises(ct.CtError):
        g4.set_slabs(-1)
