"""Full-size parity of the CUDA path (through the C ABI) against the float64 oracle.

* the cone 256^3 x 360-view workload the benchmark times, and the two 2D workloads: EVERY ray of
  A against the oracle's ray, and the WHOLE volume (image) of A^T against the oracle's
  backprojection (relative L2);
* the two 512^3 workloads (jittered spiral, dual-axis tilt series): every ray of full views,
  and a few thousand voxels of A^T computed one by one by the oracle.

The oracle runs on all host cores (a thread pool over views or voxels; each ray is still computed
single-threaded in float64).  Tolerances are those of the other parity tests: per ray
|y_gpu - y_oracle| <= 1e-4 L_ray max|x| (missed rays exactly 0), and 1e-4 relative L2 for A^T.
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest

import oracle
from fan_beam_projector_siddon_b300 import workloads as W
from tests._parity import BP_RTOL, fp_violations, rel_l2, torch_cuda

pytestmark = pytest.mark.gpu

CORES = max(1, os.cpu_count() or 1)


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


def _ray_lengths(go, v0, v1):
    """Oracle chord length of every ray of views v0..v1-1, computed on all host cores."""
    edges = np.linspace(v0, v1, min(CORES, v1 - v0) + 1).round().astype(int)
    parts = [(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:]) if b > a]
    with cf.ThreadPoolExecutor(len(parts)) as ex:
        outs = list(ex.map(lambda ab: go.ray_lengths(views=ab)[0], parts))
    L = np.zeros(go.sino_shape, np.float64)
    for (a, b), o in zip(parts, outs):
        L[a:b] = o[a:b]
    return L[v0:v1]


def _project_view(go, x, k):
    """Oracle A x for every ray of view k (rays split over all host cores)."""
    iu, iv = np.meshgrid(np.arange(go.n_u, dtype=np.int32), np.arange(go.n_v, dtype=np.int32),
                         indexing="ij")
    iu, iv = iu.reshape(-1), iv.reshape(-1)
    view = np.full(iu.shape, k, np.int32)
    chunks = np.array_split(np.arange(iu.size), CORES)
    with cf.ThreadPoolExecutor(CORES) as ex:
        outs = list(ex.map(lambda c: go.project_rays(x, view[c], iu[c], iv[c]), chunks))
    return np.concatenate(outs).reshape(go.sino_shape[1:])


def _backproject_voxels(go, y, vox):
    """Oracle (A^T y) at the listed voxels, one voxel at a time, on all host cores."""
    chunks = np.array_split(np.asarray(vox, np.int64), CORES)
    with cf.ThreadPoolExecutor(CORES) as ex:
        outs = list(ex.map(lambda c: go.backproject_voxels(y, c), chunks))
    return np.concatenate(outs)


def test_cone_every_ray_of_the_benchmark_workload(ct):
    """All 53.1 M rays of the cone 256^3 x 360-view forward projection, ray by ray."""
    import torch
    w = W.config(3)
    x = w.phantom()
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    y_gpu = _cpu(g.project(torch_cuda(x)))
    torch.cuda.empty_cache()
    y_or = go.project(x, threads=CORES)
    L = _ray_lengths(go, 0, w.n_views)
    assert (L > 0).mean() > 0.5
    bad = fp_violations(y_gpu, y_or, L, float(np.abs(x).max()))
    assert bad.size == 0, (bad.size, bad[:5], y_gpu.reshape(-1)[bad[:5]],
                           y_or.reshape(-1)[bad[:5]])


def test_cone_whole_volume_backprojection_of_the_benchmark_workload(ct):
    """The whole 256^3 volume of A^T y for a dense positive random sinogram (no exact zeros, so
    every ray is scattered; no cancellation in the sums), against the oracle's float64
    backprojection."""
    import torch
    w = W.config(3)
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    y = np.abs(W.random_sinogram(w, 3))
    b_gpu = _cpu(g.backproject(torch_cuda(y)))
    torch.cuda.empty_cache()
    b_or = go.backproject(y, threads=CORES)
    assert rel_l2(b_gpu, b_or) <= BP_RTOL, rel_l2(b_gpu, b_or)
    # and voxel by voxel where the sums are large (no cancellation against a small total)
    big = np.abs(b_or) > 0.1 * np.abs(b_or).max()
    assert big.sum() > 1000
    assert np.max(np.abs(b_gpu[big] - b_or[big]) / np.abs(b_or[big])) <= 1e-3


@pytest.mark.parametrize("n,views", [(4, (0, 359, 719)), (5, (0, 69, 139, 140, 210, 279))])
def test_large_workloads_full_views_and_voxels(ct, n, views):
    """512^3 workloads: every ray of several full views (the first and last views of the orbit
    or of each tilt series and some between them), and 2000 voxels of A^T."""
    import torch
    w = W.config(n)
    x = w.phantom()
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    y_gpu = _cpu(g.project(torch_cuda(x)))
    torch.cuda.empty_cache()
    xmax = float(np.abs(x).max())
    x64, ones = x.astype(np.float64), np.ones(w.volume_shape, np.float64)
    for k in views:
        got = y_gpu[k]
        want = _project_view(go, x64, k)
        L = _project_view(go, ones, k)        # the ray's total chord length
        assert (L > 0).mean() > 0.2
        bad = fp_violations(got, want, L, xmax)
        assert bad.size == 0, (k, bad.size, bad[:5])
    del y_gpu, x64, ones
    y = np.abs(W.random_sinogram(w, 20 + n))
    b_gpu = _cpu(g.backproject(torch_cuda(y))).reshape(-1)
    torch.cuda.empty_cache()
    rng = np.random.default_rng(40 + n)
    vox = rng.choice(b_gpu.size, size=2000, replace=False)
    want = _backproject_voxels(go, y, vox)
    assert rel_l2(b_gpu[vox], want) <= BP_RTOL
    nz = np.abs(want) > 0.1 * np.abs(want).max()
    assert nz.sum() > 100
    assert np.max(np.abs(b_gpu[vox][nz] - want[nz]) / np.abs(want[nz])) <= 1e-3


@pytest.mark.parametrize("n", [1, 2])
def test_2d_workloads_every_ray_and_whole_image(ct, n):
    """The full 2D parallel (64^2, 90 views) and fan (512^2, 720 views) workloads: every ray of
    A and the whole image of A^T."""
    import torch
    w = W.config(n)
    x = w.phantom()
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    y_gpu = _cpu(g.project(torch_cuda(x)))
    y_or = go.project(x, threads=CORES)
    L = _ray_lengths(go, 0, w.n_views)
    assert (L > 0).mean() > 0.5
    bad = fp_violations(y_gpu, y_or, L, float(np.abs(x).max()))
    assert bad.size == 0, (bad.size, bad[:5])
    y = np.abs(W.random_sinogram(w, 30 + n))
    b_gpu = _cpu(g.backproject(torch_cuda(y)))
    torch.cuda.empty_cache()
    assert rel_l2(b_gpu, go.backproject(y, threads=CORES)) <= BP_RTOL
