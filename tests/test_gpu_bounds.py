"""The bounds-checking build (-DCT_DEBUG_BOUNDS) over adversarial and ordinary geometries:
every data-dependent voxel or detector index the kernels form is checked on the device, and the
count of out-of-range indices must stay 0.  This stands in for a device memory checker.  Results
must equal the release build's (the checks change no arithmetic)."""
import ctypes
import importlib.util
import os

import numpy as np
import pytest

from fan_beam_projector_siddon_b300 import workloads as W
from tests._parity import torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pair():
    """(release binding, bounds-checking binding)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fan_beam_projector_siddon_b300 import build
    build.build()
    path = build.build(debug_bounds=True)
    import fan_beam_projector_siddon_b300 as ct
    here = os.path.dirname(os.path.abspath(ct.__file__))
    spec = importlib.util.spec_from_file_location("ct_bounds_binding",
                                                  os.path.join(here, "_binding.py"))
    dbg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(dbg)
    lib = dbg.load_library(path)
    lib.ct_debug_bounds_violations.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
    lib.ct_debug_bounds_violations.restype = ctypes.c_int32
    return ct, dbg, lib


def _violations(lib):
    n = ctypes.c_uint64(0)
    assert lib.ct_debug_bounds_violations(ctypes.byref(n)) == 0
    return n.value


def _random_frames(rng, n, beam):
    views = []
    for _ in range(n):
        u = rng.standard_normal(3); u /= np.linalg.norm(u)
        v = rng.standard_normal(3); v -= (v @ u) * u; v /= np.linalg.norm(v)
        nrm = np.cross(u, v)
        if beam == W.CONE:
            views.append(np.concatenate([nrm * 9.0 + rng.uniform(-1, 1, 3),
                                         -nrm * 7.0 + rng.uniform(-1, 1, 3), u, v]))
        else:
            r = nrm + 0.4 * rng.standard_normal(3); r /= np.linalg.norm(r)
            views.append(np.concatenate([r, rng.uniform(-.2, .2, 3), u, v]))
    return np.array(views)


def _cases():
    cases = [W.small_config(n) for n in (1, 2, 3, 4, 5)]
    cases += [W.anisotropic_config(k) for k in ("cone", "tilt", "fan")]
    cases += [W.curved_config(k) for k in ("cone", "fan")]
    rng = np.random.default_rng(5)
    for shape in [(1, 1, 1), (2, 2, 2), (1, 2, 4), (8, 1, 1), (3, 1, 5)]:
        for beam in (W.CONE, W.PARALLEL3D):
            cases.append(W.Workload(f"tiny-{beam}-{shape}", beam, _random_frames(rng, 6, beam),
                                    shape, 0.5, 37, 33, 0.11, 0.13, 0, None))
    # rays exactly in cell faces and corner lines (axis-aligned parallel beam on the lattice)
    cases.append(W.Workload("faces", W.PARALLEL3D,
                            np.array([[0, 0, 1.0, 0, 0, 0, 1.0, 0, 0, 0, 1.0, 0]]), (4, 6, 8),
                            1.0, 9, 7, 1.0, 1.0, 0, None))
    return cases


@pytest.mark.parametrize("w", _cases(), ids=lambda w: w.name)
def test_projector_indices_stay_in_bounds(pair, w):
    import torch
    ct, dbg, lib = pair
    _violations(lib)
    g, gd = ct.Geometry.from_workload(w), dbg.Geometry.from_workload(w)
    x = torch_cuda(np.random.default_rng(1).uniform(0, 1, size=w.volume_shape))
    y = torch_cuda(np.random.default_rng(2).uniform(0, 1, size=w.sino_shape))
    fp, fpd = g.project(x), gd.project(x)
    bpd = gd.backproject(y)
    batch = torch.stack([x, x, x])
    gd.project(batch)
    gd.backproject(torch.stack([y, y, y]))
    ws = gd.new_workspace(sirt=True)
    xs = torch.zeros_like(x)
    gd.sirt(xs, y, 2, ws, initialised=False)
    wc = gd.new_workspace(cgls=True)
    xc = torch.zeros_like(x)
    gd.cgls(xc, y, 2, wc, initialised=False)
    torch.cuda.synchronize()
    assert _violations(lib) == 0
    assert torch.equal(fp, fpd)
    assert bpd.abs().sum() >= 0


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_fbp_indices_stay_in_bounds(pair, n):
    import torch
    ct, dbg, lib = pair
    _violations(lib)
    w = W.small_config(n)
    g, gd = ct.Geometry.from_workload(w), dbg.Geometry.from_workload(w)
    y = torch_cuda(W.random_sinogram(w, 3))
    x = torch_cuda(W.random_volume(w, 4))
    f, fd = g.fbp(y, window="shepp-logan"), gd.fbp(y, window="shepp-logan")
    gd.fbp_transpose(x)
    gd.fbp_gradients(y, x)
    # a voxel grid much larger than the field of view: most projections land off the detector
    import dataclasses
    big = dataclasses.replace(w, vol_shape=(w.vol_shape[0], 3 * w.vol_shape[1], 3 * w.vol_shape[2]),
                              voxel_spacing=2.0)
    gb = dbg.Geometry.from_workload(big)
    gb.fbp(y)
    gb.fbp_transpose(torch_cuda(W.random_volume(big, 5)))
    torch.cuda.synchronize()
    assert _violations(lib) == 0
    assert torch.equal(f, fd)


def _slab_cases():
    from tests.test_gpu_slabs import _tall_cone
    return [W.small_config(3), W.small_config(4), _tall_cone()]


@pytest.mark.parametrize("w", _slab_cases(), ids=lambda w: w.name)
@pytest.mark.parametrize("cells", [32, 64])
def test_slab_tiled_walks_stay_in_bounds(pair, w, cells):
    """The slab-tiled walks restart every ray inside each slab: every index they form stays in
    bounds, and the results equal the release build's (forward bit for bit)."""
    import torch
    ct, dbg, lib = pair
    _violations(lib)
    g, gd = ct.Geometry.from_workload(w), dbg.Geometry.from_workload(w)
    g.set_slabs(cells)
    gd.set_slabs(cells)
    assert gd.info.n_slabs >= 1
    x = torch_cuda(np.random.default_rng(1).uniform(0, 1, size=w.volume_shape))
    y = torch_cuda(np.random.default_rng(2).uniform(0, 1, size=w.sino_shape))
    fp, fpd = g.project(x), gd.project(x)
    gd.backproject(y)
    gd.project(torch.stack([x, x]))
    gd.backproject(torch.stack([y, y]))
    torch.cuda.synchronize()
    assert _violations(lib) == 0
    assert torch.equal(fp, fpd)


def _line_cases():
    from tests.test_gpu_lines import CASES, _cone_through_faces
    cases = [make() for _, make, _ in CASES]
    views = W.circular_cone(13, 40.0, 90.0).copy()
    views[:, 2] += 60.0
    views[:, 5] -= 20.0
    cases.append(W.Workload("faces-slab", W.CONE, views, (6, 47, 53), 1.0, 61, 67, 1.1, 1.4, 0,
                            None))
    for shape in [(2, 1, 1), (2, 2, 3), (7, 1, 1), (3, 4, 2)]:
        cases.append(W.Workload(f"tiny-lines-{shape}", W.CONE, W.circular_cone(11, 12.0, 24.0),
                                shape, 1.0, 19, 13, 0.9, 0.7, 0, None))
    return cases


@pytest.mark.parametrize("w", _line_cases(), ids=lambda w: w.name)
def test_shared_line_walks_stay_in_bounds(pair, w):
    """The shared-line walks (list projection, the backprojection over the line parameters, the
    batched forms and the per-ray fallback of short chords): every voxel index stays in bounds,
    and the forward results equal the release build's bit for bit."""
    import torch
    ct, dbg, lib = pair
    _violations(lib)
    g, gd = ct.Geometry.from_workload(w), dbg.Geometry.from_workload(w)
    assert g.info.shared_lines > 0 and gd.info.shared_lines == g.info.shared_lines
    x = torch_cuda(np.random.default_rng(1).uniform(0, 1, size=w.volume_shape))
    y = torch_cuda(np.random.default_rng(2).uniform(0, 1, size=w.sino_shape))
    fp, fpd = g.project(x), gd.project(x)
    gd.backproject(y)
    fb, fbd = g.project(torch.stack([x, x])), gd.project(torch.stack([x, x]))
    gd.backproject(torch.stack([y, y, y, y]))
    torch.cuda.synchronize()
    assert _violations(lib) == 0
    assert torch.equal(fp, fpd) and torch.equal(fb, fbd)
    assert torch.equal(fb[1], fp)
