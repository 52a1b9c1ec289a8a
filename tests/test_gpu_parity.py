"""CUDA path (through the C ABI) against the float64 oracle.

* small twins of the five workloads (several tiles plus ragged tails): every ray of A, the whole
  volume of A^T, the GPU adjoint identity;
* the five full-size workloads, in the launch configuration the benchmark times: sampled rays of
  A and sampled voxels of A^T against the oracle one by one, plus the adjoint identity;
* edge cases: 1-8-voxel volumes, rays in cell faces, rays that all miss, bad pointers, aliasing,
  short workspaces, determinism, non-default streams.
"""
import math

import numpy as np
import pytest

import oracle
from fan_beam_projector_siddon_b300 import workloads as W
from tests._parity import (ADJ_RTOL, BP_RTOL, adjoint_gap, fp_violations, rel_l2, sample_rays,
                           sino_at, torch_cuda)

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


# ---------------------------------------------------------------------------------------------
# small twins: elementwise
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_small_forward_every_ray(ct, n):
    w = W.small_config(n)
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    x = w.phantom()
    y_gpu = _cpu(g.project(torch_cuda(x)))
    y_or = go.project(x, threads=8)
    L, _ = go.ray_lengths()
    bad = fp_violations(y_gpu, y_or, L, float(np.abs(x).max()))
    assert bad.size == 0, (bad[:10], y_gpu.reshape(-1)[bad[:10]], y_or.reshape(-1)[bad[:10]])
    assert (L > 0).mean() > 0.3


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_small_backprojection_whole_volume(ct, n):
    w = W.small_config(n)
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    for y in (W.random_sinogram(w, 5), np.abs(W.random_sinogram(w, 6))):
        b_gpu = _cpu(g.backproject(torch_cuda(y)))
        b_or = go.backproject(y, threads=8)
        assert rel_l2(b_gpu, b_or) <= BP_RTOL


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_small_adjoint_identity_on_gpu(ct, n):
    w = W.small_config(n)
    g = ct.Geometry.from_workload(w)
    rng = np.random.default_rng(n)
    for lo in (0.0, -1.0):
        x = rng.uniform(lo, 1.0, size=w.volume_shape).astype(np.float32)
        y = rng.uniform(lo, 1.0, size=w.sino_shape).astype(np.float32)
        Ax = _cpu(g.project(torch_cuda(x)))
        Aty = _cpu(g.backproject(torch_cuda(y)))
        gap, lhs, rhs = adjoint_gap(Ax, y, x, Aty)
        assert gap <= ADJ_RTOL, (gap, lhs, rhs)


def test_layouts_chosen_per_geometry(ct):
    assert ct.Geometry.from_workload(W.config(3)).info.volume_layout == 1      # z fastest
    assert ct.Geometry.from_workload(W.config(5)).info.volume_layout == 0      # caller order
    assert ct.Geometry.from_workload(W.config(1)).info.volume_layout == 0
    g = ct.Geometry.from_workload(W.config(3))
    assert g.workspace_bytes >= 256 ** 3 * 4


# ---------------------------------------------------------------------------------------------
# full-size workloads: sampled
# ---------------------------------------------------------------------------------------------

_PHANTOMS = {}


def _phantom(n):
    if n not in _PHANTOMS:
        _PHANTOMS.clear()
        _PHANTOMS[n] = W.config(n).phantom()
    return _PHANTOMS[n]


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_full_forward_sampled_rays(ct, n):
    import torch
    w = W.config(n)
    x = _phantom(n)
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    y_gpu = g.project(torch_cuda(x))
    view, iu, iv = sample_rays(w, 4000, seed=n)
    got = sino_at(_cpu(y_gpu), w, view, iu, iv)
    want = go.project_rays(x, view, iu, iv)
    L = go.project_rays(np.ones(w.volume_shape), view, iu, iv)
    bad = fp_violations(got, want, L, float(np.abs(x).max()))
    assert bad.size == 0, (bad[:5], got[bad[:5]], want[bad[:5]])
    # every ray is written (no stale values): a second projection into a poisoned buffer agrees
    out = torch.full(w.sino_shape, float("nan"), device="cuda")
    g.project(torch_cuda(x), out=out)
    assert torch.equal(out, y_gpu)
    del y_gpu, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_full_backprojection_sampled_voxels(ct, n):
    import torch
    w = W.config(n)
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    y = W.random_sinogram(w, 10 + n)
    y = np.abs(y)   # positive: per-voxel sums without cancellation
    b_gpu = _cpu(g.backproject(torch_cuda(y))).reshape(-1)
    rng = np.random.default_rng(n)
    vox = rng.choice(b_gpu.size, size=60 if n >= 4 else 150, replace=False)
    want = go.backproject_voxels(y, vox)
    assert rel_l2(b_gpu[vox], want) <= BP_RTOL
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_full_adjoint_identity(ct, n):
    import torch
    w = W.config(n)
    g = ct.Geometry.from_workload(w)
    x = W.random_volume(w, 1) * 0.5 + 0.5
    y = W.random_sinogram(w, 2) * 0.5 + 0.5
    Ax = _cpu(g.project(torch_cuda(x)))
    Aty = _cpu(g.backproject(torch_cuda(y)))
    gap, lhs, rhs = adjoint_gap(Ax, y, x, Aty)
    assert gap <= ADJ_RTOL, (gap, lhs, rhs)
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------------------------

def _random_frames(rng, n, beam):
    views = []
    for _ in range(n):
        u = rng.standard_normal(3); u /= np.linalg.norm(u)
        v = rng.standard_normal(3); v -= (v @ u) * u; v /= np.linalg.norm(v)
        nrm = np.cross(u, v)
        if beam == W.CONE:
            views.append(np.concatenate([-5.0 * nrm + rng.uniform(-.3, .3, 3), 4.0 * nrm, u, v]))
        else:
            r = nrm + 0.4 * rng.standard_normal(3); r /= np.linalg.norm(r)
            views.append(np.concatenate([r, rng.uniform(-.2, .2, 3), u, v]))
    return np.array(views)


@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 2, 2), (1, 2, 4), (8, 1, 1), (1, 1, 8),
                                   (3, 1, 5)])
@pytest.mark.parametrize("beam", [W.CONE, W.PARALLEL3D])
def test_tiny_volumes(ct, shape, beam):
    rng = np.random.default_rng(sum(shape) * 7 + beam)
    views = _random_frames(rng, 6, beam)
    s = 0.5
    g = ct.Geometry(beam, views, shape, s, 37, 33, 0.11, 0.13)
    go = oracle.Geometry(beam, views, shape, s, 37, 33, 0.11, 0.13)
    x = rng.uniform(0.1, 1.0, size=shape).astype(np.float32)
    y_gpu = _cpu(g.project(torch_cuda(x)))
    y_or = go.project(x)
    L, _ = go.ray_lengths()
    assert fp_violations(y_gpu, y_or, L, float(x.max())).size == 0
    yy = rng.uniform(0.1, 1.0, size=go.sino_shape).astype(np.float32)
    assert rel_l2(_cpu(g.backproject(torch_cuda(yy))), go.backproject(yy)) <= BP_RTOL


def test_face_rays_follow_the_half_open_rule(ct):
    """Axis-aligned parallel rays lying exactly in cell faces belong to the + side cell."""
    nz, ny, nx = 4, 6, 8
    s = 1.0
    x = np.random.default_rng(0).uniform(0, 1, size=(nz, ny, nx)).astype(np.float32)
    # rays along +z; pixels on the integer lattice x, y in {-4..4} x {-3..3}: every ray lies in
    # the corner line of four cells (or on the outer faces)
    rec = np.array([[0, 0, 1.0, 0, 0, 0, 1.0, 0, 0, 0, 1.0, 0]])
    g = ct.Geometry(W.PARALLEL3D, rec, (nz, ny, nx), s, 9, 7, 1.0, 1.0)
    go = oracle.Geometry(W.PARALLEL3D, rec, (nz, ny, nx), s, 9, 7, 1.0, 1.0)
    y_gpu = _cpu(g.project(torch_cuda(x)))[0]
    y_or = go.project(x)[0]
    np.testing.assert_allclose(y_gpu, y_or, rtol=1e-6, atol=1e-6)
    # column u = 8 (x = +4) and row v = 6 (y = +3) lie on the outer + faces: exactly 0
    assert np.all(y_gpu[8, :] == 0) and np.all(y_gpu[:, 6] == 0)
    # the others equal the column sum of the + side cell
    np.testing.assert_allclose(y_gpu[:8, :6], x.sum(axis=0).T, rtol=1e-6)
    # 2D: rays along +x in the face planes y = k
    rec2 = np.array([[1.0, 0, 0, 0, 0, 1.0]])
    g2 = ct.Geometry(W.PARALLEL2D, rec2, (1, ny, nx), s, 7, 1, 1.0, 1.0)
    img = x[0]
    y2 = _cpu(g2.project(torch_cuda(img)))[0]
    np.testing.assert_allclose(y2[:6], img.sum(axis=1), rtol=1e-6)
    assert y2[6] == 0


def test_rays_that_miss_give_exact_zeros(ct):
    w = W.small_config(3)
    views = w.views.copy()
    views[:, 3:6] += np.array([0.0, 0.0, 400.0])     # detector far above: every ray misses
    views[:, 0:3] += np.array([0.0, 0.0, 400.0])
    g = ct.Geometry(W.CONE, views, w.vol_shape, 1.0, w.n_u, w.n_v, w.du, w.dv)
    y = _cpu(g.project(torch_cuda(w.phantom())))
    assert np.all(y == 0)
    b = _cpu(g.backproject(torch_cuda(np.ones(w.sino_shape, np.float32))))
    assert np.all(b == 0)


def test_forward_is_deterministic_and_stream_aware(ct):
    import torch
    w = W.small_config(4)
    g = ct.Geometry.from_workload(w)
    x = torch_cuda(w.phantom())
    a = g.project(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = g.project(x, stream=s)
    s.synchronize()
    assert torch.equal(a, b)


def test_bad_pointers_aliasing_and_workspace(ct):
    import torch
    w = W.small_config(3)
    g = ct.Geometry.from_workload(w)
    vol = torch_cuda(w.phantom())
    sino = torch.empty(w.sino_shape, device="cuda")
    ws = g.new_workspace()
    wsb = ws.numel()
    host = np.zeros(w.sino_shape, np.float32)
    with pytest.raises(ct.CtError) as e:
        ct.ct_project(g.handle, vol.data_ptr(), host.ctypes.data, ws.data_ptr(), wsb, None)
    assert e.value.status == 3
    big = torch.empty(vol.numel() + sino.numel(), device="cuda")
    with pytest.raises(ct.CtError) as e:       # output overlaps input
        ct.ct_project(g.handle, big.data_ptr(), big.data_ptr() + 4 * 100, ws.data_ptr(), wsb,
                      None)
    assert e.value.status == 4
    with pytest.raises(ct.CtError) as e:       # workspace too small
        ct.ct_project(g.handle, vol.data_ptr(), sino.data_ptr(), ws.data_ptr(), wsb - 4, None)
    assert e.value.status == 7
    with pytest.raises(ct.CtError) as e:       # workspace overlapping the output
        ct.ct_backproject(g.handle, sino.data_ptr(), vol.data_ptr(), vol.data_ptr(), wsb, None)
    assert e.value.status in (4, 7)
    # the handle still works afterwards
    g.project(vol, out=sino, workspace=ws)
    torch.cuda.synchronize()


def test_calls_with_another_device_current_are_refused(ct):
    """A handle is bound to its creation device: with another device current every compute call
    returns CT_ERR_INVALID_ARGUMENT before queueing any work (needs two GPUs)."""
    import torch
    if torch.cuda.device_count() < 2:
        pytest.skip("needs a second GPU")
    w = W.small_config(3)
    torch.cuda.set_device(0)
    g = ct.Geometry.from_workload(w)
    vol = torch_cuda(w.phantom())
    sino = torch.empty(w.sino_shape, device="cuda:0")
    ws = g.new_workspace()
    try:
        torch.cuda.set_device(1)
        for call in (lambda: ct.ct_project(g.handle, vol.data_ptr(), sino.data_ptr(),
                                           ws.data_ptr(), ws.numel(), None),
                     lambda: ct.ct_backproject(g.handle, sino.data_ptr(), vol.data_ptr(),
                                               ws.data_ptr(), ws.numel(), None),
                     lambda: ct.ct_backproject_static(g.handle, sino.data_ptr(), vol.data_ptr(),
                                                      None)):
            with pytest.raises(ct.CtError) as e:
                call()
            assert e.value.status == 1
    finally:
        torch.cuda.set_device(0)
    g.project(vol, out=sino, workspace=ws)
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------------------------
# per-axis voxel spacing
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["cone", "tilt", "fan"])
def test_anisotropic_spacing_forward_backward_adjoint(ct, kind):
    w = W.anisotropic_config(kind)
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    x = w.phantom()
    y_gpu = _cpu(g.project(torch_cuda(x)))
    y_or = go.project(x, threads=8)
    L, _ = go.ray_lengths()
    bad = fp_violations(y_gpu, y_or, L, float(np.abs(x).max()))
    assert bad.size == 0, (bad[:5], y_gpu.reshape(-1)[bad[:5]], y_or.reshape(-1)[bad[:5]])
    yy = np.abs(W.random_sinogram(w, 4))
    assert rel_l2(_cpu(g.backproject(torch_cuda(yy))), go.backproject(yy, threads=8)) <= BP_RTOL
    rng = np.random.default_rng(5)
    xr = rng.uniform(0, 1, size=w.volume_shape).astype(np.float32)
    yr = rng.uniform(0, 1, size=w.sino_shape).astype(np.float32)
    gap, lhs, rhs = adjoint_gap(_cpu(g.project(torch_cuda(xr))), yr, xr,
                                _cpu(g.backproject(torch_cuda(yr))))
    assert gap <= ADJ_RTOL, (gap, lhs, rhs)


def test_anisotropic_spacing_rejects_bad_pitches(ct):
    w = W.anisotropic_config("cone")
    for bad in [(1.0, 0.0, 1.0), (1.0, -2.0, 1.0), (float("nan"), 1.0, 1.0)]:
        with pytest.raises(ct.CtError) as e:
            ct.Geometry(w.beam, w.views, w.vol_shape, bad, w.n_u, w.n_v, w.du, w.dv)
        assert e.value.status == 1


# ---------------------------------------------------------------------------------------------
# batches of volumes (leading dimensions)
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("n", [3, 5, 1])
def test_batched_calls_equal_single_calls(ct, n):
    """A batch of 7 volumes (chunks of 4 + 2 + 1 in the kernels) gives the single-volume forward
    results bit for bit and the single-volume backprojections to float32 summation order."""
    import torch
    w = W.small_config(n)
    g = ct.Geometry.from_workload(w)
    rng = np.random.default_rng(n)
    vols = torch_cuda(rng.uniform(0, 1, size=(7,) + tuple(w.volume_shape)))
    sinos = g.project(vols)
    assert tuple(sinos.shape) == (7,) + tuple(w.sino_shape)
    for b in range(7):
        assert torch.equal(sinos[b], g.project(vols[b].contiguous()))
    ys = torch_cuda(rng.uniform(-1, 1, size=(7,) + tuple(w.sino_shape)))
    backs = g.backproject(ys)
    for b in range(7):
        single = _cpu(g.backproject(ys[b].contiguous()))
        assert rel_l2(_cpu(backs[b]), single) <= 1e-6
    # two leading dimensions
    v2 = vols[:6].reshape((2, 3) + tuple(w.volume_shape)).contiguous()
    s2 = g.project(v2)
    assert torch.equal(s2.reshape(sinos[:6].shape), sinos[:6])


def test_batched_call_checks(ct):
    import torch
    w = W.small_config(3)
    g = ct.Geometry.from_workload(w)
    vols = torch.zeros((3,) + tuple(w.volume_shape), device="cuda")
    sinos = torch.zeros((3,) + tuple(w.sino_shape), device="cuda")
    need = ct.ct_batch_workspace_bytes(g.handle, 3)
    assert need >= 3 * w.n_voxels * 4
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(ct.CtError) as e:
        ct.ct_project_batch(g.handle, 3, vols.data_ptr(), sinos.data_ptr(), ws.data_ptr(),
                            need - 4, None)
    assert e.value.status == 7
    with pytest.raises(ct.CtError) as e:
        ct.ct_project_batch(g.handle, 0, vols.data_ptr(), sinos.data_ptr(), ws.data_ptr(), need,
                            None)
    assert e.value.status == 1


# ---------------------------------------------------------------------------------------------
# parameterized detector surfaces
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["cone", "fan"])
def test_cylindrical_detector_forward_backward_adjoint(ct, kind):
    w = W.curved_config(kind)
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    x = w.phantom()
    y_gpu = _cpu(g.project(torch_cuda(x)))
    y_or = go.project(x, threads=8)
    L, _ = go.ray_lengths()
    bad = fp_violations(y_gpu, y_or, L, float(np.abs(x).max()))
    assert bad.size == 0, (bad[:5], y_gpu.reshape(-1)[bad[:5]], y_or.reshape(-1)[bad[:5]])
    assert (L > 0).mean() > 0.5
    yy = np.abs(W.random_sinogram(w, 4))
    assert rel_l2(_cpu(g.backproject(torch_cuda(yy))), go.backproject(yy, threads=8)) <= BP_RTOL
    rng = np.random.default_rng(6)
    xr = rng.uniform(0, 1, size=w.volume_shape).astype(np.float32)
    yr = rng.uniform(0, 1, size=w.sino_shape).astype(np.float32)
    gap, lhs, rhs = adjoint_gap(_cpu(g.project(torch_cuda(xr))), yr, xr,
                                _cpu(g.backproject(torch_cuda(yr))))
    assert gap <= ADJ_RTOL, (gap, lhs, rhs)


def test_flat_offsets_surface_equals_flat_detector(ct):
    import torch
    w = W.small_config(3)
    flat = ct.Geometry.from_workload(w)
    surf = ct.Geometry(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv,
                       offsets=W.flat_offsets(w.n_u, w.n_v, w.du, w.dv))
    x = torch_cuda(w.phantom())
    a, b = _cpu(flat.project(x)), _cpu(surf.project(x))
    np.testing.assert_allclose(b, a, rtol=1e-5, atol=1e-5 * float(np.abs(a).max()))


def test_walk_specialisation_boundary(ct):
    """Parallel rays whose inner-axis crossing pitch is just above, at and just below the largest
    gap between outer-axis crossings: the warps on either side take the specialised or the
    general walk, and every ray still matches the oracle (both inner directions)."""
    nz, ny, nx = 24, 20, 28
    theta = math.radians(30.0)          # azimuth of the rays' xy direction
    m = max(math.cos(theta), math.sin(theta))
    phi_b = math.atan(m)                # tan(phi) = m: inner pitch equals the outer gap bound
    phis = [math.radians(10.0), math.radians(80.0)]
    # -1e-3 .. -1.4e-4: the pitch difference is a few times down to ~1.3x the walk's rounding
    # margin (1e-5 of the chord); -1e-6 .. 1e-3: at or below the bound
    for d in (-1e-3, -2e-4, -1.4e-4, -1e-6, 0.0, 1e-6, 1e-3):
        phis += [phi_b + d, -(phi_b + d)]
    views = []
    for phi in phis:
        r = [math.cos(theta) * math.cos(phi), math.sin(theta) * math.cos(phi), math.sin(phi)]
        du_vec = [-math.sin(theta), math.cos(theta), 0.0]
        views.append(r + [0.1, -0.2, 0.3] + du_vec + [0.0, 0.0, 1.0])
    views = np.array(views)
    args = (W.PARALLEL3D, views, (nz, ny, nx), 1.0, 40, 48, 0.7, 0.9)
    g, go = ct.Geometry(*args), oracle.Geometry(*args)
    assert g.info.volume_layout == 1  # z fastest: z is the walk's inner axis here
    rng = np.random.default_rng(11)
    x = rng.uniform(0.1, 1.0, size=(nz, ny, nx)).astype(np.float32)
    y_gpu = _cpu(g.project(torch_cuda(x)))
    y_or = go.project(x)
    L, _ = go.ray_lengths()
    assert (L > 0).mean() > 0.5
    bad = fp_violations(y_gpu, y_or, L, float(x.max()))
    assert bad.size == 0, bad[:10]
    yy = rng.uniform(0.1, 1.0, size=go.sino_shape).astype(np.float32)
    assert rel_l2(_cpu(g.backproject(torch_cuda(yy))), go.backproject(yy)) <= BP_RTOL


def test_walk_specialisation_changes_no_arithmetic(ct):
    """The same rays projected once in a warp that takes the specialised walk and once in a
    warp pushed onto the general walk give bit-identical values.  Rows 32..44 of the small cone
    all climb in z, so their warps vote for the fast walk; mirroring row 44 below the central
    row (through the detector-surface offsets, which leave every other ray's arithmetic
    untouched) gives that warp one descending ray, and the sign vote fails."""
    w = W.small_config(3)
    off1 = W.flat_offsets(w.n_u, w.n_v, w.du, w.dv)
    off2 = off1.copy()
    moved = w.n_v - 1
    off2[:, moved, 1] *= -1.0
    band = np.arange(32, w.n_v)
    # preconditions (float64, host): the band's flat rays climb and pass the one-crossing test
    # with room to spare; the moved ray descends and still crosses the volume
    V = w.views
    src, ctr, du_v, dv_v = V[:, 0:3], V[:, 3:6], V[:, 6:9], V[:, 9:12]

    def dirs(off):
        pix = (ctr[:, None, None, :] + off[None, :, :, 0:1] * du_v[:, None, None, :]
               + off[None, :, :, 1:2] * dv_v[:, None, None, :])
        return pix - src[:, None, None, :]

    d1, d2 = dirs(off1)[:, :, band], dirs(off2)[:, :, moved]
    assert np.all(d1[..., 2] > 0) and np.all(d2[..., 2] < 0)
    assert np.all(np.abs(d1[..., 2]) < 0.9 * np.maximum(np.abs(d1[..., 0]), np.abs(d1[..., 1])))
    go = oracle.Geometry(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv,
                         offsets=off2)
    L, _ = go.ray_lengths()
    assert (L[:, :, moved] > 0).mean() > 0.5
    g1 = ct.Geometry(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv,
                     offsets=off1)
    g2 = ct.Geometry(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv,
                     offsets=off2)
    assert g1.info.volume_layout == 1  # z fastest: z is the walk's inner axis
    x = torch_cuda(w.phantom())
    a, b = _cpu(g1.project(x)), _cpu(g2.project(x))
    keep = np.ones(w.n_v, bool)
    keep[moved] = False
    assert np.count_nonzero(a[:, :, band[:-1]]) > 0.3 * a[:, :, band[:-1]].size
    assert np.array_equal(a[:, :, keep], b[:, :, keep])


def _random_frames_2d(rng, n, beam):
    views = []
    for _ in range(n):
        th = rng.uniform(0, 2 * math.pi)
        u = np.array([-math.sin(th), math.cos(th)])
        if beam == W.FAN2D:
            r = rng.uniform(30, 60)
            src = r * np.array([math.cos(th), math.sin(th)]) + rng.uniform(-2, 2, 2)
            views.append(np.concatenate([src, -0.5 * src, u]))
        else:
            views.append(np.concatenate([[math.cos(th), math.sin(th)], rng.uniform(-1, 1, 2), u]))
    return np.array(views)


# (seed 493: a short chord with a grazing crossing, see test_grazing_crossings_far_along_an_axis)
@pytest.mark.parametrize("seed", [*range(8), 493])
def test_random_geometries_against_the_oracle(ct, seed):
    """Random frames, volume shapes, per-axis pitches and detectors for the four beams: every
    ray of A against the oracle and A^T in relative L2 (exercises the walk's specialised and
    general forms in whatever mix the geometry gives)."""
    rng = np.random.default_rng(1000 + seed)
    beam = [W.CONE, W.PARALLEL3D, W.FAN2D, W.PARALLEL2D][seed % 4]
    two_d = beam in (W.FAN2D, W.PARALLEL2D)
    if two_d:
        shape = (1, int(rng.integers(5, 40)), int(rng.integers(5, 40)))
        sp = (float(rng.uniform(0.5, 1.5)), float(rng.uniform(0.5, 1.5)))  # (dy, dx)
        views = _random_frames_2d(rng, 7, beam)
        n_u, n_v = int(rng.integers(20, 90)), 1
        du, dv = float(rng.uniform(0.3, 1.2)), 1.0
    else:
        shape = tuple(int(v) for v in rng.integers(4, 28, 3))
        sp = tuple(float(v) for v in rng.uniform(0.5, 1.5, 3))
        # positions scaled to the box size (the ray direction of a parallel beam stays a unit
        # vector)
        scale = [8.0, 8.0, 1.0, 1.0] if beam == W.CONE else [1.0, 8.0, 1.0, 1.0]
        views = _random_frames(rng, 5, beam) * np.repeat(scale, 3)
        n_u, n_v = int(rng.integers(20, 70)), int(rng.integers(20, 70))
        du, dv = float(rng.uniform(0.2, 0.8)), float(rng.uniform(0.2, 0.8))
    args = (beam, views, shape, sp, n_u, n_v, du, dv)
    g, go = ct.Geometry(*args), oracle.Geometry(*args)
    vol_shape = shape[1:] if two_d else shape
    x = rng.uniform(0.0, 1.0, size=vol_shape).astype(np.float32)
    y_gpu = _cpu(g.project(torch_cuda(x)))
    y_or = go.project(x)
    L, _ = go.ray_lengths()
    assert (L > 0).mean() > 0.1
    bad = fp_violations(y_gpu, y_or, L, float(x.max()))
    assert bad.size == 0, bad[:10]
    yy = rng.uniform(-1.0, 1.0, size=go.sino_shape).astype(np.float32)
    assert rel_l2(_cpu(g.backproject(torch_cuda(yy))), go.backproject(yy)) <= BP_RTOL


@pytest.mark.parametrize("make", [lambda: W.small_config(1), lambda: W.small_config(2),
                                  lambda: W.small_config(3), lambda: W.small_config(4),
                                  lambda: W.small_config(5), lambda: W.anisotropic_config("cone"),
                                  lambda: W.anisotropic_config("tilt"),
                                  lambda: W.anisotropic_config("fan")],
                         ids=["parallel2d", "fan2d", "cone", "spiral", "tilt", "cone-aniso",
                              "tilt-aniso", "fan-aniso"])
def test_matched_transpose_entry_by_entry(ct, make):
    """A^T is the transpose of A entry by entry, bit for bit: the projection of a unit voxel e_i
    read at ray r equals the backprojection of the unit ray e_r read at voxel i (the forward and
    adjoint walks take the same segments with the same operations; each entry is one segment
    length times the ray's length factor, rounded once, and the zero terms add nothing)."""
    w = make()
    g = ct.Geometry.from_workload(w)
    nvox, nray = int(np.prod(w.volume_shape)), int(np.prod(w.sino_shape))
    rng = np.random.default_rng(17)
    checked = 0
    for i in rng.choice(nvox, size=8, replace=False):
        e = np.zeros(nvox, np.float32)
        e[i] = 1.0
        col = _cpu(g.project(torch_cuda(e.reshape(w.volume_shape)))).reshape(-1)
        rays = np.nonzero(col)[0]
        for r in rng.choice(rays, size=min(6, rays.size), replace=False):
            er = np.zeros(nray, np.float32)
            er[r] = 1.0
            row = _cpu(g.backproject(torch_cuda(er.reshape(w.sino_shape)))).reshape(-1)
            assert row[i] == col[r], (int(i), int(r), float(row[i]), float(col[r]))
            checked += 1
    assert checked >= 12, checked
