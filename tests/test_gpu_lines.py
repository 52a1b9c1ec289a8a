"""Shared-line walks: when the detector axis along a block's lanes has no component on the two
outer volume axes (and the volume fits in L2), the rays of one detector line share their
outer-axis crossings: the forward projection reads them from one merged list per line, and the
backprojection walks the same segments per ray over the line's parameters (SIRT and CGLS keep the
per-ray walks).

* which handles use them (info.shared_lines) and which keep the per-ray walk;
* every ray of A and the whole volume of A^T against the oracle, and the adjoint identity, on
  geometries that exercise the lanes along v and along u, parallel lines at steep elevations,
  rays entering and leaving through the inner-axis faces (lanes that start part-way along the
  list, and short chords far along the line, which take the per-ray walk), per-axis pitches and
  batched calls; SIRT on a shared-line handle against the oracle; ten random shared-line
  geometries (cone orbits with offsets, steep parallel rays, random shapes and pitches), and the
  geometries whose short chords cross a plane at a grazing angle far along an axis.
"""
import math

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


def _phantom(shape, seed):
    return W.ellipsoids_3d(8, max(shape), np.random.default_rng(seed),
                           axis_range=(3.0, 0.45 * min(shape)))[:shape[0], :shape[1], :shape[2]].copy()


def _cone_lanes_u():
    """Circular cone with det_u along z (the lanes run along u)."""
    views = W.circular_cone(21, 150.0, 300.0).copy()
    du_vec, dv_vec = views[:, 6:9].copy(), views[:, 9:12].copy()
    views[:, 6:9], views[:, 9:12] = dv_vec, du_vec
    shape = (37, 45, 53)
    return W.Workload("cone-lanes-u", W.CONE, views, shape, 1.0, 47, 69, 1.2, 1.2, 5,
                      lambda: _phantom(shape, 5))


def _cone_through_faces():
    """Circular cone with the source above the volume and the detector below it: most rays
    enter through the top face and many leave through the bottom one."""
    views = W.circular_cone(19, 60.0, 130.0).copy()
    views[:, 2] += 40.0    # source z
    views[:, 5] -= 45.0    # detector centre z
    shape = (41, 39, 35)
    return W.Workload("cone-faces", W.CONE, views, shape, 1.0, 77, 83, 1.3, 1.1, 6,
                      lambda: _phantom(shape, 6))


def _parallel_lines():
    """Parallel rays at several azimuths and steep elevations, detector v along z."""
    views = []
    for k, (th, ph) in enumerate([(10, 5), (30, 45), (55, 70), (80, 85), (125, -60), (200, -20),
                                  (290, 30), (345, -80)]):
        th, ph = math.radians(th), math.radians(ph)
        r = [math.cos(th) * math.cos(ph), math.sin(th) * math.cos(ph), math.sin(ph)]
        views.append(r + [0.3 * k, -0.2, 0.1] + [-math.sin(th), math.cos(th), 0.0] + [0.0, 0.0, 1.0])
    shape = (26, 22, 30)
    return W.Workload("parallel-lines", W.PARALLEL3D, np.array(views), shape, 1.0, 45, 51, 0.9,
                      0.8, 7, lambda: _phantom(shape, 7))


CASES = [("cone-twin", lambda: W.small_config(3), 1), ("lanes-u", _cone_lanes_u, 2),
         ("faces", _cone_through_faces, 1), ("parallel", _parallel_lines, 1),
         ("aniso", lambda: W.anisotropic_config("cone"), 1)]


def test_which_handles_share_lines(ct):
    """Circular cone orbits with an upright detector share lines; 2D beams, the jittered spiral
    (tilted detector), the dual-axis tilt series and surface detectors keep the per-ray walk."""
    expect = {1: 0, 2: 0, 3: 1, 4: 0, 5: 0}
    for n, want in expect.items():
        assert ct.Geometry.from_workload(W.small_config(n)).info.shared_lines == want, n
    assert ct.Geometry.from_workload(W.config(3)).info.shared_lines == 1
    assert ct.Geometry.from_workload(W.config(4)).info.shared_lines == 0
    w = W.small_config(3)
    surf = ct.Geometry(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv,
                       offsets=W.flat_offsets(w.n_u, w.n_v, w.du, w.dv))
    assert surf.info.shared_lines == 0
    for _, make, want in CASES:
        assert ct.Geometry.from_workload(make()).info.shared_lines == want
    # a volume larger than L2 (untilted 512^3 helix): per-ray walks
    w4 = W.config(4)
    helix = ct.Geometry(w4.beam, W.spiral_cone(8, 320.0, 512.0, 40.0, 2.0), w4.vol_shape,
                        w4.voxel_spacing, w4.n_u, w4.n_v, w4.du, w4.dv)
    assert helix.info.shared_lines == 0
    # more outer-axis cells than a block's list holds (n_x + n_y > 6000), small enough for L2
    wide = ct.Geometry(W.CONE, W.circular_cone(4, 5000.0, 9000.0), (2, 3100, 3100), 1.0, 64, 8,
                       1.0, 1.0)
    assert wide.info.shared_lines == 0


def test_face_case_preconditions(ct):
    """The face geometry has rays that start part-way along their line (entry through the top
    face) and rays whose chord is short against their position along the line."""
    w = _cone_through_faces()
    go = oracle.Geometry.from_workload(w)
    starts, short = 0, 0
    for k in range(0, w.n_views, 3):
        for iu in range(0, w.n_u, 4):
            for iv in range(0, w.n_v, 4):
                idx, seg = go.ray_segments(k, iu, iv)
                if idx.size:
                    z_first = idx[0] // (w.vol_shape[1] * w.vol_shape[2])
                    starts += int(z_first == w.vol_shape[0] - 1)
                    short += int(seg.sum() < 1.0)
    assert starts > 200 and short > 2, (starts, short)


@pytest.mark.parametrize("name,make,want", CASES)
def test_lines_against_the_oracle(ct, name, make, want):
    w = make()
    g = ct.Geometry.from_workload(w)
    assert g.info.shared_lines == want
    go = oracle.Geometry.from_workload(w)
    x = w.phantom().astype(np.float32)
    y = _cpu(g.project(torch_cuda(x)))
    y_or = go.project(x, threads=8)
    L, _ = go.ray_lengths()
    assert (L > 0).mean() > 0.3
    bad = fp_violations(y, y_or, L, float(np.abs(x).max()))
    assert bad.size == 0, (bad.size, bad[:8])
    assert np.all(y[L == 0] == 0)
    yy = np.abs(W.random_sinogram(w, 4))
    b = _cpu(g.backproject(torch_cuda(yy)))
    assert rel_l2(b, go.backproject(yy, threads=8)) <= BP_RTOL
    rng = np.random.default_rng(9)
    xr = rng.uniform(-1, 1, size=w.volume_shape).astype(np.float32)
    yr = rng.uniform(-1, 1, size=w.sino_shape).astype(np.float32)
    gap, lhs, rhs = adjoint_gap(_cpu(g.project(torch_cuda(xr))), yr, xr,
                                _cpu(g.backproject(torch_cuda(yr))))
    assert gap <= ADJ_RTOL, (gap, lhs, rhs)


@pytest.mark.parametrize("name,make,want", CASES[:3])
def test_batched_lines_equal_single(ct, name, make, want):
    import torch
    w = make()
    g = ct.Geometry.from_workload(w)
    rng = np.random.default_rng(2)
    vols = torch_cuda(rng.uniform(0, 1, size=(7,) + tuple(w.volume_shape)))
    sinos = g.project(vols)
    for b in range(7):
        assert torch.equal(sinos[b], g.project(vols[b].contiguous()))
    ys = torch_cuda(rng.uniform(-1, 1, size=(7,) + tuple(w.sino_shape)))
    backs = g.backproject(ys)
    for b in range(7):
        assert rel_l2(_cpu(backs[b]), _cpu(g.backproject(ys[b].contiguous()))) <= 1e-6


def test_lines_are_deterministic(ct):
    w = _cone_through_faces()
    g = ct.Geometry.from_workload(w)
    x = torch_cuda(w.phantom())
    a = _cpu(g.project(x))
    for _ in range(3):
        assert np.array_equal(_cpu(g.project(x)), a)


def test_sirt_on_a_shared_line_handle(ct):
    """SIRT iterations walk per ray on every handle: on a shared-line handle they match the
    oracle's SIRT as on any other (relative L2 after 10 iterations, as the SIRT parity tests)."""
    import torch
    w = _cone_lanes_u()
    g = ct.Geometry.from_workload(w)
    assert g.info.shared_lines == 2
    go = oracle.Geometry.from_workload(w)
    y_or = go.project(w.phantom().astype(np.float32), threads=8)
    x_or, _ = go.sirt(y_or, 10)
    x = torch.zeros(tuple(w.volume_shape), dtype=torch.float32, device="cuda")
    g.sirt(x, torch_cuda(y_or), 10, g.new_workspace(sirt=True), initialised=False)
    assert rel_l2(_cpu(x), x_or) <= 1e-4


def test_line_backprojection_is_the_exact_transpose(ct):
    """The backprojection walks the list walk's segments (per-ray tiles given the line's
    parameters), so every entry of A^T is the entry of A bit for bit: the projection of a unit
    voxel e_i, read at ray r, equals the backprojection of a unit ray e_r, read at voxel i (both
    are one segment length times the ray's length factor, rounded once; the zero terms add
    nothing).  Checked on rays entering through the inner-axis faces far along their lines,
    where the line's and the per-ray parameterisations round differently, and on the cone twin."""
    import torch
    for w in (_cone_through_faces(), W.small_config(3)):
        g = ct.Geometry.from_workload(w)
        assert g.info.shared_lines == 1
        rng = np.random.default_rng(7)
        checked = 0
        for i in rng.choice(int(np.prod(w.volume_shape)), size=6, replace=False):
            e = np.zeros(int(np.prod(w.volume_shape)), np.float32)
            e[i] = 1.0
            col = _cpu(g.project(torch_cuda(e.reshape(w.volume_shape)))).reshape(-1)
            rays = np.nonzero(col)[0]
            for r in rng.choice(rays, size=min(8, rays.size), replace=False):
                er = np.zeros(col.size, np.float32)
                er[r] = 1.0
                row = _cpu(g.backproject(torch_cuda(er.reshape(w.sino_shape)))).reshape(-1)
                assert row[i] == col[r], (w.name, int(i), int(r), float(row[i]), float(col[r]))
                checked += 1
        assert checked >= 24, checked

@pytest.mark.parametrize("shape", [(2, 1, 1), (2, 2, 3), (3, 1, 2), (2, 3, 1), (5, 4, 6), (7, 1, 1)])
def test_tiny_volumes_on_shared_lines(ct, shape):
    """1-7-voxel volumes under a circular cone with an upright detector (shared lines; a volume
    one cell high keeps the caller's x-fastest order, whose lanes do not share lines): every ray
    against the oracle, the whole volume of A^T, and exact zeros for rays that miss."""
    views = W.circular_cone(11, 12.0, 24.0)
    args = (W.CONE, views, shape, 1.0, 19, 13, 0.9, 0.7)
    g, go = ct.Geometry(*args), oracle.Geometry(*args)
    assert g.info.shared_lines == 1
    rng = np.random.default_rng(sum(shape))
    x = rng.uniform(0.1, 1.0, size=shape).astype(np.float32)
    y = _cpu(g.project(torch_cuda(x)))
    L, _ = go.ray_lengths()
    assert (L > 0).any()
    bad = fp_violations(y, go.project(x), L, float(x.max()))
    assert bad.size == 0, bad[:8]
    yy = rng.uniform(0.1, 1.0, size=go.sino_shape).astype(np.float32)
    assert rel_l2(_cpu(g.backproject(torch_cuda(yy))), go.backproject(yy)) <= BP_RTOL


def test_lines_entering_through_a_face(ct):
    """A short, wide volume seen from far above: every ray of a line enters through the top face
    at its own position along the line, so no lane starts at the line's entry (each finds its
    first list entry by counting), and many chords are short (the per-ray fallback)."""
    views = W.circular_cone(13, 40.0, 90.0).copy()
    views[:, 2] += 60.0     # source z, far above the slab
    views[:, 5] -= 20.0     # detector centre z
    shape = (6, 47, 53)
    args = (W.CONE, views, shape, 1.0, 61, 67, 1.1, 1.4)
    g, go = ct.Geometry(*args), oracle.Geometry(*args)
    assert g.info.shared_lines == 1
    x = W.ellipsoids_3d(6, 53, np.random.default_rng(4), axis_range=(3.0, 20.0))[:6, :47, :53]
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = _cpu(g.project(torch_cuda(x)))
    L, _ = go.ray_lengths()
    assert (L > 0).mean() > 0.3
    bad = fp_violations(y, go.project(x, threads=8), L, float(np.abs(x).max()))
    assert bad.size == 0, (bad.size, bad[:8])
    rng = np.random.default_rng(5)
    xr = rng.uniform(-1, 1, size=shape).astype(np.float32)
    yr = rng.uniform(-1, 1, size=go.sino_shape).astype(np.float32)
    gap, lhs, rhs = adjoint_gap(_cpu(g.project(torch_cuda(xr))), yr, xr,
                                _cpu(g.backproject(torch_cuda(yr))))
    assert gap <= 1e-6, (gap, lhs, rhs)


def _random_line_geometry(seed):
    """Random geometry whose detector v axis is exactly z in every view (so its lines share
    their xy path): cone orbits with random radii, source and detector offsets (z included) and
    in-plane detector rotations, or parallel rays at random elevations; random volume shape,
    per-axis pitches, detector size and pitches."""
    rng = np.random.default_rng(5000 + seed)
    nz, ny, nx = (int(v) for v in rng.integers(3, 40, size=3))
    sp = tuple(float(v) for v in rng.uniform(0.6, 1.4, size=3))
    n_views = int(rng.integers(3, 12))
    n_u, n_v = int(rng.integers(20, 90)), int(rng.integers(20, 90))
    du, dv = float(rng.uniform(0.5, 1.5)), float(rng.uniform(0.5, 1.5))
    views = []
    for _ in range(n_views):
        th = rng.uniform(0, 2 * math.pi)
        c, s = math.cos(th), math.sin(th)
        rot = rng.uniform(-0.3, 0.3)                      # detector turned about z
        du_vec = [-math.sin(th + rot), math.cos(th + rot), 0.0]
        if seed % 2 == 0:
            sid = rng.uniform(40, 90)
            sdd = sid + rng.uniform(20, 60)
            src = [sid * c, sid * s, rng.uniform(-10, 10)]
            det = [-(sdd - sid) * c + rng.uniform(-3, 3), -(sdd - sid) * s + rng.uniform(-3, 3),
                   rng.uniform(-10, 10)]
            views.append(src + det + du_vec + [0.0, 0.0, 1.0])
        else:
            ph = rng.uniform(-1.2, 1.2)                  # elevation of the rays
            ray = [c * math.cos(ph), s * math.cos(ph), math.sin(ph)]
            views.append(ray + list(rng.uniform(-2, 2, size=3)) + du_vec + [0.0, 0.0, 1.0])
    beam = W.CONE if seed % 2 == 0 else W.PARALLEL3D
    return W.Workload(f"random-lines-{seed}", beam, np.array(views), (nz, ny, nx), sp, n_u, n_v,
                      du, dv, seed, None)


@pytest.mark.parametrize("seed", range(10))
def test_random_shared_line_geometries(ct, seed):
    w = _random_line_geometry(seed)
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    rng = np.random.default_rng(seed)
    x = rng.uniform(0.1, 1.0, size=w.volume_shape).astype(np.float32)
    L, _ = go.ray_lengths()
    if g.info.volume_layout != 1:
        pytest.skip("the volume order chosen for this shape is not z-fastest")
    assert g.info.shared_lines == 1
    assert (L > 0).mean() > 0.02
    y = _cpu(g.project(torch_cuda(x)))
    bad = fp_violations(y, go.project(x, threads=8), L, float(x.max()))
    assert bad.size == 0, (bad.size, bad[:8])
    yy = rng.uniform(0.1, 1.0, size=w.sino_shape).astype(np.float32)
    assert rel_l2(_cpu(g.backproject(torch_cuda(yy))), go.backproject(yy, threads=8)) <= BP_RTOL
    xr = rng.uniform(-1, 1, size=w.volume_shape).astype(np.float32)
    yr = rng.uniform(-1, 1, size=w.sino_shape).astype(np.float32)
    gap, lhs, rhs = adjoint_gap(_cpu(g.project(torch_cuda(xr))), yr, xr,
                                _cpu(g.backproject(torch_cuda(yr))))
    assert gap <= ADJ_RTOL, (gap, lhs, rhs)


# Seeds whose geometries have short chords with a crossing taken at a grazing angle far from the
# volume's corner (z cell 30 of 35 at 1/|dh| = 430 on seed 458): a float32 entry coordinate moved
# such a crossing by 2e-4 cells, two to four times the per-ray tolerance of those chords.
@pytest.mark.parametrize("seed", [458, 603, 649, 665, 982, 1096, 1245, 1990])
def test_grazing_crossings_far_along_an_axis(ct, seed):
    w = _random_line_geometry(seed)
    g = ct.Geometry.from_workload(w)
    go = oracle.Geometry.from_workload(w)
    x = np.random.default_rng(seed).uniform(0.1, 1.0, size=w.volume_shape).astype(np.float32)
    L, _ = go.ray_lengths()
    y = _cpu(g.project(torch_cuda(x)))
    bad = fp_violations(y, go.project(x, threads=8), L, float(x.max()))
    assert bad.size == 0, (bad.size, bad[:8])

