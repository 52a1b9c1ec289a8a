"""Pins for the float64 oracle, against facts that do not come from the oracle itself.

* closed forms: uniform box -> value x chord length, where the chord comes from an independent
  bisection on the point-in-box test; axis-aligned parallel rays -> column sums x spacing;
  the diffct quickstart square (golden rows derived from the page's setup by hand);
* brute force on 1-8-voxel volumes: every voxel's own half-open box intersected with the ray,
  in pure Python, compared voxel by voxel (covers random, corner, face and axis-parallel rays);
* the adjoint identity <A x, y> = <x, A^T y> to 1e-12 relative;
* exact invariants: ray reversal, axis permutation, mirroring;
* row sums A 1 = ray chord length; SIRT fixed point and non-increasing weighted residual.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
from fan_beam_projector_siddon_b300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------------------------
# independent helpers (no plane enumeration, no slab formula)
# ---------------------------------------------------------------------------------------------

def _inside_closed(p, half):
    return all(abs(p[a]) <= half[a] for a in range(len(half)))


def _bisect_chord(e, d, amin, amax, q_alpha, half):
    """Length of the ray p(a) = e + a d, a in [amin, amax], inside the closed box |p_a| <= half_a.

    ``q_alpha`` is a parameter whose point lies strictly inside the box; each boundary crossing is
    located by bisection between that point and the corresponding end of the parameter range.
    """
    e, d = np.asarray(e, float), np.asarray(d, float)
    p = lambda a: e + a * d

    def boundary(a_in, a_out):
        if _inside_closed(p(a_out), half):
            return a_out
        for _ in range(200):
            m = 0.5 * (a_in + a_out)
            if m == a_in or m == a_out:
                break
            if _inside_closed(p(m), half):
                a_in = m
            else:
                a_out = m
        return 0.5 * (a_in + a_out)

    assert _inside_closed(p(q_alpha), half)
    lo = boundary(q_alpha, amin)
    hi = boundary(q_alpha, amax)
    return (hi - lo) * float(np.linalg.norm(d))


def _brute_row_python(e, d, amin, amax, vol_shape, s, dims):
    """Per-voxel chord of the ray through each half-open cell, pure Python."""
    nz, ny, nx = vol_shape
    n = (nx, ny, nz)
    row = np.zeros(vol_shape, dtype=np.float64)
    dl = math.sqrt(sum(d[a] ** 2 for a in range(dims)))
    for iz in range(nz):
        for iy in range(ny):
            for ix in range(nx):
                idx = (ix, iy, iz)
                a0, a1 = amin, amax
                ok = True
                for a in range(dims):
                    lo = -n[a] * s / 2 + idx[a] * s
                    hi = lo + s
                    if d[a] == 0:
                        if not (lo <= e[a] < hi):
                            ok = False
                            break
                    else:
                        t1, t2 = (lo - e[a]) / d[a], (hi - e[a]) / d[a]
                        a0, a1 = max(a0, min(t1, t2)), min(a1, max(t1, t2))
                if ok and a1 > a0:
                    row[iz, iy, ix] = (a1 - a0) * dl
    return row


def _dense(idx, w, vol_shape):
    row = np.zeros(int(np.prod(vol_shape)), dtype=np.float64)
    np.add.at(row, idx, w)
    return row.reshape(vol_shape)


def _geom(beam, views, vol_shape, s, nu, nv, du, dv):
    return oracle.Geometry(beam, views, vol_shape, s, nu, nv, du, dv)


# ---------------------------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------------------------

def test_quickstart_square_golden():
    """diffct quickstart: 64^2 image, square [20:44, 20:44] = 1, 96 detectors at spacing 1."""
    g = _geom(W.PARALLEL2D, W.circular_parallel_2d(180), (1, 64, 64), 1.0, 96, 1, 1.0, 1.0)
    img = np.zeros((64, 64))
    img[20:44, 20:44] = 1.0
    sino = g.project(img)
    assert sino.shape == (180, 96)
    rows = [l.split() for l in open(os.path.join(GOLDEN, "quickstart_parallel64_square.txt"))
            if not l.startswith("#")]
    for r in rows:
        view, vals = int(r[0]), np.array([float(v) for v in r[1:]])
        np.testing.assert_allclose(sino[view], vals, rtol=0, atol=1e-12)


@pytest.mark.parametrize("s", [1.0, 0.5])
def test_axis_aligned_2d_row_and_column_sums(s):
    """Rays along +x see row sums, rays along +y see (mirrored) column sums, times the spacing."""
    rng = np.random.default_rng(7)
    ny, nx = 6, 9
    img = rng.uniform(-1, 1, size=(ny, nx))
    # along +x: det_u = (0, 1); U = ny pixels at the row centres
    g = _geom(W.PARALLEL2D, np.array([[1.0, 0, 0, 0, 0, 1.0]]), (1, ny, nx), s, ny, 1, s, s)
    np.testing.assert_allclose(g.project(img)[0], s * img.sum(axis=1), rtol=0, atol=1e-12)
    # along +y: det_u = (-1, 0); pixel u sits at x = -(u - (nx-1)/2) s, i.e. column nx-1-u
    g = _geom(W.PARALLEL2D, np.array([[0, 1.0, 0, 0, -1.0, 0]]), (1, ny, nx), s, nx, 1, s, s)
    np.testing.assert_allclose(g.project(img)[0], s * img.sum(axis=0)[::-1], rtol=0, atol=1e-12)
    # fan beam: source far on -x, detector on +x; central pixel of an odd detector hits row
    # centre when ny is odd -> use a 7-row image
    img7 = rng.uniform(-1, 1, size=(7, nx))
    g = _geom(W.FAN2D, np.array([[-50.0, 0, 40.0, 0, 0, 1.0]]), (1, 7, nx), s, 5, 1, 1.0, 1.0)
    np.testing.assert_allclose(g.project(img7)[0, 2], s * img7[3].sum(), rtol=0, atol=1e-12)


def test_axis_aligned_3d_column_sums():
    """parallel3d along z / x / y and a cone's central ray: column sums x spacing ([z, y, x])."""
    rng = np.random.default_rng(11)
    nz, ny, nx = 5, 7, 9
    vol = rng.uniform(-1, 1, size=(nz, ny, nx))
    s = 0.5
    # ray +z, det_u = +x, det_v = +y: sino[u, v] = s * sum_z vol[:, v, u]
    rec = np.array([[0, 0, 1.0, 0, 0, 0, 1.0, 0, 0, 0, 1.0, 0]])
    g = _geom(W.PARALLEL3D, rec, (nz, ny, nx), s, nx, ny, s, s)
    np.testing.assert_allclose(g.project(vol)[0], s * vol.sum(axis=0).T, rtol=0, atol=1e-12)
    # ray +x, det_u = +y, det_v = +z: sino[u, v] = s * sum_x vol[v, u, :]
    rec = np.array([[1.0, 0, 0, 0, 0, 0, 0, 1.0, 0, 0, 0, 1.0]])
    g = _geom(W.PARALLEL3D, rec, (nz, ny, nx), s, ny, nz, s, s)
    np.testing.assert_allclose(g.project(vol)[0], s * vol.sum(axis=2).T, rtol=0, atol=1e-12)
    # ray -y, det_u = +z, det_v = +x: sino[u, v] = s * sum_y vol[u, :, v]
    rec = np.array([[0, -1.0, 0, 0, 0, 0, 0, 0, 1.0, 1.0, 0, 0]])
    g = _geom(W.PARALLEL3D, rec, (nz, ny, nx), s, nz, nx, s, s)
    np.testing.assert_allclose(g.project(vol)[0], s * vol.sum(axis=1), rtol=0, atol=1e-12)
    # cone: source on -x axis, detector plane x = +30, odd detector -> the central pixel's ray is
    # the x axis through the central voxel column (odd sizes put it on voxel centres)
    rec = np.array([[-40.0, 0, 0, 30.0, 0, 0, 0, 1.0, 0, 0, 0, 1.0]])
    g = _geom(W.CONE, rec, (nz, ny, nx), s, 3, 3, 0.7, 0.7)
    np.testing.assert_allclose(g.project(vol)[0, 1, 1], s * vol[2, 3, :].sum(), rtol=0,
                               atol=1e-12)


def _random_rays(rng, n, half, segment):
    """Rays through a random interior point q; segment rays get endpoints outside the box."""
    out = []
    R = 4.0 * float(np.linalg.norm(half))
    for _ in range(n):
        q = rng.uniform(-0.98, 0.98, size=3) * half
        d = rng.standard_normal(3)
        d /= np.linalg.norm(d)
        if segment:
            a0, a1 = rng.uniform(1.0, 2.0) * R, rng.uniform(1.0, 2.0) * R
            src = q - a0 * d
            pix = q + a1 * d
            out.append((src, pix - src, 0.0, 1.0, a0 / (a0 + a1)))
        else:
            e = q + rng.uniform(-R, R) * d
            out.append((e, d, -np.inf, np.inf, float((q - e) @ d)))
    return out


@pytest.mark.parametrize("segment", [False, True])
def test_uniform_box_equals_value_times_bisection_chord(segment):
    rng = np.random.default_rng(3)
    vol_shape, s, c = (6, 10, 14), 0.75, 2.5
    half = 0.5 * s * np.array(vol_shape[::-1], dtype=float)
    vol = np.full(vol_shape, c)
    for e, d, amin, amax, qa in _random_rays(rng, 200, half, segment):
        idx, w = oracle.line_segments(e, d, amin, amax, vol_shape, s)
        y = float((vol.reshape(-1)[idx] * w).sum())
        big = 10.0 * float(np.linalg.norm(half)) / float(np.linalg.norm(d))
        lo = max(amin, qa - big)
        hi = min(amax, qa + big)
        L = _bisect_chord(e, d, lo, hi, qa, half)
        assert abs(y - c * L) <= 1e-12 * max(1.0, c * L)


def test_uniform_volume_rows_equal_ray_lengths_on_workloads():
    """A 1 == per-ray chord length == bisection chord for rays of the small workloads."""
    rng = np.random.default_rng(5)
    for n in (2, 3, 4, 5):
        w = W.small_config(n)
        g = oracle.Geometry.from_workload(w)
        ones = g.project(np.ones(w.volume_shape), views=(0, 3))
        length, _ = g.ray_lengths(views=(0, 3))
        np.testing.assert_allclose(ones[:3], length[:3], rtol=1e-13, atol=1e-13)
        assert (length[:3] > 0).mean() > 0.3


# ---------------------------------------------------------------------------------------------
# brute force on tiny volumes
# ---------------------------------------------------------------------------------------------

TINY_SHAPES = [(1, 1, 1), (2, 2, 2), (1, 2, 4), (4, 2, 1), (8, 1, 1), (1, 1, 8), (2, 1, 3)]


@pytest.mark.parametrize("vol_shape", TINY_SHAPES)
def test_brute_force_random_rays(vol_shape):
    rng = np.random.default_rng(sum(vol_shape))
    s = 0.5
    half = 0.5 * s * np.array(vol_shape[::-1], dtype=float)
    for segment in (False, True):
        for e, d, amin, amax, _ in _random_rays(rng, 60, half, segment):
            idx, w = oracle.line_segments(e, d, amin, amax, vol_shape, s)
            got = _dense(idx, w, vol_shape)
            ref = _brute_row_python(e, d, amin, amax, vol_shape, s, 3)
            np.testing.assert_allclose(got, ref, rtol=0, atol=1e-14)


def test_brute_force_face_corner_and_axis_rays():
    """Rays in cell faces go to the + side cell; the outer + face owns nothing; corner rays."""
    vol_shape, s = (2, 2, 2), 1.0
    cases = [
        # along x inside the face y = 0 (between iy = 0 and iy = 1) -> cells with iy = 1
        ((-5.0, 0.0, 0.3), (1.0, 0.0, 0.0)),
        # along x in the outer + face y = +1 -> nothing
        ((-5.0, 1.0, 0.3), (1.0, 0.0, 0.0)),
        # along x in the outer - face y = -1 -> cells with iy = 0
        ((-5.0, -1.0, -0.4), (1.0, 0.0, 0.0)),
        # along z on the edge x = 0, y = 0 -> cells (ix = 1, iy = 1)
        ((0.0, 0.0, -3.0), (0.0, 0.0, 1.0)),
        # main diagonal through the centre corner and two outer corners
        ((-2.0, -2.0, -2.0), (1.0, 1.0, 1.0)),
        # diagonal in the plane z = 0 through the central edge
        ((-2.0, -2.0, 0.0), (1.0, 1.0, 0.0)),
        # axis-parallel through cell interiors, negative direction
        ((0.5, -0.5, 4.0), (0.0, 0.0, -1.0)),
    ]
    for e, d in cases:
        idx, w = oracle.line_segments(e, d, -np.inf, np.inf, vol_shape, s)
        got = _dense(idx, w, vol_shape)
        ref = _brute_row_python(e, d, -np.inf, np.inf, vol_shape, s, 3)
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-14)
    # spot values (z, y, x) for the first and the diagonal case
    idx, w = oracle.line_segments(cases[0][0], cases[0][1], -np.inf, np.inf, vol_shape, s)
    row = _dense(idx, w, vol_shape)
    assert row[1, 1, 0] == 1.0 and row[1, 1, 1] == 1.0 and row.sum() == 2.0
    idx, w = oracle.line_segments(cases[1][0], cases[1][1], -np.inf, np.inf, vol_shape, s)
    assert len(idx) == 0
    idx, w = oracle.line_segments(cases[4][0], cases[4][1], -np.inf, np.inf, vol_shape, s)
    row = _dense(idx, w, vol_shape)
    assert abs(row[0, 0, 0] - math.sqrt(3)) < 1e-14 and abs(row[1, 1, 1] - math.sqrt(3)) < 1e-14
    assert abs(row.sum() - 2 * math.sqrt(3)) < 1e-14


@pytest.mark.parametrize("beam", [W.CONE, W.PARALLEL3D, W.FAN2D, W.PARALLEL2D])
def test_brute_force_geometry_rows(beam):
    """Whole rows of A via view records: Siddon traversal vs the C brute force vs Python."""
    rng = np.random.default_rng(beam + 20)
    if beam in (W.CONE, W.PARALLEL3D):
        vol_shape, s = (2, 3, 2), 0.5
        views = []
        for _ in range(4):
            u = rng.standard_normal(3); u /= np.linalg.norm(u)
            v = rng.standard_normal(3); v -= (v @ u) * u; v /= np.linalg.norm(v)
            n = np.cross(u, v)
            if beam == W.CONE:
                views.append(np.concatenate([-4.0 * n + rng.uniform(-.2, .2, 3), 3.0 * n, u, v]))
            else:
                r = n + 0.3 * rng.standard_normal(3); r /= np.linalg.norm(r)
                views.append(np.concatenate([r, rng.uniform(-.1, .1, 3), u, v]))
        g = _geom(beam, np.array(views), vol_shape, s, 5, 4, 0.37, 0.41)
    else:
        vol_shape, s = (1, 3, 4), 0.5
        views = []
        for _ in range(4):
            th = rng.uniform(0, 2 * math.pi)
            r = np.array([math.cos(th), math.sin(th)])
            u = np.array([-r[1], r[0]])
            if beam == W.FAN2D:
                views.append(np.concatenate([-4.0 * r, 3.0 * r, u]))
            else:
                views.append(np.concatenate([r, rng.uniform(-.1, .1, 2), u]))
        g = _geom(beam, np.array(views), vol_shape, s, 7, 1, 0.33, 1.0)
    for view in range(g.n_views):
        for iu in range(g.n_u):
            for iv in range(g.n_v):
                idx, w = g.ray_segments(view, iu, iv)
                got = _dense(idx, w, g.volume_shape)
                ref = g.brute_row(view, iu, iv)
                np.testing.assert_allclose(got, ref, rtol=0, atol=1e-14)
    # Python brute force on one ray per view, using the page's pixel formula
    for view in range(g.n_views):
        rec = g.views[view]
        iu, iv = 3, min(1, g.n_v - 1)
        if g.is_2d:
            first, ctr, du = (np.r_[rec[0:2], 0], np.r_[rec[2:4], 0], np.r_[rec[4:6], 0])
            pix = ctr + (iu - (g.n_u - 1) / 2) * 0.33 * du
        else:
            first, ctr, du, dv = rec[0:3], rec[3:6], rec[6:9], rec[9:12]
            pix = (ctr + (iu - (g.n_u - 1) / 2) * 0.37 * du + (iv - (g.n_v - 1) / 2) * 0.41 * dv)
        if beam in (W.PARALLEL2D, W.PARALLEL3D):
            e, d, amin, amax = pix, first, -np.inf, np.inf
        else:
            e, d, amin, amax = first, pix - first, 0.0, 1.0
        ref = _brute_row_python(e, d, amin, amax, vol_shape, s, 2 if g.is_2d else 3)
        idx, w = g.ray_segments(view, iu, iv)
        np.testing.assert_allclose(_dense(idx, w, g.volume_shape).reshape(vol_shape), ref,
                                   rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------------------------
# adjoint identity, invariants
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_adjoint_identity_small_workloads(n):
    w = W.small_config(n)
    g = oracle.Geometry.from_workload(w)
    rng = np.random.default_rng(n)
    x = rng.uniform(-1, 1, size=w.volume_shape)
    y = rng.uniform(-1, 1, size=w.sino_shape)
    lhs = float((g.project(x, threads=4) * y).sum())
    rhs = float((x * g.backproject(y, threads=4)).sum())
    assert abs(lhs - rhs) <= 1e-12 * max(abs(lhs), abs(rhs))


def test_threaded_views_match_single_thread():
    w = W.small_config(3)
    g = oracle.Geometry.from_workload(w)
    x = w.phantom()
    np.testing.assert_array_equal(g.project(x, threads=1), g.project(x, threads=3))
    y = W.random_sinogram(w, 1)
    np.testing.assert_allclose(g.backproject(y, threads=1), g.backproject(y, threads=3),
                               rtol=1e-13, atol=1e-13)


def test_invariants_reversal_permutation_mirror():
    rng = np.random.default_rng(9)
    vol_shape, s = (5, 7, 6), 0.8
    vol = rng.uniform(-1, 1, size=vol_shape)
    half = 0.5 * s * np.array(vol_shape[::-1], dtype=float)

    def integral(v, e, d, amin, amax):
        idx, w = oracle.line_segments(e, d, amin, amax, v.shape, s)
        return float((v.reshape(-1)[idx] * w).sum())

    for e, d, amin, amax, _ in _random_rays(rng, 50, half, True):
        y = integral(vol, e, d, amin, amax)
        # reversal: walk from the pixel back to the source
        assert abs(integral(vol, e + d, -d, 0.0, 1.0) - y) <= 1e-12 * max(1, abs(y))
        # permutation of Cartesian axes (x, y, z) -> (y, z, x) with the matching volume transpose
        perm = [1, 2, 0]                      # new component k is old component perm[k]
        ep, dp = e[perm], d[perm]
        # volume [z, y, x]: new x = old y, new y = old z, new z = old x -> new [z,y,x] = old [x,z,y]
        volp = np.ascontiguousarray(np.transpose(vol, (2, 0, 1)))
        assert abs(integral(volp, ep, dp, 0.0, 1.0) - y) <= 1e-12 * max(1, abs(y))
        # mirror x -> -x with the volume flipped along x
        em, dm = e * np.array([-1, 1, 1]), d * np.array([-1, 1, 1])
        assert abs(integral(vol[:, :, ::-1].copy(), em, dm, 0.0, 1.0) - y) <= 1e-12 * max(1, abs(y))


# ---------------------------------------------------------------------------------------------
# sampled-voxel adjoint, SIRT
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_backproject_voxels_matches_full_backprojection(n):
    w = W.small_config(n)
    g = oracle.Geometry.from_workload(w)
    y = W.random_sinogram(w, 3)
    full = g.backproject(y, threads=4).reshape(-1)
    vox = np.random.default_rng(n).choice(full.size, size=40, replace=False)
    np.testing.assert_allclose(g.backproject_voxels(y, vox), full[vox], rtol=1e-12, atol=1e-12)


def test_sirt_fixed_point_and_monotone_residual():
    w = W.small_config(5)
    g = oracle.Geometry.from_workload(w)
    x_true = w.phantom().astype(np.float64)
    y = g.project(x_true, threads=4)
    # fixed point: starting at x_true with consistent data, x does not move
    x1, res = g.sirt(y, 2, x0=x_true)
    np.testing.assert_allclose(x1, x_true, rtol=0, atol=1e-12)
    assert res.max() < 1e-20
    # from zero: the R-weighted residual never increases (relaxation in (0, 2))
    x, res = g.sirt(y, 8)
    assert np.all(np.diff(res) <= 1e-12 * res[0])
    assert res[-1] < 0.5 * res[0]


@pytest.mark.parametrize("beam", [W.CONE, W.FAN2D])
def test_segment_reading_detector_inside_volume(beam):
    """Fan/cone rays are the source-to-pixel segment: with the source and the detector plane both
    inside the box, voxels beyond either end get nothing (reading of the pages' silence)."""
    rng = np.random.default_rng(31)
    if beam == W.CONE:
        vol_shape, s = (3, 4, 5), 1.0
        rec = np.array([[-1.3, 0.2, 0.1, 1.1, 0.0, 0.0, 0.0, 1.0, 0.0, 0.0, 0.0, 1.0]])
        g = _geom(beam, rec, vol_shape, s, 5, 3, 0.6, 0.6)
        dims = 3
    else:
        vol_shape, s = (1, 4, 5), 1.0
        rec = np.array([[-1.3, 0.2, 1.1, 0.0, 0.0, 1.0]])
        g = _geom(beam, rec, vol_shape, s, 5, 1, 0.6, 1.0)
        dims = 2
    vol = rng.uniform(0.5, 1.0, size=g.volume_shape)
    sino = g.project(vol)
    for iu in range(g.n_u):
        for iv in range(g.n_v):
            src = np.r_[rec[0, :dims], [0.0] * (3 - dims)]
            ctr = np.r_[rec[0, dims:2 * dims], [0.0] * (3 - dims)]
            du = np.r_[rec[0, 2 * dims:3 * dims], [0.0] * (3 - dims)]
            dv = np.r_[rec[0, 9:12]] if dims == 3 else np.zeros(3)
            dvs = 0.6 if dims == 3 else 0.0
            pix = ctr + (iu - (g.n_u - 1) / 2) * 0.6 * du + (iv - (g.n_v - 1) / 2) * dvs * dv
            ref = _brute_row_python(src, pix - src, 0.0, 1.0, vol_shape, s, dims)
            want = float((ref.reshape(g.volume_shape) * vol).sum())
            got = sino[0, iu] if dims == 2 else sino[0, iu, iv]
            assert abs(got - want) < 1e-13


def test_sirt_one_step_closed_forms():
    """Cases whose first SIRT update is known by hand.

    * One voxel, several rays with chords l_i and consistent data y_i = c l_i: R_i = 1/l_i,
      C = 1/sum l_i, so x_1 = sum(y_i / l_i * l_i) / sum l_i = c after one update.
    * parallel3d rays along z through each column centre of a (1, 2, 3) volume: A is diagonal with
      chord s, so x_1 = y / s exactly, whatever y is.
    """
    rec = []
    for th in (0.1, 0.7, 1.3, 2.9):
        r = np.array([math.cos(th), math.sin(th), 0.3])
        r /= np.linalg.norm(r)
        u = np.array([-math.sin(th), math.cos(th), 0.0])
        v = np.cross(r, u)
        rec.append(np.concatenate([r, np.zeros(3), u, v]))
    g = _geom(W.PARALLEL3D, np.array(rec), (1, 1, 1), 0.8, 3, 3, 0.05, 0.05)
    c = 1.7
    y = g.project(np.full((1, 1, 1), c))
    assert (y > 0).all()
    x1, _ = g.sirt(y, 1)
    np.testing.assert_allclose(x1, c, rtol=1e-14)
    s = 0.5
    rec = np.array([[0, 0, 1.0, 0, 0, 0, 1.0, 0, 0, 0, 1.0, 0]])
    g = _geom(W.PARALLEL3D, rec, (1, 2, 3), s, 3, 2, s, s)
    y = np.random.default_rng(2).uniform(-1, 1, size=(1, 3, 2))
    x1, _ = g.sirt(y, 1)
    np.testing.assert_allclose(x1[0], y[0].T / s, rtol=1e-14)


# ---------------------------------------------------------------------------------------------
# CGLS
# ---------------------------------------------------------------------------------------------

def _dense_matrix(g):
    """Rows of A for every ray by the C brute force (tiny problems only)."""
    rows = []
    for view in range(g.n_views):
        for iu in range(g.n_u):
            for iv in range(g.n_v):
                rows.append(g.brute_row(view, iu, iv).reshape(-1))
    return np.array(rows)


def test_sirt_converges_to_the_weighted_least_squares_solution():
    """SIRT from x = 0 with relaxation in (0, 2) converges to the minimiser of the R-weighted
    residual ||A x - y||_R (R = 1 / row sums); with A of full column rank and inconsistent data
    that is the unique solution of A^T R A x = A^T R y.  A and R come from the per-voxel brute
    force; the unweighted least-squares solution differs by ~0.7 here, so a wrong R fails."""
    rng = np.random.default_rng(31)
    rec = []
    for th in np.linspace(0.1, 3.0, 7):
        r = np.array([math.cos(th), math.sin(th), 0.35])
        r /= np.linalg.norm(r)
        u = np.array([-math.sin(th), math.cos(th), 0.0])
        rec.append(np.concatenate([r, rng.uniform(-0.2, 0.2, 3), u, np.cross(r, u)]))
    g = _geom(W.PARALLEL3D, np.array(rec), (2, 3, 3), 1.0, 6, 5, 0.7, 0.7)
    A = _dense_matrix(g)
    assert np.linalg.matrix_rank(A) == A.shape[1]
    y = rng.uniform(0.5, 1.5, size=g.sino_shape)
    rs = A.sum(axis=1)
    R = np.where(rs > 0, 1.0 / np.where(rs > 0, rs, 1.0), 0.0)
    x_ls = np.linalg.solve(A.T @ (R[:, None] * A), A.T @ (R * y.reshape(-1)))
    x, _ = g.sirt(y, 6000)
    np.testing.assert_allclose(x.reshape(-1), x_ls, rtol=0, atol=1e-9)
    x_un = np.linalg.lstsq(A, y.reshape(-1), rcond=None)[0]
    assert np.abs(x_un - x_ls).max() > 0.1


def test_cgls_reaches_the_least_squares_solution():
    """In exact arithmetic CGLS from x = 0 reaches the minimum-norm least-squares solution of
    min ||A x - y|| within rank(A) steps; checked against numpy's SVD-based lstsq of the explicit
    matrix (rows from the per-voxel brute force) on a 3x3x2-voxel cone problem."""
    rng = np.random.default_rng(4)
    views = []
    for k in range(5):
        th = 2 * math.pi * k / 5
        src = np.array([6 * math.cos(th), 6 * math.sin(th), 0.7 * math.sin(3 * th)])
        u = np.array([-math.sin(th), math.cos(th), 0.0])
        v = np.array([0.0, 0.0, 1.0])
        views.append(np.concatenate([src, -4 * src / 6, u, v]))
    g = _geom(W.CONE, np.array(views), (2, 3, 3), 0.8, 4, 3, 0.9, 0.9)
    A = _dense_matrix(g)
    y = rng.uniform(0, 1, size=A.shape[0])
    x_ls = np.linalg.lstsq(A, y, rcond=None)[0]
    rank = np.linalg.matrix_rank(A)
    x, res = g.cgls(y.reshape(g.sino_shape), rank + 2)
    np.testing.assert_allclose(x.reshape(-1), x_ls, rtol=0, atol=1e-8 * np.abs(x_ls).max())
    # the residual norm never increases
    assert np.all(np.diff(res) <= 1e-12 * res[0])
    # A x agrees with the oracle's own projection of x (CGLS used A, not a stand-in)
    np.testing.assert_allclose(A @ x.reshape(-1), g.project(x).reshape(-1), rtol=1e-12,
                               atol=1e-12)


def test_cgls_fixed_point_and_first_step():
    """Consistent data from x_true is a fixed point; the first step from 0 is the exact line
    search along A^T y: x_1 = (|A^T y|^2 / |A A^T y|^2) A^T y."""
    w = W.small_config(1)
    g = oracle.Geometry.from_workload(w)
    x_true = w.phantom().astype(np.float64)
    y = g.project(x_true)
    x1, res = g.cgls(y, 2, x0=x_true)
    np.testing.assert_allclose(x1, x_true, rtol=0, atol=1e-12)
    assert res.max() < 1e-20
    s = g.backproject(y)
    q = g.project(s)
    want = (np.sum(s * s) / np.sum(q * q)) * s
    x1, _ = g.cgls(y, 1)
    np.testing.assert_allclose(x1, want, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------------------------
# per-axis voxel spacing
# ---------------------------------------------------------------------------------------------

def _brute_row_python_aniso(e, d, amin, amax, vol_shape, s_xyz, dims):
    """Per-voxel chord through half-open cells with spacing s_xyz = (sx, sy, sz), pure Python."""
    nz, ny, nx = vol_shape
    n = (nx, ny, nz)
    row = np.zeros(vol_shape, dtype=np.float64)
    dl = math.sqrt(sum(d[a] ** 2 for a in range(dims)))
    for iz in range(nz):
        for iy in range(ny):
            for ix in range(nx):
                idx = (ix, iy, iz)
                a0, a1, ok = amin, amax, True
                for a in range(dims):
                    lo = -n[a] * s_xyz[a] / 2 + idx[a] * s_xyz[a]
                    hi = lo + s_xyz[a]
                    if d[a] == 0:
                        if not (lo <= e[a] < hi):
                            ok = False
                            break
                    else:
                        t1, t2 = (lo - e[a]) / d[a], (hi - e[a]) / d[a]
                        a0, a1 = max(a0, min(t1, t2)), min(a1, max(t1, t2))
                if ok and a1 > a0:
                    row[iz, iy, ix] = (a1 - a0) * dl
    return row


def test_anisotropic_axis_aligned_column_sums():
    """With spacing (dz, dy, dx) the column sum along an axis is scaled by that axis's pitch."""
    rng = np.random.default_rng(13)
    nz, ny, nx = 5, 7, 9
    dz, dy, dx = 0.5, 0.8, 1.25
    vol = rng.uniform(-1, 1, size=(nz, ny, nx))
    rec = np.array([[0, 0, 1.0, 0, 0, 0, 1.0, 0, 0, 0, 1.0, 0]])              # along +z
    g = _geom(W.PARALLEL3D, rec, (nz, ny, nx), (dz, dy, dx), nx, ny, dx, dy)
    np.testing.assert_allclose(g.project(vol)[0], dz * vol.sum(axis=0).T, rtol=0, atol=1e-12)
    rec = np.array([[1.0, 0, 0, 0, 0, 0, 0, 1.0, 0, 0, 0, 1.0]])              # along +x
    g = _geom(W.PARALLEL3D, rec, (nz, ny, nx), (dz, dy, dx), ny, nz, dy, dz)
    np.testing.assert_allclose(g.project(vol)[0], dx * vol.sum(axis=2).T, rtol=0, atol=1e-12)
    rec = np.array([[0, -1.0, 0, 0, 0, 0, 0, 0, 1.0, 1.0, 0, 0]])             # along -y
    g = _geom(W.PARALLEL3D, rec, (nz, ny, nx), (dz, dy, dx), nz, nx, dz, dx)
    np.testing.assert_allclose(g.project(vol)[0], dy * vol.sum(axis=1), rtol=0, atol=1e-12)
    # 2D, (dy, dx): rays along +x see dx * row sums
    img = rng.uniform(-1, 1, size=(ny, nx))
    g = _geom(W.PARALLEL2D, np.array([[1.0, 0, 0, 0, 0, 1.0]]), (1, ny, nx), (dy, dx), ny, 1,
              dy, 1.0)
    np.testing.assert_allclose(g.project(img)[0], dx * img.sum(axis=1), rtol=0, atol=1e-12)


@pytest.mark.parametrize("segment", [False, True])
def test_anisotropic_uniform_box_and_brute_force(segment):
    rng = np.random.default_rng(17)
    vol_shape, s_zyx = (2, 3, 4), (0.7, 1.3, 0.45)
    s_xyz = s_zyx[::-1]
    half = 0.5 * np.array(vol_shape[::-1], dtype=float) * np.array(s_xyz)
    c = 1.75
    vol = np.full(vol_shape, c)
    for e, d, amin, amax, qa in _random_rays(rng, 80, half, segment):
        idx, w = oracle.line_segments(e, d, amin, amax, vol_shape, s_zyx)
        got = _dense(idx, w, vol_shape)
        np.testing.assert_allclose(got, _brute_row_python_aniso(e, d, amin, amax, vol_shape,
                                                                s_xyz, 3), rtol=0, atol=1e-14)
        big = 10.0 * float(np.linalg.norm(half)) / float(np.linalg.norm(d))
        L = _bisect_chord(e, d, max(amin, qa - big), min(amax, qa + big), qa, half)
        assert abs(float((vol.reshape(-1)[idx] * w).sum()) - c * L) <= 1e-12 * max(1.0, c * L)


@pytest.mark.parametrize("kind", ["cone", "tilt", "fan"])
def test_anisotropic_adjoint_and_rows(kind):
    w = W.anisotropic_config(kind)
    g = oracle.Geometry.from_workload(w)
    rng = np.random.default_rng(3)
    x = rng.uniform(-1, 1, size=w.volume_shape)
    y = rng.uniform(-1, 1, size=w.sino_shape)
    lhs = float((g.project(x, threads=4) * y).sum())
    rhs = float((x * g.backproject(y, threads=4)).sum())
    assert abs(lhs - rhs) <= 1e-12 * max(abs(lhs), abs(rhs))
    # a few whole rows against the per-voxel brute force
    for k in range(4):
        view, iu = int(rng.integers(w.n_views)), int(rng.integers(w.n_u))
        iv = int(rng.integers(w.n_v))
        idx, wt = g.ray_segments(view, iu, iv)
        np.testing.assert_allclose(_dense(idx, wt, g.volume_shape), g.brute_row(view, iu, iv),
                                   rtol=0, atol=1e-13)


def test_grazing_crossings_far_along_an_axis():
    """Short chords that cross a plane at a grazing angle far from the volume's corner (the
    crossing's position along the ray is the plane distance over a tiny direction component):
    the oracle's segments equal the pure-Python per-voxel clip.  The first ray is a corner clip of
    a 6 x 9 x 35 volume that crosses z plane 30 at 1/|dz| = 430 voxel lengths per cell.  Both
    sides round plane positions of ~10 units in float64 and a grazing crossing multiplies that by
    up to 1/|dz| = 1000, hence 1e-10 (a float32 plane position would be off by 1e-4)."""
    vol_shape, s_zyx = (35, 9, 6), (0.6582214119560114, 1.1847855166608365, 0.8213995296135223)
    s_xyz = s_zyx[::-1]
    rays = [(np.array([78.47037568, -29.22880575, 8.03421051]),
             np.array([-112.59456299, 50.87213812, 0.28538153]))]
    rng = np.random.default_rng(29)
    half = 0.5 * np.array(vol_shape[::-1], dtype=float) * np.array(s_xyz)
    for _ in range(12):
        # through a point near a vertical edge of the box, almost level, crossing a high z plane
        th = rng.uniform(0, 2 * math.pi)
        d = np.array([math.cos(th), math.sin(th), rng.choice([-1, 1]) * rng.uniform(1e-3, 3e-3)])
        edge = np.array([rng.choice([-1, 1]) * half[0], rng.choice([-1, 1]) * half[1],
                         (rng.integers(20, 34) - vol_shape[0] / 2) * s_zyx[0]])
        p = edge + rng.uniform(-0.3, 0.3, 3) * np.array([1, 1, 0]) + np.array([0, 0, 1e-4])
        rays.append((p - 40.0 * d, d))
    hit = 0
    for e, d in rays:
        idx, w = oracle.line_segments(e, d, -np.inf, np.inf, vol_shape, s_zyx)
        ref = _brute_row_python_aniso(e, d, -np.inf, np.inf, vol_shape, s_xyz, 3)
        np.testing.assert_allclose(_dense(idx, w, vol_shape), ref, rtol=0, atol=1e-10)
        hit += int(len(set((np.nonzero(ref.reshape(-1))[0] // (9 * 6)).tolist())) >= 2)
    assert hit >= 4   # rays whose chord crosses a z plane


# ---------------------------------------------------------------------------------------------
# parameterized detector surfaces
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_flat_detector_as_offsets_equals_flat_formula(n):
    """The page's flat pixel formula and the same detector given as per-pixel offsets."""
    w = W.small_config(n)
    flat = oracle.Geometry.from_workload(w)
    off = W.flat_offsets(w.n_u, w.n_v, w.du, w.dv)
    surf = oracle.Geometry(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du,
                           w.dv, offsets=off)
    x = w.phantom()
    np.testing.assert_allclose(surf.project(x, views=(0, 4)), flat.project(x, views=(0, 4)),
                               rtol=1e-12, atol=1e-10)


@pytest.mark.parametrize("kind", ["cone", "fan"])
def test_cylinder_centred_on_source(kind):
    """Radius = source-detector distance: every pixel is that far from the source across the
    cylinder's axis (det_v), and the projection obeys the adjoint identity, brute-force rows
    and the bisection chord of a uniform box."""
    w = W.curved_config(kind)
    g = oracle.Geometry.from_workload(w)
    k = 2 if w.is_2d else 3
    sdd = float(np.linalg.norm(w.views[0, 0:k] - w.views[0, k:2 * k]))
    rng = np.random.default_rng(1)
    for _ in range(40):
        view, iu, iv = int(rng.integers(w.n_views)), int(rng.integers(w.n_u)), int(rng.integers(w.n_v))
        e, d, (a0, a1) = g.ray(view, iu, iv)
        if not w.is_2d:
            axis = w.views[view, 9:12]
            d = d - (d @ axis) * axis
        assert abs(np.linalg.norm(d) - sdd) <= 1e-9 * sdd
    x = rng.uniform(-1, 1, size=w.volume_shape)
    y = rng.uniform(-1, 1, size=w.sino_shape)
    lhs = float((g.project(x, threads=4) * y).sum())
    rhs = float((x * g.backproject(y, threads=4)).sum())
    assert abs(lhs - rhs) <= 1e-12 * max(abs(lhs), abs(rhs))
    for _ in range(3):
        view, iu = int(rng.integers(w.n_views)), int(rng.integers(w.n_u))
        iv = int(rng.integers(w.n_v))
        idx, wt = g.ray_segments(view, iu, iv)
        np.testing.assert_allclose(_dense(idx, wt, g.volume_shape), g.brute_row(view, iu, iv),
                                   rtol=0, atol=1e-12)
    # uniform volume: each ray's line integral is value x its chord through the box, found by
    # bisection along the oracle's own ray
    c = 1.5
    ones = g.project(np.full(w.volume_shape, c), views=(0, 2))
    nz, ny, nx = w.vol_shape
    half = 0.5 * np.array([nx, ny, nz], dtype=float) * 1.0
    dims = 2 if w.is_2d else 3
    for iu in range(0, w.n_u, 7):
        e, d, (a0, a1) = g.ray(1, iu, w.n_v // 2)
        ts = np.linspace(a0, a1, 4001)[1:-1]
        inside = [t for t in ts if _inside_closed((e + t * d)[:dims], half[:dims])]
        if not inside:
            continue
        L = _bisect_chord(e[:dims], d[:dims], a0, a1, inside[len(inside) // 2], half[:dims])
        got = ones[1, iu] if w.is_2d else ones[1, iu, w.n_v // 2]
        assert abs(got - c * L) <= 1e-9 * max(1.0, c * L)
