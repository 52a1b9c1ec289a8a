"""Pins for the float64 FBP/FDK reference (oracle/fbp.py).

* filter taps from quadrature against the textbook closed forms of the band-limited Ram-Lak and
  Shepp-Logan kernels (Kak & Slaney), and every window's taps against a direct Riemann sum of
  their frequency response;
* reconstructions of analytically projected objects (a disk in parallel and fan geometry, a ball
  in cone geometry -- sinograms from chord lengths, not from any projector) come back close to 1
  inside and close to 0 outside; this pins the filter scale, the view weights, the cosine weights
  and the distance weights together.
"""
import math

import numpy as np
import pytest

from fan_beam_projector_siddon_b300 import workloads as W
from oracle import fbp as F


@pytest.mark.parametrize("tau,n_u", [(1.0, 10), (0.5, 10), (1.3, 10), (1.2, 384)])
def test_ramlak_and_shepp_logan_taps_match_closed_forms(tau, n_u):
    n = np.arange(-(n_u - 1), n_u)
    h = F.ramp_taps(n_u, tau, "ram-lak")
    nn = np.where(n == 0, 1, n).astype(float)
    want = np.where(n == 0, 1.0 / (4 * tau * tau),
                    np.where(n % 2 == 0, 0.0, -1.0 / (np.pi ** 2 * nn ** 2 * tau ** 2)))
    np.testing.assert_allclose(h, want, rtol=1e-9, atol=1e-12 / tau ** 2)
    h = F.ramp_taps(n_u, tau, "shepp-logan")
    want = -2.0 / (np.pi ** 2 * tau ** 2 * (4 * n.astype(float) ** 2 - 1))
    np.testing.assert_allclose(h, want, rtol=1e-9, atol=1e-12 / tau ** 2)


@pytest.mark.parametrize("window", F.WINDOWS)
def test_window_taps_against_riemann_sum(window):
    tau = 0.8
    h = F.ramp_taps(6, tau, window)
    f = (np.arange(200000) + 0.5) / 200000 * (0.5 / tau)
    df = (0.5 / tau) / 200000
    for n in range(6):
        want = 2 * np.sum(f * F.window_response(window, f, tau) * np.cos(2 * np.pi * f * n * tau)) * df
        assert abs(h[5 + n] - want) <= 1e-8 / tau ** 2


def _disk_parallel_sino(views, n_u, du, R):
    t = (np.arange(n_u) - (n_u - 1) / 2.0) * du
    row = 2 * np.sqrt(np.clip(R * R - t * t, 0, None))
    return np.tile(row, (views.shape[0], 1))


def _chord_ball(src, pix, R):
    """Chord of the segment src -> pix through the ball |x| <= R (all arrays (..., 3))."""
    d = pix - src
    L = np.linalg.norm(d, axis=-1)
    dh = d / L[..., None]
    b = np.sum(src * dh, axis=-1)
    c = np.sum(src * src, axis=-1) - R * R
    disc = b * b - c
    return 2 * np.sqrt(np.clip(disc, 0, None))


def _radius_grid(n, s):
    c = (np.arange(n) + 0.5 - n / 2.0) * s
    return c


def test_parallel_fbp_of_a_disk():
    n, R = 64, 20.0
    views = W.circular_parallel_2d(180)
    sino = _disk_parallel_sino(views, 129, 0.5, R)
    img = F.fbp(0, views, (1, n, n), 1.0, 129, 1, 0.5, 1.0, sino)
    c = _radius_grid(n, 1.0)
    r = np.hypot(*np.meshgrid(c, c, indexing="ij"))
    assert abs(np.median(img[r < 0.8 * R]) - 1.0) < 0.01
    assert np.abs(img[r < 0.8 * R] - 1.0).max() < 0.05
    fov = 0.95 * 64 * 0.5 / 2 * 2           # inside the detector's half-width (32)
    assert np.abs(img[(r > 1.25 * R) & (r < fov)]).max() < 0.05


def test_fan_fbp_of_a_disk():
    n, R, sid, sdd = 64, 20.0, 160.0, 256.0
    views = W.circular_fan_2d(240, sid, sdd)
    n_u, du = 161, 0.8
    sino = np.zeros((240, n_u))
    uu = (np.arange(n_u) - (n_u - 1) / 2.0) * du
    for k in range(240):
        src = np.r_[views[k, 0:2], 0.0]
        pix = np.r_[views[k, 2:4], 0.0][None, :] + uu[:, None] * np.r_[views[k, 4:6], 0.0][None, :]
        sino[k] = _chord_ball(src[None, :], pix, R)      # a disk is the ball's z = 0 section
    img = F.fbp(1, views, (1, n, n), 1.0, n_u, 1, du, 1.0, sino)
    c = _radius_grid(n, 1.0)
    r = np.hypot(*np.meshgrid(c, c, indexing="ij"))
    assert abs(np.median(img[r < 0.8 * R]) - 1.0) < 0.01
    assert np.abs(img[r < 0.8 * R] - 1.0).max() < 0.05
    fov = 0.95 * (n_u - 1) / 2 * du * sid / sdd    # radius seen by every view
    assert np.abs(img[(r > 1.25 * R) & (r < fov)]).max() < 0.05


def test_cone_fdk_of_a_ball():
    n, R, sid, sdd = 40, 12.0, 120.0, 200.0
    views = W.circular_cone(120, sid, sdd)
    n_u, n_v, du = 97, 81, 0.8
    uu = (np.arange(n_u) - (n_u - 1) / 2.0) * du
    vv = (np.arange(n_v) - (n_v - 1) / 2.0) * du
    sino = np.zeros((120, n_u, n_v))
    for k in range(120):
        src, ctr, u, v = views[k, 0:3], views[k, 3:6], views[k, 6:9], views[k, 9:12]
        pix = ctr + uu[:, None, None] * u + vv[None, :, None] * v
        sino[k] = _chord_ball(src[None, None, :], pix, R)
    vol = F.fbp(2, views, (n, n, n), 1.0, n_u, n_v, du, du, sino, window="hann")
    c = _radius_grid(n, 1.0)
    Z, Y, X = np.meshgrid(c, c, c, indexing="ij")
    r = np.sqrt(X * X + Y * Y + Z * Z)
    central = np.abs(Z) < 1.0
    assert abs(np.median(vol[central & (r < 0.7 * R)]) - 1.0) < 0.02
    assert abs(np.median(vol[r < 0.7 * R]) - 1.0) < 0.03
    fov = 0.95 * (n_u - 1) / 2 * du * sid / sdd
    rxy = np.sqrt(X * X + Y * Y)
    assert np.abs(vol[(r > 1.4 * R) & (rxy < fov) & central]).max() < 0.1


def _fan_disk_sino(views, n_u, du, R, centre):
    sino = np.zeros((views.shape[0], n_u))
    uu = (np.arange(n_u) - (n_u - 1) / 2.0) * du
    c3 = np.r_[centre, 0.0]
    for k in range(views.shape[0]):
        src = np.r_[views[k, 0:2], 0.0] - c3
        pix = (np.r_[views[k, 2:4], 0.0] - c3)[None, :] + uu[:, None] * np.r_[views[k, 4:6], 0.0]
        sino[k] = _chord_ball(src[None, :], pix, R)
    return sino


def test_fan_fbp_with_anisotropic_pixels_and_a_shifted_rotation_centre():
    """A scanner rotating about c0 != 0 reconstructs a disk centred at c0 once the isocentre is
    passed; pixels of (dy, dx) = (0.9, 0.7) place the voxel centres per axis."""
    ny, nx, R, sid, sdd = 48, 64, 14.0, 160.0, 256.0
    c0 = np.array([3.0, -2.0])
    views = W.circular_fan_2d(240, sid, sdd)
    views[:, 0:2] += c0
    views[:, 2:4] += c0
    n_u, du = 161, 0.8
    sino = _fan_disk_sino(views, n_u, du, R, c0)
    img = F.fbp(1, views, (1, ny, nx), (0.9, 0.7), n_u, 1, du, 1.0, sino, isocenter=c0)
    ys = (np.arange(ny) + 0.5 - ny / 2.0) * 0.9
    xs = (np.arange(nx) + 0.5 - nx / 2.0) * 0.7
    Y, X = np.meshgrid(ys, xs, indexing="ij")
    r = np.hypot(X - c0[0], Y - c0[1])
    assert abs(np.median(img[r < 0.8 * R]) - 1.0) < 0.01
    assert np.abs(img[r < 0.8 * R] - 1.0).max() < 0.05
    assert np.abs(img[(r > 1.3 * R) & (r < 19.0)]).max() < 0.05


def test_voxel_subset_equals_the_grid():
    w = W.small_config(3)
    sino = np.random.default_rng(3).uniform(-1, 1, size=w.sino_shape)
    full = F.fbp(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv, sino)
    idx = np.array([[0, 0, 0], [3, 5, 7], [w.vol_shape[0] - 1, w.vol_shape[1] - 1, 2]])
    sub = F.fbp(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv, sino,
                voxels=idx)
    np.testing.assert_allclose(sub, full[idx[:, 0], idx[:, 1], idx[:, 2]], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n", [1, 2, 3])
def test_transpose_satisfies_the_adjoint_identity(n):
    """<F y, x> = <y, F^T x> for random y, x: pins fbp_transpose to fbp (already pinned by the
    reconstructions above) in every stage (scatter coefficients, weights, filter, cosines)."""
    w = W.small_config(n)
    rng = np.random.default_rng(50 + n)
    y = rng.standard_normal(w.sino_shape)
    vol_shape = (w.vol_shape[1], w.vol_shape[2]) if w.beam in (0, 1) else w.vol_shape
    x = rng.standard_normal(vol_shape)
    kw = dict(window="hann", view_weights=rng.uniform(0.01, 0.1, w.views.shape[0]),
              isocenter=(0.7, -1.1, 0.4)[: 2 if w.beam in (0, 1) else 3])
    Fy = F.fbp(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv, y, **kw)
    Ftx = F.fbp_transpose(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du,
                          w.dv, x, **kw)
    lhs, rhs = float(np.sum(Fy * x)), float(np.sum(y * Ftx))
    assert abs(lhs - rhs) <= 1e-11 * np.linalg.norm(Fy) * np.linalg.norm(x), (lhs, rhs)


def test_isocenter_estimate_from_detector_normals():
    """Circular orbits about the origin give the origin; an orbit about c0 gives c0 (2D and 3D);
    a single view gives the point of its normal line nearest the origin (minimum norm)."""
    v2 = W.circular_fan_2d(90, 160.0, 256.0)
    np.testing.assert_allclose(F.estimate_isocenter(1, v2), 0.0, atol=1e-9)
    c0 = np.array([3.0, -2.0])
    s2 = v2.copy(); s2[:, 0:2] += c0; s2[:, 2:4] += c0
    np.testing.assert_allclose(F.estimate_isocenter(1, s2)[:2], c0, atol=1e-6)
    v3 = W.circular_cone(60, 120.0, 200.0)
    c3 = np.array([1.5, 2.0, -4.0])
    s3 = v3.copy(); s3[:, 0:3] += c3; s3[:, 3:6] += c3
    np.testing.assert_allclose(F.estimate_isocenter(2, s3), c3, atol=1e-6)
    one = v2[:1]                       # line through det_center (-96, 0) along x: nearest (0, 0)
    np.testing.assert_allclose(F.estimate_isocenter(1, one)[:2], [0.0, 0.0], atol=1e-6)
    one_off = one.copy(); one_off[0, 1] += 5.0; one_off[0, 3] += 5.0   # line y = 5
    np.testing.assert_allclose(F.estimate_isocenter(1, one_off)[:2], [0.0, 5.0], atol=1e-6)


def test_fan_fbp_about_a_shifted_centre_with_the_estimated_isocentre():
    """The shifted-orbit disk reconstructs without passing the isocentre."""
    n, R, sid, sdd = 64, 14.0, 160.0, 256.0
    c0 = np.array([3.0, -2.0])
    views = W.circular_fan_2d(240, sid, sdd)
    views[:, 0:2] += c0
    views[:, 2:4] += c0
    n_u, du = 161, 0.8
    sino = _fan_disk_sino(views, n_u, du, R, c0)
    img = F.fbp(1, views, (1, n, n), 1.0, n_u, 1, du, 1.0, sino)
    c = _radius_grid(n, 1.0)
    Y, X = np.meshgrid(c, c, indexing="ij")
    r = np.hypot(X - c0[0], Y - c0[1])
    assert abs(np.median(img[r < 0.8 * R]) - 1.0) < 0.01


# ---- Parker short-scan weights ----------------------------------------------------------------

def test_parker_formula_weights_of_conjugate_rays_sum_to_one():
    """A ray (beta, gamma) and its conjugate (beta + pi + 2 gamma, -gamma) (or beta - pi + 2 gamma)
    carry weights summing to 1; rays without a conjugate in the scan weigh 1."""
    rng = np.random.default_rng(1)
    delta = 0.3
    beta = rng.uniform(0, np.pi + 2 * delta, 20000)
    gamma = rng.uniform(-delta, delta, 20000)
    w = F.parker_formula(beta, gamma, delta)
    fwd = beta + np.pi + 2 * gamma
    back = beta - np.pi + 2 * gamma
    conj = np.where(fwd <= np.pi + 2 * delta, fwd, back)
    has = (fwd <= np.pi + 2 * delta) | (back >= 0)
    wc = F.parker_formula(conj, -gamma, delta)
    np.testing.assert_allclose((w + wc)[has], 1.0, atol=1e-12)
    np.testing.assert_allclose(w[~has], 1.0, atol=0)
    assert w.min() >= 0 and w.max() <= 1


def _fan_short_scan(n_views, sid, sdd, n_u, du, margin=0.02):
    """A circular fan scan over pi + 2 delta (+ margin), delta the detector's half fan angle."""
    half = (n_u - 1) / 2.0 * du
    delta = np.arctan(half / sdd)
    span = np.pi + 2 * delta + margin
    views = W.circular_fan_2d(n_views, sid, sdd, span=span * n_views / (n_views - 1))
    return views, delta


def test_parker_geometry_matches_the_geometric_conjugate_ray():
    """beta and gamma taken from the records obey the conjugate relation of the actual lines:
    the second intersection of a ray's line with the source circle sits at beta + pi + 2 gamma,
    and the ray back from there has fan angle -gamma.  This pins the signs of beta and gamma."""
    views, _ = _fan_short_scan(360, 160.0, 256.0, 129, 0.8)
    beta, gamma, delta, span = F.parker_geometry(1, views, 129, 0.8)
    R = 160.0
    th0 = np.arctan2(views[0, 1], views[0, 0])
    for k, j in [(3, 10), (100, 64), (200, 120), (350, 5)]:
        s = views[k, 0:2]
        c, u = views[k, 2:4], views[k, 4:6]
        P = c + (j - 64) * 0.8 * u
        d = (P - s) / np.linalg.norm(P - s)
        t = -2 * (s @ d)                       # |s + t d| = R, other root than t = 0
        s2 = s + t * d
        assert abs(np.linalg.norm(s2) - R) < 1e-9
        b2 = (np.arctan2(s2[1], s2[0]) - th0) % (2 * np.pi)
        want = (beta[k] + np.pi + 2 * gamma[k, j]) % (2 * np.pi)
        assert abs(np.angle(np.exp(1j * (b2 - want)))) < 1e-9
        a2, d2 = -s2, s - s2                   # back along the line from s2: central ray vs ray
        g2 = np.arctan2(a2[0] * d2[1] - a2[1] * d2[0], a2 @ d2)
        assert abs(g2 + gamma[k, j]) < 1e-9
    assert delta < span - np.pi


def test_short_scan_fan_fbp_of_a_disk_with_parker_weights():
    n, R, sid, sdd, n_u, du = 64, 20.0, 160.0, 256.0, 161, 0.8
    views, _ = _fan_short_scan(240, sid, sdd, n_u, du)
    beta, _, _, span = F.parker_geometry(1, views, n_u, du)
    pw = F.parker_weights(1, views, n_u, du)
    sino = np.zeros((views.shape[0], n_u))
    uu = (np.arange(n_u) - (n_u - 1) / 2.0) * du
    for k in range(views.shape[0]):
        src = np.r_[views[k, 0:2], 0.0]
        pix = np.r_[views[k, 2:4], 0.0][None, :] + uu[:, None] * np.r_[views[k, 4:6], 0.0][None, :]
        sino[k] = _chord_ball(src[None, :], pix, R)
    dbeta = span / (views.shape[0] - 1)
    img = F.fbp(1, views, (1, n, n), 1.0, n_u, 1, du, 1.0, sino,
                view_weights=np.full(views.shape[0], dbeta), pixel_weights=pw)
    c = _radius_grid(n, 1.0)
    r = np.hypot(*np.meshgrid(c, c, indexing="ij"))
    assert abs(np.median(img[r < 0.8 * R]) - 1.0) < 0.01
    assert np.abs(img[r < 0.8 * R] - 1.0).max() < 0.05
    fov = 0.95 * (n_u - 1) / 2 * du * sid / sdd
    assert np.abs(img[(r > 1.25 * R) & (r < fov)]).max() < 0.05
    # without the Parker weights the doubly measured wedge shows
    bad = F.fbp(1, views, (1, n, n), 1.0, n_u, 1, du, 1.0, sino,
                view_weights=np.full(views.shape[0], dbeta))
    assert np.abs(bad[r < 0.8 * R] - 1.0).max() > 0.2


def test_parker_rejects_short_and_non_circular_scans():
    views, delta = _fan_short_scan(100, 160.0, 256.0, 161, 0.8, margin=-0.2)
    with pytest.raises(ValueError):
        F.parker_weights(1, views, 161, 0.8)
    bad = W.circular_fan_2d(100, 160.0, 256.0)
    bad[7, 0:2] *= 1.01
    with pytest.raises(ValueError):
        F.parker_weights(1, bad, 161, 0.8)


# ---- caller filter kernels and gradients ---------------------------------------------------------

def test_default_kernel_is_the_scaled_window_taps():
    w = W.small_config(2)
    y = W.random_sinogram(w, 1).astype(np.float64)
    a = F.fbp(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv, y,
              window="cosine")
    k = w.du * F.ramp_taps(w.n_u, w.du, "cosine")
    b = F.fbp(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv, y,
              kernel=k)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12 * np.abs(a).max())


@pytest.mark.parametrize("n", [1, 2, 3])
def test_transpose_with_an_asymmetric_kernel_satisfies_the_adjoint_identity(n):
    w = W.small_config(n)
    rng = np.random.default_rng(70 + n)
    y = rng.standard_normal(w.sino_shape)
    vol_shape = (w.vol_shape[1], w.vol_shape[2]) if w.beam in (0, 1) else w.vol_shape
    x = rng.standard_normal(vol_shape)
    kern = rng.standard_normal(2 * w.n_u - 1)
    Fy = F.fbp(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv, y,
               kernel=kern)
    Ftx = F.fbp_transpose(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du,
                          w.dv, x, kernel=kern)
    lhs, rhs = float(np.sum(Fy * x)), float(np.sum(y * Ftx))
    assert abs(lhs - rhs) <= 1e-11 * np.linalg.norm(Fy) * np.linalg.norm(x)


@pytest.mark.parametrize("n", [1, 2, 3])
def test_gradients_equal_linear_probes(n):
    """f is linear in the kernel and in the view weights, so dL/dkernel[t] = <grad, f(kernel=e_t)>
    and dL/dw_k = <grad, f(view_weights=e_k)> exactly; checked on sampled t and k with pixel
    weights and an isocentre in play."""
    w = W.small_config(n)
    rng = np.random.default_rng(80 + n)
    y = W.random_sinogram(w, 2).astype(np.float64)
    vol_shape = (w.vol_shape[1], w.vol_shape[2]) if w.beam in (0, 1) else w.vol_shape
    grad = rng.standard_normal(vol_shape)
    nviews = w.views.shape[0]
    wts = rng.uniform(0.01, 0.05, nviews)
    pw = rng.uniform(0.5, 1.5, (nviews, w.n_u))
    iso = (0.4, -0.3, 0.2)[: 2 if w.beam in (0, 1) else 3]
    kern = F.filter_kernel(w.n_u, w.du, "hamming")
    kw = dict(view_weights=wts, isocenter=iso, pixel_weights=pw)
    gk, gw = F.fbp_gradients(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du,
                             w.dv, y, grad, kernel=kern, **kw)
    args = (w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv, y)
    for t in (0, w.n_u - 1, w.n_u + 2, 2 * w.n_u - 2):
        e = np.zeros_like(kern); e[t] = 1.0
        want = float(np.sum(F.fbp(*args, kernel=e, **kw) * grad))
        assert abs(gk[t] - want) <= 1e-10 * (abs(want) + np.abs(gk).max())
    for k in (0, nviews // 2, nviews - 1):
        e = np.zeros(nviews); e[k] = 1.0
        want = float(np.sum(F.fbp(*args, kernel=kern, view_weights=e, isocenter=iso,
                                  pixel_weights=pw) * grad))
        assert abs(gw[k] - want) <= 1e-10 * (abs(want) + np.abs(gw).max())
