"""Float64 reference of filtered backprojection (parallel FBP, fan FBP, cone FDK).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Plain numpy; it shares nothing with the
CUDA path.  The pages (diffct "Differentiable analytical reconstruction" and the parallel/fan/
cone FBP example pages) name the stages -- detector cosine weights, a ramp filter along the
detector u axis with physical sample spacing and an optional window (ram-lak, shepp-logan,
cosine, hamming, hann), angular integration weights, and a voxel-driven distance-weighted gather
-- without printing formulas.  This module writes out the textbook forms:

* cosine weight of pixel p (fan/cone):  |(c - s) . n| / |p - s|, n the detector normal;
* filter: Q(u_i) = tau * sum_j h((i - j) tau) p(u_j), with h the band-limited ramp
  h(x) = 2 * int_0^{1/(2 tau)} f W(f) cos(2 pi f x) df, tau = du, evaluated here by adaptive
  quadrature (scipy.integrate.quad) -- not by closed forms;
* view weight w_k (default pi / n_views: a uniformly sampled full scan, i.e. pi for parallel
  beams over 180 degrees, and 2 pi with the 1/2 redundancy factor for fan/cone over 360);
* isocentre (fan/cone): the caller's point, else estimated from the detector normals (the pages'
  default) as the least-squares point nearest the lines {c_k + s n_k}, with a 1e-9 ridge so that
  rank-deficient sets (one view, parallel normals) give the minimum-norm point;
* optional per (view, detector column) weights before filtering, e.g. Parker's short-scan
  weights (Parker 1982) for circular fan/cone orbits spanning pi + 2 delta;
* optional caller filter kernel replacing the windowed ramp (a learned filter), and the
  gradients of a loss with respect to that kernel and to the view weights (`fbp_gradients`);
* gather: f(X) = sum_k w_k g_k(X) Q_k(u_k(X), v_k(X)) with bilinear interpolation (0 outside the
  detector), g = 1 for parallel beams and, for fan/cone, g = (D_sd / D_so) / U(X)^2 with
  U(X) = ((X - s) . n) / ((iso - s) . n), D_so = |(iso - s) . n|, D_sd = |(c - s) . n|
  (Feldkamp's distance weight for a detector at distance D_sd; the D_sd / D_so factor converts a
  filter applied in physical detector units to the isocentre plane).
"""
from __future__ import annotations

import math

import numpy as np

WINDOWS = ("ram-lak", "shepp-logan", "cosine", "hamming", "hann")


def window_response(name: str, f: np.ndarray, tau: float) -> np.ndarray:
    """W(f) on [0, 1/(2 tau)] for the named window (frequency in cycles per unit length)."""
    x = f * tau  # in [0, 1/2]
    if name == "ram-lak":
        return np.ones_like(f)
    if name == "shepp-logan":
        return np.sinc(x)                     # sin(pi x) / (pi x)
    if name == "cosine":
        return np.cos(np.pi * x)
    if name == "hamming":
        return 0.54 + 0.46 * np.cos(2 * np.pi * x)
    if name == "hann":
        return 0.5 + 0.5 * np.cos(2 * np.pi * x)
    raise ValueError(name)


def ramp_taps(n_u: int, tau: float, window: str) -> np.ndarray:
    """h(n tau) for n = -(n_u - 1) .. n_u - 1, by quadrature of the band-limited windowed ramp."""
    from scipy.integrate import quad
    F = 0.5 / tau

    def g(f):
        return f * window_response(window, np.array([f]), tau)[0]

    taps = np.zeros(2 * n_u - 1)
    for n in range(n_u):
        x = n * tau
        if n == 0:
            val, _ = quad(g, 0.0, F, limit=400, epsabs=1e-14, epsrel=1e-12)
        else:  # the cos(2 pi f x) factor as the rule's oscillatory weight (QAWO)
            val, _ = quad(g, 0.0, F, weight="cos", wvar=2 * math.pi * x, limit=400,
                          epsabs=1e-14)
        taps[n_u - 1 + n] = taps[n_u - 1 - n] = 2.0 * val
    return taps


def estimate_isocenter(beam: int, views: np.ndarray) -> np.ndarray:
    """Least-squares point nearest the lines through each detector centre along its normal:
    (sum_k P_k + eps I) x = sum_k P_k c_k with P_k = I - n_k n_k^T (unit n_k) and
    eps = 1e-9 * trace(sum_k P_k) / dim; 2D geometries solve in the plane (z = 0)."""
    dim = 2 if beam in (0, 1) else 3
    M = np.zeros((dim, dim))
    b = np.zeros(dim)
    for rec in views:
        _, ctr, _, _, n = _frames(beam, rec)
        n = n[:dim] / np.linalg.norm(n[:dim])
        P = np.eye(dim) - np.outer(n, n)
        M += P
        b += P @ ctr[:dim]
    M += 1e-9 * np.trace(M) / dim * np.eye(dim)
    x = np.linalg.solve(M, b)
    return np.r_[x, [0.0] * (3 - dim)]


def parker_formula(beta, gamma, delta):
    """Parker's short-scan weight for source angle beta in [0, pi + 2 delta] and fan angle gamma
    (same rotational sense as beta), half fan angle delta; 0 outside the scan."""
    beta, gamma = np.broadcast_arrays(np.asarray(beta, float), np.asarray(gamma, float))
    w = np.zeros(beta.shape)
    a = delta - gamma
    b = delta + gamma
    r1 = (beta >= 0) & (beta < 2 * a)
    r2 = (beta >= 2 * a) & (beta <= np.pi - 2 * gamma)
    r3 = (beta > np.pi - 2 * gamma) & (beta <= np.pi + 2 * delta)
    w[r1] = np.sin(np.pi / 4 * beta[r1] / a[r1]) ** 2
    w[r2] = 1.0
    w[r3] = np.sin(np.pi / 4 * (np.pi + 2 * delta - beta[r3]) / b[r3]) ** 2
    return w


def parker_geometry(beam: int, views: np.ndarray, n_u: int, du: float, isocenter=None):
    """(beta (n_views,), gamma (n_views, n_u), delta, span) of a circular fan or cone orbit in
    the xy-plane: beta the source angle about the isocentre from the first view, in the sense of
    rotation; gamma the fan angle of each detector column (the column's centre line) from the
    central ray (source to isocentre), in the same sense; delta the largest |gamma|; span the last
    view's beta.  Raises ValueError if the orbit is not a circle about the isocentre."""
    assert beam in (1, 2), "fan and cone beams"
    iso = (estimate_isocenter(beam, views) if isocenter is None else
           np.r_[np.asarray(isocenter, float), [0.0] * (3 - len(isocenter))])
    src = np.array([_frames(beam, r)[0] for r in views])
    rel = src[:, :2] - iso[:2]
    radius = np.hypot(rel[:, 0], rel[:, 1])
    if np.ptp(radius) > 1e-6 * radius.mean() or (beam == 2 and np.ptp(src[:, 2]) > 1e-6 * radius.mean()):
        raise ValueError("not a circular orbit in the xy-plane about the isocentre")
    beta = np.unwrap(np.arctan2(rel[:, 1], rel[:, 0]))
    sense = 1.0 if beta[-1] >= beta[0] else -1.0
    beta = (beta - beta[0]) * sense
    cu = (n_u - 1) / 2.0
    gamma = np.zeros((views.shape[0], n_u))
    for k, rec in enumerate(views):
        first, ctr, u, _, _ = _frames(beam, rec)
        a = (iso - first)[:2]
        P = ctr[None, :] + ((np.arange(n_u) - cu) * du)[:, None] * u[None, :]
        b = (P - first)[:, :2]
        gamma[k] = sense * np.arctan2(a[0] * b[:, 1] - a[1] * b[:, 0], b @ a)
    return beta, gamma, float(np.abs(gamma).max()), float(beta[-1])


def parker_weights(beam: int, views: np.ndarray, n_u: int, du: float, isocenter=None):
    """Per (view, column) Parker weights of a circular short scan (pages: short-scan Parker
    weighting before filtering).  With a span above pi + 2 delta the effective half fan angle is
    (span - pi) / 2, which keeps conjugate rays' weights summing to 1.  Raises ValueError if the
    span is shorter than pi + 2 delta."""
    beta, gamma, delta, span = parker_geometry(beam, views, n_u, du, isocenter)
    if span < np.pi + 2 * delta - 1e-9:
        raise ValueError("the scan spans less than pi + 2 delta")
    return parker_formula(beta[:, None], gamma, (span - np.pi) / 2)


def _frames(beam: int, rec: np.ndarray):
    if beam in (0, 1):
        first, ctr, u = np.r_[rec[0:2], 0.0], np.r_[rec[2:4], 0.0], np.r_[rec[4:6], 0.0]
        v = np.array([0.0, 0.0, 1.0])
        n = np.array([u[1], -u[0], 0.0])
    else:
        first, ctr, u, v = rec[0:3], rec[3:6], rec[6:9], rec[9:12]
        n = np.cross(u, v)
    return first, ctr, u, v, n


def filter_kernel(n_u: int, du: float, window: str = "ram-lak", kernel=None) -> np.ndarray:
    """The discrete filter applied along u: Q_i = sum_j kernel[i - j + n_u - 1] p_j.  Default:
    du * h((i - j) du), the band-limited windowed ramp; a caller's kernel (2 n_u - 1 values, e.g.
    a learned filter) replaces it."""
    if kernel is not None:
        k = np.asarray(kernel, dtype=np.float64).reshape(-1)
        assert k.size == 2 * n_u - 1
        return k
    return du * ramp_taps(n_u, du, window)


def fbp(beam: int, views: np.ndarray, vol_shape, spacing, n_u: int, n_v: int, du: float,
        dv: float, sino: np.ndarray, window: str = "ram-lak", view_weights=None, isocenter=None,
        voxels=None, pixel_weights=None, kernel=None):
    """Filtered backprojection of `sino` ((views, U) or (views, U, V)) onto the volume grid.

    `spacing` is one pitch or per-axis pitches in tensor order ((dz, dy, dx), 2D (dy, dx)); voxel
    centres sit at (i + 1/2 - n/2) * pitch on each axis.  With `voxels` (an (m, 3) array of
    (iz, iy, ix) indices) only those voxels are reconstructed and an (m,) array is returned."""
    assert beam in (0, 1, 2), "parallel (2D), fan (2D) and cone beams"
    two_d = beam in (0, 1)
    nz, ny, nx = vol_shape
    n_views = views.shape[0]
    p = np.asarray(sino, dtype=np.float64).reshape(n_views, n_u, 1 if two_d else n_v)
    V = p.shape[2]
    w = (np.full(n_views, math.pi / n_views) if view_weights is None
         else np.asarray(view_weights, dtype=np.float64))
    iso = (estimate_isocenter(beam, views) if isocenter is None else
           np.r_[np.asarray(isocenter, float), [0.0] * (3 - len(isocenter))])
    cu, cv = (n_u - 1) / 2.0, (V - 1) / 2.0
    uu = (np.arange(n_u) - cu) * du
    vv = (np.arange(V) - cv) * dv if not two_d else np.zeros(1)
    kern = filter_kernel(n_u, du, window, kernel)
    sp = np.broadcast_to(np.asarray(spacing, dtype=np.float64), (2 if two_d else 3,))
    sz, sy, sx = (1.0, sp[0], sp[1]) if two_d else (sp[0], sp[1], sp[2])
    # voxel centres
    zs = (np.arange(nz) + 0.5 - nz / 2.0) * sz if not two_d else np.zeros(1)
    ys = (np.arange(ny) + 0.5 - ny / 2.0) * sy
    xs = (np.arange(nx) + 0.5 - nx / 2.0) * sx
    if voxels is None:
        Z, Y, X = np.meshgrid(zs, ys, xs, indexing="ij")
        P = np.stack([X, Y, Z], axis=-1)                           # (nz|1, ny, nx, 3)
    else:
        vi = np.asarray(voxels, dtype=np.int64).reshape(-1, 3)
        P = np.stack([xs[vi[:, 2]], ys[vi[:, 1]], zs[vi[:, 0]]], axis=-1)[None, None]  # (1,1,m,3)
    out = np.zeros(P.shape[:3])
    for k in range(n_views):
        first, ctr, u, v, n = _frames(beam, views[k])
        q = p[k].copy()
        if beam != 0:                                              # cosine pre-weights
            pix = ctr[None, None, :] + uu[:, None, None] * u + vv[None, :, None] * v
            q *= abs((ctr - first) @ n) / np.linalg.norm(pix - first, axis=-1)
        if pixel_weights is not None:                              # e.g. Parker weights
            q *= np.asarray(pixel_weights, dtype=np.float64)[k][:, None]
        # filter every detector column along u (linear convolution, no wrap-around)
        Q = np.empty_like(q)
        for j in range(V):
            Q[:, j] = np.convolve(q[:, j], kern, mode="full")[n_u - 1:2 * n_u - 1]
        # gather
        if beam == 0:
            upix = ((P - ctr) @ u) / du + cu
            vpix = np.zeros_like(upix)
            g = np.ones_like(upix)
        else:
            a = P - first
            den = a @ n
            D = (ctr - first) @ n
            upix = ((first - ctr) @ u + D * (a @ u) / den) / du + cu
            vpix = (((first - ctr) @ v + D * (a @ v) / den) / dv + cv) if not two_d else np.zeros_like(upix)
            Uw = den / ((iso - first) @ n)
            g = (abs(D) / abs((iso - first) @ n)) / (Uw * Uw)
        out += w[k] * g * _bilinear(Q, upix, vpix)
    if voxels is not None:
        return out[0, 0]
    return out[0] if two_d else out


def _bilinear(Q: np.ndarray, up: np.ndarray, vp: np.ndarray) -> np.ndarray:
    """Bilinear interpolation of Q[u, v] at fractional pixel indices, 0 outside the grid."""
    nU, nV = Q.shape
    u0 = np.floor(up).astype(np.int64)
    v0 = np.floor(vp).astype(np.int64)
    fu, fv = up - u0, vp - v0
    res = np.zeros(up.shape)
    for du_, wu in ((0, 1 - fu), (1, fu)):
        for dv_, wv in ((0, 1 - fv), (1, fv)):
            iu, iv = u0 + du_, v0 + dv_
            ok = (iu >= 0) & (iu < nU) & (iv >= 0) & (iv < nV)
            vals = np.zeros(up.shape)
            vals[ok] = Q[iu[ok], iv[ok]]
            res += wu * wv * vals
    return res


def fbp_transpose(beam: int, views: np.ndarray, vol_shape, spacing, n_u: int, n_v: int,
                  du: float, dv: float, vol: np.ndarray, window: str = "ram-lak",
                  view_weights=None, isocenter=None, pixel_weights=None, kernel=None):
    """The transpose of `fbp` as a linear map from sinograms to volumes: volume -> sinogram.

    The pages state that the analytical operator's backward pass scatters the same interpolation
    coefficients, distance weights and normalisation (diffct "Differentiable analytical
    reconstruction"; "Analytical Reconstruction Helpers": dedicated transpose kernels).  Written
    as the transposes of the three stages in reverse order: the gather's bilinear coefficients
    times w_k g_k(X) scattered onto each view's detector, the filter (its matrix
    tau h((i - j) tau) is symmetric because h is even), then the cosine weights (diagonal).
    """
    assert beam in (0, 1, 2), "parallel (2D), fan (2D) and cone beams"
    two_d = beam in (0, 1)
    nz, ny, nx = vol_shape
    n_views = views.shape[0]
    V = 1 if two_d else n_v
    f = np.asarray(vol, dtype=np.float64).reshape(1 if two_d else nz, ny, nx)
    w = (np.full(n_views, math.pi / n_views) if view_weights is None
         else np.asarray(view_weights, dtype=np.float64))
    iso = (estimate_isocenter(beam, views) if isocenter is None else
           np.r_[np.asarray(isocenter, float), [0.0] * (3 - len(isocenter))])
    cu, cv = (n_u - 1) / 2.0, (V - 1) / 2.0
    uu = (np.arange(n_u) - cu) * du
    vv = (np.arange(V) - cv) * dv if not two_d else np.zeros(1)
    kern = filter_kernel(n_u, du, window, kernel)
    sp = np.broadcast_to(np.asarray(spacing, dtype=np.float64), (2 if two_d else 3,))
    sz, sy, sx = (1.0, sp[0], sp[1]) if two_d else (sp[0], sp[1], sp[2])
    zs = (np.arange(nz) + 0.5 - nz / 2.0) * sz if not two_d else np.zeros(1)
    ys = (np.arange(ny) + 0.5 - ny / 2.0) * sy
    xs = (np.arange(nx) + 0.5 - nx / 2.0) * sx
    Z, Y, X = np.meshgrid(zs, ys, xs, indexing="ij")
    P = np.stack([X, Y, Z], axis=-1)
    out = np.zeros((n_views, n_u, V))
    for k in range(n_views):
        first, ctr, u, v, n = _frames(beam, views[k])
        if beam == 0:
            upix = ((P - ctr) @ u) / du + cu
            vpix = np.zeros_like(upix)
            g = np.ones_like(upix)
        else:
            a = P - first
            den = a @ n
            D = (ctr - first) @ n
            upix = ((first - ctr) @ u + D * (a @ u) / den) / du + cu
            vpix = (((first - ctr) @ v + D * (a @ v) / den) / dv + cv) if not two_d else np.zeros_like(upix)
            Uw = den / ((iso - first) @ n)
            g = (abs(D) / abs((iso - first) @ n)) / (Uw * Uw)
        # transpose of the gather: scatter w g f with the bilinear coefficients
        Q = _bilinear_transpose(w[k] * g * f, upix, vpix, n_u, V)
        # transpose of the filter (the kernel reversed; the windowed ramps are symmetric), then of
        # the cosine weights
        q = np.empty_like(Q)
        for j in range(V):
            q[:, j] = np.convolve(Q[:, j], kern[::-1], mode="full")[n_u - 1:2 * n_u - 1]
        if beam != 0:
            pix = ctr[None, None, :] + uu[:, None, None] * u + vv[None, :, None] * v
            q *= abs((ctr - first) @ n) / np.linalg.norm(pix - first, axis=-1)
        if pixel_weights is not None:
            q *= np.asarray(pixel_weights, dtype=np.float64)[k][:, None]
        out[k] = q
    return out[:, :, 0] if two_d else out


def _bilinear_transpose(vals: np.ndarray, up: np.ndarray, vp: np.ndarray, nU: int, nV: int):
    """Adds vals at fractional pixel indices into an (nU, nV) grid with the bilinear
    coefficients of `_bilinear` (contributions off the grid are dropped)."""
    u0 = np.floor(up).astype(np.int64)
    v0 = np.floor(vp).astype(np.int64)
    fu, fv = up - u0, vp - v0
    res = np.zeros((nU, nV))
    for du_, wu in ((0, 1 - fu), (1, fu)):
        for dv_, wv in ((0, 1 - fv), (1, fv)):
            iu, iv = u0 + du_, v0 + dv_
            ok = (iu >= 0) & (iu < nU) & (iv >= 0) & (iv < nV)
            np.add.at(res, (iu[ok], iv[ok]), (wu * wv * vals)[ok])
    return res


def fbp_gradients(beam: int, views: np.ndarray, vol_shape, spacing, n_u: int, n_v: int,
                  du: float, dv: float, sino: np.ndarray, grad_vol: np.ndarray,
                  window: str = "ram-lak", view_weights=None, isocenter=None,
                  pixel_weights=None, kernel=None):
    """Gradients of L(f) with f = fbp(sino, ...) with respect to the filter kernel and the view
    weights, given dL/df = grad_vol (the pages: filter and explicit weight gradients propagate
    through the analytical pipeline).  f is linear in both: with q_k the pre-weighted sinogram,
    Q_k = H q_k the filtered one and G_k the view's gather without its weight,
    dL/dw_k = <G_k^T grad, Q_k> and dL/dkernel[d + n_u - 1] = sum_k w_k sum_i (G_k^T grad)_i
    q_k[i - d].  Returns (grad_kernel (2 n_u - 1,), grad_view_weights (n_views,))."""
    assert beam in (0, 1, 2)
    two_d = beam in (0, 1)
    n_views = views.shape[0]
    V = 1 if two_d else n_v
    w = (np.full(n_views, math.pi / n_views) if view_weights is None
         else np.asarray(view_weights, dtype=np.float64))
    ones = np.ones(n_views)
    # G_k^T grad for every view (unit view weights) through the transpose with an identity filter
    # and no cosine or pixel weights
    ident = np.zeros(2 * n_u - 1)
    ident[n_u - 1] = 1.0
    gq = np.asarray(fbp_transpose(beam, views, vol_shape, spacing, n_u, n_v, du, dv, grad_vol,
                                  view_weights=ones, isocenter=isocenter, kernel=ident,
                                  pixel_weights=None), dtype=np.float64)
    gq = gq.reshape(n_views, n_u, V)
    if beam != 0:  # undo the cosine weights the transpose applied
        for k in range(n_views):
            first, ctr, u, v, n = _frames(beam, views[k])
            cu, cv = (n_u - 1) / 2.0, (V - 1) / 2.0
            uu = (np.arange(n_u) - cu) * du
            vv = (np.arange(V) - cv) * dv if not two_d else np.zeros(1)
            pix = ctr[None, None, :] + uu[:, None, None] * u + vv[None, :, None] * v
            gq[k] /= abs((ctr - first) @ n) / np.linalg.norm(pix - first, axis=-1)
    kern = filter_kernel(n_u, du, window, kernel)
    p = np.asarray(sino, dtype=np.float64).reshape(n_views, n_u, V)
    g_kern = np.zeros(2 * n_u - 1)
    g_w = np.zeros(n_views)
    for k in range(n_views):
        first, ctr, u, v, n = _frames(beam, views[k])
        q = p[k].copy()
        if beam != 0:
            cu, cv = (n_u - 1) / 2.0, (V - 1) / 2.0
            uu = (np.arange(n_u) - cu) * du
            vv = (np.arange(V) - cv) * dv if not two_d else np.zeros(1)
            pix = ctr[None, None, :] + uu[:, None, None] * u + vv[None, :, None] * v
            q *= abs((ctr - first) @ n) / np.linalg.norm(pix - first, axis=-1)
        if pixel_weights is not None:
            q *= np.asarray(pixel_weights, dtype=np.float64)[k][:, None]
        for j in range(V):
            Qj = np.convolve(q[:, j], kern, mode="full")[n_u - 1:2 * n_u - 1]
            g_w[k] += gq[k][:, j] @ Qj
            # sum_i gq_i q_{i-d} for d = -(n_u-1) .. n_u-1
            g_kern += w[k] * np.correlate(gq[k][:, j], q[:, j], mode="full")
    return g_kern, g_w
