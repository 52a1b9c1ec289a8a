"""Seeded synthetic inputs: acquisition geometries (per-view vector records) and phantoms.

This module only *generates inputs*.  It holds none of the projector's arithmetic (no ray
set-up, clipping or traversal), so it is the one module that both the CUDA library's tests and
the float64 oracle's tests may share.

Geometry records follow the per-view trajectory layout of the diffct documentation
("Trajectories and Geometry", *Trajectory format* table): one row per view,

* 3D (cone, parallel3d): ``[e(3), det_center(3), det_u(3), det_v(3)]`` (12 doubles), where ``e`` is
  ``src_pos`` for cone beams and ``ray_dir`` for parallel3d,
* 2D (parallel, fan): ``[e(2), det_center(2), det_u(2)]`` (6 doubles), where ``e`` is ``ray_dir``
  for parallel beams (the page calls its detector point ``det_origin``) and ``src_pos`` for fan.

Coordinates are Cartesian ``(x, y[, z])`` with the origin at the volume centre; volumes are
indexed ``[z, y, x]`` (2D: ``[y, x]``) and sinograms ``[view, u, v]`` (2D: ``[view, u]``).

The circular/spiral generator formulas are not printed on the pages (only their names and
signatures, e.g. ``spiral_trajectory_3d(n, sid, sdd, z_range, n_turns)``); the formulas below are
the plain reading: source on a circle of radius ``sid``, detector centre diametrically opposite
at distance ``sdd - sid`` from the origin, ``det_u`` tangential and ``det_v`` along +z.
The dual-axis tilt vectors follow the ``parallel3d_vec`` construction printed on the ASTRA
HAADF-STEM article (section 2, dual-axis geometry code).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable

import numpy as np

# Beam identifiers.  They equal the values of the C enum ``ct_beam`` so that a record array and
# its beam id can be passed unchanged to either side.
PARALLEL2D = 0
FAN2D = 1
CONE = 2
PARALLEL3D = 3
BEAM_NAMES = {PARALLEL2D: "parallel", FAN2D: "fan", CONE: "cone", PARALLEL3D: "parallel3d"}


def record_width(beam: int) -> int:
    """Doubles per view record: 6 for the 2D beams, 12 for the 3D beams."""
    return 6 if beam in (PARALLEL2D, FAN2D) else 12


@dataclasses.dataclass
class Workload:
    """One synthetic acquisition: geometry records, volume/detector sizes and a phantom recipe."""

    name: str
    beam: int
    views: np.ndarray            # (n_views, 6|12) float64, C-contiguous
    vol_shape: tuple             # (nz, ny, nx); 2D problems have nz == 1
    voxel_spacing: float | tuple # scalar, or per axis in tensor order: (dy, dx) / (dz, dy, dx)
    n_u: int
    n_v: int                     # 1 for 2D problems
    du: float
    dv: float
    seed: int
    phantom_fn: Callable[[], np.ndarray] | None = None
    offsets: np.ndarray | None = None  # (n_u, n_v, 3) local (u, v, n) pixel offsets, or flat

    @property
    def n_views(self) -> int:
        return int(self.views.shape[0])

    @property
    def is_2d(self) -> bool:
        return self.beam in (PARALLEL2D, FAN2D)

    @property
    def n_rays(self) -> int:
        return self.n_views * self.n_u * self.n_v

    @property
    def n_voxels(self) -> int:
        nz, ny, nx = self.vol_shape
        return nz * ny * nx

    @property
    def sino_shape(self) -> tuple:
        return (self.n_views, self.n_u) if self.is_2d else (self.n_views, self.n_u, self.n_v)

    @property
    def volume_shape(self) -> tuple:
        """Tensor shape of the volume: (ny, nx) for 2D, (nz, ny, nx) for 3D."""
        return self.vol_shape[1:] if self.is_2d else self.vol_shape

    def phantom(self) -> np.ndarray:
        assert self.phantom_fn is not None
        img = self.phantom_fn()
        assert img.dtype == np.float32 and img.shape == self.volume_shape
        return np.ascontiguousarray(img)

    def subset(self, view_ids) -> "Workload":
        """The same acquisition restricted to the given views (records copied, phantom shared)."""
        view_ids = np.asarray(view_ids, dtype=np.int64)
        return dataclasses.replace(self, name=f"{self.name}[{len(view_ids)} views]",
                                   views=np.ascontiguousarray(self.views[view_ids]))


# ----------------------------------------------------------------------------------------------
# Trajectories
# ----------------------------------------------------------------------------------------------

def circular_parallel_2d(n_views: int, span: float = math.pi) -> np.ndarray:
    """2D parallel beam: ``ray_dir = (cos t, sin t)``, ``det_u = (-sin t, cos t)``, origin 0."""
    th = np.arange(n_views, dtype=np.float64) * (span / n_views)
    c, s = np.cos(th), np.sin(th)
    z = np.zeros_like(th)
    return np.ascontiguousarray(np.stack([c, s, z, z, -s, c], axis=1))


def circular_fan_2d(n_views: int, sid: float, sdd: float, span: float = 2 * math.pi) -> np.ndarray:
    """2D fan beam on a circle: source at radius sid, detector centre opposite at sdd - sid."""
    th = np.arange(n_views, dtype=np.float64) * (span / n_views)
    c, s = np.cos(th), np.sin(th)
    r = sdd - sid
    return np.ascontiguousarray(np.stack([sid * c, sid * s, -r * c, -r * s, -s, c], axis=1))


def circular_cone(n_views: int, sid: float, sdd: float, span: float = 2 * math.pi) -> np.ndarray:
    """3D cone beam, circular orbit in the z = 0 plane, ``det_v = +z``."""
    th = np.arange(n_views, dtype=np.float64) * (span / n_views)
    c, s = np.cos(th), np.sin(th)
    z, o = np.zeros_like(th), np.ones_like(th)
    r = sdd - sid
    return np.ascontiguousarray(np.stack(
        [sid * c, sid * s, z, -r * c, -r * s, z, -s, c, z, z, z, o], axis=1))


def _rot(axis: np.ndarray, ang: float) -> np.ndarray:
    """Rodrigues rotation matrix about a unit axis (input generation only)."""
    a = axis / np.linalg.norm(axis)
    k = np.array([[0, -a[2], a[1]], [a[2], 0, -a[0]], [-a[1], a[0], 0]])
    return np.eye(3) + math.sin(ang) * k + (1 - math.cos(ang)) * (k @ k)


def spiral_cone(n_views: int, sid: float, sdd: float, z_range: float, n_turns: float,
                rng: np.random.Generator | None = None, src_jitter: float = 0.0,
                det_tilt_deg: float = 0.0) -> np.ndarray:
    """Helical cone trajectory with optional seeded per-view jitter.

    ``theta_k = 2 pi n_turns k / n``, ``z_k = -z_range/2 + z_range k / (n-1)``; source and detector
    centre share ``z_k``.  Jitter: the source moves by U[-j, j]^3; the detector frame (det_u, det_v)
    is rotated by three small angles U[-a, a] about u, v and n, then re-orthonormalised
    (Gram-Schmidt).
    """
    out = np.empty((n_views, 12), dtype=np.float64)
    r = sdd - sid
    for k in range(n_views):
        th = 2 * math.pi * n_turns * k / n_views
        zk = -z_range / 2 + z_range * k / max(n_views - 1, 1)
        c, s = math.cos(th), math.sin(th)
        src = np.array([sid * c, sid * s, zk])
        ctr = np.array([-r * c, -r * s, zk])
        u = np.array([-s, c, 0.0])
        v = np.array([0.0, 0.0, 1.0])
        if rng is not None:
            src = src + rng.uniform(-src_jitter, src_jitter, size=3)
            n = np.cross(u, v)
            ang = np.deg2rad(rng.uniform(-det_tilt_deg, det_tilt_deg, size=3))
            R = _rot(u, ang[0]) @ _rot(v, ang[1]) @ _rot(n, ang[2])
            u, v = R @ u, R @ v
            u = u / np.linalg.norm(u)
            v = v - (v @ u) * u
            v = v / np.linalg.norm(v)
        out[k] = np.concatenate([src, ctr, u, v])
    return np.ascontiguousarray(out)


def dual_axis_tilt(angles1_deg, angles2_deg) -> np.ndarray:
    """parallel3d dual-axis tilt series, vectors as printed on the ASTRA dual-axis article.

    Series 1: ray (sin a, 0, -cos a), det_u (cos a, 0, sin a), det_v (0, 1, 0).
    Series 2: ray (0, -sin a, -cos a), det_u (0, -cos a, sin a), det_v (1, 0, 0).
    Detector centre at the origin.
    """
    rows = []
    for a in np.deg2rad(np.asarray(angles1_deg, dtype=np.float64)):
        sa, ca = math.sin(a), math.cos(a)
        rows.append([sa, 0, -ca, 0, 0, 0, ca, 0, sa, 0, 1, 0])
    for a in np.deg2rad(np.asarray(angles2_deg, dtype=np.float64)):
        sa, ca = math.sin(a), math.cos(a)
        rows.append([0, -sa, -ca, 0, 0, 0, 0, -ca, sa, 1, 0, 0])
    return np.ascontiguousarray(np.array(rows, dtype=np.float64))


# ----------------------------------------------------------------------------------------------
# Phantoms (all float32; evaluated at voxel centres, coordinates in voxel units about the centre)
# ----------------------------------------------------------------------------------------------

def uniform_image(shape, rng: np.random.Generator) -> np.ndarray:
    """i.i.d. U[0, 1) values."""
    return rng.random(shape).astype(np.float32)


def _centres(n: int) -> np.ndarray:
    return np.arange(n, dtype=np.float64) + 0.5 - n / 2.0


def ellipses_2d(n_shapes: int, n: int, rng: np.random.Generator,
                axis_range=(5.0, 150.0), value_range=(-0.5, 1.0)) -> np.ndarray:
    """Sum of random filled ellipses on a zero background (n x n pixels)."""
    img = np.zeros((n, n), dtype=np.float64)
    ys, xs = _centres(n)[:, None], _centres(n)[None, :]
    for _ in range(n_shapes):
        cx, cy = rng.uniform(-0.4 * n, 0.4 * n, size=2)
        a, b = rng.uniform(*axis_range, size=2)
        phi = rng.uniform(0.0, math.pi)
        val = rng.uniform(*value_range)
        c, s = math.cos(phi), math.sin(phi)
        xr = (xs - cx) * c + (ys - cy) * s
        yr = -(xs - cx) * s + (ys - cy) * c
        img += val * ((xr / a) ** 2 + (yr / b) ** 2 <= 1.0)
    return img.astype(np.float32)


def _random_rotation(rng: np.random.Generator) -> np.ndarray:
    """Uniform random rotation from a normalised Gaussian quaternion."""
    q = rng.standard_normal(4)
    w, x, y, z = q / np.linalg.norm(q)
    return np.array([
        [1 - 2 * (y * y + z * z), 2 * (x * y - z * w), 2 * (x * z + y * w)],
        [2 * (x * y + z * w), 1 - 2 * (x * x + z * z), 2 * (y * z - x * w)],
        [2 * (x * z - y * w), 2 * (y * z + x * w), 1 - 2 * (x * x + y * y)]])


def ellipsoids_3d(n_shapes: int, n: int, rng: np.random.Generator,
                  axis_range=(8.0, 100.0), value_range=(0.0, 1.0)) -> np.ndarray:
    """Sum of random filled ellipsoids in an n^3 volume ([z, y, x] order).

    Each ellipsoid is drawn on its own axis-aligned bounding box, slab by slab, so that a 512^3
    phantom needs a few hundred MB of scratch at most.
    """
    vol = np.zeros((n, n, n), dtype=np.float32)
    cen = _centres(n)
    for _ in range(n_shapes):
        c = rng.uniform(-0.4 * n, 0.4 * n, size=3)          # (x, y, z)
        ax = rng.uniform(*axis_range, size=3)
        R = _random_rotation(rng)
        val = np.float32(rng.uniform(*value_range))
        # bounding half-extents of the rotated ellipsoid along x, y, z
        half = np.sqrt(((R * ax[None, :]) ** 2).sum(axis=1))
        lo = np.clip(np.floor(c - half + n / 2.0).astype(int), 0, n)
        hi = np.clip(np.ceil(c + half + n / 2.0).astype(int) + 1, 0, n)
        if np.any(hi <= lo):
            continue
        xs = (cen[lo[0]:hi[0]] - c[0])[None, None, :]
        ys = (cen[lo[1]:hi[1]] - c[1])[None, :, None]
        M = R / ax[None, :]            # local coordinate j = sum_i R[i, j] p_i / ax[j]
        for z0 in range(lo[2], hi[2], 32):
            z1 = min(z0 + 32, hi[2])
            zs = (cen[z0:z1] - c[2])[:, None, None]
            q = np.zeros((z1 - z0, hi[1] - lo[1], hi[0] - lo[0]), dtype=np.float64)
            for j in range(3):
                lj = M[0, j] * xs + M[1, j] * ys + M[2, j] * zs
                q += lj * lj
            vol[z0:z1, lo[1]:hi[1], lo[0]:hi[0]] += val * (q <= 1.0)
    return vol


def spheres_slab(n_spheres: int, n: int, rng: np.random.Generator, radius_range=(3.0, 20.0),
                 density_range=(0.5, 1.0), half_thickness: float = 64.0) -> np.ndarray:
    """Random spheres wholly inside the slab |z| <= half_thickness (voxels); overlaps take max."""
    vol = np.zeros((n, n, n), dtype=np.float32)
    cen = _centres(n)
    for _ in range(n_spheres):
        r = rng.uniform(*radius_range)
        cx, cy = rng.uniform(-n / 2 + r, n / 2 - r, size=2)
        cz = rng.uniform(-half_thickness + r, half_thickness - r)
        dens = np.float32(rng.uniform(*density_range))
        c = np.array([cx, cy, cz])
        lo = np.clip(np.floor(c - r + n / 2.0).astype(int), 0, n)
        hi = np.clip(np.ceil(c + r + n / 2.0).astype(int) + 1, 0, n)
        xs = (cen[lo[0]:hi[0]] - cx)[None, None, :]
        ys = (cen[lo[1]:hi[1]] - cy)[None, :, None]
        zs = (cen[lo[2]:hi[2]] - cz)[:, None, None]
        inside = (xs * xs + ys * ys + zs * zs) <= r * r
        sub = vol[lo[2]:hi[2], lo[1]:hi[1], lo[0]:hi[0]]
        np.maximum(sub, np.where(inside, dens, np.float32(0)), out=sub)
    return vol


# ----------------------------------------------------------------------------------------------
# The five benchmark/parity workloads
# ----------------------------------------------------------------------------------------------

def config(n: int, seed: int | None = None) -> Workload:
    """Workload ``n`` (1..5) with its default seed (= n) unless ``seed`` is given."""
    seed = n if seed is None else seed
    if n == 1:
        views = circular_parallel_2d(90)
        return Workload("parallel2d-64x64-90v", PARALLEL2D, views, (1, 64, 64), 1.0, 96, 1, 1.0,
                        1.0, seed,
                        lambda: uniform_image((64, 64), np.random.default_rng(seed)))
    if n == 2:
        views = circular_fan_2d(720, 1000.0, 1500.0)
        return Workload("fan2d-512x512-720v", FAN2D, views, (1, 512, 512), 1.0, 768, 1, 1.0, 1.0,
                        seed, lambda: ellipses_2d(10, 512, np.random.default_rng(seed)))
    if n == 3:
        views = circular_cone(360, 500.0, 1000.0)
        return Workload("cone-256^3-360v-384x384", CONE, views, (256, 256, 256), 1.0, 384, 384,
                        1.2, 1.2, seed,
                        lambda: ellipsoids_3d(12, 256, np.random.default_rng(seed)))
    if n == 4:
        jit = np.random.default_rng(1000 + seed)
        views = spiral_cone(720, 320.0, 512.0, 40.0, 2.0, rng=jit, src_jitter=0.5,
                            det_tilt_deg=0.5)
        return Workload("spiral-512^3-720v-768x512", CONE, views, (512, 512, 512), 0.5, 768, 512,
                        0.8, 0.8, seed,
                        lambda: ellipsoids_3d(12, 512, np.random.default_rng(seed),
                                              axis_range=(16.0, 200.0)))
    if n == 5:
        ang = np.arange(-70, 70, dtype=np.float64)
        views = dual_axis_tilt(ang, ang)
        return Workload("parallel3d-tilt-512^3-280v-512x512", PARALLEL3D, views, (512, 512, 512),
                        1.0, 512, 512, 1.0, 1.0, seed,
                        lambda: spheres_slab(400, 512, np.random.default_rng(seed)))
    raise ValueError(f"unknown workload {n}")


def small_config(n: int, seed: int | None = None) -> Workload:
    """A scaled-down twin of workload ``n`` that the oracle runs in about a second.

    Same beam type and the same kind of geometry and phantom, with sizes that still span several
    kernel tiles plus a ragged tail (odd detector sizes, non-cubic volumes).
    """
    seed = 100 + n if seed is None else seed
    rng = np.random.default_rng(seed)
    if n == 1:
        views = circular_parallel_2d(37)
        return Workload("parallel2d-small", PARALLEL2D, views, (1, 45, 61), 1.0, 83, 1, 1.0, 1.0,
                        seed, lambda: uniform_image((45, 61), np.random.default_rng(seed)))
    if n == 2:
        views = circular_fan_2d(41, 300.0, 450.0)
        return Workload("fan2d-small", FAN2D, views, (1, 77, 93), 1.0, 131, 1, 1.0, 1.0, seed,
                        lambda: ellipses_2d(6, 93, np.random.default_rng(seed),
                                            axis_range=(2.0, 30.0))[:77])
    if n == 3:
        views = circular_cone(23, 150.0, 300.0)
        return Workload("cone-small", CONE, views, (37, 45, 53), 1.0, 71, 45, 1.2, 1.2, seed,
                        lambda: _crop(ellipsoids_3d(8, 53, np.random.default_rng(seed),
                                                    axis_range=(3.0, 20.0)), (37, 45, 53)))
    if n == 4:
        views = spiral_cone(29, 64.0, 102.4, 8.0, 2.0, rng=rng, src_jitter=0.5, det_tilt_deg=0.5)
        return Workload("spiral-small", CONE, views, (40, 48, 56), 0.5, 75, 43, 0.8, 0.8, seed,
                        lambda: _crop(ellipsoids_3d(8, 56, np.random.default_rng(seed),
                                                    axis_range=(4.0, 25.0)), (40, 48, 56)))
    if n == 5:
        ang = np.arange(-70, 70, 7, dtype=np.float64)
        views = dual_axis_tilt(ang, ang)
        return Workload("parallel3d-tilt-small", PARALLEL3D, views, (48, 56, 52), 1.0, 67, 61, 1.0,
                        1.0, seed,
                        lambda: _crop(spheres_slab(40, 56, np.random.default_rng(seed),
                                                   radius_range=(2.0, 6.0), half_thickness=12.0),
                                      (48, 56, 52)))
    raise ValueError(f"unknown workload {n}")


def anisotropic_config(kind: str, seed: int = 7) -> Workload:
    """Small workloads with a different voxel spacing per axis (tensor order), for parity tests:
    'cone' (spacing (dz, dy, dx) = (1.1, 0.8, 0.6)), 'tilt' (parallel3d, (0.7, 1.3, 0.9)) and
    'fan' (2D, (dy, dx) = (0.9, 0.7))."""
    if kind == "cone":
        views = circular_cone(19, 120.0, 240.0)
        return Workload("cone-aniso", CONE, views, (29, 37, 41), (1.1, 0.8, 0.6), 63, 41, 1.0,
                        1.3, seed, lambda: _crop(ellipsoids_3d(8, 41, np.random.default_rng(seed),
                                                              axis_range=(3.0, 18.0)),
                                                 (29, 37, 41)))
    if kind == "tilt":
        ang = np.arange(-60, 61, 10, dtype=np.float64)
        views = dual_axis_tilt(ang, ang)
        return Workload("tilt-aniso", PARALLEL3D, views, (23, 31, 27), (0.7, 1.3, 0.9), 49, 45,
                        0.9, 1.1, seed,
                        lambda: _crop(spheres_slab(30, 31, np.random.default_rng(seed),
                                                   radius_range=(2.0, 5.0),
                                                   half_thickness=10.0), (23, 31, 27)))
    if kind == "fan":
        views = circular_fan_2d(29, 200.0, 300.0)
        return Workload("fan-aniso", FAN2D, views, (1, 53, 67), (0.9, 0.7), 97, 1, 0.8, 1.0,
                        seed, lambda: ellipses_2d(6, 67, np.random.default_rng(seed),
                                                  axis_range=(3.0, 20.0))[:53])
    raise ValueError(kind)


def flat_offsets(n_u: int, n_v: int, du: float, dv: float) -> np.ndarray:
    """The flat detector written as per-pixel (u, v, n) offsets: ((u - (U-1)/2) du,
    (v - (V-1)/2) dv, 0)."""
    ou = (np.arange(n_u) - (n_u - 1) / 2.0) * du
    ov = (np.arange(n_v) - (n_v - 1) / 2.0) * dv
    off = np.zeros((n_u, n_v, 3))
    off[:, :, 0] = ou[:, None]
    off[:, :, 1] = ov[None, :]
    return off


def cylindrical_offsets(views: np.ndarray, is_2d: bool, n_u: int, n_v: int, du: float,
                        dv: float, radius: float) -> np.ndarray:
    """Cylindrical detector (axis along det_v) of the given radius, as in the diffct
    detector-surface example: at arc length u, offsets (R sin(u/R), v, +/-R (1 - cos(u/R))).
    The normal offset bends the detector towards the source (the sign follows the generated
    frame's normal, checked on view 0), so radius = sdd centres the cylinder on the source."""
    r = views[0]
    if is_2d:
        src, ctr, u = np.r_[r[0:2], 0.0], np.r_[r[2:4], 0.0], np.r_[r[4:6], 0.0]
        nrm = np.array([u[1], -u[0], 0.0])
    else:
        src, ctr, u, v = r[0:3], r[3:6], r[6:9], r[9:12]
        nrm = np.cross(u, v)
    towards = 1.0 if float(nrm @ (src - ctr)) > 0 else -1.0
    ang = (np.arange(n_u) - (n_u - 1) / 2.0) * du / radius
    ov = (np.arange(n_v) - (n_v - 1) / 2.0) * dv if not is_2d else np.zeros(1)
    off = np.zeros((n_u, n_v, 3))
    off[:, :, 0] = (radius * np.sin(ang))[:, None]
    off[:, :, 1] = ov[None, :]
    off[:, :, 2] = (towards * radius * (1.0 - np.cos(ang)))[:, None]
    return off


def curved_config(kind: str, seed: int = 9) -> Workload:
    """Small workloads with a cylindrical detector centred on the source ('cone', 'fan')."""
    if kind == "cone":
        views = circular_cone(17, 150.0, 300.0)
        w = Workload("cone-cylindrical", CONE, views, (33, 41, 45), 1.0, 71, 37, 1.4, 1.2, seed,
                     lambda: _crop(ellipsoids_3d(8, 45, np.random.default_rng(seed),
                                                 axis_range=(3.0, 18.0)), (33, 41, 45)))
        w.offsets = cylindrical_offsets(views, False, 71, 37, 1.4, 1.2, 300.0)
        return w
    if kind == "fan":
        views = circular_fan_2d(23, 200.0, 350.0)
        w = Workload("fan-cylindrical", FAN2D, views, (1, 57, 63), 1.0, 101, 1, 1.3, 1.0, seed,
                     lambda: ellipses_2d(6, 63, np.random.default_rng(seed),
                                         axis_range=(3.0, 20.0))[:57])
        w.offsets = cylindrical_offsets(views, True, 101, 1, 1.3, 1.0, 350.0)
        return w
    raise ValueError(kind)


def _crop(vol: np.ndarray, shape) -> np.ndarray:
    """Centre crop of a cubic phantom to a non-cubic shape (for ragged-size tests)."""
    out = []
    for n_have, n_want in zip(vol.shape, shape):
        o = (n_have - n_want) // 2
        out.append(slice(o, o + n_want))
    return np.ascontiguousarray(vol[tuple(out)])


def random_sinogram(w: Workload, seed: int) -> np.ndarray:
    """i.i.d. U[-1, 1) float32 sinogram of the workload's shape (adjoint tests)."""
    return np.random.default_rng(seed).uniform(-1.0, 1.0, size=w.sino_shape).astype(np.float32)


def random_volume(w: Workload, seed: int) -> np.ndarray:
    """i.i.d. U[-1, 1) float32 volume of the workload's shape (adjoint tests)."""
    return np.random.default_rng(seed).uniform(-1.0, 1.0, size=w.volume_shape).astype(np.float32)
