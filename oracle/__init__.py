"""Float64 CPU oracle for the Siddon projector (ctypes loader for ``siddon_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg use it; the library (``fan_beam_projector_siddon_b300``) never imports it.  It shares no code
with the CUDA path.  Parity of every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, brute force, invariants and the adjoint identity.

All arrays crossing this boundary are float64 (inputs are converted), volumes ``[z, y, x]``
(2D ``[y, x]``), sinograms ``[view, u, v]`` (2D ``[view, u]``).
"""
from __future__ import annotations

import concurrent.futures as _cf
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "siddon_oracle.c")
_LIB = os.path.join(_HERE, "libsiddon_oracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math) into ``oracle/libsiddon_oracle.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Geom(ctypes.Structure):
    _fields_ = [("beam", ctypes.c_int32), ("n_views", ctypes.c_int32),
                ("views", ctypes.POINTER(ctypes.c_double)),
                ("nz", ctypes.c_int32), ("ny", ctypes.c_int32), ("nx", ctypes.c_int32),
                ("s", ctypes.c_double * 3), ("nu", ctypes.c_int32), ("nv", ctypes.c_int32),
                ("du", ctypes.c_double), ("dv", ctypes.c_double),
                ("offsets", ctypes.POINTER(ctypes.c_double))]


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.POINTER
        dp, gp = P(ctypes.c_double), P(_Geom)
        i32p, i64p = P(ctypes.c_int32), P(ctypes.c_int64)
        L.oracle_project.argtypes = [gp, dp, dp, ctypes.c_int32, ctypes.c_int32]
        L.oracle_project_rays.argtypes = [gp, dp, ctypes.c_int64, i32p, i32p, i32p, dp]
        L.oracle_backproject.argtypes = [gp, dp, dp, ctypes.c_int32, ctypes.c_int32]
        L.oracle_ray_segments.argtypes = [gp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          i64p, dp, ctypes.c_int64]
        L.oracle_ray_segments.restype = ctypes.c_int64
        L.oracle_line_segments.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, dp, dp, dp,
                                           ctypes.c_double, ctypes.c_double, i64p, dp,
                                           ctypes.c_int64]
        L.oracle_line_segments.restype = ctypes.c_int64
        L.oracle_ray_lengths.argtypes = [gp, ctypes.c_int32, ctypes.c_int32, dp, i64p]
        L.oracle_brute_row.argtypes = [gp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, dp]
        L.oracle_backproject_voxels.argtypes = [gp, dp, ctypes.c_int64, i64p, dp]
        L.oracle_sirt.argtypes = [gp, dp, dp, ctypes.c_int32, ctypes.c_double, dp]
        L.oracle_cgls.argtypes = [gp, dp, dp, ctypes.c_int32, dp]
        L.oracle_ray.argtypes = [gp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, dp, dp, dp]
        _lib = L
    return _lib


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def spacing_xyz(voxel_spacing, is_2d: bool):
    """(sx, sy, sz) from a scalar or a tuple in tensor order: (dy, dx) for 2D, (dz, dy, dx) for
    3D (diffct "Trajectories and Geometry", voxel spacing)."""
    if np.ndim(voxel_spacing) == 0:
        s = float(voxel_spacing)
        return (s, s, s)
    vs = [float(v) for v in voxel_spacing]
    if is_2d:
        assert len(vs) == 2
        return (vs[1], vs[0], 1.0)
    assert len(vs) == 3
    return (vs[2], vs[1], vs[0])


class Geometry:
    """Oracle-side view of an acquisition (same record layout as the C library's input)."""

    def __init__(self, beam: int, views, vol_shape, voxel_spacing, n_u: int, n_v: int,
                 du: float, dv: float, offsets=None):
        self.beam = int(beam)
        self.views = np.ascontiguousarray(np.asarray(views, dtype=np.float64))
        nz, ny, nx = vol_shape
        self.vol_shape = (int(nz), int(ny), int(nx))
        self.is_2d = self.beam in (0, 1)
        self.n_u, self.n_v = int(n_u), (1 if self.is_2d else int(n_v))
        self.spacing_xyz = spacing_xyz(voxel_spacing, self.is_2d)
        # per-pixel (u, v, n) offsets of a parameterized detector surface, (n_u, n_v, 3)
        self.offsets = None
        if offsets is not None:
            self.offsets = np.ascontiguousarray(
                np.asarray(offsets, dtype=np.float64).reshape(self.n_u, self.n_v, 3))
        self._g = _Geom(self.beam, self.views.shape[0], _dp(self.views), self.vol_shape[0],
                        self.vol_shape[1], self.vol_shape[2],
                        (ctypes.c_double * 3)(*self.spacing_xyz), self.n_u, self.n_v,
                        float(du), float(dv),
                        _dp(self.offsets) if self.offsets is not None else None)

    @classmethod
    def from_workload(cls, w) -> "Geometry":
        return cls(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv,
                   getattr(w, "offsets", None))

    def ray(self, view: int, iu: int, iv: int = 0):
        """(origin e, direction d, (amin, amax)) of one pixel's ray."""
        L = _load()
        e, d, rg = np.zeros(3), np.zeros(3), np.zeros(2)
        L.oracle_ray(ctypes.byref(self._g), view, iu, iv, _dp(e), _dp(d), _dp(rg))
        return e, d, (rg[0], rg[1])

    @property
    def n_views(self) -> int:
        return int(self.views.shape[0])

    @property
    def sino_shape(self):
        return (self.n_views, self.n_u) if self.is_2d else (self.n_views, self.n_u, self.n_v)

    @property
    def volume_shape(self):
        return self.vol_shape[1:] if self.is_2d else self.vol_shape

    # -- operators ------------------------------------------------------------------------------
    def project(self, x, views=None, threads: int = 1) -> np.ndarray:
        """A x for all views (or the view range ``views=(v0, v1)``); rows outside stay 0."""
        L = _load()
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64).reshape(self.volume_shape))
        out = np.zeros(self.sino_shape, dtype=np.float64)
        v0, v1 = (0, self.n_views) if views is None else views
        if threads <= 1:
            L.oracle_project(ctypes.byref(self._g), _dp(x), _dp(out), v0, v1)
        else:
            with _cf.ThreadPoolExecutor(threads) as ex:
                list(ex.map(lambda ab: L.oracle_project(ctypes.byref(self._g), _dp(x), _dp(out),
                                                        ab[0], ab[1]), _split(v0, v1, threads)))
        return out

    def backproject(self, sino, views=None, threads: int = 1) -> np.ndarray:
        """A^T sino (views restricted to ``views=(v0, v1)`` if given)."""
        L = _load()
        sino = np.ascontiguousarray(np.asarray(sino, dtype=np.float64).reshape(self.sino_shape))
        v0, v1 = (0, self.n_views) if views is None else views
        if threads <= 1:
            out = np.zeros(self.volume_shape, dtype=np.float64)
            L.oracle_backproject(ctypes.byref(self._g), _dp(sino), _dp(out), v0, v1)
            return out
        parts = _split(v0, v1, threads)
        outs = [np.zeros(self.volume_shape, dtype=np.float64) for _ in parts]
        with _cf.ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(lambda k: L.oracle_backproject(ctypes.byref(self._g), _dp(sino),
                                                       _dp(outs[k]), parts[k][0], parts[k][1]),
                        range(len(parts))))
        return np.sum(outs, axis=0)

    def project_rays(self, x, view, iu, iv) -> np.ndarray:
        L = _load()
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64).reshape(self.volume_shape))
        view = np.ascontiguousarray(view, dtype=np.int32)
        iu = np.ascontiguousarray(iu, dtype=np.int32)
        iv = np.ascontiguousarray(iv, dtype=np.int32)
        out = np.zeros(view.shape[0], dtype=np.float64)
        i32 = ctypes.POINTER(ctypes.c_int32)
        L.oracle_project_rays(ctypes.byref(self._g), _dp(x), view.shape[0],
                              view.ctypes.data_as(i32), iu.ctypes.data_as(i32),
                              iv.ctypes.data_as(i32), _dp(out))
        return out

    def ray_segments(self, view: int, iu: int, iv: int = 0):
        """(voxel indices, chord lengths) of one ray in traversal order."""
        L = _load()
        cap = sum(self.vol_shape) + 4
        idx = np.zeros(cap, dtype=np.int64)
        w = np.zeros(cap, dtype=np.float64)
        cnt = L.oracle_ray_segments(ctypes.byref(self._g), view, iu, iv,
                                    idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _dp(w),
                                    cap)
        assert cnt <= cap
        return idx[:cnt].copy(), w[:cnt].copy()

    def ray_lengths(self, views=None):
        """(total chord length, positive-length segment count) per ray, sinogram-shaped."""
        L = _load()
        v0, v1 = (0, self.n_views) if views is None else views
        length = np.zeros(self.sino_shape, dtype=np.float64)
        segs = np.zeros(self.sino_shape, dtype=np.int64)
        L.oracle_ray_lengths(ctypes.byref(self._g), v0, v1, _dp(length),
                             segs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
        return length, segs

    def brute_row(self, view: int, iu: int, iv: int = 0) -> np.ndarray:
        """Row of A for one ray by per-voxel box intersection (tiny volumes only)."""
        L = _load()
        row = np.zeros(self.volume_shape, dtype=np.float64)
        L.oracle_brute_row(ctypes.byref(self._g), view, iu, iv, _dp(row))
        return row

    def backproject_voxels(self, sino, voxels) -> np.ndarray:
        """(A^T sino) at the given linear voxel indices, one voxel at a time."""
        L = _load()
        sino = np.ascontiguousarray(np.asarray(sino, dtype=np.float64).reshape(self.sino_shape))
        voxels = np.ascontiguousarray(voxels, dtype=np.int64)
        out = np.zeros(voxels.shape[0], dtype=np.float64)
        L.oracle_backproject_voxels(ctypes.byref(self._g), _dp(sino), voxels.shape[0],
                                    voxels.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                    _dp(out))
        return out

    def sirt(self, y, n_iter: int, x0=None, relax: float = 1.0):
        """(x after n_iter SIRT updates, R-weighted squared residual before each update)."""
        L = _load()
        y = np.ascontiguousarray(np.asarray(y, dtype=np.float64).reshape(self.sino_shape))
        x = (np.zeros(self.volume_shape, dtype=np.float64) if x0 is None
             else np.array(x0, dtype=np.float64).reshape(self.volume_shape))
        res = np.zeros(max(n_iter, 1), dtype=np.float64)
        L.oracle_sirt(ctypes.byref(self._g), _dp(y), _dp(x), n_iter, relax, _dp(res))
        return x, res[:n_iter]

    def cgls(self, y, n_iter: int, x0=None):
        """(x after n_iter CGLS steps, ||y - A x||^2 before the first and after each step)."""
        L = _load()
        y = np.ascontiguousarray(np.asarray(y, dtype=np.float64).reshape(self.sino_shape))
        x = (np.zeros(self.volume_shape, dtype=np.float64) if x0 is None
             else np.array(x0, dtype=np.float64).reshape(self.volume_shape))
        res = np.zeros(n_iter + 1, dtype=np.float64)
        L.oracle_cgls(ctypes.byref(self._g), _dp(y), _dp(x), n_iter, _dp(res))
        return x, res


def line_segments(e, d, amin, amax, vol_shape, spacing, dims=3):
    """Segments (voxel indices, chords) of an explicit ray p(a) = e + a d, a in [amin, amax];
    `spacing` is a scalar or (dz, dy, dx)."""
    L = _load()
    nz, ny, nx = vol_shape
    sp = np.ascontiguousarray(spacing_xyz(spacing, False) if dims == 3 or np.ndim(spacing) == 0
                              else spacing_xyz(spacing, True), dtype=np.float64)
    e = np.ascontiguousarray(np.resize(np.asarray(e, dtype=np.float64), 3))
    d = np.ascontiguousarray(np.resize(np.asarray(d, dtype=np.float64), 3))
    cap = nx + ny + nz + 4
    idx = np.zeros(cap, dtype=np.int64)
    w = np.zeros(cap, dtype=np.float64)
    cnt = L.oracle_line_segments(dims, nz, ny, nx, _dp(sp), _dp(e), _dp(d), float(amin),
                                 float(amax), idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                 _dp(w), cap)
    return idx[:cnt].copy(), w[:cnt].copy()


def _split(v0: int, v1: int, parts: int):
    parts = max(1, min(parts, v1 - v0))
    edges = np.linspace(v0, v1, parts + 1).round().astype(int)
    return [(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:]) if b > a]
