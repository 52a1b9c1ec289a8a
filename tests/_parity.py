"""Shared helpers for the GPU parity tests and the smoke check (CUDA path vs float64 oracle).

Tolerances (from the projector's stated accuracy):
* forward projection, per ray: |y_gpu - y_oracle| <= 1e-4 * L_ray * max|x|, with L_ray the ray's
  total chord length from the oracle; rays the oracle finds missing (L = 0) must be exactly 0;
* backprojection: ||b_gpu - b_oracle||_2 <= 1e-4 ||b_oracle||_2;
* adjoint identity on the GPU: |<Ax, y> - <x, A^T y>| <= 1e-5 max(|<Ax, y>|, |<x, A^T y>|), both
  inner products accumulated in float64 on the host.
"""
import numpy as np

FP_RTOL = 1e-4
BP_RTOL = 1e-4
ADJ_RTOL = 1e-5


def torch_cuda(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def fp_violations(y_gpu, y_or, L, xmax):
    """Indices of rays that break the forward tolerance (flattened)."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64).reshape(-1)
    y_or = np.asarray(y_or, dtype=np.float64).reshape(-1)
    L = np.asarray(L, dtype=np.float64).reshape(-1)
    err = np.abs(y_gpu - y_or)
    bad = err > FP_RTOL * L * xmax
    bad |= (L == 0) & (y_gpu != 0)
    return np.nonzero(bad)[0]


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def adjoint_gap(Ax, y, x, Aty):
    lhs = float(np.dot(np.asarray(Ax, np.float64).reshape(-1), np.asarray(y, np.float64).reshape(-1)))
    rhs = float(np.dot(np.asarray(x, np.float64).reshape(-1), np.asarray(Aty, np.float64).reshape(-1)))
    return abs(lhs - rhs) / max(abs(lhs), abs(rhs)), lhs, rhs


def sample_rays(w, n, seed):
    rng = np.random.default_rng(seed)
    view = rng.integers(0, w.n_views, size=n).astype(np.int32)
    iu = rng.integers(0, w.n_u, size=n).astype(np.int32)
    iv = rng.integers(0, w.n_v, size=n).astype(np.int32)
    return view, iu, iv


def sino_at(sino, w, view, iu, iv):
    s = np.asarray(sino)
    return s[view, iu] if w.is_2d else s[view, iu, iv]
