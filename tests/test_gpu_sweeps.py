"""Seeded random-geometry sweeps of the CUDA path against the oracle, wider than the hand-made
cases of the other modules (each sweep a few seconds on one GPU):

* shared-line geometries (cone orbits with offsets and in-plane detector turns, steep parallel
  rays, random shapes and per-axis pitches): every ray of A, the whole volume of A^T, and entries
  of A against A^T bit for bit;
* random frames of the four beams walked per ray: every ray of A and the whole volume of A^T;
* tall volumes with forced 32- or 64-cell slabs: every ray of A and A^T, and the batched call equal
  to single calls with slabs on and off;
* perturbed cylindrical detector surfaces of random radius, all four beams;
* FBP/FDK and its transpose on random parallel, fan and cone frames with random windows;
* SIRT, ten iterations, against the oracle's iterate.

Geometries that miss the volume almost entirely (a tenth of the rays or fewer hitting) are
skipped, since they test little; the sweeps assert that most seeds are kept.
"""
import numpy as np
import pytest

import oracle
from fan_beam_projector_siddon_b300 import workloads as W
from oracle import fbp as F
from tests._parity import BP_RTOL, fp_violations, rel_l2, torch_cuda
from tests.test_gpu_lines import _random_line_geometry
from tests.test_gpu_parity import _random_frames, _random_frames_2d

pytestmark = pytest.mark.gpu

FBP_REL_L2 = 2e-4   # the tolerances of test_gpu_fbp.py (float32 filter and gather)
FBP_MAX_REL = 2e-3
SIRT_RTOL = 1e-4    # test_gpu_sirt.py's


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


def _frames_case(rng, beam, n_views=5, tall=False):
    """Random frames, shape, pitches and detector for one beam (the per-ray parity generator's
    recipe; `tall` stretches the volume along z and the geometry with it)."""
    two_d = beam in (W.FAN2D, W.PARALLEL2D)
    if two_d:
        shape = (1, int(rng.integers(5, 40)), int(rng.integers(5, 40)))
        sp = (float(rng.uniform(0.5, 1.5)), float(rng.uniform(0.5, 1.5)))
        views = _random_frames_2d(rng, n_views, beam)
        return beam, views, shape, sp, int(rng.integers(20, 90)), 1, float(rng.uniform(0.3, 1.2)), 1.0
    nz = int(rng.integers(33, 110)) if tall else int(rng.integers(4, 28))
    shape = (nz, int(rng.integers(4, 30 if tall else 28)), int(rng.integers(4, 30 if tall else 28)))
    sp = tuple(float(v) for v in rng.uniform(0.5, 1.5, 3))
    scale = [8.0, 8.0, 1.0, 1.0] if beam == W.CONE else [1.0, 8.0, 1.0, 1.0]
    views = _random_frames(rng, n_views, beam) * np.repeat(scale, 3)
    k = max(1.0, nz / 30.0) if tall else 1.0   # keep the sources outside the taller boxes
    if beam == W.CONE:
        views[:, 0:6] *= k
    else:
        views[:, 3:6] *= k
    n_u, n_v = int(rng.integers(20, 70)), int(rng.integers(20, 70))
    du, dv = float(rng.uniform(0.2, 0.8)), float(rng.uniform(0.2, 0.8)) * k
    return beam, views, shape, sp, n_u, n_v, du, dv


def _forward_backward(g, go, x, rng):
    """(rays outside the per-ray tolerance, A^T relative L2 error) of one geometry."""
    L, _ = go.ray_lengths()
    y = _cpu(g.project(torch_cuda(x)))
    bad = fp_violations(y, go.project(x, threads=8), L, float(np.abs(x).max()))
    yy = rng.uniform(-1.0, 1.0, size=go.sino_shape).astype(np.float32)
    return bad.size, rel_l2(_cpu(g.backproject(torch_cuda(yy))), go.backproject(yy, threads=8))


@pytest.mark.parametrize("chunk", range(3))
def test_shared_line_sweep(ct, chunk):
    kept = 0
    for seed in range(100 + 100 * chunk, 200 + 100 * chunk):
        w = _random_line_geometry(seed)
        go = oracle.Geometry.from_workload(w)
        L, _ = go.ray_lengths()
        if (L > 0).mean() <= 0.1:
            continue
        kept += 1
        g = ct.Geometry.from_workload(w)
        rng = np.random.default_rng(seed)
        x = rng.uniform(0.1, 1.0, size=w.volume_shape).astype(np.float32)
        nbad, bp = _forward_backward(g, go, x, rng)
        assert nbad == 0 and bp <= BP_RTOL, (seed, nbad, bp)
        if g.info.shared_lines:
            # two entries of A against A^T, bit for bit
            nvox, nray = int(np.prod(w.volume_shape)), int(np.prod(w.sino_shape))
            e = np.zeros(nvox, np.float32)
            i = int(rng.integers(nvox))
            e[i] = 1.0
            col = _cpu(g.project(torch_cuda(e.reshape(w.volume_shape)))).reshape(-1)
            rays = np.nonzero(col)[0]
            for r in rays[:: max(1, rays.size // 2)][:2]:
                er = np.zeros(nray, np.float32)
                er[r] = 1.0
                row = _cpu(g.backproject(torch_cuda(er.reshape(w.sino_shape)))).reshape(-1)
                assert row[i] == col[r], (seed, i, r, row[i], col[r])
    assert kept >= 80


@pytest.mark.parametrize("chunk", range(2))
def test_per_ray_sweep(ct, chunk):
    kept = 0
    for seed in range(100 + 150 * chunk, 250 + 150 * chunk):
        rng = np.random.default_rng(1000 + seed)
        args = _frames_case(rng, [W.CONE, W.PARALLEL3D, W.FAN2D, W.PARALLEL2D][seed % 4])
        go = oracle.Geometry(*args)
        L, _ = go.ray_lengths()
        if (L > 0).mean() <= 0.1:
            continue
        kept += 1
        g = ct.Geometry(*args)
        vol_shape = args[2][1:] if args[0] in (W.FAN2D, W.PARALLEL2D) else args[2]
        x = rng.uniform(0.0, 1.0, size=vol_shape).astype(np.float32)
        nbad, bp = _forward_backward(g, go, x, rng)
        assert nbad == 0 and bp <= BP_RTOL, (seed, nbad, bp)
    assert kept >= 100


def test_slab_sweep(ct):
    kept = 0
    for seed in range(0, 1500):
        rng = np.random.default_rng(7000 + seed)
        args = _frames_case(rng, W.CONE if seed % 2 == 0 else W.PARALLEL3D, tall=True)
        g = ct.Geometry(*args)
        if g.info.volume_layout != 1:
            continue   # slab tiling needs the z-fastest internal order
        go = oracle.Geometry(*args)
        L, _ = go.ray_lengths()
        if (L > 0).mean() <= 0.1:
            continue
        kept += 1
        cells = int(rng.choice([32, 64]))
        g.set_slabs(cells if args[2][0] > cells else 32)   # at least two slabs (nz >= 33)
        assert g.info.n_slabs >= 2
        x = rng.uniform(0.0, 1.0, size=args[2]).astype(np.float32)
        nbad, bp = _forward_backward(g, go, x, rng)
        assert nbad == 0 and bp <= BP_RTOL, (seed, nbad, bp)
        xs = torch_cuda(np.stack([x, x[::-1].copy()]))
        for cells in (None, 0):
            if cells is not None:
                g.set_slabs(cells)
            single = _cpu(g.project(torch_cuda(x)))
            assert np.array_equal(_cpu(g.project(xs))[0], single), seed
    assert kept >= 100


def test_surface_sweep(ct):
    for seed in range(300):
        rng = np.random.default_rng(9000 + seed)
        beam = [W.CONE, W.FAN2D, W.PARALLEL3D, W.PARALLEL2D][seed % 4]
        two_d = beam in (W.FAN2D, W.PARALLEL2D)
        args = _frames_case(rng, beam, n_views=6 if two_d else 5)
        _, views, shape, sp, n_u, n_v, du, dv = args
        off = W.cylindrical_offsets(views, two_d, n_u, n_v, du, dv, float(rng.uniform(5.0, 60.0)))
        off = off + rng.uniform(-0.2, 0.2, size=off.shape) * np.array(
            [du, 0.0 if two_d else dv, 0.5])
        g, go = ct.Geometry(*args, offsets=off), oracle.Geometry(*args, offsets=off)
        x = rng.uniform(0.0, 1.0, size=shape[1:] if two_d else shape).astype(np.float32)
        nbad, bp = _forward_backward(g, go, x, rng)
        assert nbad == 0 and bp <= BP_RTOL, (seed, nbad, bp)


def test_fbp_sweep(ct):
    windows = ["ram-lak", "shepp-logan", "cosine", "hamming", "hann"]
    for seed in range(300):
        rng = np.random.default_rng(11000 + seed)
        beam = [W.CONE, W.FAN2D, W.PARALLEL2D][seed % 3]
        two_d = beam != W.CONE
        args = _frames_case(rng, beam, n_views=int(rng.integers(3, 12 if two_d else 10)))
        _, views, shape, sp, n_u, n_v, du, dv = args
        win = windows[int(rng.integers(0, 5))]
        g = ct.Geometry(*args)
        sino_shape = (views.shape[0], n_u) if two_d else (views.shape[0], n_u, n_v)
        sino = rng.uniform(-1, 1, size=sino_shape).astype(np.float32)
        got = _cpu(g.fbp(torch_cuda(sino), window=win))
        want = F.fbp(*args, sino.astype(np.float64), window=win)
        xr = rng.uniform(-1, 1, size=shape[1:] if two_d else shape).astype(np.float32)
        got_t = _cpu(g.fbp_transpose(torch_cuda(xr), window=win))
        want_t = F.fbp_transpose(*args, xr.astype(np.float64), window=win)
        for a, b in ((got, want), (got_t, want_t)):
            mx = float(np.abs(a - b).max()) / max(float(np.abs(b).max()), 1e-30)
            assert rel_l2(a, b) <= FBP_REL_L2 and mx <= FBP_MAX_REL, (seed, win, rel_l2(a, b), mx)


def test_sirt_sweep(ct):
    import torch
    for seed in range(100):
        rng = np.random.default_rng(13000 + seed)
        args = _frames_case(rng, [W.CONE, W.PARALLEL3D, W.FAN2D, W.PARALLEL2D][seed % 4],
                            n_views=7 if seed % 4 >= 2 else 5)
        g, go = ct.Geometry(*args), oracle.Geometry(*args)
        vol_shape = args[2][1:] if args[0] in (W.FAN2D, W.PARALLEL2D) else args[2]
        x_true = rng.uniform(0, 1, size=vol_shape).astype(np.float32)
        x_or, _ = go.sirt(go.project(x_true, threads=8), 10)
        x = torch.zeros(vol_shape, dtype=torch.float32, device="cuda")
        g.sirt(x, g.project(torch_cuda(x_true)), 10, g.new_workspace(sirt=True),
               initialised=False)
        assert rel_l2(_cpu(x), x_or) <= SIRT_RTOL, seed
