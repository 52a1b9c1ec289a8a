"""Filtered backprojection (FBP / FDK) through the C ABI against the float64 oracle (oracle/fbp.py).

Tolerance.  The GPU path filters and gathers in float32; the oracle in float64.  The gather's
fractional detector index u(X) carries a float32 rounding error of a few ulp of the largest
coordinate involved (about 1e-6 pixel for these sizes); the ramp-filtered sinogram changes by at
most ~2 max|Q| per pixel, and the filter's float32 sums of n_u terms add ~n_u eps relative to
sum|h p|.  Over a whole volume both stay below 1e-4 of the result's L2 norm, so small cases are
compared at rel L2 <= 2e-4 and max |diff| <= 2e-3 max |f|, both scaled by n_u / 400 for wider
detectors; sampled voxels of the full-size cone case at max |diff| <= 2e-3 max |f|.
"""
import math

import numpy as np
import pytest

from fan_beam_projector_siddon_b300 import workloads as W
from oracle import fbp as F
from tests._parity import rel_l2, torch_cuda

pytestmark = pytest.mark.gpu

REL_L2 = 2e-4
MAX_REL = 2e-3


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


def _oracle(w, sino, **kw):
    return F.fbp(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv, sino,
                 **kw)


def _check(got, want, n_u=0):
    # the filter's float32 sums of n_u terms: the bound grows linearly with n_u (above 400)
    grow = max(1.0, n_u / 400.0)
    err = rel_l2(got, want)
    mx = float(np.abs(got - want).max()) / max(float(np.abs(want).max()), 1e-30)
    assert err <= REL_L2 * grow and mx <= MAX_REL * grow, (err, mx)


def _phantom_sino(w):
    """Sinogram of the workload's phantom by the oracle's own Siddon projector (float64)."""
    import oracle
    return oracle.Geometry.from_workload(w).project(w.phantom(), threads=8)


@pytest.mark.parametrize("n", [1, 2, 3])
def test_small_phantom_matches_oracle(ct, n):
    w = W.small_config(n)
    sino = _phantom_sino(w)
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp(torch_cuda(sino.astype(np.float32))))
    want = _oracle(w, sino.astype(np.float32).astype(np.float64))
    _check(got, want)


@pytest.mark.parametrize("window", ["ram-lak", "shepp-logan", "cosine", "hamming", "hann"])
@pytest.mark.parametrize("n", [2, 3])
def test_windows_on_random_sinograms(ct, n, window):
    w = W.small_config(n)
    sino = W.random_sinogram(w, 40 + n)
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp(torch_cuda(sino), window=window))
    _check(got, _oracle(w, sino.astype(np.float64), window=window))


@pytest.mark.parametrize("n", [2, 3])
def test_view_weights_and_isocentre(ct, n):
    w = W.small_config(n)
    sino = W.random_sinogram(w, 7)
    wts = np.random.default_rng(8).uniform(0.0, 0.05, size=w.views.shape[0]).astype(np.float32)
    iso = (1.5, -2.25, 0.75)[: 2 if n == 2 else 3]
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp(torch_cuda(sino), window="hann", view_weights=torch_cuda(wts),
                     isocenter=iso))
    want = _oracle(w, sino.astype(np.float64), window="hann",
                   view_weights=wts.astype(np.float64), isocenter=iso)
    _check(got, want)


@pytest.mark.parametrize("kind", ["cone", "fan"])
def test_anisotropic_voxels(ct, kind):
    w = W.anisotropic_config(kind)
    sino = W.random_sinogram(w, 11)
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp(torch_cuda(sino)))
    _check(got, _oracle(w, sino.astype(np.float64)), n_u=w.n_u)


def test_full_size_cone_sampled_voxels(ct):
    """The 256^3, 360-view cone workload (the benchmark's), sampled voxels against the oracle."""
    w = W.config(3)
    sino = W.random_sinogram(w, 5)
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp(torch_cuda(sino)))
    rng = np.random.default_rng(6)
    idx = np.stack([rng.integers(0, s, 48) for s in w.vol_shape], axis=1)
    idx = np.concatenate([idx, [[0, 0, 0], [255, 255, 255], [128, 0, 255]]])
    want = _oracle(w, sino.astype(np.float64), voxels=idx)
    scale = float(np.abs(got).max())
    diff = np.abs(got[idx[:, 0], idx[:, 1], idx[:, 2]] - want)
    assert diff.max() <= MAX_REL * scale, (diff.max(), scale)


def test_batch_dims_and_determinism(ct):
    w = W.small_config(3)
    s = np.stack([W.random_sinogram(w, 1), W.random_sinogram(w, 2)])
    g = ct.Geometry.from_workload(w)
    st = torch_cuda(s)
    a = _cpu(g.fbp(st))
    b = _cpu(g.fbp(st))
    assert np.array_equal(a, b)
    one = _cpu(g.fbp(torch_cuda(s[1])))
    assert np.array_equal(a[1], one)


def test_linearity(ct):
    w = W.small_config(2)
    a, b = W.random_sinogram(w, 3), W.random_sinogram(w, 4)
    g = ct.Geometry.from_workload(w)
    fa, fb = _cpu(g.fbp(torch_cuda(a))), _cpu(g.fbp(torch_cuda(b)))
    fab = _cpu(g.fbp(torch_cuda(2.0 * a - b)))
    assert rel_l2(fab, 2.0 * fa - fb) < 1e-5


def test_errors(ct):
    import torch
    w = W.small_config(3)
    g = ct.Geometry.from_workload(w)
    sino = torch.zeros(g.sino_shape, device="cuda")
    vol = torch.zeros(g.volume_shape, device="cuda")
    need = ct.ct_fbp_workspace_bytes(g.handle)
    assert need >= 4 * sino.numel()
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def call(status, **kw):
        args = dict(d_sino=sino.data_ptr(), d_volume=vol.data_ptr(), d_view_weights=None,
                    d_pixel_weights=None, d_kernel=None, isocenter=None, window=0,
                    d_workspace=ws.data_ptr(), workspace_bytes=need)
        args.update(kw)
        opts, keep = ct.fbp_options(args["window"], args["d_view_weights"],
                                    args["d_pixel_weights"], args["d_kernel"], args["isocenter"])
        with pytest.raises(ct.CtError) as ei:
            ct.ct_fbp(g.handle, args["d_sino"], args["d_volume"], opts, args["d_workspace"],
                      args["workspace_bytes"], s)
        assert ei.value.status == status

    call(7, workspace_bytes=need - 1)
    # the transpose needs its own (larger) scratch: the parity copies of the detector
    need_t = ct.ct_fbp_transpose_workspace_bytes(g.handle)
    assert need_t > need
    with pytest.raises(ct.CtError) as ei:
        ct.ct_fbp_transpose(g.handle, vol.data_ptr(), sino.data_ptr(), None, ws.data_ptr(),
                            need, s)
    assert ei.value.status == 7
    call(1, window=5)
    call(1, isocenter=(math.nan, 0.0, 0.0))
    call(4, d_volume=ws.data_ptr())
    host = np.zeros(4, np.float32)
    call(3, d_view_weights=host.ctypes.data)
    call(3, d_pixel_weights=host.ctypes.data)
    call(4, d_pixel_weights=vol.data_ptr())
    call(3, d_kernel=host.ctypes.data)
    call(4, d_kernel=ws.data_ptr())
    # gradients: at least one output; their own (larger) scratch
    need_g = ct.ct_fbp_gradients_workspace_bytes(g.handle)
    wsg = torch.empty(need_g, dtype=torch.uint8, device="cuda")
    gk = torch.empty(2 * w.n_u - 1, device="cuda")
    for args, status in (((None, None, wsg.data_ptr(), need_g), 1),
                         ((gk.data_ptr(), None, wsg.data_ptr(), need_g - 1), 7),
                         ((gk.data_ptr(), gk.data_ptr(), wsg.data_ptr(), need_g), 4)):
        with pytest.raises(ct.CtError) as ei:
            ct.ct_fbp_gradients(g.handle, sino.data_ptr(), vol.data_ptr(), None, *args, s)
        assert ei.value.status == status
    # Parker weights: parallel beams have none
    with pytest.raises(ct.CtError) as ei:
        ct.Geometry.from_workload(W.small_config(1)).parker_weights()
    assert ei.value.status == 1
    # parallel3d and surface detectors have no FBP here
    p = W.small_config(5)
    gp = ct.Geometry.from_workload(p)
    with pytest.raises(ct.CtError) as ei:
        gp.fbp(torch.zeros(gp.sino_shape, device="cuda"))
    assert ei.value.status == 1
    c = W.curved_config("cone")
    gc = ct.Geometry.from_workload(c)
    with pytest.raises(ct.CtError) as ei:
        gc.fbp(torch.zeros(gc.sino_shape, device="cuda"))
    assert ei.value.status == 1


@pytest.mark.parametrize("n,shape", [(3, (50, 21, 19)), (3, (101, 13, 17)), (3, (200, 7, 9)),
                                     (4, (50, 9, 11)), (4, (101, 5, 7)), (4, (200, 7, 9)),
                                     (2, (1, 130, 41)), (1, (1, 131, 37))])
def test_gather_variants(ct, n, shape):
    """Volumes that select the other gather shapes (2, 4 and 8 voxels a thread along z; 4 rows a
    thread in 2D), with ragged tails; the circular orbit (workload 3) takes the z-independent
    path, the jittered helix (workload 4, tilted detectors) the general one."""
    import dataclasses
    w = dataclasses.replace(W.small_config(n), vol_shape=shape)
    sino = W.random_sinogram(w, 21)
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp(torch_cuda(sino), window="shepp-logan"))
    _check(got, _oracle(w, sino.astype(np.float64), window="shepp-logan"))


def test_wide_detector_uses_the_plain_filter(ct):
    """n_u = 1601 exceeds the blocked filter's shared memory; the per-output filter runs."""
    import dataclasses
    base = W.small_config(3)
    w = dataclasses.replace(base, n_u=1601, n_v=5, du=0.05, views=base.views[:4],
                            vol_shape=(4, 9, 11))
    sino = W.random_sinogram(w, 22)
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp(torch_cuda(sino)))
    _check(got, _oracle(w, sino.astype(np.float64)), n_u=w.n_u)


# ---------------------------------------------------------------------------------------------
# transpose (volume -> sinogram)
# ---------------------------------------------------------------------------------------------

def _oracle_t(w, vol, **kw):
    return F.fbp_transpose(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du,
                           w.dv, vol, **kw)


def _vol(w, seed):
    return W.random_volume(w, seed)


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_transpose_matches_oracle(ct, n):
    w = W.small_config(n)
    x = _vol(w, 60 + n)
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp_transpose(torch_cuda(x), window="cosine"))
    _check(got, _oracle_t(w, x.astype(np.float64), window="cosine"))


@pytest.mark.parametrize("n,shape", [(3, (50, 21, 19)), (3, (101, 13, 17)), (3, (200, 7, 9)),
                                     (4, (200, 7, 9)), (2, (1, 130, 41)), (1, (1, 131, 37))])
def test_transpose_variants(ct, n, shape):
    import dataclasses
    w = dataclasses.replace(W.small_config(n), vol_shape=shape)
    x = _vol(w, 23)
    wts = np.random.default_rng(9).uniform(0.0, 0.05, size=w.views.shape[0]).astype(np.float32)
    iso = (0.5, 1.25, -0.75)[: 2 if w.beam in (0, 1) else 3]
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp_transpose(torch_cuda(x), view_weights=torch_cuda(wts), isocenter=iso))
    _check(got, _oracle_t(w, x.astype(np.float64), view_weights=wts.astype(np.float64),
                          isocenter=iso))


@pytest.mark.parametrize("full", [False, True])
def test_adjoint_identity_on_the_gpu(ct, full):
    """<F y, x> = <y, F^T x> with both sides computed by the CUDA path; at full size (the cone
    256^3 x 360 workload) this is the transpose's check, the oracle being too slow there."""
    w = W.config(3) if full else W.small_config(3)
    g = ct.Geometry.from_workload(w)
    y = W.random_sinogram(w, 31)
    x = _vol(w, 32)
    Fy = _cpu(g.fbp(torch_cuda(y), window="hamming")).astype(np.float64)
    Ftx = _cpu(g.fbp_transpose(torch_cuda(x), window="hamming")).astype(np.float64)
    lhs, rhs = float(np.sum(Fy * x)), float(np.sum(y * Ftx))
    scale = np.linalg.norm(Fy) * np.linalg.norm(x)
    assert abs(lhs - rhs) <= 1e-5 * scale, (lhs, rhs, scale)


# ---------------------------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("case", ["one_view", "one_row", "one_voxel", "one_column"])
def test_degenerate_shapes(ct, case):
    import dataclasses
    base = W.small_config(3)
    if case == "one_view":
        w = dataclasses.replace(base, views=base.views[:1])
    elif case == "one_row":
        w = dataclasses.replace(base, n_v=1, vol_shape=(5, 21, 23))
    elif case == "one_voxel":
        w = dataclasses.replace(base, vol_shape=(1, 1, 1), voxel_spacing=3.0)
    else:
        w = dataclasses.replace(base, n_u=1, vol_shape=(9, 4, 5))
    y = W.random_sinogram(w, 3)
    x = W.random_volume(w, 4)
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp(torch_cuda(y), window="hann"))
    want = _oracle(w, y.astype(np.float64), window="hann")
    if np.abs(want).max() > 0:
        _check(got, want)
    else:
        assert np.abs(got).max() == 0
    got_t = _cpu(g.fbp_transpose(torch_cuda(x), window="hann"))
    want_t = _oracle_t(w, x.astype(np.float64), window="hann")
    if np.abs(want_t).max() > 0:
        _check(got_t, want_t)
    else:
        assert np.abs(got_t).max() == 0


def test_zero_weights_and_empty_batch(ct):
    import torch
    w = W.small_config(2)
    g = ct.Geometry.from_workload(w)
    y = torch_cuda(W.random_sinogram(w, 5))
    zero = torch.zeros(w.views.shape[0], device="cuda")
    assert _cpu(g.fbp(y, view_weights=zero)).max() == 0
    assert _cpu(g.fbp_transpose(torch_cuda(W.random_volume(w, 6)), view_weights=zero)).max() == 0
    empty = torch.zeros((0,) + tuple(g.sino_shape), device="cuda")
    assert g.fbp(empty).shape == (0,) + tuple(g.volume_shape)


@pytest.mark.parametrize("n", [2, 3])
def test_estimated_isocentre_matches_oracle(ct, n):
    """Without an isocentre both sides estimate it from the detector normals; a shifted orbit
    makes the estimate matter (the distance weights depend on it)."""
    import dataclasses
    base = W.small_config(n)
    views = base.views.copy()
    shift = np.array([2.5, -1.5, 0.75])[: 2 if n == 2 else 3]
    d = len(shift)
    views[:, 0:d] += shift
    views[:, d:2 * d] += shift
    w = dataclasses.replace(base, views=views)
    y = W.random_sinogram(w, 8)
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp(torch_cuda(y)))
    _check(got, _oracle(w, y.astype(np.float64)))
    x = W.random_volume(w, 9)
    got_t = _cpu(g.fbp_transpose(torch_cuda(x)))
    _check(got_t, _oracle_t(w, x.astype(np.float64)))



# ---------------------------------------------------------------------------------------------
# short scans with Parker weights
# ---------------------------------------------------------------------------------------------

def _short_scan(n, margin=0.03):
    """Workload n (2: fan, 3: cone) on a circular orbit spanning pi + 2 delta + margin."""
    import dataclasses
    base = W.small_config(n)
    src = base.views[0, 0:2] if n == 2 else base.views[0, 0:3]
    d = 2 if n == 2 else 3
    sid = float(np.linalg.norm(base.views[0, 0:2]))
    sdd = sid + float(np.linalg.norm(base.views[0, d:d + 2]))
    delta = np.arctan(((base.n_u - 1) / 2.0 * base.du) / sdd)
    span = np.pi + 2 * delta + margin
    nv = base.views.shape[0]
    full = span * nv / (nv - 1)
    views = (W.circular_fan_2d(nv, sid, sdd, span=full) if n == 2 else
             W.circular_cone(nv, sid, sdd, span=full))
    return dataclasses.replace(base, views=views), span


@pytest.mark.parametrize("n", [2, 3])
def test_parker_weights_match_oracle(ct, n):
    w, _ = _short_scan(n)
    g = ct.Geometry.from_workload(w)
    got = g.parker_weights()
    want = F.parker_weights(w.beam, w.views, w.n_u, w.du)
    np.testing.assert_allclose(got, want, atol=2e-6)
    assert got.min() >= 0 and got.max() <= 1 and (got < 0.5).any()


@pytest.mark.parametrize("n", [2, 3])
def test_short_scan_fbp_and_transpose_with_parker_weights(ct, n):
    w, span = _short_scan(n)
    g = ct.Geometry.from_workload(w)
    pw = g.parker_weights()
    vw = np.full(w.views.shape[0], span / (w.views.shape[0] - 1), dtype=np.float32)
    y = W.random_sinogram(w, 12)
    got = _cpu(g.fbp(torch_cuda(y), view_weights=torch_cuda(vw), pixel_weights=torch_cuda(pw)))
    _check(got, _oracle(w, y.astype(np.float64), view_weights=vw.astype(np.float64),
                        pixel_weights=pw.astype(np.float64)))
    x = W.random_volume(w, 13)
    got_t = _cpu(g.fbp_transpose(torch_cuda(x), view_weights=torch_cuda(vw),
                                 pixel_weights=torch_cuda(pw)))
    _check(got_t, _oracle_t(w, x.astype(np.float64), view_weights=vw.astype(np.float64),
                            pixel_weights=pw.astype(np.float64)))


def test_parker_rejects_short_and_non_circular_scans(ct):
    import dataclasses
    w, _ = _short_scan(2, margin=-0.3)
    with pytest.raises(ct.CtError) as ei:
        ct.Geometry.from_workload(w).parker_weights()
    assert ei.value.status == 2
    base = W.small_config(2)
    bad = base.views.copy()
    bad[3, 0:2] *= 1.01
    with pytest.raises(ct.CtError) as ei:
        ct.Geometry.from_workload(dataclasses.replace(base, views=bad)).parker_weights()
    assert ei.value.status == 2



# ---------------------------------------------------------------------------------------------
# caller filter kernels and gradients
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3])
def test_caller_kernel_forward_and_transpose(ct, n):
    """An asymmetric caller kernel: the forward filter uses it as given, the transpose reversed."""
    w = W.small_config(n)
    rng = np.random.default_rng(90 + n)
    kern = (rng.standard_normal(2 * w.n_u - 1) / w.n_u).astype(np.float32)
    y = W.random_sinogram(w, 5)
    x = W.random_volume(w, 6)
    g = ct.Geometry.from_workload(w)
    got = _cpu(g.fbp(torch_cuda(y), kernel=torch_cuda(kern)))
    _check(got, _oracle(w, y.astype(np.float64), kernel=kern.astype(np.float64)))
    got_t = _cpu(g.fbp_transpose(torch_cuda(x), kernel=torch_cuda(kern)))
    _check(got_t, _oracle_t(w, x.astype(np.float64), kernel=kern.astype(np.float64)))


@pytest.mark.parametrize("n", [1, 2, 3])
def test_gradients_match_oracle(ct, n):
    w = W.small_config(n)
    rng = np.random.default_rng(100 + n)
    nv = w.views.shape[0]
    y = W.random_sinogram(w, 7)
    grad = W.random_volume(w, 8)
    wts = rng.uniform(0.01, 0.05, nv).astype(np.float32)
    pw = rng.uniform(0.5, 1.5, (nv, w.n_u)).astype(np.float32)
    kern = (w.du * F.ramp_taps(w.n_u, w.du, "hann")).astype(np.float32)
    iso = (0.4, -0.3, 0.2)[: 2 if n < 3 else 3]
    g = ct.Geometry.from_workload(w)
    gk, gw = g.fbp_gradients(torch_cuda(y), torch_cuda(grad), view_weights=torch_cuda(wts),
                             pixel_weights=torch_cuda(pw), kernel=torch_cuda(kern),
                             isocenter=iso)
    want_k, want_w = F.fbp_gradients(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u,
                                     w.n_v, w.du, w.dv, y.astype(np.float64),
                                     grad.astype(np.float64), kernel=kern.astype(np.float64),
                                     view_weights=wts.astype(np.float64), isocenter=iso,
                                     pixel_weights=pw.astype(np.float64))
    assert rel_l2(_cpu(gk), want_k) < 1e-4
    assert rel_l2(_cpu(gw), want_w) < 1e-4
    # one output at a time gives the same values
    gk2, none = g.fbp_gradients(torch_cuda(y), torch_cuda(grad), view_weights=torch_cuda(wts),
                                pixel_weights=torch_cuda(pw), kernel=torch_cuda(kern),
                                isocenter=iso, want_view_weights=False)
    assert none is None and rel_l2(_cpu(gk2), _cpu(gk)) < 1e-6
