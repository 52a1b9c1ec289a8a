"""The backprojection entry point that allocates nothing (ct_backproject_static).

It serves callers that cannot allocate device memory when they backproject (a plugin handed only
a stream and its buffers, a real-time loop that forbids allocation after start-up, a program
that keeps all device memory in its own pool).  Its scratch is one static device array shared by
every call, so these tests check it against ct_backproject on two calls in a row with different
sinograms: a second call that saw the first call's sums would fail.  This file is collected last
so that a run stopping at the first failure has run every other test before it.
"""
import numpy as np
import pytest

from fan_beam_projector_siddon_b300 import workloads as W
from tests._parity import BP_RTOL, rel_l2, torch_cuda

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


# (workload, whether its internal volume order differs from the caller's): the cone and spiral
# twins walk a z-fastest volume, so their sums go through the static array; the tilt-series and
# 2D twins keep the caller's order and accumulate straight into the output
@pytest.mark.parametrize("n,uses_array", [(3, True), (4, True), (5, False), (1, False)])
def test_static_backprojection_matches_workspace_entry_point(ct, n, uses_array):
    import torch
    w = W.small_config(n)
    g = ct.Geometry.from_workload(w)
    assert (g.info.volume_layout != 0) == uses_array
    assert g.info.n_voxels <= (1 << 22)
    stream = torch.cuda.current_stream().cuda_stream
    for seed in (11, 12):                        # two calls in a row, different inputs
        y = torch_cuda(W.random_sinogram(w, seed))
        want = g.backproject(y)
        got = torch.full(w.volume_shape, float("nan"), device="cuda")
        ct.ct_backproject_static(g.handle, y.data_ptr(), got.data_ptr(), stream)
        torch.cuda.synchronize()
        assert rel_l2(got.cpu().numpy(), want.cpu().numpy()) <= BP_RTOL


def test_static_backprojection_rejects_volumes_beyond_its_array(ct):
    import torch
    w = W.config(3)                              # 256^3 voxels, z-fastest order: needs scratch
    g = ct.Geometry.from_workload(w)
    assert g.info.volume_layout != 0 and g.info.n_voxels > (1 << 22)
    y = torch.zeros(w.sino_shape, device="cuda")
    out = torch.zeros(w.volume_shape, device="cuda")
    with pytest.raises(ct.CtError) as e:
        ct.ct_backproject_static(g.handle, y.data_ptr(), out.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert e.value.status == 7
