"""The compute calls are asynchronous, allocate nothing and never synchronise, so a caller can
capture them into a CUDA graph once and replay it: replays must reproduce the eager results
(forward bit for bit; atomic backprojections to float32 rounding)."""
import numpy as np
import pytest

from fan_beam_projector_siddon_b300 import workloads as W
from tests._parity import rel_l2, torch_cuda

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


def _capture(torch, fn):
    """Capture fn() on a side stream (after one eager warm-up call there) into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        fn()
    return graph


@pytest.mark.parametrize("n", [1, 3])
def test_project_backproject_graph_replay(ct, n):
    import torch
    w = W.small_config(n)
    g = ct.Geometry.from_workload(w)
    vol = torch_cuda(w.phantom())
    sino = torch.empty(g.sino_shape, device="cuda")
    back = torch.empty(g.volume_shape, device="cuda")
    ws = g.new_workspace()

    def step():
        g.project(vol, out=sino, workspace=ws)
        g.backproject(sino, out=back, workspace=ws)

    step()
    torch.cuda.synchronize()
    sino_eager, back_eager = sino.clone(), back.clone()
    graph = _capture(torch, step)
    for _ in range(3):
        sino.zero_()
        back.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(sino, sino_eager)
    assert rel_l2(back.cpu().numpy(), back_eager.cpu().numpy()) < 1e-6
    # new inputs in the captured buffers flow through the replay
    vol.mul_(2.0)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.allclose(sino, 2.0 * sino_eager, rtol=1e-6, atol=0)


def test_sirt_and_cgls_graph_replay(ct):
    import torch
    w = W.small_config(3)
    g = ct.Geometry.from_workload(w)
    y = g.project(torch_cuda(w.phantom()))
    # eager: initialise, then 4 iterations
    x_e = torch.zeros(g.volume_shape, device="cuda")
    ws_e = g.new_workspace(sirt=True)
    g.sirt(x_e, y, 0, ws_e, initialised=False)
    g.sirt(x_e, y, 4, ws_e, initialised=True)
    # graph: initialise eagerly, capture 2 iterations, replay twice
    x = torch.zeros(g.volume_shape, device="cuda")
    ws = g.new_workspace(sirt=True)
    g.sirt(x, y, 0, ws, initialised=False)
    torch.cuda.synchronize()
    x_start = x.clone()
    graph = _capture(torch, lambda: g.sirt(x, y, 2, ws, initialised=True))
    x.copy_(x_start)      # undo the warm-up call's 2 iterations (C and b are unchanged)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert rel_l2(x.cpu().numpy(), x_e.cpu().numpy()) < 1e-5
    # CGLS: one captured iteration replayed after eager initialisation
    xc_e = torch.zeros(g.volume_shape, device="cuda")
    wc_e = g.new_workspace(cgls=True)
    g.cgls(xc_e, y, 3, wc_e, initialised=False)
    xc = torch.zeros(g.volume_shape, device="cuda")
    wc = g.new_workspace(cgls=True)
    g.cgls(xc, y, 1, wc, initialised=False)
    torch.cuda.synchronize()
    graph = _capture(torch, lambda: g.cgls(xc, y, 1, wc, initialised=True))
    # the warm-up inside _capture already took step 2; one replay takes step 3
    graph.replay()
    torch.cuda.synchronize()
    assert rel_l2(xc.cpu().numpy(), xc_e.cpu().numpy()) < 1e-4


def test_fdk_graph_replay(ct):
    import torch
    w = W.small_config(3)
    g = ct.Geometry.from_workload(w)
    y = torch_cuda(W.random_sinogram(w, 2))
    out = torch.empty(g.volume_shape, device="cuda")
    ws = torch.empty(ct.ct_fbp_workspace_bytes(g.handle), dtype=torch.uint8, device="cuda")
    g.fbp(y, out=out, workspace=ws)
    torch.cuda.synchronize()
    eager = out.clone()
    graph = _capture(torch, lambda: g.fbp(y, out=out, workspace=ws))
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
