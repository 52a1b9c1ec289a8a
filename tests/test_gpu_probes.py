"""The L2 roofline probes (ct_probe_l2_read, ct_probe_l2_reduce) do exactly the work they
declare: the reduction probe adds `passes` to every float it covers and nothing elsewhere, the
read probe leaves its buffer and its sink untouched."""
import numpy as np
import pytest

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


@pytest.mark.parametrize("stride", [1, 2, 8])
def test_reduce_probe_adds_passes_to_every_covered_float(ct, stride):
    import torch
    n = (1 << 20) + 37                       # a ragged tail the sweep does not cover
    buf = torch.zeros(n, device="cuda")
    ct.ct_probe_l2_reduce(buf.data_ptr(), n, 3, stride, None)
    torch.cuda.synchronize()
    got = buf.cpu().numpy()
    span = 32 * stride
    want = np.zeros(n, np.float32)
    covered = (n // span) * span
    want[:covered:stride] = 3.0
    assert np.array_equal(got, want)


def test_read_probe_writes_nothing(ct):
    import torch
    n = (1 << 20) + 6
    buf = torch.rand(n, device="cuda")
    ref = buf.clone()
    sink = torch.full((1,), 7.0, device="cuda")
    ct.ct_probe_l2_read(buf.data_ptr(), n, 2, sink.data_ptr(), None)
    torch.cuda.synchronize()
    assert torch.equal(buf, ref) and float(sink.item()) == 7.0


def test_l1_read_probe_writes_nothing(ct):
    import torch
    buf = torch.rand(4096, device="cuda")
    ref = buf.clone()
    sink = torch.full((1,), 7.0, device="cuda")
    ct.ct_probe_l1_read(buf.data_ptr(), 4096, 3, sink.data_ptr(), None)
    torch.cuda.synchronize()
    assert torch.equal(buf, ref) and float(sink.item()) == 7.0
    with pytest.raises(ct.CtError):
        ct.ct_probe_l1_read(buf.data_ptr(), 16385, 1, sink.data_ptr(), None)
