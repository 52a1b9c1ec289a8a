"""The C ABI driven from a plain C program (tests/c/abi_check.c: raw device pointers, its own
CUDA runtime and stream), compared with the ctypes binding on the same seeded inputs."""
import os
import subprocess

import numpy as np
import pytest

from tests._parity import rel_l2, torch_cuda
from tests.test_abi_cpu import build_c_check

pytestmark = pytest.mark.gpu


def test_c_program_matches_the_binding(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fan_beam_projector_siddon_b300 as ct
    exe = build_c_check(tmp_path)
    out = tmp_path / "abi_check.bin"
    r = subprocess.run([exe, str(out)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.stdout, r.stderr)
    nv, nz, ny, nx, nu, nvv = 12, 20, 24, 28, 40, 30
    raw = open(out, "rb").read()
    views = np.frombuffer(raw, dtype=np.float64, count=nv * 12).reshape(nv, 12).copy()
    rest = np.frombuffer(raw, dtype=np.float32, offset=nv * 12 * 8)
    nvox, nray = nz * ny * nx, nv * nu * nvv
    vol = rest[:nvox].reshape(nz, ny, nx).copy()
    sino_c = rest[nvox:nvox + nray].reshape(nv, nu, nvv).copy()
    back_c = rest[nvox + nray:].reshape(nz, ny, nx).copy()
    g = ct.Geometry(ct.CT_CONE, views, (nz, ny, nx), 1.0, nu, nvv, 1.5, 1.5)
    sino = g.project(torch_cuda(vol)).cpu().numpy()
    assert np.array_equal(sino, sino_c)
    back = g.backproject(torch_cuda(sino_c)).cpu().numpy()
    assert rel_l2(back, back_c) < 1e-6
    assert np.abs(sino_c).max() > 0
