"""Host-side checks of the C ABI that need no GPU: build, load, exported symbols, admission."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

from fan_beam_projector_siddon_b300 import build as ct_build
from fan_beam_projector_siddon_b300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ct_build.build()
    import fan_beam_projector_siddon_b300 as ct
    return ct


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"CT_API\s+[^;(]*?\b(ct_\w+)\s*\(", text, flags=re.S))
    return names


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert {"ct_geometry_create", "ct_project", "ct_backproject", "ct_sirt_iterate"} <= declared
    so = ctypes.CDLL(ct_build.LIB)
    for name in sorted(declared):
        assert hasattr(so, name), f"{name} declared in include/ but not exported"


def test_status_strings(lib):
    assert lib.ct_status_string(0) == "CT_OK"
    assert lib.ct_status_string(2) == "CT_ERR_INVALID_GEOMETRY"
    assert lib.ct_status_string(99) == "CT_ERR_UNKNOWN"


def _expect(lib, status, fn, *args):
    with pytest.raises(lib.CtError) as ei:
        fn(*args)
    assert ei.value.status == status, str(ei.value)


def test_admission_rejects_bad_geometry_before_touching_the_gpu(lib):
    INV_GEOM, INV_ARG = 2, 1
    w = W.config(3)
    create = lib.ct_geometry_create
    args = lambda views: (W.CONE, views, w.vol_shape, 1.0, 384, 384, 1.2, 1.2)
    bad = w.views.copy(); bad[5, 0] = math.nan                       # non-finite
    _expect(lib, INV_GEOM, create, *args(bad))
    bad = w.views.copy(); bad[5, 6:9] *= 1.01                        # det_u not unit
    _expect(lib, INV_GEOM, create, *args(bad))
    bad = w.views.copy(); bad[5, 9:12] = bad[5, 6:9]                 # det_u not orthogonal to v
    _expect(lib, INV_GEOM, create, *args(bad))
    bad = w.views.copy(); bad[5, 0:3] = bad[5, 3:6]                  # source on detector centre
    _expect(lib, INV_GEOM, create, *args(bad))
    bad = w.views.copy(); bad[5, 0:3] = bad[5, 3:6] + 10 * bad[5, 6:9]   # edge-on detector
    _expect(lib, INV_GEOM, create, *args(bad))
    bad = w.views.copy(); bad[5, 0:6] *= 1e7                         # both endpoints too far
    _expect(lib, INV_GEOM, create, *args(bad))
    # parallel3d: ray tangent to the detector plane
    p = W.config(5).views.copy(); p[3, 0:3] = p[3, 6:9]
    _expect(lib, INV_GEOM, create, W.PARALLEL3D, p, (8, 8, 8), 1.0, 8, 8, 1.0, 1.0)
    # 2D parallel: ray_dir not orthogonal to det_u
    q = W.circular_parallel_2d(4); q[1, 4:6] = q[1, 0:2]
    _expect(lib, INV_GEOM, create, W.PARALLEL2D, q, (1, 8, 8), 1.0, 8, 1, 1.0, 1.0)
    # sizes
    _expect(lib, INV_ARG, create, W.CONE, w.views, (0, 4, 4), 1.0, 4, 4, 1.0, 1.0)
    _expect(lib, INV_ARG, create, W.CONE, w.views, (2048, 1024, 1024), 1.0, 4, 4, 1.0, 1.0)
    _expect(lib, INV_ARG, create, W.CONE, w.views[:0], (4, 4, 4), 1.0, 4, 4, 1.0, 1.0)
    _expect(lib, INV_ARG, create, W.CONE, w.views, (4, 4, 4), -1.0, 4, 4, 1.0, 1.0)
    _expect(lib, INV_ARG, create, W.CONE, w.views, (4, 4, 4), 1.0, 4, 4, 0.0, 1.0)
    _expect(lib, INV_ARG, create, W.FAN2D, W.config(2).views, (2, 8, 8), 1.0, 8, 1, 1.0, 1.0)
    _expect(lib, INV_ARG, create, W.FAN2D, W.config(2).views, (1, 8, 8), 1.0, 8, 3, 1.0, 1.0)
    _expect(lib, INV_ARG, create, 7, w.views, (4, 4, 4), 1.0, 4, 4, 1.0, 1.0)


def test_null_arguments_are_rejected(lib):
    L = lib.load_library()
    assert L.ct_project(None, None, None, None, 0, None) == 1
    assert L.ct_backproject(None, None, None, None, 0, None) == 1
    assert L.ct_sirt_iterate(None, None, None, None, 0, 1, 1.0, 0, None) == 1
    assert L.ct_geometry_destroy(None) == 0
    assert L.ct_sirt_workspace_bytes(None) == 0
    assert L.ct_fbp(None, None, None, None, None, 0, None) == 1
    assert L.ct_fbp_workspace_bytes(None) == 0
    assert L.ct_fbp_transpose(None, None, None, None, None, 0, None) == 1
    assert L.ct_fbp_gradients(None, None, None, None, None, None, None, 0, None) == 1
    assert L.ct_fbp_gradients_workspace_bytes(None) == 0
    assert L.ct_fbp_parker_weights(None, None, None) == 1
    assert L.ct_fbp_transpose_workspace_bytes(None) == 0
    assert L.ct_probe_l2_read(None, 1024, 1, None, None) == 1
    assert L.ct_probe_l2_reduce(None, 1024, 1, 1, None) == 1
    assert L.ct_probe_l2_reduce(16, 1024, 1, 0, None) == 1       # stride out of range
    assert L.ct_probe_l2_reduce(16, 1024, 0, 1, None) == 1       # no passes
    assert L.ct_probe_l2_read(8, 1024, 1, 16, None) == 1          # not 16-byte aligned


def test_surface_admission_before_touching_the_gpu(lib):
    """Surface detectors are checked pixel by pixel on the host: non-finite offsets and a pixel
    on the source are rejected as invalid geometry."""
    w = W.curved_config("cone")
    bad = w.offsets.copy()
    bad[3, 4, 2] = np.nan
    _expect(lib, 2, lib.ct_geometry_create_surface, w.beam, w.views, w.vol_shape,
            w.voxel_spacing, w.n_u, w.n_v, bad)
    bad = w.offsets.copy()
    src, ctr, u, v = w.views[0, 0:3], w.views[0, 3:6], w.views[0, 6:9], w.views[0, 9:12]
    rel = src - ctr
    bad[0, 0] = [rel @ u, rel @ v, rel @ np.cross(u, v)]
    _expect(lib, 2, lib.ct_geometry_create_surface, w.beam, w.views, w.vol_shape,
            w.voxel_spacing, w.n_u, w.n_v, bad)
    # per-axis spacing: non-positive pitches are bad arguments
    c = W.anisotropic_config("cone")
    _expect(lib, 1, lib.ct_geometry_create, c.beam, c.views, c.vol_shape, (1.0, 0.0, 1.0),
            c.n_u, c.n_v, c.du, c.dv)


def test_header_is_strict_c99(tmp_path):
    """include/ct.h is a C header: it compiles alone under gcc -std=c99 -pedantic -Werror."""
    import subprocess
    src = tmp_path / "hdr.c"
    src.write_text('#include "ct.h"\nint main(void) { return (int)sizeof(ct_geometry_info) == 0; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-c",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o",
                        str(tmp_path / "hdr.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def build_c_check(out_dir):
    """Compile and link tests/c/abi_check.c against libctproj.so and the CUDA runtime."""
    import subprocess
    ct_build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = os.path.join(str(out_dir), "abi_check")
    pkg = os.path.dirname(ct_build.LIB)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O1",
           os.path.join(ROOT, "tests", "c", "abi_check.c"), "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), "-L", pkg, "-lctproj",
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm", "-Wl,-rpath," + pkg,
           "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_links_against_the_library(tmp_path):
    assert os.path.exists(build_c_check(tmp_path))
