"""ctypes binding of ``libctproj.so`` (declared in ``include/ct.h``).

Argument marshalling only: every step of the projector runs in the library's CUDA kernels.
PyTorch is used to allocate device memory and to name the current CUDA stream.  There is no
fallback: if the shared library is missing or cannot be loaded, importing a binding function
raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libctproj.so")

CT_PARALLEL2D, CT_FAN2D, CT_CONE, CT_PARALLEL3D = 0, 1, 2, 3
STATUS_NAMES = ["CT_OK", "CT_ERR_INVALID_ARGUMENT", "CT_ERR_INVALID_GEOMETRY",
                "CT_ERR_NOT_DEVICE_POINTER", "CT_ERR_ALIASING", "CT_ERR_OUT_OF_MEMORY",
                "CT_ERR_CUDA", "CT_ERR_WORKSPACE"]
CT_OK = 0
FBP_WINDOWS = {"ram-lak": 0, "shepp-logan": 1, "cosine": 2, "hamming": 3, "hann": 4}


class CtError(RuntimeError):
    """A libctproj call returned a status other than CT_OK."""

    def __init__(self, status: int, call: str):
        self.status = int(status)
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else f"status {status}"
        super().__init__(f"{call} failed: {name}")


class FbpOptions(ctypes.Structure):
    """``ct_fbp_options``: window code, device pointers (or None) and a host isocentre."""
    _fields_ = [("window", ctypes.c_int32), ("d_view_weights", ctypes.c_void_p),
                ("d_pixel_weights", ctypes.c_void_p), ("d_kernel", ctypes.c_void_p),
                ("isocenter", ctypes.POINTER(ctypes.c_double))]


class GeometryInfo(ctypes.Structure):
    _fields_ = [("beam", ctypes.c_int32), ("n_views", ctypes.c_int32),
                ("nz", ctypes.c_int32), ("ny", ctypes.c_int32), ("nx", ctypes.c_int32),
                ("n_u", ctypes.c_int32), ("n_v", ctypes.c_int32),
                ("volume_layout", ctypes.c_int32),
                ("n_rays", ctypes.c_int64), ("n_voxels", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t), ("sirt_workspace_bytes", ctypes.c_size_t),
                ("n_slabs", ctypes.c_int32), ("slab_cells", ctypes.c_int32),
                ("shared_lines", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libctproj once; raise ImportError if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libctproj.so not built at {path}; run "
                          "`python -m fan_beam_projector_siddon_b300.build` (nvcc, sm_103a)")
    L = ctypes.CDLL(path)
    vp, i32, i64, f32, f64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_float, ctypes.c_double, ctypes.c_size_t)
    L.ct_geometry_create.argtypes = [i32, i32, ctypes.POINTER(f64), i32, i32, i32, f64, i32, i32,
                                     f64, f64, ctypes.POINTER(vp)]
    L.ct_geometry_create.restype = i32
    L.ct_geometry_create_ex.argtypes = [i32, i32, ctypes.POINTER(f64), i32, i32, i32,
                                        ctypes.POINTER(f64), i32, i32, f64, f64,
                                        ctypes.POINTER(vp)]
    L.ct_geometry_create_ex.restype = i32
    L.ct_geometry_create_surface.argtypes = [i32, i32, ctypes.POINTER(f64), i32, i32, i32,
                                             ctypes.POINTER(f64), i32, i32, ctypes.POINTER(f64),
                                             ctypes.POINTER(vp)]
    L.ct_geometry_create_surface.restype = i32
    L.ct_geometry_destroy.argtypes = [vp]
    L.ct_geometry_destroy.restype = i32
    L.ct_geometry_get_info.argtypes = [vp, ctypes.POINTER(GeometryInfo)]
    L.ct_geometry_get_info.restype = i32
    L.ct_geometry_set_slabs.argtypes = [vp, i32]
    L.ct_geometry_set_slabs.restype = i32
    L.ct_project.argtypes = [vp, vp, vp, vp, sz, vp]
    L.ct_project.restype = i32
    L.ct_backproject.argtypes = [vp, vp, vp, vp, sz, vp]
    L.ct_backproject.restype = i32
    L.ct_sirt_workspace_bytes.argtypes = [vp]
    L.ct_sirt_workspace_bytes.restype = sz
    L.ct_sirt_iterate.argtypes = [vp, vp, vp, vp, sz, i32, f32, i32, vp]
    L.ct_sirt_iterate.restype = i32
    L.ct_batch_workspace_bytes.argtypes = [vp, i32]
    L.ct_batch_workspace_bytes.restype = sz
    L.ct_project_batch.argtypes = [vp, i32, vp, vp, vp, sz, vp]
    L.ct_project_batch.restype = i32
    L.ct_backproject_batch.argtypes = [vp, i32, vp, vp, vp, sz, vp]
    L.ct_backproject_batch.restype = i32
    L.ct_cgls_workspace_bytes.argtypes = [vp]
    L.ct_cgls_workspace_bytes.restype = sz
    L.ct_cgls_iterate.argtypes = [vp, vp, vp, vp, sz, i32, i32, vp]
    L.ct_cgls_iterate.restype = i32
    L.ct_backproject_static.argtypes = [vp, vp, vp, vp]
    L.ct_backproject_static.restype = i32
    L.ct_probe_l2_read.argtypes = [vp, sz, i32, vp, vp]
    L.ct_probe_l2_read.restype = i32
    L.ct_probe_l1_read.argtypes = [vp, sz, i32, vp, vp]
    L.ct_probe_l1_read.restype = i32
    L.ct_probe_l2_reduce.argtypes = [vp, sz, i32, i32, vp]
    L.ct_probe_l2_reduce.restype = i32
    L.ct_fbp_workspace_bytes.argtypes = [vp]
    L.ct_fbp_workspace_bytes.restype = sz
    opt = ctypes.POINTER(FbpOptions)
    L.ct_fbp.argtypes = [vp, vp, vp, opt, vp, sz, vp]
    L.ct_fbp.restype = i32
    L.ct_fbp_transpose_workspace_bytes.argtypes = [vp]
    L.ct_fbp_transpose_workspace_bytes.restype = sz
    L.ct_fbp_transpose.argtypes = [vp, vp, vp, opt, vp, sz, vp]
    L.ct_fbp_gradients_workspace_bytes.argtypes = [vp]
    L.ct_fbp_gradients_workspace_bytes.restype = sz
    L.ct_fbp_gradients.argtypes = [vp, vp, vp, opt, vp, vp, vp, sz, vp]
    L.ct_fbp_gradients.restype = i32
    L.ct_fbp_parker_weights.argtypes = [vp, ctypes.POINTER(f64), ctypes.POINTER(ctypes.c_float)]
    L.ct_fbp_parker_weights.restype = i32
    L.ct_fbp_transpose.restype = i32
    L.ct_status_string.argtypes = [i32]
    L.ct_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(status: int, call: str) -> None:
    if status != CT_OK:
        raise CtError(status, call)


# ---- the C entry points, same names, raw pointers ---------------------------------------------

def _spacing_zyx(voxel_spacing):
    if np.ndim(voxel_spacing) == 0:
        s = float(voxel_spacing)
        return (ctypes.c_double * 3)(s, s, s)
    s = [float(x) for x in voxel_spacing]
    return (ctypes.c_double * 3)(*([1.0] + s if len(s) == 2 else s))


def ct_geometry_create_surface(beam: int, views, vol_shape, voxel_spacing, n_u: int, n_v: int,
                               offsets) -> int:
    """Create a handle with a parameterized detector surface: ``offsets`` is (n_u, n_v, 3)
    local (u, v, n) pixel offsets (2D: n_v = 1)."""
    L = load_library()
    v = np.ascontiguousarray(np.asarray(views, dtype=np.float64))
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.float64).reshape(n_u, n_v, 3))
    nz, ny, nx = vol_shape
    h = ctypes.c_void_p()
    dp = ctypes.POINTER(ctypes.c_double)
    _check(L.ct_geometry_create_surface(int(beam), int(v.shape[0]), v.ctypes.data_as(dp),
                                        int(nz), int(ny), int(nx), _spacing_zyx(voxel_spacing),
                                        int(n_u), int(n_v), off.ctypes.data_as(dp),
                                        ctypes.byref(h)), "ct_geometry_create_surface")
    return h.value


def ct_geometry_create(beam: int, views, vol_shape, voxel_spacing, n_u: int, n_v: int,
                       du: float, dv: float) -> int:
    """Create a handle; ``views`` is a host (n_views, 6|12) float64 array; ``voxel_spacing`` a
    scalar (ct_geometry_create) or a tuple in tensor order, (dy, dx) for 2D or (dz, dy, dx) for
    3D (ct_geometry_create_ex).  Returns the handle."""
    L = load_library()
    v = np.ascontiguousarray(np.asarray(views, dtype=np.float64))
    nz, ny, nx = vol_shape
    h = ctypes.c_void_p()
    vp = v.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    if np.ndim(voxel_spacing) == 0:
        _check(L.ct_geometry_create(int(beam), int(v.shape[0]), vp, int(nz), int(ny), int(nx),
                                    float(voxel_spacing), int(n_u), int(n_v), float(du),
                                    float(dv), ctypes.byref(h)), "ct_geometry_create")
    else:
        s = [float(x) for x in voxel_spacing]
        s = [1.0] + s if len(s) == 2 else s
        arr = (ctypes.c_double * 3)(*s)
        _check(L.ct_geometry_create_ex(int(beam), int(v.shape[0]), vp, int(nz), int(ny), int(nx),
                                       arr, int(n_u), int(n_v), float(du), float(dv),
                                       ctypes.byref(h)), "ct_geometry_create_ex")
    return h.value


def ct_geometry_destroy(handle: int) -> None:
    _check(load_library().ct_geometry_destroy(handle), "ct_geometry_destroy")


def ct_geometry_get_info(handle: int) -> GeometryInfo:
    info = GeometryInfo()
    _check(load_library().ct_geometry_get_info(handle, ctypes.byref(info)),
           "ct_geometry_get_info")
    return info


def ct_geometry_set_slabs(handle: int, slab_cells: int) -> None:
    """Slab height of the tiled walks, 0 = no tiling (see ``include/ct.h``)."""
    _check(load_library().ct_geometry_set_slabs(handle, int(slab_cells)), "ct_geometry_set_slabs")


def ct_project(handle: int, d_volume: int, d_sino: int, d_workspace: int | None,
               workspace_bytes: int, stream: int | None) -> None:
    _check(load_library().ct_project(handle, d_volume, d_sino, d_workspace, workspace_bytes,
                                     stream), "ct_project")


def ct_backproject(handle: int, d_sino: int, d_volume: int, d_workspace: int | None,
                   workspace_bytes: int, stream: int | None) -> None:
    _check(load_library().ct_backproject(handle, d_sino, d_volume, d_workspace,
                                         workspace_bytes, stream), "ct_backproject")


def ct_backproject_static(handle: int, d_sino: int, d_volume: int, stream: int | None) -> None:
    """Backprojection without allocation or workspace (see ``include/ct.h``)."""
    _check(load_library().ct_backproject_static(handle, d_sino, d_volume, stream),
           "ct_backproject_static")


def ct_probe_l2_read(d_buf: int, n_floats: int, passes: int, d_sink: int,
                     stream: int | None) -> None:
    """L2 read-bandwidth probe (see ``include/ct.h``)."""
    _check(load_library().ct_probe_l2_read(d_buf, int(n_floats), int(passes), d_sink, stream),
           "ct_probe_l2_read")


def ct_probe_l1_read(d_buf: int, n_floats: int, passes: int, d_sink: int,
                     stream: int | None) -> None:
    """L1 read-bandwidth probe (see ``include/ct.h``)."""
    _check(load_library().ct_probe_l1_read(d_buf, int(n_floats), int(passes), d_sink, stream),
           "ct_probe_l1_read")


def ct_probe_l2_reduce(d_buf: int, n_floats: int, passes: int, stride: int,
                       stream: int | None) -> None:
    """L2 reduction-throughput probe (see ``include/ct.h``)."""
    _check(load_library().ct_probe_l2_reduce(d_buf, int(n_floats), int(passes), int(stride),
                                             stream), "ct_probe_l2_reduce")


def ct_sirt_workspace_bytes(handle: int) -> int:
    return int(load_library().ct_sirt_workspace_bytes(handle))


def ct_sirt_iterate(handle: int, d_x: int, d_y: int, d_workspace: int, workspace_bytes: int,
                    n_iters: int, relaxation: float, workspace_initialised: bool,
                    stream: int | None) -> None:
    _check(load_library().ct_sirt_iterate(handle, d_x, d_y, d_workspace, workspace_bytes,
                                          int(n_iters), float(relaxation),
                                          1 if workspace_initialised else 0, stream),
           "ct_sirt_iterate")


def ct_batch_workspace_bytes(handle: int, batch: int) -> int:
    return int(load_library().ct_batch_workspace_bytes(handle, int(batch)))


def ct_project_batch(handle: int, batch: int, d_volumes: int, d_sinos: int,
                     d_workspace: int | None, workspace_bytes: int, stream: int | None) -> None:
    _check(load_library().ct_project_batch(handle, int(batch), d_volumes, d_sinos, d_workspace,
                                           workspace_bytes, stream), "ct_project_batch")


def ct_backproject_batch(handle: int, batch: int, d_sinos: int, d_volumes: int,
                         d_workspace: int | None, workspace_bytes: int,
                         stream: int | None) -> None:
    _check(load_library().ct_backproject_batch(handle, int(batch), d_sinos, d_volumes,
                                               d_workspace, workspace_bytes, stream),
           "ct_backproject_batch")


def ct_cgls_workspace_bytes(handle: int) -> int:
    return int(load_library().ct_cgls_workspace_bytes(handle))


def ct_cgls_iterate(handle: int, d_x: int, d_y: int, d_workspace: int, workspace_bytes: int,
                    n_iters: int, workspace_initialised: bool, stream: int | None) -> None:
    _check(load_library().ct_cgls_iterate(handle, d_x, d_y, d_workspace, workspace_bytes,
                                          int(n_iters), 1 if workspace_initialised else 0,
                                          stream), "ct_cgls_iterate")


def ct_fbp_workspace_bytes(handle: int) -> int:
    return int(load_library().ct_fbp_workspace_bytes(handle))


def _fbp_args(isocenter, window):
    code = FBP_WINDOWS[window] if isinstance(window, str) else int(window)
    iso = None
    if isocenter is not None:
        arr = np.zeros(3, dtype=np.float64)
        vals = np.asarray(isocenter, dtype=np.float64).ravel()
        arr[:len(vals)] = vals
        iso = arr
    return code, iso


def _dptr(arr):
    return None if arr is None else arr.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def fbp_options(window="ram-lak", d_view_weights: int | None = None,
                d_pixel_weights: int | None = None, d_kernel: int | None = None,
                isocenter=None):
    """(FbpOptions, keep-alive) for the FBP calls; keep the second item alive during the call."""
    code, iso = _fbp_args(isocenter, window)
    o = FbpOptions(code, d_view_weights, d_pixel_weights, d_kernel, _dptr(iso))
    return o, iso


def ct_fbp(handle: int, d_sino: int, d_volume: int, options: "FbpOptions | None",
           d_workspace: int, workspace_bytes: int, stream: int | None) -> None:
    """Filtered backprojection with ``options`` (``fbp_options(...)[0]``, or None for the
    defaults)."""
    _check(load_library().ct_fbp(handle, d_sino, d_volume,
                                 None if options is None else ctypes.byref(options),
                                 d_workspace, workspace_bytes, stream), "ct_fbp")


def ct_fbp_transpose_workspace_bytes(handle: int) -> int:
    return int(load_library().ct_fbp_transpose_workspace_bytes(handle))


def ct_fbp_transpose(handle: int, d_volume: int, d_sino: int, options: "FbpOptions | None",
                     d_workspace: int, workspace_bytes: int, stream: int | None) -> None:
    """Transpose of ``ct_fbp`` (volume -> sinogram), same options."""
    _check(load_library().ct_fbp_transpose(handle, d_volume, d_sino,
                                           None if options is None else ctypes.byref(options),
                                           d_workspace, workspace_bytes, stream),
           "ct_fbp_transpose")


def ct_fbp_gradients_workspace_bytes(handle: int) -> int:
    return int(load_library().ct_fbp_gradients_workspace_bytes(handle))


def ct_fbp_gradients(handle: int, d_sino: int, d_grad_volume: int,
                     options: "FbpOptions | None", d_grad_kernel: int | None,
                     d_grad_view_weights: int | None, d_workspace: int, workspace_bytes: int,
                     stream: int | None) -> None:
    """dL/dkernel and dL/dview_weights of the FBP of ``d_sino`` given dL/df = ``d_grad_volume``."""
    _check(load_library().ct_fbp_gradients(handle, d_sino, d_grad_volume,
                                           None if options is None else ctypes.byref(options),
                                           d_grad_kernel, d_grad_view_weights, d_workspace,
                                           workspace_bytes, stream), "ct_fbp_gradients")


def ct_fbp_parker_weights(handle: int, n_views: int, n_u: int, isocenter=None) -> np.ndarray:
    """Parker short-scan weights, a host (n_views, n_u) float32 array."""
    _, iso = _fbp_args(isocenter, 0)
    out = np.empty((n_views, n_u), dtype=np.float32)
    _check(load_library().ct_fbp_parker_weights(
        handle, _dptr(iso), out.ctypes.data_as(ctypes.POINTER(ctypes.c_float))),
        "ct_fbp_parker_weights")
    return out


def ct_status_string(status: int) -> str:
    return load_library().ct_status_string(int(status)).decode()


# ---- a small object wrapper over torch tensors -------------------------------------------------

class Geometry:
    """Owns one ``ct_geometry`` handle; methods take and return CUDA float32 torch tensors."""

    def __init__(self, beam: int, views, vol_shape, voxel_spacing, n_u: int, n_v: int,
                 du: float, dv: float, offsets=None):
        if offsets is None:
            self.handle = ct_geometry_create(beam, views, vol_shape, voxel_spacing, n_u, n_v, du,
                                             dv)
        else:
            self.handle = ct_geometry_create_surface(beam, views, vol_shape, voxel_spacing, n_u,
                                                     n_v, offsets)
        self.info = ct_geometry_get_info(self.handle)
        self.beam = int(beam)
        self.is_2d = self.beam in (CT_PARALLEL2D, CT_FAN2D)

    @classmethod
    def from_workload(cls, w) -> "Geometry":
        return cls(w.beam, w.views, w.vol_shape, w.voxel_spacing, w.n_u, w.n_v, w.du, w.dv,
                   getattr(w, "offsets", None))

    def set_slabs(self, slab_cells: int) -> None:
        """Override the slab tiling of the walks (0 = off); refreshes ``info``."""
        ct_geometry_set_slabs(self.handle, slab_cells)
        self.info = ct_geometry_get_info(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            ct_geometry_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def volume_shape(self):
        i = self.info
        return (i.ny, i.nx) if self.is_2d else (i.nz, i.ny, i.nx)

    @property
    def sino_shape(self):
        i = self.info
        return (i.n_views, i.n_u) if self.is_2d else (i.n_views, i.n_u, i.n_v)

    @property
    def workspace_bytes(self) -> int:
        return int(self.info.workspace_bytes)

    @property
    def sirt_workspace_bytes(self) -> int:
        return int(self.info.sirt_workspace_bytes)

    @property
    def cgls_workspace_bytes(self) -> int:
        return ct_cgls_workspace_bytes(self.handle)

    def new_workspace(self, sirt: bool = False, cgls: bool = False):
        import torch
        n = (self.cgls_workspace_bytes if cgls else
             self.sirt_workspace_bytes if sirt else self.workspace_bytes)
        return torch.empty(max(n, 1), dtype=torch.uint8, device="cuda") if n else None

    @staticmethod
    def _stream(stream):
        import torch
        s = torch.cuda.current_stream() if stream is None else stream
        return s.cuda_stream

    def _ws(self, workspace, sirt=False):
        need = self.sirt_workspace_bytes if sirt else self.workspace_bytes
        if need == 0:
            return None, 0
        if workspace is None:
            workspace = self.new_workspace(sirt)
        return workspace.data_ptr(), workspace.numel() * workspace.element_size()

    def _batch_ws(self, batch, workspace):
        need = ct_batch_workspace_bytes(self.handle, batch)
        if need == 0:
            return None, 0
        if workspace is None:
            import torch
            workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
        return workspace.data_ptr(), workspace.numel() * workspace.element_size()

    def project(self, volume, out=None, workspace=None, stream=None):
        """A volume -> sinogram; leading batch/channel dimensions are kept."""
        import torch
        assert volume.is_cuda and volume.dtype == torch.float32 and volume.is_contiguous()
        nd = len(self.volume_shape)
        assert tuple(volume.shape[volume.dim() - nd:]) == tuple(self.volume_shape)
        lead = tuple(volume.shape[:volume.dim() - nd])
        if out is None:
            out = torch.empty(lead + tuple(self.sino_shape), dtype=torch.float32,
                              device=volume.device)
        batch = int(np.prod(lead)) if lead else 0
        if batch == 0 and lead:
            return out
        if not lead:
            ws, wsb = self._ws(workspace)
            ct_project(self.handle, volume.data_ptr(), out.data_ptr(), ws, wsb,
                       self._stream(stream))
        else:
            ws, wsb = self._batch_ws(batch, workspace)
            ct_project_batch(self.handle, batch, volume.data_ptr(), out.data_ptr(), ws, wsb,
                             self._stream(stream))
        return out

    def backproject(self, sino, out=None, workspace=None, stream=None):
        """A^T sinogram -> volume; leading batch/channel dimensions are kept."""
        import torch
        assert sino.is_cuda and sino.dtype == torch.float32 and sino.is_contiguous()
        nd = len(self.sino_shape)
        assert tuple(sino.shape[sino.dim() - nd:]) == tuple(self.sino_shape)
        lead = tuple(sino.shape[:sino.dim() - nd])
        if out is None:
            out = torch.empty(lead + tuple(self.volume_shape), dtype=torch.float32,
                              device=sino.device)
        batch = int(np.prod(lead)) if lead else 0
        if batch == 0 and lead:
            return out
        if not lead:
            ws, wsb = self._ws(workspace)
            ct_backproject(self.handle, sino.data_ptr(), out.data_ptr(), ws, wsb,
                           self._stream(stream))
        else:
            ws, wsb = self._batch_ws(batch, workspace)
            ct_backproject_batch(self.handle, batch, sino.data_ptr(), out.data_ptr(), ws, wsb,
                                 self._stream(stream))
        return out

    def cgls(self, x, y, n_iters: int, workspace, initialised: bool, stream=None):
        """``n_iters`` CGLS steps on ``x`` in place; ``workspace`` carries the state between
        calls (``initialised=False`` on the first call)."""
        import torch
        assert x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()
        assert y.is_cuda and y.dtype == torch.float32 and y.is_contiguous()
        ws, wsb = workspace.data_ptr(), workspace.numel() * workspace.element_size()
        ct_cgls_iterate(self.handle, x.data_ptr(), y.data_ptr(), ws, wsb, n_iters, initialised,
                        self._stream(stream))
        return x

    def sirt(self, x, y, n_iters: int, workspace, initialised: bool, relaxation: float = 1.0,
             stream=None):
        """``n_iters`` SIRT updates of ``x`` in place; ``workspace`` caches C between calls."""
        import torch
        assert x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()
        assert y.is_cuda and y.dtype == torch.float32 and y.is_contiguous()
        ws, wsb = workspace.data_ptr(), workspace.numel() * workspace.element_size()
        ct_sirt_iterate(self.handle, x.data_ptr(), y.data_ptr(), ws, wsb, n_iters, relaxation,
                        initialised, self._stream(stream))
        return x

    def _fbp_inputs(self, device, view_weights, pixel_weights, kernel):
        """Device float32 tensors (or None) for the optional FBP inputs, checked for size."""
        import torch
        out = []
        for t, n in ((view_weights, self.info.n_views),
                     (pixel_weights, self.info.n_views * self.info.n_u),
                     (kernel, 2 * self.info.n_u - 1)):
            if t is not None:
                t = torch.as_tensor(t, dtype=torch.float32, device=device).contiguous()
                assert t.numel() == n
            out.append(t)
        return out

    def _fbp_call(self, fn, need, src, src_shape, dst_shape, out, window, view_weights,
                  isocenter, workspace, stream, pixel_weights=None, kernel=None):
        import torch
        assert src.is_cuda and src.dtype == torch.float32 and src.is_contiguous()
        nd = len(src_shape)
        assert tuple(src.shape[src.dim() - nd:]) == tuple(src_shape)
        lead = tuple(src.shape[:src.dim() - nd])
        if out is None:
            out = torch.empty(lead + tuple(dst_shape), dtype=torch.float32, device=src.device)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=src.device)
        ws, wsb = workspace.data_ptr(), workspace.numel() * workspace.element_size()
        vw, pw, kn = self._fbp_inputs(src.device, view_weights, pixel_weights, kernel)
        opts, keep = fbp_options(window, None if vw is None else vw.data_ptr(),
                                 None if pw is None else pw.data_ptr(),
                                 None if kn is None else kn.data_ptr(), isocenter)
        s2 = src.reshape((-1,) + tuple(src_shape))
        o2 = out.view((-1,) + tuple(dst_shape))
        for b in range(s2.shape[0]):
            fn(self.handle, s2[b].data_ptr(), o2[b].data_ptr(), opts, ws, wsb,
               self._stream(stream))
        del keep
        return out

    def fbp(self, sino, out=None, window="ram-lak", view_weights=None, isocenter=None,
            workspace=None, stream=None, pixel_weights=None, kernel=None):
        """Filtered backprojection (FBP / FDK) of a sinogram; leading dimensions are kept and
        reconstructed one after another with the same workspace.  ``kernel`` (2 n_u - 1 values)
        replaces the windowed ramp."""
        return self._fbp_call(ct_fbp, ct_fbp_workspace_bytes(self.handle), sino,
                              self.sino_shape, self.volume_shape, out, window, view_weights,
                              isocenter, workspace, stream, pixel_weights, kernel)

    def fbp_transpose(self, volume, out=None, window="ram-lak", view_weights=None,
                      isocenter=None, workspace=None, stream=None, pixel_weights=None,
                      kernel=None):
        """Transpose of ``fbp`` (volume -> sinogram); leading dimensions are kept."""
        return self._fbp_call(ct_fbp_transpose, ct_fbp_transpose_workspace_bytes(self.handle),
                              volume, self.volume_shape, self.sino_shape, out, window,
                              view_weights, isocenter, workspace, stream, pixel_weights, kernel)

    def fbp_gradients(self, sino, grad_volume, window="ram-lak", view_weights=None,
                      isocenter=None, pixel_weights=None, kernel=None, want_kernel=True,
                      want_view_weights=True, workspace=None, stream=None):
        """(dL/dkernel, dL/dview_weights) of ``fbp(sino, ...)`` given dL/df = ``grad_volume``;
        an entry is None when not wanted."""
        import torch
        for t, shape in ((sino, self.sino_shape), (grad_volume, self.volume_shape)):
            assert t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()
            assert tuple(t.shape) == tuple(shape)
        dev = sino.device
        if workspace is None:
            workspace = torch.empty(ct_fbp_gradients_workspace_bytes(self.handle),
                                    dtype=torch.uint8, device=dev)
        vw, pw, kn = self._fbp_inputs(dev, view_weights, pixel_weights, kernel)
        opts, keep = fbp_options(window, None if vw is None else vw.data_ptr(),
                                 None if pw is None else pw.data_ptr(),
                                 None if kn is None else kn.data_ptr(), isocenter)
        gk = torch.empty(2 * self.info.n_u - 1, device=dev) if want_kernel else None
        gw = torch.empty(self.info.n_views, device=dev) if want_view_weights else None
        ct_fbp_gradients(self.handle, sino.data_ptr(), grad_volume.data_ptr(), opts,
                         None if gk is None else gk.data_ptr(),
                         None if gw is None else gw.data_ptr(), workspace.data_ptr(),
                         workspace.numel(), self._stream(stream))
        del keep
        return gk, gw

    def parker_weights(self, isocenter=None) -> np.ndarray:
        """Parker short-scan weights (n_views, n_u) for ``fbp(..., pixel_weights=)``."""
        return ct_fbp_parker_weights(self.handle, self.info.n_views, self.info.n_u, isocenter)
