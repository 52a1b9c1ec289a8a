"""B300-native cell-constant Siddon CT projector: forward A, matched adjoint A^T, SIRT, CGLS,
and filtered backprojection (FBP / FDK).

The compute path is the C-ABI library ``libctproj.so`` (CUDA, sm_103a); this package is its
thin ctypes binding plus the seeded input generators in ``workloads``.
"""
from ._binding import (CT_CONE, CT_FAN2D, CT_PARALLEL2D, CT_PARALLEL3D, FBP_WINDOWS, CtError,
                       FbpOptions, ct_fbp_gradients, ct_fbp_gradients_workspace_bytes, fbp_options,
                       Geometry, GeometryInfo, ct_backproject, ct_backproject_batch,
                       ct_backproject_static, ct_batch_workspace_bytes, ct_cgls_iterate,
                       ct_cgls_workspace_bytes, ct_fbp, ct_fbp_parker_weights, ct_fbp_transpose,
                       ct_fbp_transpose_workspace_bytes, ct_fbp_workspace_bytes,
                       ct_geometry_create, ct_geometry_create_surface, ct_geometry_destroy,
                       ct_geometry_set_slabs,
                       ct_geometry_get_info, ct_probe_l1_read, ct_probe_l2_read, ct_probe_l2_reduce, ct_project,
                       ct_project_batch, ct_sirt_iterate,
                       ct_sirt_workspace_bytes, ct_status_string, load_library)

__all__ = ["CT_CONE", "CT_FAN2D", "CT_PARALLEL2D", "CT_PARALLEL3D", "FBP_WINDOWS", "CtError",
           "FbpOptions", "ct_fbp_gradients", "ct_fbp_gradients_workspace_bytes", "fbp_options",
           "Geometry", "GeometryInfo", "ct_backproject", "ct_backproject_batch",
           "ct_backproject_static", "ct_batch_workspace_bytes", "ct_cgls_iterate",
           "ct_cgls_workspace_bytes", "ct_fbp", "ct_fbp_parker_weights", "ct_fbp_transpose",
           "ct_fbp_transpose_workspace_bytes", "ct_fbp_workspace_bytes",
           "ct_geometry_create",
           "ct_geometry_create_surface", "ct_geometry_destroy", "ct_geometry_get_info",
           "ct_geometry_set_slabs",
           "ct_probe_l1_read", "ct_probe_l2_read", "ct_probe_l2_reduce", "ct_project", "ct_project_batch",
           "ct_sirt_iterate", "ct_sirt_workspace_bytes", "ct_status_string", "load_library"]
