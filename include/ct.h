/*
 * ct.h -- C ABI of libctproj: the cell-constant Siddon CT forward projector A, its matched
 * adjoint A^T, SIRT and CGLS built on the pair, batched volumes, per-axis voxel pitches,
 * parameterised detector surfaces, and filtered backprojection (FBP/FDK, short scans) with its
 * transpose, for one NVIDIA B300 (sm_103a).
 *
 * Operator (diffct documentation, "Differentiable analytical reconstruction", first paragraph:
 * "cell-constant Siddon forward operator and its matched adjoint"; "Trajectories and Geometry",
 * detector-surface section: one ray per detector pixel, no detector-area integration):
 *
 *     y_ray = sum_v x_v * l_v(ray)          (A, ct_project)
 *     b_v   = sum_ray y_ray * l_v(ray)      (A^T, ct_backproject)
 *
 * where l_v is the physical length of the ray inside voxel v of a piecewise-constant volume
 * (half-open cells: a ray that lies exactly in a cell face belongs to the cell on the + side).
 *
 * Frame (diffct "Trajectories and Geometry", trajectory-format table and pixel formula):
 * Cartesian (x, y[, z]), origin at the volume centre, one length unit for positions and both
 * spacings.  Voxel i of an axis with n cells spans [-n s/2 + i s, -n s/2 + (i+1) s).
 * Detector pixel (u, v) lies at
 *     det_center + (u - (U-1)/2) du det_u + (v - (V-1)/2) dv det_v.
 * Parallel beams: the ray is the infinite line through the pixel along ray_dir.
 * Fan/cone beams: the ray is the segment from the source to the pixel.
 *
 * Layouts (all float32, C order, device memory owned by the caller):
 *     volume    3D [z][y][x] = (nz, ny, nx);  2D [y][x] = (ny, nx)
 *     sinogram  3D [view][u][v] (v fastest);  2D [view][u]
 *
 * Threading and streams: a geometry handle is immutable after creation; calls on different
 * streams may share a handle, but not a workspace.  Every compute call is asynchronous on the
 * given stream (NULL = legacy default stream), allocates nothing and never synchronises, so the
 * projector, SIRT, CGLS and FBP calls can be recorded into a CUDA graph by stream capture
 * (thread-local capture mode) and replayed; a replay reads the buffers' current contents.
 * A handle is bound to the device that was current when it was created: every compute call
 * must be made with that device current, else it returns CT_ERR_INVALID_ARGUMENT before
 * queueing anything.
 * Asynchronous CUDA errors surface as CT_ERR_CUDA on a later call.  No call aborts the process.
 */
#ifndef CT_H
#define CT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t is `struct CUstream_st *`; pass it (or NULL) wherever `stream` appears. */
struct CUstream_st;

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define CT_API __attribute__((visibility("default")))
#else
#define CT_API
#endif

/* Beam kinds (diffct "Trajectories and Geometry", trajectory-format table). */
typedef enum {
    CT_PARALLEL2D = 0, /* record: ray_dir(2), det_origin(2), det_u(2)             */
    CT_FAN2D = 1,      /* record: src_pos(2), det_center(2), det_u(2)             */
    CT_CONE = 2,       /* record: src_pos(3), det_center(3), det_u(3), det_v(3)   */
    CT_PARALLEL3D = 3  /* record: ray_dir(3), det_center(3), det_u(3), det_v(3)   */
} ct_beam;

typedef enum {
    CT_OK = 0,
    CT_ERR_INVALID_ARGUMENT = 1,   /* NULL handle/pointer, bad size, bad enum, overflow, or a
                                      compute call with another device current than the
                                      handle's                                                  */
    CT_ERR_INVALID_GEOMETRY = 2,   /* a view record fails the admission checks below          */
    CT_ERR_NOT_DEVICE_POINTER = 3, /* a buffer is not device (or managed) memory of the
                                      handle's device                                          */
    CT_ERR_ALIASING = 4,           /* input, output and workspace ranges overlap               */
    CT_ERR_OUT_OF_MEMORY = 5,      /* cudaMalloc failed in ct_geometry_create                  */
    CT_ERR_CUDA = 6,               /* any other CUDA runtime error (incl. earlier async ones)  */
    CT_ERR_WORKSPACE = 7           /* workspace missing or smaller than the reported size      */
} ct_status;

typedef struct ct_geometry ct_geometry; /* opaque, immutable after ct_geometry_create */

/* Read-only description of a handle. */
typedef struct {
    int32_t beam;             /* ct_beam                                                  */
    int32_t n_views;
    int32_t nz, ny, nx;       /* 2D: nz == 1                                              */
    int32_t n_u, n_v;         /* 2D: n_v == 1                                             */
    int32_t volume_layout;    /* internal volume order used by the kernels:
                                 0 = [z][y][x] (caller's order, no copy),
                                 1 = [y][x][z] (z fastest), 2 = [z][x][y] (y fastest)      */
    int64_t n_rays;           /* n_views * n_u * n_v                                      */
    int64_t n_voxels;         /* nz * ny * nx                                             */
    size_t workspace_bytes;   /* scratch needed by ct_project / ct_backproject            */
    size_t sirt_workspace_bytes;
    int32_t n_slabs;          /* slabs of the inner axis the projector walks one at a time
                                 (1: the whole volume at once); see ct_geometry_set_slabs  */
    int32_t slab_cells;       /* cells of the inner axis per slab (the last may be shorter) */
    int32_t shared_lines;     /* 1 (2): in every view the detector's v (u) axis has no
                                 component on the two outer volume axes, so the rays of one
                                 detector column (row) share their outer-axis crossings, and the
                                 volume fits in the device's L2: the untiled forward projection
                                 reads them from one list per line, and the backprojection
                                 walks the same segments per ray (still the exact transpose).
                                 0: per-ray parameters only.  The two parameterisations agree
                                 within float32 rounding of the crossing positions; SIRT and
                                 CGLS always use the per-ray one.                          */
} ct_geometry_info;

/*
 * Create a geometry handle.
 *
 * beam, n_views   ct_beam and number of views (> 0).
 * views           HOST pointer, row-major n_views x 12 doubles (3D) or n_views x 6 (2D), one
 *                 record per view as listed in ct_beam.  Copied; the caller keeps ownership.
 * nz, ny, nx      volume size in voxels (2D: nz must be 1); nz*ny*nx < 2^31.
 * voxel_spacing   scalar voxel pitch (> 0), same unit as the records.
 * n_u, n_v        detector size in pixels (2D: n_v must be 1).
 * du, dv          detector pitch along det_u / det_v (> 0; dv ignored for 2D).
 * out             receives the handle on CT_OK, NULL otherwise.
 *
 * Admission checks, in float64 on the host (diffct "Trajectories and Geometry", the paragraph
 * after the custom-acquisition example): every value finite; det_u (and det_v, ray_dir) unit
 * length within 1e-6; 2D parallel: ray_dir . det_u = 0 within 1e-6; 3D: det_u . det_v = 0 within
 * 1e-6; parallel3d: |ray_dir . (det_u x det_v)| > 1e-6 (not tangent to the detector); fan/cone:
 * source and detector centre distinct, the detector not seen edge-on
 * (|(det_center - src) . n| > 1e-6 |det_center - src|), and the nearer of the two within 1e6
 * voxel spacings of the origin, both within 1e15; parallel beams: det_center within 1e6 voxel
 * spacings.  Failing records give CT_ERR_INVALID_GEOMETRY; sizes give CT_ERR_INVALID_ARGUMENT.
 *
 * The handle allocates a small device table of per-view records on the current device and
 * uploads it synchronously; the handle is bound to that device.
 */
CT_API ct_status ct_geometry_create(ct_beam beam, int32_t n_views, const double *views, int32_t nz,
                             int32_t ny, int32_t nx, double voxel_spacing, int32_t n_u,
                             int32_t n_v, double du, double dv, ct_geometry **out);

/*
 * As ct_geometry_create, with a voxel spacing per axis ("Trajectories and Geometry": voxel
 * spacing is a positive scalar or a positive per-axis tuple in tensor order).
 *
 * spacing_zyx   HOST pointer to 3 doubles (dz, dy, dx), each > 0; for 2D beams dz is ignored.
 * Voxel i of an axis with n cells and pitch s spans [-n s/2 + i s, -n s/2 + (i+1) s); chord
 * lengths are physical.  The admission distance limit uses the smallest pitch.
 */
CT_API ct_status ct_geometry_create_ex(ct_beam beam, int32_t n_views, const double *views,
                                       int32_t nz, int32_t ny, int32_t nx,
                                       const double *spacing_zyx, int32_t n_u, int32_t n_v,
                                       double du, double dv, ct_geometry **out);

/*
 * As ct_geometry_create_ex, with a parameterized detector surface instead of the flat detector
 * ("Trajectories and Geometry", detector surfaces): pixel (u, v) of a view sits at
 *     det_center + o_u det_u + o_v det_v + o_n n,   n = det_u x det_v  (2D: (det_u_y, -det_u_x))
 * with the pixel's local offsets o = offsets_uvn[(u * n_v + v) * 3 + {0, 1, 2}] (physical units,
 * shared by all views; 2D: o_v is ignored).  A cylinder of radius R about det_v, for example, has
 * o = (R sin(s/R), v, +-R (1 - cos(s/R))) at arc length s.  The record's det_u/det_v must still
 * be orthonormal; instead of the flat edge-on test every source/pixel pair is checked: distinct
 * in float32, nearer endpoint within 1e6 voxel spacings of the origin, both within 1e15.
 * offsets_uvn is a HOST pointer to n_u x n_v x 3 doubles, copied to a device table that the
 * handle owns.
 */
CT_API ct_status ct_geometry_create_surface(ct_beam beam, int32_t n_views, const double *views,
                                            int32_t nz, int32_t ny, int32_t nx,
                                            const double *spacing_zyx, int32_t n_u, int32_t n_v,
                                            const double *offsets_uvn, ct_geometry **out);

/* Free a handle and its device table (synchronous).  NULL is accepted. */
CT_API ct_status ct_geometry_destroy(ct_geometry *geom);

/* Fill *info for a handle. */
CT_API ct_status ct_geometry_get_info(const ct_geometry *geom, ct_geometry_info *info);

/*
 * Slab tiling of the forward projection and backprojection, for volumes larger than the L2 cache
 * (diffct "Large Volumes and Chunked Execution": spatial tiles keep the working set bounded).
 * Off by default.  With slab_cells > 0 (rounded up to a multiple of 32, so that slabs hold whole
 * 128-byte lines of the z-fastest order) ct_project, ct_backproject and the batched calls run
 * one launch per slab of the inner axis (z) over the detector tiles whose rays can reach it
 * (found on the host from the planes that hold each detector row's rays), every ray walking only
 * its part inside the slab, so that the cells a launch touches stay in L2.  Each walk restarts
 * from the whole ray's own crossing values, so every ray-voxel segment carries the same weight as
 * without slabs; the forward projection adds the slabs' partial sums in slab order
 * (deterministic; the last bits may differ from an untiled run).  SIRT, CGLS and the FBP calls do
 * not use slabs.  On the 512^3 spiral workload (512 MiB) 64-cell slabs cut the walks' DRAM
 * traffic about threefold but take about four times as long: every slab re-clips its rays in
 * float64, and sloped rays of one detector column enter a slab at different points of their
 * shared path, so the lanes of a warp no longer walk in lock-step.
 *
 * slab_cells = 0 turns tiling off.  Only for handles with info.volume_layout == 1 and a flat
 * detector (else CT_ERR_INVALID_ARGUMENT).  It replaces the handle's small device table of
 * per-slab tile lists (synchronous), so call it before any compute call is queued with the
 * handle, never while one may be running.
 */
CT_API ct_status ct_geometry_set_slabs(ct_geometry *geom, int32_t slab_cells);

/*
 * Forward projection: d_sino = A d_volume.
 *
 * d_volume   device, (nz, ny, nx) float32, read only.
 * d_sino     device, (n_views, n_u, n_v) float32; every entry is overwritten, rays that miss
 *            the volume get 0 (diffct "Memory and chunking", resident layouts: forward kernels
 *            overwrite each active ray, including missed rays).
 * d_workspace, workspace_bytes
 *            device scratch of at least info.workspace_bytes (may be NULL when that is 0);
 *            used for the kernels' internal volume order.  Must not overlap the other buffers.
 * Float32 walk with float64 entry/exit clipping (the entry and exit cells and the distance to
 * each axis's first plane are also taken in float64, so a plane crossed at a grazing angle keeps
 * its position); per-ray results match the float64 definition within 1e-4 of (ray chord length
 * x max |x|).
 */
CT_API ct_status ct_project(const ct_geometry *geom, const float *d_volume, float *d_sino,
                     void *d_workspace, size_t workspace_bytes, struct CUstream_st *stream);

/*
 * Matched adjoint: d_volume = A^T d_sino, with exactly the chord weights of ct_project (the same
 * traversal code and the same float32 arithmetic).  d_volume is overwritten (cleared on the
 * stream, then accumulated with float32 atomics, so the summation order, and thus the last bits,
 * may vary from run to run).  Arguments as for ct_project.
 */
CT_API ct_status ct_backproject(const ct_geometry *geom, const float *d_sino, float *d_volume,
                         void *d_workspace, size_t workspace_bytes,
                         struct CUstream_st *stream);

/* Scratch bytes needed by ct_sirt_iterate (= info.sirt_workspace_bytes). */
CT_API size_t ct_sirt_workspace_bytes(const ct_geometry *geom);

/*
 * SIRT: n_iters updates  x <- x + relaxation * C . A^T( R . (y - A x) ),
 * R = 1/(A 1) per ray, C = 1/(A^T 1) per voxel, each 0 where the sum is 0.  The pages name SIRT
 * (ASTRA SIRT3D_CUDA in the HAADF-STEM article's timing table; diffct.solvers.sirt) without
 * printing it; this is the textbook simultaneous iteration with those row/column normalisers.
 *
 * d_x        device volume, updated in place (start from zeros for a plain SIRT run).
 * d_y        device sinogram (measurements), read only.
 * d_workspace, workspace_bytes
 *            at least ct_sirt_workspace_bytes(geom) of device scratch.  It caches C between
 *            calls: pass workspace_initialised = 0 on the first call with a workspace (C is then
 *            computed), 1 on later calls with the same handle and workspace.
 * relaxation in (0, 2); n_iters >= 0.
 */
CT_API ct_status ct_sirt_iterate(const ct_geometry *geom, float *d_x, const float *d_y,
                          void *d_workspace, size_t workspace_bytes, int32_t n_iters,
                          float relaxation, int32_t workspace_initialised,
                          struct CUstream_st *stream);

/*
 * Batches of volumes ("Leading batch/channel dimensions are preserved", diffct quickstart):
 * d_volumes holds `batch` volumes back to back, (batch, nz, ny, nx); d_sinos holds `batch`
 * sinograms, (batch, n_views, n_u, n_v).  Results equal `batch` separate ct_project /
 * ct_backproject calls (the forward results bit for bit); the kernels walk each ray once for up
 * to 4 volumes, so the per-update cost of the traversal is shared.  Workspace: at least
 * ct_batch_workspace_bytes(geom, batch) (0 when the internal volume order is the caller's).
 * Semantics, ownership and errors as for the single-volume calls.
 */
CT_API size_t ct_batch_workspace_bytes(const ct_geometry *geom, int32_t batch);
CT_API ct_status ct_project_batch(const ct_geometry *geom, int32_t batch,
                                  const float *d_volumes, float *d_sinos, void *d_workspace,
                                  size_t workspace_bytes, struct CUstream_st *stream);
CT_API ct_status ct_backproject_batch(const ct_geometry *geom, int32_t batch,
                                      const float *d_sinos, float *d_volumes, void *d_workspace,
                                      size_t workspace_bytes, struct CUstream_st *stream);

/* Scratch bytes needed by ct_cgls_iterate. */
CT_API size_t ct_cgls_workspace_bytes(const ct_geometry *geom);

/*
 * CGLS: n_iters steps of conjugate gradients on the normal equations A^T A x = A^T y, in the
 * form that never forms A^T A (r = y - A x, s = A^T r, p = s, gamma = |s|^2; each step:
 * q = A p, alpha = gamma / |q|^2, x += alpha p, r -= alpha q, s = A^T r, beta = |s|^2 / gamma,
 * p = s + beta p).  The pages list a CGLS solver on this operator pair (diffct "Solvers" API
 * entries cgls / cgls_into) and time one CGLS iteration in their performance table; they do not
 * print the recurrences, which are the textbook ones.  Norms are accumulated in float64 on the
 * device; alpha, beta and gamma stay on the device (no host synchronisation).  A zero
 * denominator (an exact solution) gives alpha = 0 or beta = 0.
 *
 * d_x        device volume, updated in place; the starting point (zeros for a plain run).
 * d_y        device sinogram (measurements), read only.
 * d_workspace, workspace_bytes
 *            at least ct_cgls_workspace_bytes(geom).  It carries the CGLS state (r, p, gamma)
 *            between calls: pass workspace_initialised = 0 on the first call (the state is
 *            set up from d_x), 1 to continue a run with the same handle, workspace and d_y, and
 *            with d_x unchanged since the previous call.
 * n_iters >= 0.
 */
CT_API ct_status ct_cgls_iterate(const ct_geometry *geom, float *d_x, const float *d_y,
                                 void *d_workspace, size_t workspace_bytes, int32_t n_iters,
                                 int32_t workspace_initialised, struct CUstream_st *stream);

/*
 * Backprojection that allocates nothing: d_volume = A^T d_sino, the same operator, kernels and
 * weights as ct_backproject, for callers that cannot allocate device memory at the time they
 * backproject (code that receives only a stream and its input/output pointers from a host
 * framework, real-time pipelines that forbid allocation after start-up, programs that keep all
 * device memory in their own pool).  It takes no workspace: when the geometry's internal volume
 * order differs from the caller's (info.volume_layout != 0) the accumulator lives in one static
 * device array of CT_STATIC_SCRATCH_VOXELS floats (16 MiB) that every GPU which loads the library
 * holds until the process exits.  The pages describe no such entry point; it has no counterpart
 * there.
 *
 * d_sino, d_volume  device buffers as for ct_backproject; d_volume is overwritten.
 * Errors: CT_ERR_WORKSPACE if the geometry needs the static array and has more than
 * CT_STATIC_SCRATCH_VOXELS voxels; CT_ERR_INVALID_ARGUMENT if the handle's device is not the
 * current device; otherwise as ct_backproject.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress, which may
 * load the module on that device); make that first call before any stream capture.  The address
 * is kept per device and CUDA context: after a device reset the next call runs in a new context
 * and looks it up again (again outside any capture).  Every call
 * shares the one array: it is cleared on the stream at the start of each call, and calls whose
 * work overlaps on the GPU (different streams, or graphs replayed concurrently) race on it.
 */
#define CT_STATIC_SCRATCH_VOXELS (1u << 22)
CT_API ct_status ct_backproject_static(const ct_geometry *geom, const float *d_sino,
                                       float *d_volume, struct CUstream_st *stream);

/*
 * Filtered backprojection: parallel-beam FBP (CT_PARALLEL2D), fan-beam FBP (CT_FAN2D) and
 * Feldkamp-Davis-Kress cone-beam reconstruction (CT_CONE), on flat detectors.  The pages list the
 * stages (diffct "Differentiable analytical reconstruction" and the FBP/FDK example pages:
 * detector cosine weights, a ramp filter with physical sample spacing and an optional window,
 * angular integration weights and a voxel-driven distance-weighted gather) without formulas;
 * this is the textbook form:
 *
 *   1. fan/cone: p'(u, v) = p(u, v) |(c - s) . n| / |P(u, v) - s|   (s source, c detector
 *      centre, n detector normal, P the pixel);
 *   2. Q(u_i, v) = sum_j k[i - j + n_u - 1] p'(u_j, v), a linear convolution along u (no
 *      wrap-around) with the discrete kernel k[m] = du h((m - n_u + 1) du), h the band-limited
 *      ramp h(x) = 2 int_0^{1/(2 du)} f W(f) cos(2 pi f x) df with window W (ct_fbp_window), or
 *      the caller's kernel (e.g. a learned filter);
 *   3. f(X) = sum_k w_k g_k(X) Q_k(u_k(X), v_k(X)): X projected onto view k's detector through
 *      the source (parallel: along the ray), Q interpolated bilinearly (0 off the detector),
 *      g = 1 for parallel beams, else g = (D_sd / D_so) / U(X)^2 with
 *      U(X) = ((X - s) . n) / ((iso - s) . n), D_so = |(iso - s) . n|, D_sd = |(c - s) . n|.
 *
 * This is an approximate inverse, not the Siddon adjoint.  Voxel centres as in the frame above
 * (per-axis pitches of ct_geometry_create_ex are honoured).
 *
 * d_sino       device sinogram, read only.
 * d_volume     device volume, overwritten.
 * options      NULL for the defaults, or (fields):
 *   window          ct_fbp_window of the ramp (used when d_kernel is NULL).
 *   d_view_weights  device, n_views floats, or NULL for the uniform full-scan quadrature
 *                   w_k = pi / n_views (a 180-degree parallel scan, or a 360-degree fan/cone scan
 *                   with the 1/2 redundancy factor).  Short scans pass the angular step instead.
 *   d_pixel_weights device, n_views x n_u floats, or NULL: weights per view and detector column
 *                   applied with the cosine weights before filtering, e.g. Parker's short-scan
 *                   weights from ct_fbp_parker_weights.
 *   d_kernel        device, 2 n_u - 1 floats, or NULL: the discrete filter k above (offset
 *                   m - n_u + 1 at index m), replacing the windowed ramp.
 *   isocenter       host, 3 doubles (x, y, z; z ignored in 2D), or NULL: the point whose
 *                   detector-plane distance sets D_so (fan/cone; unused for parallel beams).
 *                   NULL estimates it from the detector normals, as the pages' default does: the
 *                   least-squares point nearest the lines through each detector centre along its
 *                   normal (the origin for circular orbits about it); one view, or views whose
 *                   normals are all parallel, give that set's minimum-norm point, so pass the
 *                   isocentre explicitly for such geometries.
 * Workspace: at least ct_fbp_workspace_bytes(geom) (the filtered sinogram, per-view constants
 * and the filter taps).
 * Errors: CT_ERR_INVALID_ARGUMENT for CT_PARALLEL3D, surface detectors, an unknown window, or
 * n_u > 16384, or a grid beyond the gather launch (3D: ny > 65535 or nx > 524280; 2D:
 * ny > 524280); otherwise as ct_backproject.
 */
typedef enum {
    CT_WINDOW_RAM_LAK = 0,     /* W(f) = 1                                          */
    CT_WINDOW_SHEPP_LOGAN = 1, /* W(f) = sin(pi f du) / (pi f du)                   */
    CT_WINDOW_COSINE = 2,      /* W(f) = cos(pi f du)                               */
    CT_WINDOW_HAMMING = 3,     /* W(f) = 0.54 + 0.46 cos(2 pi f du)                 */
    CT_WINDOW_HANN = 4         /* W(f) = 0.5 + 0.5 cos(2 pi f du)                   */
} ct_fbp_window;

typedef struct {
    ct_fbp_window window;
    const float *d_view_weights;
    const float *d_pixel_weights;
    const float *d_kernel;
    const double *isocenter;
} ct_fbp_options;

CT_API size_t ct_fbp_workspace_bytes(const ct_geometry *geom);
CT_API ct_status ct_fbp(const ct_geometry *geom, const float *d_sino, float *d_volume,
                        const ct_fbp_options *options, void *d_workspace, size_t workspace_bytes,
                        struct CUstream_st *stream);

/*
 * Transpose of ct_fbp as a linear map (sinogram -> volume), for gradients with respect to the
 * sinogram: d_sino = F^T d_volume, so that <F y, x> = <y, F^T x>.  The pages state that the
 * analytical operator's backward pass scatters the same interpolation coefficients, distance
 * weights and normalisation, with dedicated transpose kernels (diffct "Differentiable analytical
 * reconstruction"; "Analytical Reconstruction Helpers").  Steps: every voxel adds
 * w_k g_k(X) f(X) times its four bilinear coefficients onto view k's detector (atomic adds;
 * contributions off the detector are dropped), the filter with its kernel reversed (the
 * windowed ramps are symmetric), then the cosine and pixel weights.  Arguments and errors as for
 * ct_fbp, with d_volume read and d_sino overwritten; the workspace is at least
 * ct_fbp_transpose_workspace_bytes(geom) (per view and detector pixel 4 floats for cone beams, 2
 * for 2D, plus the per-view constants and taps).  The atomic adds make the float32 result depend
 * on the order in which they land (run-to-run differences of a few ulp).
 */
CT_API size_t ct_fbp_transpose_workspace_bytes(const ct_geometry *geom);
CT_API ct_status ct_fbp_transpose(const ct_geometry *geom, const float *d_volume, float *d_sino,
                                  const ct_fbp_options *options, void *d_workspace,
                                  size_t workspace_bytes, struct CUstream_st *stream);

/*
 * Gradients of a loss L(f), f = ct_fbp(d_sino, options), with respect to the filter kernel and
 * the view weights, given dL/df = d_grad_volume (the pages: filter and explicit weight gradients
 * propagate through the analytical pipeline, "Differentiable analytical reconstruction").  f is
 * linear in both: with q_k the cosine- and pixel-weighted sinogram of view k, Q_k its filtered
 * columns and G_k the view's gather without its weight,
 *     dL/dw_k = <G_k^T grad, Q_k>,
 *     dL/dk[d + n_u - 1] = sum_k w_k sum_v sum_i (G_k^T grad)(u_i, v) q_k(u_{i - d}, v).
 * d_grad_kernel (device, 2 n_u - 1 floats) and d_grad_view_weights (device, n_views floats) are
 * overwritten; either may be NULL, not both.  Workspace: ct_fbp_gradients_workspace_bytes(geom).
 * The kernel gradient sums float32 partials (one block's tile of the products over a chunk of
 * views) into float64 with atomic adds, so results differ run to run in the last bits.  Errors
 * as for ct_fbp.
 */
CT_API size_t ct_fbp_gradients_workspace_bytes(const ct_geometry *geom);
CT_API ct_status ct_fbp_gradients(const ct_geometry *geom, const float *d_sino,
                                  const float *d_grad_volume, const ct_fbp_options *options,
                                  float *d_grad_kernel, float *d_grad_view_weights,
                                  void *d_workspace, size_t workspace_bytes,
                                  struct CUstream_st *stream);

/*
 * Parker's short-scan weights (Parker 1982) for a circular fan or cone scan, host-computed in
 * float64: the pages add them before filtering for short scans ("Differentiable analytical
 * reconstruction": short_scan).  beta = source angle about the isocentre from the first view,
 * in the sense of rotation; gamma = fan angle of detector column u (its centre line) from the
 * central ray, in the same sense; delta = max |gamma|.  With the last view at beta = span
 * >= pi + 2 delta the weights use the effective half fan angle d = (span - pi) / 2:
 *     w = sin^2(pi/4 * beta / (d - gamma))                0 <= beta < 2 (d - gamma)
 *       = 1                                                up to beta = pi - 2 gamma
 *       = sin^2(pi/4 * (pi + 2 d - beta) / (d + gamma))    up to beta = pi + 2 d
 * so that the two measurements of every line weigh 1 together.  Use them as ct_fbp's
 * d_pixel_weights with view weights equal to the angular step (no 1/2 factor).
 *
 * isocenter  host, 3 doubles, or NULL to estimate it as ct_fbp does.
 * out        HOST, n_views x n_u floats (view-major), written on CT_OK.
 * Errors: CT_ERR_INVALID_ARGUMENT for parallel beams, surface detectors or NULL pointers;
 * CT_ERR_INVALID_GEOMETRY if the sources are not on a circle in the xy-plane about the
 * isocentre (relative tolerance 1e-6) or the scan spans less than pi + 2 delta.
 */
CT_API ct_status ct_fbp_parker_weights(const ct_geometry *geom, const double *isocenter,
                                       float *out);

/*
 * Bounds-checking builds (the library compiled with -DCT_DEBUG_BOUNDS; the package's build
 * script does that with debug_bounds=True): every data-dependent voxel or detector index the
 * kernels form is checked before use, and an index outside its array skips the access and is
 * counted on the device instead of faulting.  This call synchronises the device and returns the
 * count since the previous call (then resets it).  Release builds return CT_ERR_INVALID_ARGUMENT
 * with *count = 0.  The pages have no counterpart; it stands in for a memory checker.
 */
CT_API ct_status ct_debug_bounds_violations(uint64_t *count);

/* Static, human-readable name of a status code. */
CT_API const char *ct_status_string(ct_status status);

/*
 * Roofline probes.  The pages give no counterpart: these calls exist so that a benchmark
 * can measure, on the GPU at hand and with CUDA events on `stream`, the rates of the access
 * patterns the projector's kernels press on, and use them as the denominators of their roofline
 * fractions.  Use a buffer that fits in L2 (64 MiB on a B300) and warm it once first.
 *
 * ct_probe_l2_read:   passes x n_floats/4 sixteen-byte loads that bypass L1 (ld.global.cg),
 *                     grid-stride over d_buf by every resident thread (a multiple of the SM
 *                     count).  d_buf: device, n_floats >= 4 floats, 16-byte aligned, read only;
 *                     d_sink: device, one float, written only if the loaded values sum to -1
 *                     per thread (never, for non-negative contents).  Traffic per call:
 *                     16 * floor(n_floats / 4) * passes bytes.
 * ct_probe_l1_read:   the same loads, but allocating in L1 (ld.global.ca), every block re-reading
 *                     the same first n_floats (4 <= n_floats <= 16384, 16-byte aligned) floats of
 *                     d_buf, so that after the first pass every load hits in L1.  Traffic per
 *                     call: 16 * floor(n_floats / 4) * passes bytes per block, blocks = 4 per SM.
 * ct_probe_l2_reduce: passes sweeps of red.global.add.f32 (+1.0) over d_buf, each warp
 *                     instruction updating 32 floats `stride` apart (1 <= stride <= 32;
 *                     stride 1 puts 8 updates in each 32-byte sector, stride 2 four).  Updates
 *                     per call: 32 * floor(n_floats / (32 stride)) * passes; d_buf is modified.
 * Errors: CT_ERR_INVALID_ARGUMENT (NULL, sizes, passes <= 0, alignment, stride),
 * CT_ERR_NOT_DEVICE_POINTER, CT_ERR_ALIASING, CT_ERR_CUDA.
 */
CT_API ct_status ct_probe_l2_read(const float *d_buf, size_t n_floats, int32_t passes,
                                  float *d_sink, struct CUstream_st *stream);
CT_API ct_status ct_probe_l1_read(const float *d_buf, size_t n_floats, int32_t passes,
                                  float *d_sink, struct CUstream_st *stream);
CT_API ct_status ct_probe_l2_reduce(float *d_buf, size_t n_floats, int32_t passes,
                                    int32_t stride, struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* CT_H */
