// Internal declarations shared by the C-ABI layer and the kernels of libctproj.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace ct {

// Bounds-checking builds (compiled with -DCT_DEBUG_BOUNDS): every data-dependent voxel or detector
// index the kernels form is checked before use; an index outside its array skips the access and
// increments a per-file device counter (no trap).  Release builds compile the checks away.
// Counters of the kernel files, read and reset from the host (0 in release builds).
uint64_t siddon_bounds_violations(bool reset);
uint64_t fbp_bounds_violations(bool reset);

// Streaming multiprocessors of the current device (queried once per device, then cached); grid
// sizes of the grid-stride kernels are multiples of it.
int device_sm_count();

// Internal volume orders (the kernels' memory layout of the volume).
enum Layout : int32_t {
    LAYOUT_ZYX = 0,  // caller's order, x fastest
    LAYOUT_YXZ = 1,  // z fastest: one 2D transpose of (nz) x (ny*nx)
    LAYOUT_ZXY = 2,  // y fastest: nz transposes of (ny) x (nx)
};

// Per-view record as the kernels read it.  All positions are in voxel units, with the origin at
// the volume's lower corner, so the volume is the box [0, nx] x [0, ny] x [0, nz] and voxel
// (i, j, k) is the unit cell [i, i+1) x [j, j+1) x [k, k+1).  Pixel (u, v) sits at
//     flat detector:  P(u, v) = pb + u * pu + v * pv   (pb holds the -(U-1)/2, -(V-1)/2 offsets)
//     surface:        P(u, v) = pb + o_u * pu + o_v * pv + o_n * pn   (per-pixel offsets o)
// Parallel beams: the ray is P(u, v) + t * q   (q = ray direction), t over all reals.
// Point sources:  the ray is q + a * (P(u, v) - q) for a in [0, 1]; pb is stored minus q, so
//                 the direction is directly P(u, v).
struct ViewRec {
    double pb[3];
    double pu[3];
    double pv[3];
    double pn[3];           // detector normal (surface detectors only)
    double q[3];
    int32_t lanes_along_v;  // 1: a warp's 32 lanes take 32 consecutive v; 0: consecutive u
    int32_t pad;
};
static_assert(sizeof(ViewRec) == 128, "ViewRec layout");

// Volume grid as the kernels see it.
struct Grid {
    int32_t n[3];        // cells along x, y, z
    int32_t stride[3];   // element stride of x, y, z in the internal layout
    double nd[3];        // n as doubles (box upper corner)
    float sp[3];         // physical voxel pitch along x, y, z
    int32_t iso;         // 1 when the three pitches are equal
    int32_t parallel;    // 1: infinite lines, 0: source-to-pixel segments
    int32_t fast;        // axis that is fastest in memory (0 x, 1 y, 2 z): the walk's inner axis
    const double* offsets;  // surface detectors: (n_u, n_v, 3) local offsets; flat: nullptr
    int32_t nv;             // detector pixels along v (row pitch of the offsets table)
};

// Detector tiling of one launch.
struct Tiling {
    int32_t n_views;
    int32_t n_u, n_v;
    int32_t tiles_u, tiles_v;  // 32 x 32 pixel tiles (2D: 256 x 1)
    int32_t two_d;
    // Shared-line forward projections (siddon_kernels.cu): 0 off; 1 every view's rays of one
    // detector column (fixed u) share their outer-axis line, lanes along v; 2 the same for rows
    // (fixed v), lanes along u.  Blocks take kLinePixels pixels along the lanes times kLineRows
    // lines.
    int32_t line;
    int32_t line_lane_tiles, line_row_tiles;
    // 3D backprojection tiles whose warps take every second pixel along the lanes' axis (two
    // warps interleave over 64 pixels): 0 off; 1 lanes along v in every view, 16 (u) x 64 (v)
    // tiles; 2 lanes along u, 64 x 16 tiles.  Counts of those tiles.
    int32_t spread;
    int32_t spread_tiles_u, spread_tiles_v;
};

// Shared-line tiles: pixels along the lanes per block (its threads), lines per block, and the
// largest outer-axis cell count n_a + n_b whose crossing list (8 bytes per entry) a block keeps.
constexpr int kLinePixels = 128;
constexpr int kLineRows = 8;
constexpr int kLineMaxCells = 6000;

// One slab of the inner (fastest) axis for the slab-tiled walks: the walks of a launch are
// restricted to the inner-axis cells [c0, c1), over the detector tiles whose rays can reach the
// slab: tiles[i] = view * tiles_v + v_tile for i < n_tiles, and block b takes the u-tile
// b % tiles_u of entry b / tiles_u.
struct SlabArgs {
    int32_t c0, c1;
    const int32_t* tiles;
    int32_t n_tiles;
};

// Launchers (kernels in siddon_kernels.cu).  All asynchronous on `stream`.
cudaError_t launch_project(const ViewRec* views, const Grid& g, const Tiling& t,
                           const float* vol, float* sino, cudaStream_t stream);
cudaError_t launch_backproject(const ViewRec* views, const Grid& g, const Tiling& t,
                               const float* sino, float* vol, cudaStream_t stream);
cudaError_t launch_backproject_ones(const ViewRec* views, const Grid& g, const Tiling& t,
                                    float* vol, cudaStream_t stream);
// Batched forms: nb (1, 2 or 4) volumes at vol + b * vstride (internal order) and sinograms at
// sino + b * sstride, one walk per ray for all of them.
cudaError_t launch_project_batch(const ViewRec* views, const Grid& g, const Tiling& t, int nb,
                                 const float* vol, int64_t vstride, float* sino, int64_t sstride,
                                 cudaStream_t stream);
cudaError_t launch_backproject_batch(const ViewRec* views, const Grid& g, const Tiling& t, int nb,
                                     const float* sino, int64_t sstride, float* vol,
                                     int64_t vstride, cudaStream_t stream);
// Slab-tiled forms (3D, z-fastest internal order only): the projection ADDS each ray's partial
// line integral over the slab to sino (which the caller clears before the first slab), the
// backprojection scatters the slab's segments.  nb as for the batched forms.
cudaError_t launch_project_slab(const ViewRec* views, const Grid& g, const Tiling& t, int nb,
                                const float* vol, int64_t vstride, float* sino, int64_t sstride,
                                const SlabArgs& slab, cudaStream_t stream);
cudaError_t launch_backproject_slab(const ViewRec* views, const Grid& g, const Tiling& t, int nb,
                                    const float* sino, int64_t sstride, float* vol,
                                    int64_t vstride, const SlabArgs& slab, cudaStream_t stream);
cudaError_t launch_project_residual(const ViewRec* views, const Grid& g, const Tiling& t,
                                    const float* x, const float* y, float* r,
                                    cudaStream_t stream);
// CGLS pieces.  Scalars (float64, device): [gamma, delta, alpha, beta].
int64_t project_blocks(const Tiling& t);  // blocks (= partial sums) of one projection launch
int norm_blocks(int sm_count);              // blocks (= partial sums) of launch_norm_partials
cudaError_t launch_project_norm(const ViewRec* views, const Grid& g, const Tiling& t,
                                const float* vol, float* sino, double* partials,
                                cudaStream_t stream);
cudaError_t launch_backproject_residual(const ViewRec* views, const Grid& g, const Tiling& t,
                                        float* r, const float* q, const double* scal, float* vol,
                                        cudaStream_t stream);
cudaError_t launch_norm_partials(const float* v, int64_t n, double* partials, int sm_count,
                                 cudaStream_t stream);
cudaError_t launch_cgls_scalars(const double* partials, int64_t n, double* scal, int which,
                                cudaStream_t stream);
cudaError_t launch_cgls_update(float* x, float* p, float* s, const double* scal, int64_t n,
                               cudaStream_t stream);
cudaError_t launch_sub(float* r, const float* y, const float* q, int64_t n, cudaStream_t stream);
cudaError_t launch_invert(float* c, int64_t n, cudaStream_t stream);
cudaError_t launch_sirt_update(float* x, float* b, const float* c, float relax, int64_t n,
                               cudaStream_t stream);
// out[b][c][r] = in[b][r][c] for b < batch, r < rows, c < cols.
cudaError_t launch_transpose(const float* in, float* out, int64_t rows, int64_t cols,
                             int64_t batch, cudaStream_t stream);

// L2 roofline probes (kernels in probe_kernels.cu): 16-byte L1-bypassing loads over `buf`
// (n_floats, 16-byte aligned) `passes` times; red.global.add.f32 of 1.0 over `buf` with the lanes
// of a warp `stride` floats apart, `passes` sweeps.
cudaError_t launch_l2_read(const float* buf, int64_t n_floats, int32_t passes, float* sink,
                           cudaStream_t stream);
cudaError_t launch_l2_reduce(float* buf, int64_t n_floats, int32_t passes, int32_t stride,
                             cudaStream_t stream);
// Every block reads the same first n_floats floats of `buf` (L1-resident) `passes` times.
cudaError_t launch_l1_read(const float* buf, int64_t n_floats, int32_t passes, float* sink,
                           cudaStream_t stream);

// Filtered backprojection (kernels in fbp_kernels.cu).  Physical units, origin at the volume
// centre (the caller's frame, not the Siddon kernels' voxel frame).
enum FbpWindow : int32_t {
    FBP_RAM_LAK = 0,
    FBP_SHEPP_LOGAN = 1,
    FBP_COSINE = 2,
    FBP_HAMMING = 3,
    FBP_HANN = 4,
};
struct FbpParams {
    int32_t n_views, n_u, n_v;
    int32_t nx, ny, nz;
    int32_t two_d, parallel, window;
    int32_t rows, cols;  // padded filtered sinogram per view: rows = n_u + 3, cols = n_v + 3 (2D: 1)
    int32_t bu, bv;      // transpose: 2 x 2 blocks per view and copy along u, v (2D: pairs, bv = 1)
    double du, dv;
    double iso[3];
    float sx, sy, sz;  // voxel pitches along x, y, z
    const float* pixel_weights;  // optional (n_views, n_u) weights before filtering, or nullptr
    const float* kernel;  // optional caller filter (2 n_u - 1), replacing the window, or nullptr
    int32_t reverse_kernel;  // 1: the taps are stored reversed (the transpose's filter)
    int32_t unit_weights;    // 1: every view weight is 1 (gradient scatter)
};
// Per-view constants of the gather (64 bytes, read as four float4).
struct FbpView {
    float s[3];      // source (fan/cone)
    float n[3];      // detector normal
    float eu[3];     // det_u / du
    float ev[3];     // det_v / dv (cone)
    float D;         // (c - s) . n
    float ku0, kv0;  // additive terms of the fractional pixel indices
    float wg;        // view weight times the constant part of the distance weight
};
static_assert(sizeof(FbpView) == 64, "FbpView layout");
// Per-view constants of the cosine pre-weights (48 bytes).
struct FbpCosine {
    float pc[3];   // pixel (0, 0) minus source
    float pdu[3];  // du det_u
    float pdv[3];  // dv det_v
    float D;       // |(c - s) . n|
    float pad[2];
};
static_assert(sizeof(FbpCosine) == 48, "FbpCosine layout");
// Filtered sinogram layout: view k, pixel (u, v) at
//     filtered[(k * rows + u + 1) * cols + v + 1]            (3D)
//     filtered[k * rows + u + 1]                             (2D)
// with zero pads one pixel before and two after each axis, so that a bilinear read at any index
// clamped to [-1, n] stays in bounds and reads 0 off the detector.
// Scratch: views (n_views FbpView), cosine records (n_views FbpCosine), taps (2 n_u - 1 floats),
// filtered sinogram (n_views * rows * cols floats).
cudaError_t launch_fbp(const FbpParams& p, const double* raw_views, const float* view_weights,
                       FbpView* views, FbpCosine* cosines, float* taps, const float* sino,
                       float* filtered, float* vol, cudaStream_t stream);
// Transpose of the same operator: volume -> sinogram.  `scattered` holds the parity copies of
// the padded detector (layout in fbp_kernels.cu, fbp_copies_floats floats); it is cleared on the
// stream first.
size_t fbp_copies_floats(const FbpParams& p);
// Gradients of a loss L(f), f = the FBP of `sino`, given dL/df = grad_vol: dL/dkernel (2 n_u - 1
// floats, or nullptr) and dL/dview_weights (n_views floats, or nullptr).  Scratch: the transpose's
// (copies) plus the padded filtered sinogram (`filtered`) and 2 n_u - 1 doubles (`acc`).
cudaError_t launch_fbp_gradients(const FbpParams& p, const double* raw_views,
                                 const float* view_weights, FbpView* views, FbpCosine* cosines,
                                 float* taps, const float* sino, const float* grad_vol,
                                 float* copies, float* filtered, double* acc, float* grad_kernel,
                                 float* grad_view_weights, cudaStream_t stream);
cudaError_t launch_fbp_transpose(const FbpParams& p, const double* raw_views,
                                 const float* view_weights, FbpView* views, FbpCosine* cosines,
                                 float* taps, const float* vol, float* scattered, float* sino,
                                 cudaStream_t stream);

}  // namespace ct
