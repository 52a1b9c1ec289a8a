// C ABI of libctproj (declared in include/ct.h): geometry admission, per-view record staging,
// internal volume order, workspace carving and kernel dispatch.  Host code only.
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <utility>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "ct.h"
#include "ct_internal.h"

struct ct_geometry {
    ct_geometry_info info;
    double spacing;
    double du, dv;
    int device;
    int sm_count;           // streaming multiprocessors of that device
    ct::Grid grid;          // strides of the internal layout
    ct::Tiling tiling;
    ct::ViewRec* d_views;   // device table, n_views records
    double* d_offsets;      // surface detectors: device (n_u, n_v, 3) offsets; else nullptr
    double* d_raw;          // device copy of the caller's view records (physical units)
    int32_t* d_slab_tiles;  // slab-tiled walks: per slab, the (view, v-tile) entries reaching it
    std::vector<int64_t> slab_off;  // slab s owns d_slab_tiles[slab_off[s] .. slab_off[s + 1])
    std::vector<double> host_views;
    std::vector<ct::ViewRec> recs;  // host copy of the device records (voxel units)
};

namespace {

using ct::Layout;

constexpr size_t kAlign = 256;

size_t align_up(size_t n) { return (n + kAlign - 1) / kAlign * kAlign; }

bool is_2d(int beam) { return beam == CT_PARALLEL2D || beam == CT_FAN2D; }
bool is_parallel(int beam) { return beam == CT_PARALLEL2D || beam == CT_PARALLEL3D; }

double dot3(const double* a, const double* b) { return a[0] * b[0] + a[1] * b[1] + a[2] * b[2]; }
double norm3(const double* a) { return std::sqrt(dot3(a, a)); }
void cross3(const double* a, const double* b, double* c) {
    c[0] = a[1] * b[2] - a[2] * b[1];
    c[1] = a[2] * b[0] - a[0] * b[2];
    c[2] = a[0] * b[1] - a[1] * b[0];
}

// Unpack one record into 3-vectors (2D records get z = 0; their det_v is +z, unused).
void unpack(int beam, const double* r, double* first, double* ctr, double* u, double* v) {
    if (is_2d(beam)) {
        first[0] = r[0]; first[1] = r[1]; first[2] = 0.0;
        ctr[0] = r[2]; ctr[1] = r[3]; ctr[2] = 0.0;
        u[0] = r[4]; u[1] = r[5]; u[2] = 0.0;
        v[0] = 0.0; v[1] = 0.0; v[2] = 1.0;
    } else {
        for (int k = 0; k < 3; ++k) {
            first[k] = r[k]; ctr[k] = r[3 + k]; u[k] = r[6 + k]; v[k] = r[9 + k];
        }
    }
}

// Admission checks (diffct "Trajectories and Geometry", validation paragraph), float64.
bool admit_view(int beam, const double* r, double s, bool surface) {
    const int w = is_2d(beam) ? 6 : 12;
    for (int k = 0; k < w; ++k)
        if (!std::isfinite(r[k])) return false;
    double first[3], ctr[3], u[3], v[3];
    unpack(beam, r, first, ctr, u, v);
    const double tol = 1e-6;
    if (std::fabs(norm3(u) - 1.0) > tol) return false;
    if (!is_2d(beam) && std::fabs(norm3(v) - 1.0) > tol) return false;
    if (!is_2d(beam) && std::fabs(dot3(u, v)) > tol) return false;
    double n[3];
    if (is_2d(beam)) {
        n[0] = u[1]; n[1] = -u[0]; n[2] = 0.0;
    } else {
        cross3(u, v, n);
    }
    if (is_parallel(beam)) {
        if (std::fabs(norm3(first) - 1.0) > tol) return false;
        if (beam == CT_PARALLEL2D && std::fabs(dot3(first, u)) > tol) return false;
        if (beam == CT_PARALLEL3D && std::fabs(dot3(first, n)) <= tol) return false;
        if (norm3(ctr) > 1e6 * s) return false;
    } else {
        double sd[3] = {ctr[0] - first[0], ctr[1] - first[1], ctr[2] - first[2]};
        const double dist = norm3(sd);
        if (!(dist > 0.0)) return false;
        if (!surface && std::fabs(dot3(sd, n)) <= tol * dist) return false;  // edge-on detector
        const double rs = norm3(first), rc = norm3(ctr);
        if ((rs < rc ? rs : rc) > 1e6 * s) return false;
        if ((rs > rc ? rs : rc) > 1e15 * s) return false;
    }
    return true;
}

// Internal volume order: the axis that the 32 lanes of a warp run along (det_v or det_u,
// whichever is better aligned with it, view by view) should be the fastest in memory, so that
// a warp's 32 gathers or atomics fall into one or two 128-byte lines.
Layout choose_layout(int beam, int n_views, const double* views, int nz) {
    if (is_2d(beam) || nz == 1) return ct::LAYOUT_ZYX;
    const int w = 12;
    double score[3] = {0, 0, 0};
    for (int i = 0; i < n_views; ++i) {
        double first[3], ctr[3], u[3], v[3];
        unpack(beam, views + (int64_t)i * w, first, ctr, u, v);
        for (int a = 0; a < 3; ++a) score[a] += std::fmax(std::fabs(u[a]), std::fabs(v[a]));
    }
    // keep the caller's order unless another axis is clearly better (it costs two copies)
    int best = 0;
    for (int a = 1; a < 3; ++a)
        if (score[a] > 1.1 * score[best] && score[a] > score[best]) best = a;
    if (best == 2) return ct::LAYOUT_YXZ;
    if (best == 1) return ct::LAYOUT_ZXY;
    return ct::LAYOUT_ZYX;
}

void strides_for(Layout L, int nx, int ny, int nz, int32_t st[3]) {
    switch (L) {
        case ct::LAYOUT_YXZ:  // [y][x][z]
            st[2] = 1; st[0] = nz; st[1] = nz * nx;
            break;
        case ct::LAYOUT_ZXY:  // [z][x][y]
            st[1] = 1; st[0] = ny; st[2] = nx * ny;
            break;
        default:              // [z][y][x]
            st[0] = 1; st[1] = nx; st[2] = nx * ny;
            break;
    }
}

ct_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return CT_OK;
    if (e == cudaErrorMemoryAllocation) return CT_ERR_OUT_OF_MEMORY;
    return CT_ERR_CUDA;
}

// A pointer must be device or managed memory of the handle's device.
ct_status check_device_ptr(const void* p, int device) {
    if (p == nullptr) return CT_ERR_INVALID_ARGUMENT;
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CT_ERR_NOT_DEVICE_POINTER;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
        return CT_ERR_NOT_DEVICE_POINTER;
    if (at.type == cudaMemoryTypeDevice && at.device != device) return CT_ERR_NOT_DEVICE_POINTER;
    return CT_OK;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
    const uintptr_t x0 = (uintptr_t)a, x1 = x0 + na, y0 = (uintptr_t)b, y1 = y0 + nb;
    return x0 < y1 && y0 < x1;
}

size_t volume_bytes(const ct_geometry* g) { return (size_t)g->info.n_voxels * sizeof(float); }
size_t sino_bytes(const ct_geometry* g) { return (size_t)g->info.n_rays * sizeof(float); }

// Convert between the caller's [z][y][x] order and the internal order.
cudaError_t to_internal(const ct_geometry* g, const float* src, float* dst, cudaStream_t s) {
    const int64_t nx = g->info.nx, ny = g->info.ny, nz = g->info.nz;
    switch (g->info.volume_layout) {
        case ct::LAYOUT_YXZ: return ct::launch_transpose(src, dst, nz, ny * nx, 1, s);
        case ct::LAYOUT_ZXY: return ct::launch_transpose(src, dst, ny, nx, nz, s);
        default: return cudaErrorInvalidValue;
    }
}
cudaError_t from_internal(const ct_geometry* g, const float* src, float* dst, cudaStream_t s) {
    const int64_t nx = g->info.nx, ny = g->info.ny, nz = g->info.nz;
    switch (g->info.volume_layout) {
        case ct::LAYOUT_YXZ: return ct::launch_transpose(src, dst, ny * nx, nz, 1, s);
        case ct::LAYOUT_ZXY: return ct::launch_transpose(src, dst, nx, ny, nz, s);
        default: return cudaErrorInvalidValue;
    }
}

// Common argument checks for project/backproject.
ct_status check_call(const ct_geometry* g, const void* in, size_t in_bytes, const void* out,
                     size_t out_bytes, const void* ws, size_t ws_bytes, size_t ws_needed) {
    if (g == nullptr || in == nullptr || out == nullptr) return CT_ERR_INVALID_ARGUMENT;
    // kernels launch on the current device and read the handle's record table: they must be
    // the same device (checked before anything is queued)
    int current = -1;
    if (cudaGetDevice(&current) != cudaSuccess) {
        cudaGetLastError();
        return CT_ERR_CUDA;
    }
    if (current != g->device) return CT_ERR_INVALID_ARGUMENT;
    ct_status st;
    if ((st = check_device_ptr(in, g->device)) != CT_OK) return st;
    if ((st = check_device_ptr(out, g->device)) != CT_OK) return st;
    if (ws_needed > 0) {
        if (ws == nullptr || ws_bytes < ws_needed) return CT_ERR_WORKSPACE;
        if ((st = check_device_ptr(ws, g->device)) != CT_OK) return st;
    }
    if (overlap(in, in_bytes, out, out_bytes)) return CT_ERR_ALIASING;
    if (ws_needed > 0 && (overlap(ws, ws_needed, in, in_bytes) ||
                          overlap(ws, ws_needed, out, out_bytes)))
        return CT_ERR_ALIASING;
    // surface errors of earlier asynchronous work before queueing more
    cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CT_ERR_CUDA;
    }
    return CT_OK;
}

}  // namespace

extern "C" {

const char* ct_status_string(ct_status s) {
    switch (s) {
        case CT_OK: return "CT_OK";
        case CT_ERR_INVALID_ARGUMENT: return "CT_ERR_INVALID_ARGUMENT";
        case CT_ERR_INVALID_GEOMETRY: return "CT_ERR_INVALID_GEOMETRY";
        case CT_ERR_NOT_DEVICE_POINTER: return "CT_ERR_NOT_DEVICE_POINTER";
        case CT_ERR_ALIASING: return "CT_ERR_ALIASING";
        case CT_ERR_OUT_OF_MEMORY: return "CT_ERR_OUT_OF_MEMORY";
        case CT_ERR_CUDA: return "CT_ERR_CUDA";
        case CT_ERR_WORKSPACE: return "CT_ERR_WORKSPACE";
    }
    return "CT_ERR_UNKNOWN";
}

ct_status ct_geometry_create(ct_beam beam, int32_t n_views, const double* views, int32_t nz,
                             int32_t ny, int32_t nx, double voxel_spacing, int32_t n_u,
                             int32_t n_v, double du, double dv, ct_geometry** out) {
    const double s3[3] = {voxel_spacing, voxel_spacing, voxel_spacing};
    return ct_geometry_create_ex(beam, n_views, views, nz, ny, nx, s3, n_u, n_v, du, dv, out);
}

}  // extern "C"

namespace {

// Per-pixel admission for surface detectors ("Trajectories and Geometry": surface detectors
// validate each actual source/pixel pair): finite world points; for point sources every pixel
// distinct from the source in float32; the nearer endpoint within 1e6 voxel spacings of the
// origin and both within 1e15.
bool admit_surface(int beam, int32_t n_views, const double* views, int32_t n_u, int32_t n_v,
                   const double* off, double s) {
    const int w = is_2d(beam) ? 6 : 12;
    for (int64_t k = 0; k < (int64_t)n_u * n_v * 3; ++k)
        if (!std::isfinite(off[k])) return false;
    for (int i = 0; i < n_views; ++i) {
        double first[3], ctr[3], u[3], v[3], n[3];
        unpack(beam, views + (int64_t)i * w, first, ctr, u, v);
        if (is_2d(beam)) {
            n[0] = u[1]; n[1] = -u[0]; n[2] = 0.0;
        } else {
            cross3(u, v, n);
        }
        for (int64_t p = 0; p < (int64_t)n_u * n_v; ++p) {
            const double* o = off + p * 3;
            double pix[3];
            for (int a = 0; a < 3; ++a)
                pix[a] = ctr[a] + o[0] * u[a] + (is_2d(beam) ? 0.0 : o[1] * v[a]) + o[2] * n[a];
            if (!(std::isfinite(pix[0]) && std::isfinite(pix[1]) && std::isfinite(pix[2])))
                return false;
            const double rp = norm3(pix);
            if (is_parallel(beam)) {
                if (rp > 1e6 * s) return false;
            } else {
                if ((float)pix[0] == (float)first[0] && (float)pix[1] == (float)first[1] &&
                    (float)pix[2] == (float)first[2])
                    return false;
                const double rs = norm3(first);
                if ((rs < rp ? rs : rp) > 1e6 * s) return false;
                if ((rs > rp ? rs : rp) > 1e15 * s) return false;
            }
        }
    }
    return true;
}

// ---- slab tiling of the walks --------------------------------------------------------------

// Slab tiling is opt-in (ct_geometry_set_slabs): measured on the 512^3 spiral it cuts the walks'
// DRAM traffic about threefold but takes about four times as long, because every slab re-clips
// its rays in float64 and sloped rays of one detector column enter a slab at different points of
// their shared column path, so the lanes of a warp lose their lock-step.

// Per (view, detector v-tile), the first and last slab that the tile's rays can reach.  The
// rays of one detector row of a flat detector lie in one plane (through the source and the row,
// or through the row along the ray direction); the z of that plane over the box's xy rectangle
// is affine, so its extremes are at the rectangle's corners.  The union over the tile's rows,
// widened by two cells, bounds the z of every ray of the tile inside the box.
std::vector<int2> slab_ranges(const ct_geometry* g, int32_t h, int32_t n_slabs) {
    const ct_geometry_info& I = g->info;
    const int tiles_v = g->tiling.tiles_v;
    std::vector<int2> out((size_t)I.n_views * (size_t)tiles_v);
    const bool par = g->grid.parallel != 0;
    const double cx[2] = {0.0, (double)I.nx}, cy[2] = {0.0, (double)I.ny};
    for (int i = 0; i < I.n_views; ++i) {
        const ct::ViewRec& R = g->recs[(size_t)i];
        for (int vt = 0; vt < tiles_v; ++vt) {
            double zlo = INFINITY, zhi = -INFINITY;
            const int v1 = std::min(I.n_v, 32 * (vt + 1));
            for (int v = 32 * vt; v < v1; ++v) {
                double X0[3], D[3], N[3];
                for (int a = 0; a < 3; ++a) {
                    const double row = R.pb[a] + (double)v * R.pv[a];
                    X0[a] = par ? row : R.q[a];
                    D[a] = par ? R.q[a] : row;
                }
                cross3(D, R.pu, N);
                const double nn = norm3(N);
                if (!(nn > 0.0) || !(std::fabs(N[2]) > 1e-9 * nn)) {  // plane (nearly) contains z
                    zlo = -INFINITY;
                    zhi = INFINITY;
                    break;
                }
                for (int cxi = 0; cxi < 2; ++cxi)
                    for (int cyi = 0; cyi < 2; ++cyi) {
                        const double z = X0[2] - (N[0] * (cx[cxi] - X0[0]) +
                                                  N[1] * (cy[cyi] - X0[1])) / N[2];
                        zlo = std::min(zlo, z);
                        zhi = std::max(zhi, z);
                    }
            }
            int lo, hi;
            if (!(zhi >= -2.0) || !(zlo <= (double)I.nz + 2.0)) {
                lo = 1;  // no slab
                hi = 0;
            } else {
                const double a = std::max(zlo - 2.0, 0.0), b = std::min(zhi + 2.0, (double)I.nz);
                lo = std::min((int)std::floor(a / h), n_slabs - 1);
                hi = std::min((int)std::floor(b / h), n_slabs - 1);
            }
            out[(size_t)i * tiles_v + vt] = make_int2(lo, hi);
        }
    }
    return out;
}

// Sets the handle's slab height (0: no tiling) and uploads its per-slab tile lists
// (synchronous).  Within a slab the entries run v-tile first, then view, like the untiled grid.
ct_status set_slabs(ct_geometry* g, int32_t h) {
    int32_t* table = nullptr;
    int32_t n_slabs = 1;
    std::vector<int64_t> off;
    if (h > 0) {
        n_slabs = (int32_t)((g->info.nz + h - 1) / h);
        const std::vector<int2> r = slab_ranges(g, h, n_slabs);
        const int tiles_v = g->tiling.tiles_v;
        std::vector<int32_t> list;
        off.push_back(0);
        for (int32_t s = 0; s < n_slabs; ++s) {
            for (int vt = 0; vt < tiles_v; ++vt)
                for (int i = 0; i < g->info.n_views; ++i) {
                    const int2 rg = r[(size_t)i * tiles_v + vt];
                    if (s >= rg.x && s <= rg.y) list.push_back(i * tiles_v + vt);
                }
            off.push_back((int64_t)list.size());
        }
        cudaError_t e = cudaMalloc(&table, sizeof(int32_t) * std::max<size_t>(list.size(), 1));
        if (e == cudaSuccess && !list.empty())
            e = cudaMemcpy(table, list.data(), sizeof(int32_t) * list.size(),
                           cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            cudaGetLastError();
            if (table) cudaFree(table);
            return from_cuda(e);
        }
    }
    if (g->d_slab_tiles) cudaFree(g->d_slab_tiles);
    g->d_slab_tiles = table;
    g->slab_off = std::move(off);
    g->info.n_slabs = h > 0 ? n_slabs : 1;
    g->info.slab_cells = h > 0 ? h : g->info.nz;
    return CT_OK;
}

ct::SlabArgs slab_args(const ct_geometry* g, int32_t s) {
    ct::SlabArgs a;
    a.c0 = s * g->info.slab_cells;
    a.c1 = std::min(g->info.nz, (s + 1) * g->info.slab_cells);
    a.tiles = g->d_slab_tiles + g->slab_off[(size_t)s];
    a.n_tiles = (int32_t)(g->slab_off[(size_t)s + 1] - g->slab_off[(size_t)s]);
    return a;
}

ct_status create_impl(ct_beam beam, int32_t n_views, const double* views, int32_t nz, int32_t ny,
                      int32_t nx, const double* spacing_zyx, int32_t n_u, int32_t n_v, double du,
                      double dv, const double* offsets, ct_geometry** out) {
    if (out == nullptr) return CT_ERR_INVALID_ARGUMENT;
    *out = nullptr;
    const int b = (int)beam;
    if (b < CT_PARALLEL2D || b > CT_PARALLEL3D) return CT_ERR_INVALID_ARGUMENT;
    if (views == nullptr || n_views <= 0 || nz <= 0 || ny <= 0 || nx <= 0 || n_u <= 0 ||
        n_v <= 0)
        return CT_ERR_INVALID_ARGUMENT;
    if (is_2d(b)) {
        if (nz != 1 || n_v != 1) return CT_ERR_INVALID_ARGUMENT;
        dv = 1.0;
    }
    if (spacing_zyx == nullptr) return CT_ERR_INVALID_ARGUMENT;
    // spacing along x, y, z; a 2D grid has no z extent, its z pitch is unused (set to 1)
    const double sp[3] = {spacing_zyx[2], spacing_zyx[1], is_2d(b) ? 1.0 : spacing_zyx[0]};
    for (int a = 0; a < 3; ++a)
        if (!(std::isfinite(sp[a]) && sp[a] > 0.0)) return CT_ERR_INVALID_ARGUMENT;
    if (!(std::isfinite(du) && du > 0.0) || !(std::isfinite(dv) && dv > 0.0))
        return CT_ERR_INVALID_ARGUMENT;
    const double sp_min = std::min(sp[0], std::min(sp[1], is_2d(b) ? sp[1] : sp[2]));
    const bool iso = sp[0] == sp[1] && (is_2d(b) || sp[1] == sp[2]);
    const int64_t nvox = (int64_t)nz * ny * nx;
    if (nvox > (int64_t)INT32_MAX) return CT_ERR_INVALID_ARGUMENT;  // 32-bit voxel indices
    const int64_t tiles_u = is_2d(b) ? (n_u + 255) / 256 : (n_u + 31) / 32;
    const int64_t tiles_v = is_2d(b) ? 1 : (n_v + 31) / 32;
    if (tiles_u * tiles_v * n_views > (int64_t)INT32_MAX) return CT_ERR_INVALID_ARGUMENT;
    const int w = is_2d(b) ? 6 : 12;
    const bool surface = offsets != nullptr;
    for (int i = 0; i < n_views; ++i)
        if (!admit_view(b, views + (int64_t)i * w, sp_min, surface))
            return CT_ERR_INVALID_GEOMETRY;
    if (surface && !admit_surface(b, n_views, views, n_u, n_v, offsets, sp_min))
        return CT_ERR_INVALID_GEOMETRY;

    ct_geometry* g = new (std::nothrow) ct_geometry();
    if (g == nullptr) return CT_ERR_OUT_OF_MEMORY;
    g->host_views.assign(views, views + (int64_t)n_views * w);
    g->spacing = sp_min;
    g->du = du;
    g->dv = dv;
    ct_geometry_info& I = g->info;
    I.beam = b;
    I.n_views = n_views;
    I.nz = nz; I.ny = ny; I.nx = nx;
    I.n_u = n_u; I.n_v = n_v;
    I.n_rays = (int64_t)n_views * n_u * n_v;
    I.n_voxels = nvox;
    I.volume_layout = choose_layout(b, n_views, views, nz);
    I.workspace_bytes = I.volume_layout == ct::LAYOUT_ZYX ? 0 : align_up(volume_bytes(g));
    // SIRT: C, b (and x in the internal order), residual sinogram
    I.sirt_workspace_bytes = 2 * align_up(volume_bytes(g)) +
                             (I.volume_layout == ct::LAYOUT_ZYX ? 0 : align_up(volume_bytes(g))) +
                             align_up(sino_bytes(g));

    ct::Grid& G = g->grid;
    G.n[0] = nx; G.n[1] = ny; G.n[2] = nz;
    G.nd[0] = nx; G.nd[1] = ny; G.nd[2] = nz;
    strides_for((Layout)I.volume_layout, nx, ny, nz, G.stride);
    for (int a = 0; a < 3; ++a) G.sp[a] = (float)sp[a];
    G.iso = iso ? 1 : 0;
    G.parallel = is_parallel(b) ? 1 : 0;
    G.fast = I.volume_layout == ct::LAYOUT_YXZ ? 2 : (I.volume_layout == ct::LAYOUT_ZXY ? 1 : 0);
    ct::Tiling& T = g->tiling;
    T.n_views = n_views;
    T.n_u = n_u; T.n_v = n_v;
    T.tiles_u = (int32_t)tiles_u;
    T.tiles_v = (int32_t)tiles_v;
    T.two_d = is_2d(b) ? 1 : 0;

    // Per-view records in voxel units, origin at the lower box corner.
    const int fast = G.fast;
    std::vector<ct::ViewRec> recs((size_t)n_views);
    const double half[3] = {0.5 * nx * sp[0], 0.5 * ny * sp[1], 0.5 * nz * sp[2]};
    const double is[3] = {1.0 / sp[0], 1.0 / sp[1], 1.0 / sp[2]};
    for (int i = 0; i < n_views; ++i) {
        double first[3], ctr[3], u[3], v[3];
        unpack(b, views + (int64_t)i * w, first, ctr, u, v);
        ct::ViewRec& R = recs[(size_t)i];
        std::memset(&R, 0, sizeof(R));
        // coordinates in voxel units per axis (p_a + half_a) / spacing_a
        if (!surface) {
            const double cu = 0.5 * (n_u - 1), cv = is_2d(b) ? 0.0 : 0.5 * (n_v - 1);
            const double dvv = is_2d(b) ? 0.0 : dv;
            for (int a = 0; a < 3; ++a) {
                R.pu[a] = du * is[a] * u[a];
                R.pv[a] = dvv * is[a] * v[a];
                R.pb[a] = (ctr[a] + half[a]) * is[a] - cu * R.pu[a] - cv * R.pv[a];
            }
        } else {
            double n[3];
            if (is_2d(b)) {
                n[0] = u[1]; n[1] = -u[0]; n[2] = 0.0;
            } else {
                cross3(u, v, n);
            }
            for (int a = 0; a < 3; ++a) {
                R.pu[a] = is[a] * u[a];
                R.pv[a] = is_2d(b) ? 0.0 : is[a] * v[a];
                R.pn[a] = is[a] * n[a];
                R.pb[a] = (ctr[a] + half[a]) * is[a];
            }
        }
        if (is_parallel(b)) {
            // unit direction in physical space, expressed in voxel units per axis (for an
            // isotropic grid this is the physical unit vector itself)
            const double nr = norm3(first);
            for (int a = 0; a < 3; ++a) R.q[a] = iso ? first[a] / nr : first[a] / nr * is[a];
        } else {
            for (int a = 0; a < 3; ++a) {
                R.q[a] = (first[a] + half[a]) * is[a];
                R.pb[a] -= R.q[a];
            }
        }
        R.lanes_along_v = (!is_2d(b) && std::fabs(v[fast]) >= std::fabs(u[fast])) ? 1 : 0;
    }
    // The device's L2 size: the shared-line walks and the spread tiles widen the detector band
    // that resident blocks walk, which pays only while the volume stays in L2.
    int l2_bytes = 0;
    {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
            cudaGetLastError();
            l2_bytes = 0;
        }
    }
    const bool fits_l2 = nvox * (int64_t)sizeof(float) <= (int64_t)l2_bytes;
    // Spread backprojection tiles (a warp's lanes two pixels apart): 3D volumes that fit in L2,
    // every view running its lanes along the same detector axis (the tile shape follows it).
    // Measured: cone 256^3 backprojection 17.8 -> 17.1 ms; a 512^3 spiral 149 -> 200 ms and the
    // 2D fan 1.13 -> 1.55 ms, so neither takes them.
    if (!is_2d(b) && fits_l2) {
        bool same = true;
        for (int i = 1; same && i < n_views; ++i)
            same = recs[(size_t)i].lanes_along_v == recs[0].lanes_along_v;
        if (same) {
            const bool along_v = recs[0].lanes_along_v != 0;
            const int64_t su = along_v ? (n_u + 15) / 16 : (n_u + 63) / 64;
            const int64_t sv = along_v ? (n_v + 63) / 64 : (n_v + 15) / 16;
            if (su * sv * n_views <= (int64_t)INT32_MAX) {
                T.spread = along_v ? 1 : 2;
                T.spread_tiles_u = (int32_t)su;
                T.spread_tiles_v = (int32_t)sv;
            }
        }
    }
    // Shared-line forward projections: 3D flat detectors whose lane-axis vector (pv for lanes
    // along v, else pu) has no component on either outer axis in every view, with the lanes along
    // the same detector axis in every view, so that the pixels of one detector line share their
    // outer-axis line; and a volume no larger than L2 (measured: a 256^3 cone projects 22 %
    // faster, a 512^3 helix 12 % slower, its lines' wider bands outgrowing L2).
    {
        const int oa = fast == 0 ? 1 : 0, ob = fast == 2 ? 1 : 2;
        bool line = !is_2d(b) && !surface && nx + ny + nz - G.n[fast] <= ct::kLineMaxCells &&
                    fits_l2;
        for (int i = 0; line && i < n_views; ++i) {
            const ct::ViewRec& R = recs[(size_t)i];
            const double* lane = R.lanes_along_v ? R.pv : R.pu;
            line = lane[oa] == 0.0 && lane[ob] == 0.0 && R.lanes_along_v == recs[0].lanes_along_v;
        }
        if (line) {
            const int64_t n_lane = recs[0].lanes_along_v ? n_v : n_u;
            const int64_t n_line = recs[0].lanes_along_v ? n_u : n_v;
            const int64_t lane_tiles = (n_lane + ct::kLinePixels - 1) / ct::kLinePixels;
            const int64_t line_tiles = (n_line + ct::kLineRows - 1) / ct::kLineRows;
            if (lane_tiles * line_tiles * n_views <= (int64_t)INT32_MAX) {
                T.line = recs[0].lanes_along_v ? 1 : 2;
                I.shared_lines = T.line;
                T.line_lane_tiles = (int32_t)lane_tiles;
                T.line_row_tiles = (int32_t)line_tiles;
            }
        }
    }
    cudaError_t e = cudaGetDevice(&g->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&g->sm_count, cudaDevAttrMultiProcessorCount, g->device);
    if (e == cudaSuccess) e = cudaMalloc(&g->d_views, sizeof(ct::ViewRec) * (size_t)n_views);
    if (e == cudaSuccess)
        e = cudaMemcpy(g->d_views, recs.data(), sizeof(ct::ViewRec) * (size_t)n_views,
                       cudaMemcpyHostToDevice);
    const size_t raw_bytes = sizeof(double) * (size_t)n_views * (size_t)w;
    if (e == cudaSuccess) e = cudaMalloc(&g->d_raw, raw_bytes);
    if (e == cudaSuccess) e = cudaMemcpy(g->d_raw, views, raw_bytes, cudaMemcpyHostToDevice);
    const size_t off_bytes = sizeof(double) * 3 * (size_t)n_u * (size_t)n_v;
    if (e == cudaSuccess && surface) e = cudaMalloc(&g->d_offsets, off_bytes);
    if (e == cudaSuccess && surface)
        e = cudaMemcpy(g->d_offsets, offsets, off_bytes, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaGetLastError();
        if (g->d_views) cudaFree(g->d_views);
        if (g->d_offsets) cudaFree(g->d_offsets);
        if (g->d_raw) cudaFree(g->d_raw);
        delete g;
        return from_cuda(e);
    }
    G.offsets = g->d_offsets;
    G.nv = n_v;
    g->recs = std::move(recs);
    g->info.n_slabs = 1;
    g->info.slab_cells = nz;
    *out = g;
    return CT_OK;
}

// The handle's tiling with the shared-line walks off: the SIRT and CGLS iterations, whose fused
// kernels walk per ray, take every walk that way so that their A^T is the transpose of their A.
ct::Tiling per_ray_tiling(const ct_geometry* g) {
    ct::Tiling t = g->tiling;
    t.line = 0;
    return t;
}

}  // namespace

extern "C" {

ct_status ct_geometry_create_ex(ct_beam beam, int32_t n_views, const double* views, int32_t nz,
                                int32_t ny, int32_t nx, const double* spacing_zyx, int32_t n_u,
                                int32_t n_v, double du, double dv, ct_geometry** out) {
    return create_impl(beam, n_views, views, nz, ny, nx, spacing_zyx, n_u, n_v, du, dv, nullptr,
                       out);
}

ct_status ct_geometry_create_surface(ct_beam beam, int32_t n_views, const double* views,
                                     int32_t nz, int32_t ny, int32_t nx,
                                     const double* spacing_zyx, int32_t n_u, int32_t n_v,
                                     const double* offsets_uvn, ct_geometry** out) {
    if (offsets_uvn == nullptr) {
        if (out) *out = nullptr;
        return CT_ERR_INVALID_ARGUMENT;
    }
    return create_impl(beam, n_views, views, nz, ny, nx, spacing_zyx, n_u, n_v, 1.0, 1.0,
                       offsets_uvn, out);
}

ct_status ct_geometry_destroy(ct_geometry* g) {
    if (g == nullptr) return CT_OK;
    cudaError_t e = cudaSuccess;
    if (g->d_views) e = cudaFree(g->d_views);
    if (g->d_slab_tiles) {
        const cudaError_t e2 = cudaFree(g->d_slab_tiles);
        if (e == cudaSuccess) e = e2;
    }
    if (g->d_offsets) {
        const cudaError_t e2 = cudaFree(g->d_offsets);
        if (e == cudaSuccess) e = e2;
    }
    if (g->d_raw) {
        const cudaError_t e2 = cudaFree(g->d_raw);
        if (e == cudaSuccess) e = e2;
    }
    delete g;
    return from_cuda(e);
}

ct_status ct_geometry_get_info(const ct_geometry* g, ct_geometry_info* info) {
    if (g == nullptr || info == nullptr) return CT_ERR_INVALID_ARGUMENT;
    *info = g->info;
    return CT_OK;
}

ct_status ct_geometry_set_slabs(ct_geometry* g, int32_t slab_cells) {
    if (g == nullptr || slab_cells < 0) return CT_ERR_INVALID_ARGUMENT;
    if (g->info.volume_layout != ct::LAYOUT_YXZ || g->d_offsets != nullptr)
        return CT_ERR_INVALID_ARGUMENT;
    int current = -1;
    if (cudaGetDevice(&current) != cudaSuccess) {
        cudaGetLastError();
        return CT_ERR_CUDA;
    }
    if (current != g->device) return CT_ERR_INVALID_ARGUMENT;
    int64_t h = slab_cells == 0 ? 0 : ((int64_t)slab_cells + 31) / 32 * 32;
    if (h >= g->info.nz) h = 0;  // one slab: no tiling
    return set_slabs(g, (int32_t)h);
}

ct_status ct_project(const ct_geometry* g, const float* d_volume, float* d_sino,
                     void* d_workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (g == nullptr) return CT_ERR_INVALID_ARGUMENT;
    ct_status st = check_call(g, d_volume, volume_bytes(g), d_sino, sino_bytes(g), d_workspace,
                              workspace_bytes, g->info.workspace_bytes);
    if (st != CT_OK) return st;
    const float* vol = d_volume;
    if (g->info.volume_layout != ct::LAYOUT_ZYX) {
        float* tmp = static_cast<float*>(d_workspace);
        if ((st = from_cuda(to_internal(g, d_volume, tmp, stream))) != CT_OK) return st;
        vol = tmp;
    }
    if (g->info.n_slabs > 1) {
        // every ray's partial sums over the slabs are added to its cleared entry, slab by slab
        cudaError_t e = cudaMemsetAsync(d_sino, 0, sino_bytes(g), stream);
        for (int32_t s = 0; s < g->info.n_slabs && e == cudaSuccess; ++s)
            e = ct::launch_project_slab(g->d_views, g->grid, g->tiling, 1, vol, 0, d_sino, 0,
                                        slab_args(g, s), stream);
        return from_cuda(e);
    }
    return from_cuda(ct::launch_project(g->d_views, g->grid, g->tiling, vol, d_sino, stream));
}

ct_status ct_backproject(const ct_geometry* g, const float* d_sino, float* d_volume,
                         void* d_workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (g == nullptr) return CT_ERR_INVALID_ARGUMENT;
    ct_status st = check_call(g, d_sino, sino_bytes(g), d_volume, volume_bytes(g), d_workspace,
                              workspace_bytes, g->info.workspace_bytes);
    if (st != CT_OK) return st;
    float* acc = g->info.volume_layout == ct::LAYOUT_ZYX ? d_volume
                                                          : static_cast<float*>(d_workspace);
    if ((st = from_cuda(cudaMemsetAsync(acc, 0, volume_bytes(g), stream))) != CT_OK) return st;
    if (g->info.n_slabs > 1) {
        cudaError_t e = cudaSuccess;
        for (int32_t s = 0; s < g->info.n_slabs && e == cudaSuccess; ++s)
            e = ct::launch_backproject_slab(g->d_views, g->grid, g->tiling, 1, d_sino, 0, acc, 0,
                                            slab_args(g, s), stream);
        if ((st = from_cuda(e)) != CT_OK) return st;
    } else if ((st = from_cuda(ct::launch_backproject(g->d_views, g->grid, g->tiling, d_sino, acc,
                                                      stream))) != CT_OK) {
        return st;
    }
    if (acc != d_volume) return from_cuda(from_internal(g, acc, d_volume, stream));
    return CT_OK;
}

size_t ct_sirt_workspace_bytes(const ct_geometry* g) {
    return g == nullptr ? 0 : g->info.sirt_workspace_bytes;
}

ct_status ct_sirt_iterate(const ct_geometry* g, float* d_x, const float* d_y, void* d_workspace,
                          size_t workspace_bytes, int32_t n_iters, float relaxation,
                          int32_t workspace_initialised, cudaStream_t stream) {
    if (g == nullptr || n_iters < 0 || !(relaxation > 0.0f && relaxation < 2.0f))
        return CT_ERR_INVALID_ARGUMENT;
    ct_status st = check_call(g, d_y, sino_bytes(g), d_x, volume_bytes(g), d_workspace,
                              workspace_bytes, g->info.sirt_workspace_bytes);
    if (st != CT_OK) return st;
    if (overlap(d_x, volume_bytes(g), d_y, sino_bytes(g))) return CT_ERR_ALIASING;
    const int64_t nvox = g->info.n_voxels;
    const size_t vb = align_up(volume_bytes(g));
    char* ws = static_cast<char*>(d_workspace);
    float* C = reinterpret_cast<float*>(ws);
    float* B = reinterpret_cast<float*>(ws + vb);
    const bool native = g->info.volume_layout == ct::LAYOUT_ZYX;
    float* X = native ? d_x : reinterpret_cast<float*>(ws + 2 * vb);
    float* Rres = reinterpret_cast<float*>(ws + (native ? 2 : 3) * vb);
    // the fused solver kernels walk per ray, so every walk of the iteration does
    const ct::Tiling rays = per_ray_tiling(g);
    cudaError_t e = cudaSuccess;
    if (!workspace_initialised) {
        // C = 1 / (A^T 1), b = 0
        e = cudaMemsetAsync(C, 0, volume_bytes(g), stream);
        if (e == cudaSuccess) e = ct::launch_backproject_ones(g->d_views, g->grid, rays, C, stream);
        if (e == cudaSuccess) e = ct::launch_invert(C, nvox, stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(B, 0, volume_bytes(g), stream);
        if (e != cudaSuccess) return from_cuda(e);
    }
    if (n_iters == 0) return CT_OK;
    if (!native && (e = to_internal(g, d_x, X, stream)) != cudaSuccess) return from_cuda(e);
    for (int it = 0; it < n_iters && e == cudaSuccess; ++it) {
        e = ct::launch_project_residual(g->d_views, g->grid, rays, X, d_y, Rres, stream);
        if (e == cudaSuccess) e = ct::launch_backproject(g->d_views, g->grid, rays, Rres, B, stream);
        if (e == cudaSuccess) e = ct::launch_sirt_update(X, B, C, relaxation, nvox, stream);
    }
    if (e == cudaSuccess && !native) e = from_internal(g, X, d_x, stream);
    return from_cuda(e);
}

// ---- batches of volumes ---------------------------------------------------------------------

// Volumes per batched launch: 4, 2 or 1 (the kernels are instantiated for these).
static int chunk_of(int remaining) { return remaining >= 4 ? 4 : (remaining >= 2 ? 2 : 1); }

size_t ct_batch_workspace_bytes(const ct_geometry* g, int32_t batch) {
    if (g == nullptr || batch <= 0) return 0;
    if (g->info.volume_layout == ct::LAYOUT_ZYX) return 0;
    return (size_t)std::min(batch, 4) * align_up(volume_bytes(g));
}

// The byte sizes of `batch` volumes and sinograms fit in size_t.
static bool batch_fits(const ct_geometry* g, int32_t batch) {
    const size_t most = std::max(volume_bytes(g), sino_bytes(g));
    return most == 0 || (size_t)batch <= SIZE_MAX / most;
}

ct_status ct_project_batch(const ct_geometry* g, int32_t batch, const float* d_volumes,
                           float* d_sinos, void* d_workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
    if (g == nullptr || batch <= 0 || !batch_fits(g, batch)) return CT_ERR_INVALID_ARGUMENT;
    ct_status st = check_call(g, d_volumes, (size_t)batch * volume_bytes(g), d_sinos,
                              (size_t)batch * sino_bytes(g), d_workspace, workspace_bytes,
                              ct_batch_workspace_bytes(g, batch));
    if (st != CT_OK) return st;
    const int64_t nvox = g->info.n_voxels, nray = g->info.n_rays;
    const bool native = g->info.volume_layout == ct::LAYOUT_ZYX;
    const int64_t wstride = (int64_t)(align_up(volume_bytes(g)) / sizeof(float));
    float* ws = static_cast<float*>(d_workspace);
    cudaError_t e = cudaSuccess;
    for (int b0 = 0; b0 < batch && e == cudaSuccess;) {
        const int nb = chunk_of(batch - b0);
        const float* vol = d_volumes + (int64_t)b0 * nvox;
        int64_t vstride = nvox;
        if (!native) {
            for (int j = 0; j < nb && e == cudaSuccess; ++j)
                e = to_internal(g, d_volumes + (int64_t)(b0 + j) * nvox, ws + j * wstride, stream);
            vol = ws;
            vstride = wstride;
        }
        float* sinos = d_sinos + (int64_t)b0 * nray;
        if (e == cudaSuccess && g->info.n_slabs > 1) {
            e = cudaMemsetAsync(sinos, 0, (size_t)nb * sino_bytes(g), stream);
            for (int32_t s = 0; s < g->info.n_slabs && e == cudaSuccess; ++s)
                e = ct::launch_project_slab(g->d_views, g->grid, g->tiling, nb, vol, vstride, sinos,
                                            nray, slab_args(g, s), stream);
        } else if (e == cudaSuccess) {
            e = ct::launch_project_batch(g->d_views, g->grid, g->tiling, nb, vol, vstride, sinos,
                                         nray, stream);
        }
        b0 += nb;
    }
    return from_cuda(e);
}

ct_status ct_backproject_batch(const ct_geometry* g, int32_t batch, const float* d_sinos,
                               float* d_volumes, void* d_workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
    if (g == nullptr || batch <= 0 || !batch_fits(g, batch)) return CT_ERR_INVALID_ARGUMENT;
    ct_status st = check_call(g, d_sinos, (size_t)batch * sino_bytes(g), d_volumes,
                              (size_t)batch * volume_bytes(g), d_workspace, workspace_bytes,
                              ct_batch_workspace_bytes(g, batch));
    if (st != CT_OK) return st;
    const int64_t nvox = g->info.n_voxels, nray = g->info.n_rays;
    const bool native = g->info.volume_layout == ct::LAYOUT_ZYX;
    const int64_t wstride = (int64_t)(align_up(volume_bytes(g)) / sizeof(float));
    float* ws = static_cast<float*>(d_workspace);
    cudaError_t e = cudaSuccess;
    for (int b0 = 0; b0 < batch && e == cudaSuccess;) {
        const int nb = chunk_of(batch - b0);
        float* acc = native ? d_volumes + (int64_t)b0 * nvox : ws;
        const int64_t vstride = native ? nvox : wstride;
        e = cudaMemsetAsync(acc, 0, (size_t)((nb - 1) * vstride + nvox) * sizeof(float), stream);
        const float* sinos = d_sinos + (int64_t)b0 * nray;
        if (e == cudaSuccess && g->info.n_slabs > 1) {
            for (int32_t s = 0; s < g->info.n_slabs && e == cudaSuccess; ++s)
                e = ct::launch_backproject_slab(g->d_views, g->grid, g->tiling, nb, sinos, nray, acc,
                                                vstride, slab_args(g, s), stream);
        } else if (e == cudaSuccess) {
            e = ct::launch_backproject_batch(g->d_views, g->grid, g->tiling, nb, sinos, nray, acc,
                                             vstride, stream);
        }
        if (!native)
            for (int j = 0; j < nb && e == cudaSuccess; ++j)
                e = from_internal(g, ws + j * wstride, d_volumes + (int64_t)(b0 + j) * nvox,
                                  stream);
        b0 += nb;
    }
    return from_cuda(e);
}

// ---- CGLS -------------------------------------------------------------------------------------

// Workspace of ct_cgls_iterate: x in the internal order (unless that is the caller's), p, s,
// r, q, the partial sums of one reduction, and the four float64 scalars.
struct CglsLayout {
    size_t x, p, s, r, q, partials, scal, total;
};

static CglsLayout cgls_layout(const ct_geometry* g) {
    const size_t vb = align_up(volume_bytes(g)), sb = align_up(sino_bytes(g));
    const int64_t parts =
        std::max<int64_t>(ct::project_blocks(g->tiling), ct::norm_blocks(g->sm_count));
    CglsLayout L{};
    size_t off = 0;
    const bool native = g->info.volume_layout == ct::LAYOUT_ZYX;
    L.x = off; off += native ? 0 : vb;
    L.p = off; off += vb;
    L.s = off; off += vb;
    L.r = off; off += sb;
    L.q = off; off += sb;
    L.partials = off; off += align_up((size_t)parts * sizeof(double));
    L.scal = off; off += align_up(4 * sizeof(double));
    L.total = off;
    return L;
}

size_t ct_cgls_workspace_bytes(const ct_geometry* g) {
    return g == nullptr ? 0 : cgls_layout(g).total;
}

ct_status ct_cgls_iterate(const ct_geometry* g, float* d_x, const float* d_y, void* d_workspace,
                          size_t workspace_bytes, int32_t n_iters, int32_t workspace_initialised,
                          cudaStream_t stream) {
    if (g == nullptr || n_iters < 0) return CT_ERR_INVALID_ARGUMENT;
    const CglsLayout L = cgls_layout(g);
    ct_status st = check_call(g, d_y, sino_bytes(g), d_x, volume_bytes(g), d_workspace,
                              workspace_bytes, L.total);
    if (st != CT_OK) return st;
    const int64_t nvox = g->info.n_voxels, nray = g->info.n_rays;
    char* ws = static_cast<char*>(d_workspace);
    const bool native = g->info.volume_layout == ct::LAYOUT_ZYX;
    float* X = native ? d_x : reinterpret_cast<float*>(ws + L.x);
    float* P = reinterpret_cast<float*>(ws + L.p);
    float* S = reinterpret_cast<float*>(ws + L.s);
    float* R = reinterpret_cast<float*>(ws + L.r);
    float* Q = reinterpret_cast<float*>(ws + L.q);
    double* parts = reinterpret_cast<double*>(ws + L.partials);
    double* scal = reinterpret_cast<double*>(ws + L.scal);
    // the fused solver kernels walk per ray, so every walk of the iteration does
    const ct::Tiling rays = per_ray_tiling(g);
    const int64_t fp_parts = ct::project_blocks(rays),
                  nrm_parts = ct::norm_blocks(g->sm_count);
    const ct::ViewRec* V = g->d_views;
    cudaError_t e = cudaSuccess;
    if (!native) e = to_internal(g, d_x, X, stream);
    if (e == cudaSuccess && !workspace_initialised) {
        // r = y - A x;  s = A^T r;  p = s;  gamma = |s|^2
        e = ct::launch_project(V, g->grid, rays, X, Q, stream);
        if (e == cudaSuccess) e = ct::launch_sub(R, d_y, Q, nray, stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(S, 0, volume_bytes(g), stream);
        if (e == cudaSuccess) e = ct::launch_backproject(V, g->grid, rays, R, S, stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(P, 0, volume_bytes(g), stream);
        if (e == cudaSuccess) e = ct::launch_norm_partials(S, nvox, parts, g->sm_count, stream);
        if (e == cudaSuccess) e = ct::launch_cgls_scalars(parts, nrm_parts, scal, 2, stream);
        if (e == cudaSuccess) e = ct::launch_cgls_update(X, P, S, scal, nvox, stream);
    }
    for (int it = 0; it < n_iters && e == cudaSuccess; ++it) {
        // q = A p, delta = |q|^2, alpha = gamma / delta
        e = ct::launch_project_norm(V, g->grid, rays, P, Q, parts, stream);
        if (e == cudaSuccess) e = ct::launch_cgls_scalars(parts, fp_parts, scal, 0, stream);
        // r -= alpha q, s = A^T r (s is zero here)
        if (e == cudaSuccess)
            e = ct::launch_backproject_residual(V, g->grid, rays, R, Q, scal, S, stream);
        // beta = |s|^2 / gamma, gamma = |s|^2
        if (e == cudaSuccess) e = ct::launch_norm_partials(S, nvox, parts, g->sm_count, stream);
        if (e == cudaSuccess) e = ct::launch_cgls_scalars(parts, nrm_parts, scal, 1, stream);
        // x += alpha p, p = s + beta p, s = 0
        if (e == cudaSuccess) e = ct::launch_cgls_update(X, P, S, scal, nvox, stream);
    }
    if (e == cudaSuccess && !native) e = from_internal(g, X, d_x, stream);
    return from_cuda(e);
}

}  // extern "C"

// ---- backprojection without allocation (scratch in a fixed device array) -------------------
//
// Some callers cannot allocate device memory when they backproject: code running inside a
// framework that hands it only a stream and its input/output pointers (a plugin or operator with
// no access to an allocator), real-time pipelines that forbid allocation after start-up, and
// programs that keep every device byte in a pool of their own.  For them the accumulator that
// ct_backproject keeps in the caller's workspace lives here in one static device array instead.
namespace {

__device__ __align__(256) float g_ct_static_scratch[CT_STATIC_SCRATCH_VOXELS];

constexpr int kMaxStaticDevices = 64;
std::mutex g_static_mu;
// Device address of the array per device, and the id of the context it was looked up in.  A
// device reset destroys the context (and with it the module and the address); the next call
// then runs in a new context with another id and looks the address up again.
float* g_static_scratch_ptr[kMaxStaticDevices];
unsigned long long g_static_scratch_ctx[kMaxStaticDevices];

// Driver entry points for the current context's id, fetched through the runtime (the library
// does not link the driver library itself).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

ct_status current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    if (get_current == nullptr || get_id == nullptr) {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault,
                                             &q1) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
                cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess ||
            f1 == nullptr || f2 == nullptr) {
            cudaGetLastError();
            return CT_ERR_CUDA;
        }
        get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
        get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return CT_ERR_CUDA;
    if (get_id(ctx, id) != CUDA_SUCCESS) return CT_ERR_CUDA;
    return CT_OK;
}

// Device address of the static array on `device`, which must be the current device.  The
// first call per device and context looks the address up (this may load the module on that
// device); later calls in the same context reuse it.
ct_status static_scratch_on(int device, float** out) {
    if (device < 0 || device >= kMaxStaticDevices) return CT_ERR_INVALID_ARGUMENT;
    std::lock_guard<std::mutex> lock(g_static_mu);
    unsigned long long ctx = 0;
    const ct_status st = current_context_id(&ctx);
    if (st != CT_OK) return st;
    if (g_static_scratch_ptr[device] == nullptr || g_static_scratch_ctx[device] != ctx) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_ct_static_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return CT_ERR_CUDA;
        }
        g_static_scratch_ptr[device] = static_cast<float*>(p);
        g_static_scratch_ctx[device] = ctx;
    }
    *out = g_static_scratch_ptr[device];
    return CT_OK;
}

}  // namespace

extern "C" ct_status ct_backproject_static(const ct_geometry* g, const float* d_sino,
                                           float* d_volume, cudaStream_t stream) {
    if (g == nullptr) return CT_ERR_INVALID_ARGUMENT;
    int current = -1;
    if (cudaGetDevice(&current) != cudaSuccess) {
        cudaGetLastError();
        return CT_ERR_CUDA;
    }
    if (current != g->device) return CT_ERR_INVALID_ARGUMENT;
    ct_status st = check_call(g, d_sino, sino_bytes(g), d_volume, volume_bytes(g), nullptr, 0, 0);
    if (st != CT_OK) return st;
    if (g->info.volume_layout == ct::LAYOUT_ZYX) {
        // this geometry needs no scratch: accumulate straight into the caller's volume
        cudaError_t e = cudaMemsetAsync(d_volume, 0, volume_bytes(g), stream);
        if (e == cudaSuccess)
            e = ct::launch_backproject(g->d_views, g->grid, g->tiling, d_sino, d_volume, stream);
        return from_cuda(e);
    }
    if (g->info.n_voxels > (int64_t)CT_STATIC_SCRATCH_VOXELS) return CT_ERR_WORKSPACE;
    float* acc = nullptr;
    if ((st = static_scratch_on(g->device, &acc)) != CT_OK) return st;
    // the array keeps the previous call's sums: clear the part this call accumulates into
    cudaError_t e = cudaMemsetAsync(acc, 0, volume_bytes(g), stream);
    if (e == cudaSuccess)
        e = ct::launch_backproject(g->d_views, g->grid, g->tiling, d_sino, acc, stream);
    if (e == cudaSuccess) e = from_internal(g, acc, d_volume, stream);
    return from_cuda(e);
}

// ---------------------------------------------------------------------------------------------
// Filtered backprojection.

namespace {

enum FbpMode { kFbpForward = 0, kFbpTranspose = 1, kFbpGradients = 2 };

struct FbpLayout {
    int32_t rows, cols;  // padded filtered sinogram of one view
    int32_t bu, bv;      // 2 x 2 blocks (2D: pairs) per view and parity copy
    size_t views, cosines, taps, filtered, copies, acc, total;
};

// Scratch: per-view constants and taps, then (forward) the padded filtered sinogram, (transpose)
// the parity copies of the padded detector (4 copies of 2 x 2 blocks; 2D 2 copies of pairs), or
// (gradients) both plus 2 n_u - 1 doubles.
FbpLayout fbp_layout(const ct_geometry* g, FbpMode mode) {
    FbpLayout L;
    const size_t nv = (size_t)g->info.n_views;
    const bool two_d = is_2d(g->info.beam);
    L.rows = g->info.n_u + 3;
    L.cols = two_d ? 1 : g->info.n_v + 3;
    L.bu = (g->info.n_u + 2) / 2 + 1;
    L.bv = two_d ? 1 : (g->info.n_v + 2) / 2 + 1;
    L.views = 0;
    L.cosines = align_up(sizeof(ct::FbpView) * nv);
    L.taps = L.cosines + align_up(sizeof(ct::FbpCosine) * nv);
    size_t off = L.taps + align_up(sizeof(float) * (size_t)(2 * g->info.n_u - 1));
    const size_t padded = sizeof(float) * nv * (size_t)L.rows * (size_t)L.cols;
    const size_t copies = two_d ? sizeof(float) * 4 * nv * (size_t)L.bu
                                : sizeof(float) * 16 * nv * (size_t)L.bu * (size_t)L.bv;
    L.filtered = L.copies = L.acc = off;
    if (mode != kFbpTranspose) {
        L.filtered = off;
        off += align_up(padded);
    }
    if (mode != kFbpForward) {
        L.copies = off;
        off += align_up(copies);
    }
    if (mode == kFbpGradients) {
        L.acc = off;
        off += align_up(sizeof(double) * (size_t)(2 * g->info.n_u - 1));
    }
    L.total = off;
    return L;
}

constexpr int32_t kFbpMaxU = 16384;

}  // namespace

extern "C" size_t ct_fbp_workspace_bytes(const ct_geometry* g) {
    return g == nullptr ? 0 : fbp_layout(g, kFbpForward).total;
}

extern "C" size_t ct_fbp_transpose_workspace_bytes(const ct_geometry* g) {
    return g == nullptr ? 0 : fbp_layout(g, kFbpTranspose).total;
}

extern "C" size_t ct_fbp_gradients_workspace_bytes(const ct_geometry* g) {
    return g == nullptr ? 0 : fbp_layout(g, kFbpGradients).total;
}

namespace {

// Isocentre estimated from the detector normals ("Analytical Reconstruction Helpers": the default
// isocentre is estimated from the detector normals): the least-squares point nearest the lines
// {c_k + s n_k} through each detector centre along its unit normal,
// (sum_k P_k + eps I) x = sum_k P_k c_k with P_k = I - n_k n_k^T and
// eps = 1e-9 trace(sum_k P_k) / dim, so that rank-deficient sets (one view, parallel normals) give
// the minimum-norm point.  2D geometries solve in the plane.  Float64, Gaussian elimination with
// partial pivoting on the symmetric positive definite system.
void estimate_isocenter(const ct_geometry* g, double* iso) {
    const int b = g->info.beam;
    const int dim = is_2d(b) ? 2 : 3;
    const int w = is_2d(b) ? 6 : 12;
    double M[3][3] = {}, rhs[3] = {};
    for (int k = 0; k < g->info.n_views; ++k) {
        double first[3], ctr[3], u[3], v[3], n[3];
        unpack(b, g->host_views.data() + (int64_t)k * w, first, ctr, u, v);
        if (is_2d(b)) {
            n[0] = u[1]; n[1] = -u[0]; n[2] = 0.0;
        } else {
            cross3(u, v, n);
        }
        double nn = 0.0;
        for (int a = 0; a < dim; ++a) nn += n[a] * n[a];
        nn = std::sqrt(nn);
        for (int a = 0; a < dim; ++a) n[a] /= nn;
        for (int r = 0; r < dim; ++r) {
            for (int c = 0; c < dim; ++c) {
                const double P = (r == c ? 1.0 : 0.0) - n[r] * n[c];
                M[r][c] += P;
                rhs[r] += P * ctr[c];
            }
        }
    }
    double tr = 0.0;
    for (int a = 0; a < dim; ++a) tr += M[a][a];
    for (int a = 0; a < dim; ++a) M[a][a] += 1e-9 * tr / dim;
    for (int col = 0; col < dim; ++col) {
        int piv = col;
        for (int r = col + 1; r < dim; ++r)
            if (std::fabs(M[r][col]) > std::fabs(M[piv][col])) piv = r;
        if (piv != col) {
            for (int c = 0; c < dim; ++c) std::swap(M[col][c], M[piv][c]);
            std::swap(rhs[col], rhs[piv]);
        }
        for (int r = col + 1; r < dim; ++r) {
            const double f = M[r][col] / M[col][col];
            for (int c = col; c < dim; ++c) M[r][c] -= f * M[col][c];
            rhs[r] -= f * rhs[col];
        }
    }
    for (int r = dim - 1; r >= 0; --r) {
        double acc = rhs[r];
        for (int c = r + 1; c < dim; ++c) acc -= M[r][c] * iso[c];
        iso[r] = acc / M[r][r];
    }
    if (dim == 2) iso[2] = 0.0;
}

// Device buffer of `bytes` given by the caller: device memory of the handle's device, not
// overlapping `out` or the workspace.
ct_status check_input(const ct_geometry* g, const void* ptr, size_t bytes, const void* out,
                      size_t out_bytes, const void* ws, size_t ws_bytes) {
    ct_status st = check_device_ptr(ptr, g->device);
    if (st != CT_OK) return st;
    if (overlap(ptr, bytes, out, out_bytes) || overlap(ptr, bytes, ws, ws_bytes))
        return CT_ERR_ALIASING;
    return CT_OK;
}

// Argument checks shared by the FBP entry points; fills the kernel parameters.
ct_status fbp_setup(const ct_geometry* g, const void* in, size_t in_bytes, const void* out,
                    size_t out_bytes, const ct_fbp_options* opt, const void* d_workspace,
                    size_t workspace_bytes, FbpMode mode, ct::FbpParams* P, FbpLayout* L) {
    if (g == nullptr) return CT_ERR_INVALID_ARGUMENT;
    ct_fbp_options o;
    if (opt != nullptr) {
        o = *opt;
    } else {
        std::memset(&o, 0, sizeof(o));
        o.window = CT_WINDOW_RAM_LAK;
    }
    const int b = g->info.beam;
    if (b == CT_PARALLEL3D || g->d_offsets != nullptr) return CT_ERR_INVALID_ARGUMENT;
    if ((int)o.window < CT_WINDOW_RAM_LAK || (int)o.window > CT_WINDOW_HANN)
        return CT_ERR_INVALID_ARGUMENT;
    if (g->info.n_u > kFbpMaxU) return CT_ERR_INVALID_ARGUMENT;
    // gather grid limits: 3D (ceil(nz/32), ceil(nx/8), ny), 2D (ceil(nx/32), ceil(ny/8))
    if (is_2d(b) ? (g->info.ny + 7) / 8 > 65535
                 : (g->info.nx + 7) / 8 > 65535 || g->info.ny > 65535)
        return CT_ERR_INVALID_ARGUMENT;
    double iso[3] = {0.0, 0.0, 0.0};
    if (o.isocenter != nullptr) {
        for (int a = 0; a < (is_2d(b) ? 2 : 3); ++a) {
            if (!std::isfinite(o.isocenter[a])) return CT_ERR_INVALID_ARGUMENT;
            iso[a] = o.isocenter[a];
        }
    } else if (!is_parallel(b)) {
        estimate_isocenter(g, iso);
    }
    *L = fbp_layout(g, mode);
    ct_status st = check_call(g, in, in_bytes, out, out_bytes, d_workspace, workspace_bytes,
                              L->total);
    if (st != CT_OK) return st;
    const size_t wbytes = sizeof(float) * (size_t)g->info.n_views;
    const size_t pbytes = wbytes * (size_t)g->info.n_u;
    const size_t kbytes = sizeof(float) * (size_t)(2 * g->info.n_u - 1);
    if (o.d_view_weights != nullptr &&
        (st = check_input(g, o.d_view_weights, wbytes, out, out_bytes, d_workspace, L->total)) !=
            CT_OK)
        return st;
    if (o.d_pixel_weights != nullptr &&
        (st = check_input(g, o.d_pixel_weights, pbytes, out, out_bytes, d_workspace,
                          L->total)) != CT_OK)
        return st;
    if (o.d_kernel != nullptr &&
        (st = check_input(g, o.d_kernel, kbytes, out, out_bytes, d_workspace, L->total)) != CT_OK)
        return st;
    ct::FbpParams& p = *P;
    std::memset(&p, 0, sizeof(p));
    p.n_views = g->info.n_views;
    p.n_u = g->info.n_u;
    p.n_v = g->info.n_v;
    p.nx = g->info.nx; p.ny = g->info.ny; p.nz = g->info.nz;
    p.two_d = is_2d(b) ? 1 : 0;
    p.parallel = is_parallel(b) ? 1 : 0;
    p.window = (int32_t)o.window;
    p.rows = L->rows;
    p.cols = L->cols;
    p.bu = L->bu;
    p.bv = L->bv;
    p.du = g->du;
    p.dv = g->dv;
    for (int a = 0; a < 3; ++a) p.iso[a] = iso[a];
    p.sx = g->grid.sp[0];
    p.sy = g->grid.sp[1];
    p.sz = g->grid.sp[2];
    p.pixel_weights = o.d_pixel_weights;
    p.kernel = o.d_kernel;
    return CT_OK;
}

const float* view_weights_of(const ct_fbp_options* opt) {
    return opt == nullptr ? nullptr : opt->d_view_weights;
}

}  // namespace

extern "C" ct_status ct_fbp(const ct_geometry* g, const float* d_sino, float* d_volume,
                            const ct_fbp_options* options, void* d_workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
    ct::FbpParams P;
    FbpLayout L;
    if (g == nullptr) return CT_ERR_INVALID_ARGUMENT;
    const ct_status st = fbp_setup(g, d_sino, sino_bytes(g), d_volume, volume_bytes(g), options,
                                   d_workspace, workspace_bytes, kFbpForward, &P, &L);
    if (st != CT_OK) return st;
    char* ws = static_cast<char*>(d_workspace);
    return from_cuda(ct::launch_fbp(P, g->d_raw, view_weights_of(options),
                                    reinterpret_cast<ct::FbpView*>(ws + L.views),
                                    reinterpret_cast<ct::FbpCosine*>(ws + L.cosines),
                                    reinterpret_cast<float*>(ws + L.taps), d_sino,
                                    reinterpret_cast<float*>(ws + L.filtered), d_volume, stream));
}

extern "C" ct_status ct_fbp_transpose(const ct_geometry* g, const float* d_volume, float* d_sino,
                                      const ct_fbp_options* options, void* d_workspace,
                                      size_t workspace_bytes, cudaStream_t stream) {
    ct::FbpParams P;
    FbpLayout L;
    if (g == nullptr) return CT_ERR_INVALID_ARGUMENT;
    const ct_status st = fbp_setup(g, d_volume, volume_bytes(g), d_sino, sino_bytes(g), options,
                                   d_workspace, workspace_bytes, kFbpTranspose, &P, &L);
    if (st != CT_OK) return st;
    char* ws = static_cast<char*>(d_workspace);
    return from_cuda(ct::launch_fbp_transpose(
        P, g->d_raw, view_weights_of(options), reinterpret_cast<ct::FbpView*>(ws + L.views),
        reinterpret_cast<ct::FbpCosine*>(ws + L.cosines), reinterpret_cast<float*>(ws + L.taps),
        d_volume, reinterpret_cast<float*>(ws + L.copies), d_sino, stream));
}

extern "C" ct_status ct_fbp_gradients(const ct_geometry* g, const float* d_sino,
                                      const float* d_grad_volume, const ct_fbp_options* options,
                                      float* d_grad_kernel, float* d_grad_view_weights,
                                      void* d_workspace, size_t workspace_bytes,
                                      cudaStream_t stream) {
    ct::FbpParams P;
    FbpLayout L;
    if (g == nullptr || (d_grad_kernel == nullptr && d_grad_view_weights == nullptr))
        return CT_ERR_INVALID_ARGUMENT;
    // the outputs: the kernel gradient and the view-weight gradient, checked like outputs
    float* first_out = d_grad_kernel ? d_grad_kernel : d_grad_view_weights;
    const size_t kbytes = sizeof(float) * (size_t)(2 * g->info.n_u - 1);
    const size_t wbytes = sizeof(float) * (size_t)g->info.n_views;
    const size_t first_bytes = d_grad_kernel ? kbytes : wbytes;
    ct_status st = fbp_setup(g, d_sino, sino_bytes(g), first_out, first_bytes, options,
                             d_workspace, workspace_bytes, kFbpGradients, &P, &L);
    if (st != CT_OK) return st;
    if ((st = check_device_ptr(d_grad_volume, g->device)) != CT_OK) return st;
    if (overlap(d_grad_volume, volume_bytes(g), d_workspace, L.total) ||
        overlap(d_grad_volume, volume_bytes(g), first_out, first_bytes))
        return CT_ERR_ALIASING;
    if (d_grad_kernel && d_grad_view_weights) {
        if ((st = check_device_ptr(d_grad_view_weights, g->device)) != CT_OK) return st;
        if (overlap(d_grad_view_weights, wbytes, d_grad_kernel, kbytes) ||
            overlap(d_grad_view_weights, wbytes, d_workspace, L.total) ||
            overlap(d_grad_view_weights, wbytes, d_sino, sino_bytes(g)) ||
            overlap(d_grad_view_weights, wbytes, d_grad_volume, volume_bytes(g)))
            return CT_ERR_ALIASING;
    }
    char* ws = static_cast<char*>(d_workspace);
    return from_cuda(ct::launch_fbp_gradients(
        P, g->d_raw, view_weights_of(options), reinterpret_cast<ct::FbpView*>(ws + L.views),
        reinterpret_cast<ct::FbpCosine*>(ws + L.cosines), reinterpret_cast<float*>(ws + L.taps),
        d_sino, d_grad_volume, reinterpret_cast<float*>(ws + L.copies),
        reinterpret_cast<float*>(ws + L.filtered), reinterpret_cast<double*>(ws + L.acc),
        d_grad_kernel, d_grad_view_weights, stream));
}

// ---------------------------------------------------------------------------------------------
// Parker short-scan weights ("Differentiable analytical reconstruction": short scans add Parker
// weighting before filtering; Parker 1982).

extern "C" ct_status ct_fbp_parker_weights(const ct_geometry* g, const double* isocenter,
                                           float* out) {
    if (g == nullptr || out == nullptr) return CT_ERR_INVALID_ARGUMENT;
    const int b = g->info.beam;
    if (b != CT_FAN2D && b != CT_CONE) return CT_ERR_INVALID_ARGUMENT;
    if (g->d_offsets != nullptr) return CT_ERR_INVALID_ARGUMENT;
    double iso[3] = {0.0, 0.0, 0.0};
    if (isocenter != nullptr) {
        for (int a = 0; a < (is_2d(b) ? 2 : 3); ++a) {
            if (!std::isfinite(isocenter[a])) return CT_ERR_INVALID_ARGUMENT;
            iso[a] = isocenter[a];
        }
    } else {
        estimate_isocenter(g, iso);
    }
    const int n_views = g->info.n_views, n_u = g->info.n_u;
    const int w = is_2d(b) ? 6 : 12;
    const double pi = 3.14159265358979323846;
    // source angles about the isocentre, unwrapped, in the sense of rotation; the orbit must be a
    // circle in the xy-plane about the isocentre
    std::vector<double> beta((size_t)n_views);
    double rmin = 1e300, rmax = 0.0, zmin = 1e300, zmax = -1e300;
    for (int k = 0; k < n_views; ++k) {
        double first[3], ctr[3], u[3], v[3];
        unpack(b, g->host_views.data() + (int64_t)k * w, first, ctr, u, v);
        const double rx = first[0] - iso[0], ry = first[1] - iso[1];
        const double r = std::hypot(rx, ry);
        rmin = std::min(rmin, r);
        rmax = std::max(rmax, r);
        zmin = std::min(zmin, first[2]);
        zmax = std::max(zmax, first[2]);
        double a = std::atan2(ry, rx);
        if (k > 0) {
            while (a - beta[(size_t)k - 1] > pi) a -= 2.0 * pi;
            while (a - beta[(size_t)k - 1] < -pi) a += 2.0 * pi;
        }
        beta[(size_t)k] = a;
    }
    const double rmean = 0.5 * (rmin + rmax);
    if (!(rmean > 0.0) || rmax - rmin > 1e-6 * rmean || zmax - zmin > 1e-6 * rmean)
        return CT_ERR_INVALID_GEOMETRY;
    const double sense = beta[(size_t)n_views - 1] >= beta[0] ? 1.0 : -1.0;
    const double b0 = beta[0];
    for (double& x : beta) x = (x - b0) * sense;
    // fan angle of each detector column's centre line from the central ray, same sense
    std::vector<double> gamma((size_t)n_views * (size_t)n_u);
    double delta = 0.0;
    const double cu = 0.5 * (n_u - 1);
    for (int k = 0; k < n_views; ++k) {
        double first[3], ctr[3], u[3], v[3];
        unpack(b, g->host_views.data() + (int64_t)k * w, first, ctr, u, v);
        const double ax = iso[0] - first[0], ay = iso[1] - first[1];
        for (int j = 0; j < n_u; ++j) {
            const double o = (j - cu) * g->du;
            const double bx = ctr[0] + o * u[0] - first[0], by = ctr[1] + o * u[1] - first[1];
            const double gm = sense * std::atan2(ax * by - ay * bx, ax * bx + ay * by);
            gamma[(size_t)k * n_u + j] = gm;
            delta = std::max(delta, std::fabs(gm));
        }
    }
    const double span = beta[(size_t)n_views - 1];
    if (span < pi + 2.0 * delta - 1e-9) return CT_ERR_INVALID_GEOMETRY;
    const double d = 0.5 * (span - pi);  // effective half fan angle
    for (int k = 0; k < n_views; ++k) {
        const double bk = beta[(size_t)k];
        for (int j = 0; j < n_u; ++j) {
            const double gm = gamma[(size_t)k * n_u + j];
            double wt = 0.0;
            if (bk >= 0.0 && bk < 2.0 * (d - gm)) {
                const double sn = std::sin(0.25 * pi * bk / (d - gm));
                wt = sn * sn;
            } else if (bk >= 2.0 * (d - gm) && bk <= pi - 2.0 * gm) {
                wt = 1.0;
            } else if (bk > pi - 2.0 * gm && bk <= pi + 2.0 * d) {
                const double sn = std::sin(0.25 * pi * (pi + 2.0 * d - bk) / (d + gm));
                wt = sn * sn;
            }
            out[(size_t)k * n_u + j] = (float)wt;
        }
    }
    return CT_OK;
}

// ---------------------------------------------------------------------------------------------
// L2 roofline probes.

extern "C" ct_status ct_probe_l2_read(const float* d_buf, size_t n_floats, int32_t passes,
                                      float* d_sink, cudaStream_t stream) {
    if (d_buf == nullptr || d_sink == nullptr || passes <= 0 || n_floats < 4 ||
        n_floats > (size_t)INT64_MAX || ((uintptr_t)d_buf & 15) != 0)
        return CT_ERR_INVALID_ARGUMENT;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return CT_ERR_CUDA;
    }
    ct_status st;
    if ((st = check_device_ptr(d_buf, dev)) != CT_OK) return st;
    if ((st = check_device_ptr(d_sink, dev)) != CT_OK) return st;
    if (overlap(d_buf, n_floats * sizeof(float), d_sink, sizeof(float))) return CT_ERR_ALIASING;
    return from_cuda(ct::launch_l2_read(d_buf, (int64_t)n_floats, passes, d_sink, stream));
}

extern "C" ct_status ct_probe_l1_read(const float* d_buf, size_t n_floats, int32_t passes,
                                      float* d_sink, cudaStream_t stream) {
    if (d_buf == nullptr || d_sink == nullptr || passes <= 0 || n_floats < 4 ||
        n_floats > (size_t)16384 || ((uintptr_t)d_buf & 15) != 0)
        return CT_ERR_INVALID_ARGUMENT;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return CT_ERR_CUDA;
    }
    ct_status st;
    if ((st = check_device_ptr(d_buf, dev)) != CT_OK) return st;
    if ((st = check_device_ptr(d_sink, dev)) != CT_OK) return st;
    if (overlap(d_buf, n_floats * sizeof(float), d_sink, sizeof(float))) return CT_ERR_ALIASING;
    return from_cuda(ct::launch_l1_read(d_buf, (int64_t)n_floats, passes, d_sink, stream));
}

extern "C" ct_status ct_probe_l2_reduce(float* d_buf, size_t n_floats, int32_t passes,
                                        int32_t stride, cudaStream_t stream) {
    if (d_buf == nullptr || passes <= 0 || stride < 1 || stride > 32 ||
        n_floats < (size_t)32 * (size_t)stride || n_floats > (size_t)INT64_MAX)
        return CT_ERR_INVALID_ARGUMENT;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return CT_ERR_CUDA;
    }
    const ct_status st = check_device_ptr(d_buf, dev);
    if (st != CT_OK) return st;
    return from_cuda(ct::launch_l2_reduce(d_buf, (int64_t)n_floats, passes, stride, stream));
}

// ---------------------------------------------------------------------------------------------
// Bounds-checking builds.

extern "C" ct_status ct_debug_bounds_violations(uint64_t* count) {
    if (count == nullptr) return CT_ERR_INVALID_ARGUMENT;
    *count = 0;
#ifdef CT_DEBUG_BOUNDS
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return from_cuda(e);
    *count = ct::siddon_bounds_violations(true) + ct::fbp_bounds_violations(true);
    e = cudaGetLastError();
    return from_cuda(e);
#else
    return CT_ERR_INVALID_ARGUMENT;
#endif
}
