/*
 * Float64 CPU oracle for the cell-constant Siddon projector, its matched adjoint and SIRT.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the CUDA library is
 * checked against.  Only the tests, the graft smoke check and the benchmark's CPU-baseline leg
 * load it; the library never does.  It shares no code, header, table or constant with the CUDA
 * path: geometry records are read in the page's own layout and every step is re-derived here.
 *
 * What it computes (the plain definition, which Siddon's method reaches exactly):
 *   y_ray = sum over voxels v of x_v * l_v(ray)
 * where l_v is the physical length of the part of the ray that lies inside voxel v, the volume
 * being piecewise constant on half-open cells.  diffct calls this "the cell-constant Siddon
 * forward operator and its matched adjoint" (diffct docs, "Differentiable analytical
 * reconstruction", first paragraph); one ray per detector pixel, no detector-area integration
 * ("Trajectories and Geometry", parameterized detector surfaces).  The adjoint is
 * (A^T y)_v = sum over rays of y_ray * l_v(ray) (quickstart: x.grad = A^T (A x - y)).
 *
 * Conventions (diffct "Trajectories and Geometry", trajectory format and pixel formula):
 *   - Cartesian (x, y[, z]), origin at the volume centre, one length unit throughout.
 *   - Volume [z][y][x] (2D [y][x]); voxel i on an axis with n cells of spacing s spans
 *     [-n s/2 + i s, -n s/2 + (i+1) s)  (half-open: a ray lying in a cell face belongs to the cell
 *     on the + side; the outer + face of the box belongs to no cell).  The spacing may differ per
 *     axis ("Trajectories and Geometry": a scalar or a per-axis tuple in tensor order).
 *   - Pixel (u, v) at det_center + (u - (U-1)/2) du det_u + (v - (V-1)/2) dv det_v.
 *   - parallel / parallel3d: p(a) = pixel + a * ray_dir, a over all reals (infinite line).
 *   - fan / cone: p(a) = src + a * (pixel - src), a in [0, 1] (source-to-pixel segment; the
 *     pages do not say whether the line extends past source or pixel; for every workload here
 *     the volume lies strictly between source and detector, where both readings agree).
 *   - Sinogram [view][u][v] (2D [view][u]), v fastest.
 *
 * Algorithm per ray (Siddon's original formulation, float64 throughout):
 *   1. pixel point and ray (e, d) from the view record;
 *   2. clip the parameter range against the box with the slab method;
 *   3. per axis, the parameters of all interior cell planes inside the clipped range, as an
 *      ordered list; merge the per-axis lists into one ordered list bracketed by the clip ends;
 *   4. each consecutive pair with a positive gap is one segment: its voxel is the one that holds
 *      the segment's midpoint, its length is gap * |d|.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OG_PARALLEL2D = 0, OG_FAN2D = 1, OG_CONE = 2, OG_PARALLEL3D = 3 };

/* Geometry as handed over by the Python loader (mirrors the ctypes Structure there). */
typedef struct {
    int32_t beam;
    int32_t n_views;
    const double *views;   /* n_views x (6 | 12) */
    int32_t nz, ny, nx;    /* 2D: nz == 1 */
    double s[3];           /* voxel spacing along x, y, z (2D: z unused) */
    int32_t nu, nv;        /* 2D: nv == 1 */
    double du, dv;
    const double *offsets; /* NULL: flat detector; else nu x nv x 3 local (u, v, n) offsets */
} og_geom;

static int is_2d(const og_geom *g) { return g->beam == OG_PARALLEL2D || g->beam == OG_FAN2D; }
static int is_parallel(const og_geom *g) {
    return g->beam == OG_PARALLEL2D || g->beam == OG_PARALLEL3D;
}

/* Cells per Cartesian axis: component 0 = x, 1 = y, 2 = z. */
static void axis_cells(const og_geom *g, int64_t n[3]) {
    n[0] = g->nx; n[1] = g->ny; n[2] = g->nz;
}

/* Build the ray of pixel (iu, iv) of view `view`: origin e, direction d, parameter range. */
static void make_ray(const og_geom *g, int view, int iu, int iv, double e[3], double d[3],
                     double *amin, double *amax) {
    const int w = is_2d(g) ? 6 : 12;
    const double *r = g->views + (int64_t)view * w;
    double first[3] = {0, 0, 0}, ctr[3] = {0, 0, 0}, du[3] = {0, 0, 0}, dv[3] = {0, 0, 0};
    if (is_2d(g)) {
        first[0] = r[0]; first[1] = r[1];
        ctr[0] = r[2]; ctr[1] = r[3];
        du[0] = r[4]; du[1] = r[5];
    } else {
        for (int k = 0; k < 3; ++k) {
            first[k] = r[k]; ctr[k] = r[3 + k]; du[k] = r[6 + k]; dv[k] = r[9 + k];
        }
    }
    double pix[3];
    if (g->offsets == NULL) {
        /* flat detector: the page's pixel formula */
        const double cu = ((double)iu - (g->nu - 1) / 2.0) * g->du;
        const double cv = is_2d(g) ? 0.0 : ((double)iv - (g->nv - 1) / 2.0) * g->dv;
        for (int k = 0; k < 3; ++k) pix[k] = ctr[k] + cu * du[k] + cv * dv[k];
    } else {
        /* parameterized surface ("Trajectories and Geometry", detector surfaces): the pixel's
           local (u, v, n) offsets along det_u, det_v and the normal, which is
           cross(det_u, det_v) in 3D and (det_u_y, -det_u_x) in 2D */
        const double *o = g->offsets + ((int64_t)iu * g->nv + iv) * 3;
        double nrm[3];
        if (is_2d(g)) {
            nrm[0] = du[1]; nrm[1] = -du[0]; nrm[2] = 0.0;
        } else {
            nrm[0] = du[1] * dv[2] - du[2] * dv[1];
            nrm[1] = du[2] * dv[0] - du[0] * dv[2];
            nrm[2] = du[0] * dv[1] - du[1] * dv[0];
        }
        for (int k = 0; k < 3; ++k)
            pix[k] = ctr[k] + o[0] * du[k] + (is_2d(g) ? 0.0 : o[1] * dv[k]) + o[2] * nrm[k];
    }
    if (is_parallel(g)) {
        for (int k = 0; k < 3; ++k) { e[k] = pix[k]; d[k] = first[k]; }
        *amin = -INFINITY; *amax = INFINITY;
    } else {
        for (int k = 0; k < 3; ++k) { e[k] = first[k]; d[k] = pix[k] - first[k]; }
        *amin = 0.0; *amax = 1.0;
    }
}

/* Segment visitor: voxel linear index and chord length (physical units). */
typedef void (*seg_fn)(void *ctx, int64_t voxel, double length);

/*
 * Siddon traversal of one ray through an nx*ny*nz grid of spacing s centred at the origin.
 * `dims` = 2 or 3 (2D grids ignore the z component; their single slice is z in [-s/2, s/2)).
 * Returns the number of segments with positive length.
 */
static int64_t siddon_ray(int dims, const int64_t n[3], const double s[3], const double e[3],
                          const double d[3], double amin, double amax, seg_fn fn, void *ctx) {
    double h[3];
    for (int a = 0; a < 3; ++a) h[a] = 0.5 * (double)n[a] * s[a];
    double lo = amin, hi = amax;
    for (int a = 0; a < dims; ++a) {
        if (d[a] != 0.0) {
            double t1 = (-h[a] - e[a]) / d[a];
            double t2 = (h[a] - e[a]) / d[a];
            double tn = t1 < t2 ? t1 : t2, tf = t1 < t2 ? t2 : t1;
            if (tn > lo) lo = tn;
            if (tf < hi) hi = tf;
        } else if (e[a] < -h[a] || e[a] >= h[a]) {
            return 0;              /* parallel to this slab and outside it (half-open box) */
        }
    }
    if (!(hi > lo)) return 0;

    /* Per-axis ordered lists of interior plane crossings strictly inside (lo, hi). */
    int64_t cap = 2;
    for (int a = 0; a < dims; ++a) cap += n[a];
    double *alist = (double *)malloc(sizeof(double) * (size_t)cap);
    int64_t cnt[3] = {0, 0, 0};
    double *ax[3] = {NULL, NULL, NULL};
    int64_t used = 0;
    for (int a = 0; a < dims; ++a) {
        ax[a] = alist + used;
        if (d[a] == 0.0) continue;
        for (int64_t k = 1; k < n[a]; ++k) {
            /* visit planes in the order the ray meets them */
            int64_t kk = d[a] > 0 ? k : n[a] - k;
            double al = (-h[a] + (double)kk * s[a] - e[a]) / d[a];
            if (al > lo && al < hi) ax[a][cnt[a]++] = al;
        }
        used += cnt[a];
    }
    /* Merge the (already increasing) lists together with both clip ends. */
    double *merged = (double *)malloc(sizeof(double) * (size_t)(used + 2));
    int64_t m = 0, p[3] = {0, 0, 0};
    merged[m++] = lo;
    for (;;) {
        int best = -1;
        for (int a = 0; a < dims; ++a)
            if (p[a] < cnt[a] && (best < 0 || ax[a][p[a]] < ax[best][p[best]])) best = a;
        if (best < 0) break;
        merged[m++] = ax[best][p[best]++];
    }
    merged[m++] = hi;

    double dlen = 0.0;
    for (int a = 0; a < dims; ++a) dlen += d[a] * d[a];
    dlen = sqrt(dlen);

    int64_t nseg = 0;
    for (int64_t k = 0; k + 1 < m; ++k) {
        double gap = merged[k + 1] - merged[k];
        if (!(gap > 0.0)) continue;
        double mid = 0.5 * (merged[k] + merged[k + 1]);
        int64_t idx[3] = {0, 0, 0};
        for (int a = 0; a < dims; ++a) {
            double c = (e[a] + mid * d[a] + h[a]) / s[a];
            int64_t i = (int64_t)floor(c);
            if (i < 0) i = 0;
            if (i > n[a] - 1) i = n[a] - 1;
            idx[a] = i;
        }
        int64_t lin = (idx[2] * n[1] + idx[1]) * n[0] + idx[0];
        fn(ctx, lin, gap * dlen);
        ++nseg;
    }
    free(merged);
    free(alist);
    return nseg;
}

static int dims_of(const og_geom *g) { return is_2d(g) ? 2 : 3; }

/* ---- forward projection -------------------------------------------------------------------- */

typedef struct { const double *x; double acc; } fp_ctx;
static void fp_visit(void *c, int64_t v, double l) {
    fp_ctx *f = (fp_ctx *)c;
    f->acc += f->x[v] * l;
}

/* Project views [v0, v1) of volume x (float64, [z][y][x]) into sino (full-size, [view][u][v]). */
void oracle_project(const og_geom *g, const double *x, double *sino, int32_t v0, int32_t v1) {
    int64_t n[3];
    axis_cells(g, n);
    for (int view = v0; view < v1; ++view)
        for (int iu = 0; iu < g->nu; ++iu)
            for (int iv = 0; iv < g->nv; ++iv) {
                double e[3], d[3], amin, amax;
                make_ray(g, view, iu, iv, e, d, &amin, &amax);
                fp_ctx c = {x, 0.0};
                siddon_ray(dims_of(g), n, g->s, e, d, amin, amax, fp_visit, &c);
                sino[((int64_t)view * g->nu + iu) * g->nv + iv] = c.acc;
            }
}

/* Project an explicit list of rays (view, u, v) -> out[k]. */
void oracle_project_rays(const og_geom *g, const double *x, int64_t nrays, const int32_t *view,
                         const int32_t *iu, const int32_t *iv, double *out) {
    int64_t n[3];
    axis_cells(g, n);
    for (int64_t k = 0; k < nrays; ++k) {
        double e[3], d[3], amin, amax;
        make_ray(g, view[k], iu[k], iv[k], e, d, &amin, &amax);
        fp_ctx c = {x, 0.0};
        siddon_ray(dims_of(g), n, g->s, e, d, amin, amax, fp_visit, &c);
        out[k] = c.acc;
    }
}

/* ---- adjoint (backprojection) -------------------------------------------------------------- */

typedef struct { double *vol; double y; } bp_ctx;
static void bp_visit(void *c, int64_t v, double l) {
    bp_ctx *b = (bp_ctx *)c;
    b->vol[v] += b->y * l;
}

/* vol += A^T sino restricted to views [v0, v1).  The caller zeroes vol first. */
void oracle_backproject(const og_geom *g, const double *sino, double *vol, int32_t v0,
                        int32_t v1) {
    int64_t n[3];
    axis_cells(g, n);
    for (int view = v0; view < v1; ++view)
        for (int iu = 0; iu < g->nu; ++iu)
            for (int iv = 0; iv < g->nv; ++iv) {
                double y = sino[((int64_t)view * g->nu + iu) * g->nv + iv];
                if (y == 0.0) continue;
                double e[3], d[3], amin, amax;
                make_ray(g, view, iu, iv, e, d, &amin, &amax);
                bp_ctx c = {vol, y};
                siddon_ray(dims_of(g), n, g->s, e, d, amin, amax, bp_visit, &c);
            }
}

/* ---- per-ray diagnostics -------------------------------------------------------------------- */

typedef struct { int64_t *idx; double *w; int64_t cap, cnt; double total; } list_ctx;
static void list_visit(void *c, int64_t v, double l) {
    list_ctx *L = (list_ctx *)c;
    if (L->cnt < L->cap) { L->idx[L->cnt] = v; L->w[L->cnt] = l; }
    L->cnt++;
    L->total += l;
}

/* Segments of one ray in traversal order.  Returns the segment count (may exceed cap). */
int64_t oracle_ray_segments(const og_geom *g, int32_t view, int32_t iu, int32_t iv,
                            int64_t *idx, double *w, int64_t cap) {
    int64_t n[3];
    axis_cells(g, n);
    double e[3], d[3], amin, amax;
    make_ray(g, view, iu, iv, e, d, &amin, &amax);
    list_ctx L = {idx, w, cap, 0, 0.0};
    siddon_ray(dims_of(g), n, g->s, e, d, amin, amax, list_visit, &L);
    return L.cnt;
}

/* Same for an explicit ray (e, d, [amin, amax]) through an nx*ny*nz grid (dims = 2 or 3) of
   spacing s[0..2] along x, y, z. */
int64_t oracle_line_segments(int32_t dims, int32_t nz, int32_t ny, int32_t nx, const double *s,
                             const double *e, const double *d, double amin, double amax,
                             int64_t *idx, double *w, int64_t cap) {
    int64_t n[3] = {nx, ny, nz};
    double ee[3] = {e[0], e[1], dims == 3 ? e[2] : 0.0};
    double dd[3] = {d[0], d[1], dims == 3 ? d[2] : 0.0};
    list_ctx L = {idx, w, cap, 0, 0.0};
    siddon_ray(dims, n, s, ee, dd, amin, amax, list_visit, &L);
    return L.cnt;
}

/* Per-ray total chord length (= row sum of A) and positive-length segment count. */
void oracle_ray_lengths(const og_geom *g, int32_t v0, int32_t v1, double *length,
                        int64_t *segments) {
    int64_t n[3];
    axis_cells(g, n);
    for (int view = v0; view < v1; ++view)
        for (int iu = 0; iu < g->nu; ++iu)
            for (int iv = 0; iv < g->nv; ++iv) {
                double e[3], d[3], amin, amax;
                make_ray(g, view, iu, iv, e, d, &amin, &amax);
                list_ctx L = {NULL, NULL, 0, 0, 0.0};
                siddon_ray(dims_of(g), n, g->s, e, d, amin, amax, list_visit, &L);
                int64_t k = ((int64_t)view * g->nu + iu) * g->nv + iv;
                if (length) length[k] = L.total;
                if (segments) segments[k] = L.cnt;
            }
}

/* The ray of pixel (iu, iv) of a view: origin e, direction d, parameter range (for tests). */
void oracle_ray(const og_geom *g, int32_t view, int32_t iu, int32_t iv, double *e, double *d,
                double *range) {
    make_ray(g, view, iu, iv, e, d, &range[0], &range[1]);
}

/* ---- brute force: one voxel's own box against the ray --------------------------------------- */

/*
 * Length of {p(a) : a in [amin, amax]} inside the half-open cell
 * [lo_0, hi_0) x [lo_1, hi_1) (x [lo_2, hi_2)).  Independent of the traversal above: it never
 * enumerates planes, it intersects the ray with this one cell.
 */
static double cell_chord(int dims, const double lo[3], const double hi[3], const double e[3],
                         const double d[3], double amin, double amax) {
    double a0 = amin, a1 = amax, dl = 0.0;
    for (int a = 0; a < dims; ++a) {
        dl += d[a] * d[a];
        if (d[a] == 0.0) {
            if (!(e[a] >= lo[a] && e[a] < hi[a])) return 0.0;
        } else {
            double t1 = (lo[a] - e[a]) / d[a], t2 = (hi[a] - e[a]) / d[a];
            if (t1 > t2) { double t = t1; t1 = t2; t2 = t; }
            if (t1 > a0) a0 = t1;
            if (t2 < a1) a1 = t2;
        }
    }
    return a1 > a0 ? (a1 - a0) * sqrt(dl) : 0.0;
}

/* Row of A for one ray by brute force over every voxel (tiny volumes only). */
void oracle_brute_row(const og_geom *g, int32_t view, int32_t iu, int32_t iv, double *row) {
    double e[3], d[3], amin, amax;
    make_ray(g, view, iu, iv, e, d, &amin, &amax);
    int64_t n[3];
    axis_cells(g, n);
    const int dims = dims_of(g);
    for (int64_t z = 0; z < n[2]; ++z)
        for (int64_t y = 0; y < n[1]; ++y)
            for (int64_t x = 0; x < n[0]; ++x) {
                int64_t idx[3] = {x, y, z};
                double lo[3], hi[3];
                for (int a = 0; a < 3; ++a) {
                    lo[a] = -0.5 * (double)n[a] * g->s[a] + (double)idx[a] * g->s[a];
                    hi[a] = lo[a] + g->s[a];
                }
                row[(z * n[1] + y) * n[0] + x] = cell_chord(dims, lo, hi, e, d, amin, amax);
            }
}

/*
 * (A^T sino)_v for a list of voxels, computed voxel by voxel: for each view, the voxel's corners
 * are projected onto the detector, every pixel of the (1-pixel padded) bounding rectangle is
 * tried, and the ray's chord through this one cell is accumulated.  Requires every voxel to lie
 * strictly between source and detector plane for fan/cone beams (true for all workloads here).
 */
void oracle_backproject_voxels(const og_geom *g, const double *sino, int64_t nvox,
                               const int64_t *voxel, double *out) {
    int64_t n[3];
    axis_cells(g, n);
    const int dims = dims_of(g);
    const int w = is_2d(g) ? 6 : 12;
    for (int64_t k = 0; k < nvox; ++k) {
        int64_t lin = voxel[k];
        int64_t idx[3] = {lin % n[0], (lin / n[0]) % n[1], lin / (n[0] * n[1])};
        double lo[3], hi[3];
        for (int a = 0; a < 3; ++a) {
            lo[a] = -0.5 * (double)n[a] * g->s[a] + (double)idx[a] * g->s[a];
            hi[a] = lo[a] + g->s[a];
        }
        double acc = 0.0;
        for (int view = 0; view < g->n_views; ++view) {
            const double *r = g->views + (int64_t)view * w;
            double first[3] = {0, 0, 0}, ctr[3] = {0, 0, 0}, du[3] = {0, 0, 0},
                   dv[3] = {0, 0, 0}, nrm[3];
            if (dims == 2) {
                first[0] = r[0]; first[1] = r[1]; ctr[0] = r[2]; ctr[1] = r[3];
                du[0] = r[4]; du[1] = r[5];
                nrm[0] = du[1]; nrm[1] = -du[0]; nrm[2] = 0.0;
            } else {
                for (int a = 0; a < 3; ++a) {
                    first[a] = r[a]; ctr[a] = r[3 + a]; du[a] = r[6 + a]; dv[a] = r[9 + a];
                }
                nrm[0] = du[1] * dv[2] - du[2] * dv[1];
                nrm[1] = du[2] * dv[0] - du[0] * dv[2];
                nrm[2] = du[0] * dv[1] - du[1] * dv[0];
            }
            /* detector coordinates (in pixels) of the projected corners */
            double umin = INFINITY, umax = -INFINITY, vmin = INFINITY, vmax = -INFINITY;
            int ncorner = dims == 2 ? 4 : 8;
            for (int c = 0; c < ncorner; ++c) {
                double X[3];
                for (int a = 0; a < 3; ++a) X[a] = ((c >> a) & 1) ? hi[a] : lo[a];
                if (dims == 2) X[2] = 0.0;
                double Q[3];
                if (is_parallel(g)) {
                    /* along the ray direction onto the detector plane */
                    double num = 0, den = 0;
                    for (int a = 0; a < 3; ++a) {
                        num += (ctr[a] - X[a]) * nrm[a];
                        den += first[a] * nrm[a];
                    }
                    double mu = num / den;
                    for (int a = 0; a < 3; ++a) Q[a] = X[a] + mu * first[a];
                } else {
                    double num = 0, den = 0;
                    for (int a = 0; a < 3; ++a) {
                        num += (ctr[a] - first[a]) * nrm[a];
                        den += (X[a] - first[a]) * nrm[a];
                    }
                    double lam = num / den;
                    for (int a = 0; a < 3; ++a) Q[a] = first[a] + lam * (X[a] - first[a]);
                }
                double pu = 0, pv = 0;
                for (int a = 0; a < 3; ++a) {
                    pu += (Q[a] - ctr[a]) * du[a];
                    pv += (Q[a] - ctr[a]) * dv[a];
                }
                pu = pu / g->du + (g->nu - 1) / 2.0;
                pv = dims == 2 ? 0.0 : pv / g->dv + (g->nv - 1) / 2.0;
                if (pu < umin) umin = pu;
                if (pu > umax) umax = pu;
                if (pv < vmin) vmin = pv;
                if (pv > vmax) vmax = pv;
            }
            int64_t u0 = (int64_t)floor(umin) - 1, u1 = (int64_t)ceil(umax) + 1;
            int64_t w0 = (int64_t)floor(vmin) - 1, w1 = (int64_t)ceil(vmax) + 1;
            if (g->offsets != NULL) {  /* not a plane: no bounding rectangle, try every pixel */
                u0 = 0; u1 = g->nu - 1; w0 = 0; w1 = g->nv - 1;
            }
            if (u0 < 0) u0 = 0;
            if (w0 < 0) w0 = 0;
            if (u1 > g->nu - 1) u1 = g->nu - 1;
            if (w1 > g->nv - 1) w1 = g->nv - 1;
            for (int64_t iu = u0; iu <= u1; ++iu)
                for (int64_t iv = w0; iv <= w1; ++iv) {
                    double y = sino[((int64_t)view * g->nu + iu) * g->nv + iv];
                    if (y == 0.0) continue;
                    double e[3], d[3], amin, amax;
                    make_ray(g, view, (int)iu, (int)iv, e, d, &amin, &amax);
                    acc += y * cell_chord(dims, lo, hi, e, d, amin, amax);
                }
        }
        out[k] = acc;
    }
}

/* ---- SIRT ------------------------------------------------------------------------------------ */

/*
 * n_iter SIRT updates  x <- x + relax * C (A^T (R (y - A x)))  with R = 1/(A 1) per ray and
 * C = 1/(A^T 1) per voxel, both 0 where the sum is 0.  All vectors float64.  x is updated in
 * place.  residual_norms (optional, n_iter entries) receives ||R^(1/2) (y - A x_k)||^2 before
 * each update.
 */
void oracle_sirt(const og_geom *g, const double *y, double *x, int32_t n_iter, double relax,
                 double *residual_norms) {
    int64_t n[3];
    axis_cells(g, n);
    const int64_t nvox = n[0] * n[1] * n[2];
    const int64_t nray = (int64_t)g->n_views * g->nu * g->nv;
    double *R = (double *)calloc((size_t)nray, sizeof(double));
    double *C = (double *)calloc((size_t)nvox, sizeof(double));
    double *ones_r = (double *)malloc(sizeof(double) * (size_t)nray);
    double *ones_v = (double *)malloc(sizeof(double) * (size_t)nvox);
    double *ax = (double *)malloc(sizeof(double) * (size_t)nray);
    double *b = (double *)malloc(sizeof(double) * (size_t)nvox);
    for (int64_t i = 0; i < nray; ++i) ones_r[i] = 1.0;
    for (int64_t i = 0; i < nvox; ++i) ones_v[i] = 1.0;
    /* R = 1 / (A 1),  C = 1 / (A^T 1) */
    oracle_project(g, ones_v, ax, 0, g->n_views);
    for (int64_t i = 0; i < nray; ++i) R[i] = ax[i] > 0.0 ? 1.0 / ax[i] : 0.0;
    memset(b, 0, sizeof(double) * (size_t)nvox);
    oracle_backproject(g, ones_r, b, 0, g->n_views);
    for (int64_t i = 0; i < nvox; ++i) C[i] = b[i] > 0.0 ? 1.0 / b[i] : 0.0;
    for (int it = 0; it < n_iter; ++it) {
        oracle_project(g, x, ax, 0, g->n_views);
        double rn = 0.0;
        for (int64_t i = 0; i < nray; ++i) {
            double r = y[i] - ax[i];
            rn += R[i] * r * r;
            ax[i] = R[i] * r;
        }
        if (residual_norms) residual_norms[it] = rn;
        memset(b, 0, sizeof(double) * (size_t)nvox);
        oracle_backproject(g, ax, b, 0, g->n_views);
        for (int64_t i = 0; i < nvox; ++i) x[i] += relax * C[i] * b[i];
    }
    free(R); free(C); free(ones_r); free(ones_v); free(ax); free(b);
}

/* ---- CGLS ------------------------------------------------------------------------------------ */

/*
 * n_iter steps of CGLS (conjugate gradients on the normal equations A^T A x = A^T y, in the
 * form that never forms A^T A) from the given x, all vectors float64:
 *   r = y - A x,  s = A^T r,  p = s,  gamma = <s, s>
 *   repeat: q = A p;  alpha = gamma / <q, q>;  x += alpha p;  r -= alpha q;
 *           s = A^T r;  gamma' = <s, s>;  beta = gamma' / gamma;  p = s + beta p;  gamma = gamma'
 * A zero denominator (converged) gives alpha = 0 or beta = 0.  residual_norms (optional,
 * n_iter + 1 entries) receives ||r||^2 before the first and after each step.
 */
void oracle_cgls(const og_geom *g, const double *y, double *x, int32_t n_iter,
                 double *residual_norms) {
    int64_t n[3];
    axis_cells(g, n);
    const int64_t nvox = n[0] * n[1] * n[2];
    const int64_t nray = (int64_t)g->n_views * g->nu * g->nv;
    double *r = (double *)malloc(sizeof(double) * (size_t)nray);
    double *q = (double *)malloc(sizeof(double) * (size_t)nray);
    double *s = (double *)malloc(sizeof(double) * (size_t)nvox);
    double *p = (double *)malloc(sizeof(double) * (size_t)nvox);
    oracle_project(g, x, q, 0, g->n_views);
    double rn = 0.0;
    for (int64_t i = 0; i < nray; ++i) {
        r[i] = y[i] - q[i];
        rn += r[i] * r[i];
    }
    if (residual_norms) residual_norms[0] = rn;
    memset(s, 0, sizeof(double) * (size_t)nvox);
    oracle_backproject(g, r, s, 0, g->n_views);
    double gamma = 0.0;
    for (int64_t i = 0; i < nvox; ++i) {
        p[i] = s[i];
        gamma += s[i] * s[i];
    }
    for (int it = 0; it < n_iter; ++it) {
        oracle_project(g, p, q, 0, g->n_views);
        double delta = 0.0;
        for (int64_t i = 0; i < nray; ++i) delta += q[i] * q[i];
        const double alpha = delta > 0.0 ? gamma / delta : 0.0;
        for (int64_t i = 0; i < nvox; ++i) x[i] += alpha * p[i];
        rn = 0.0;
        for (int64_t i = 0; i < nray; ++i) {
            r[i] -= alpha * q[i];
            rn += r[i] * r[i];
        }
        if (residual_norms) residual_norms[it + 1] = rn;
        memset(s, 0, sizeof(double) * (size_t)nvox);
        oracle_backproject(g, r, s, 0, g->n_views);
        double gamma_new = 0.0;
        for (int64_t i = 0; i < nvox; ++i) gamma_new += s[i] * s[i];
        const double beta = gamma > 0.0 ? gamma_new / gamma : 0.0;
        for (int64_t i = 0; i < nvox; ++i) p[i] = s[i] + beta * p[i];
        gamma = gamma_new;
    }
    free(r); free(q); free(s); free(p);
}
