// Siddon forward projector, matched adjoint and SIRT kernels for sm_103a.
//
// Operator: the cell-constant Siddon line integral (diffct documentation, "Differentiable
// analytical reconstruction": cell-constant Siddon forward operator and matched adjoint), one ray
// per detector pixel (diffct "Trajectories and Geometry", detector-surface section), pixel
// positions from that page's flat-detector formula.
//
// Per ray:
//   1. float64: pixel point, ray origin/direction, slab clip of the parameter range against the
//      box [0, nx] x [0, ny] x [0, nz] (voxel units), entry and exit points, and per axis the
//      entry and exit cells (hence the crossing count n) and the distance to the first plane;
//   2. float32: per-axis first-crossing distance t0 (that distance over the direction component)
//      and crossing pitch dt, then the incremental Siddon walk.  The k-th crossing of axis a is
//      always fmaf(k, dt_a, t0_a) (no running sums), so any kernel that walks the same ray gets
//      bit-identical crossing positions and therefore bit-identical chord weights.
// The walk takes exactly n_x + n_y + n_z steps and moves each axis at most n_a times from an
// entry voxel inside the grid towards an exit voxel inside the grid, so every index it forms is
// in bounds whatever the float rounding does to the order of near-simultaneous crossings.
#include "ct_internal.h"

#include <atomic>

#include <cuda_runtime.h>

namespace ct {
namespace {

#ifdef CT_DEBUG_BOUNDS
__device__ unsigned long long g_bounds_violations = 0;

// True when 0 <= i < n; otherwise the miss is counted and the caller skips the access.
__device__ __forceinline__ bool in_bounds(int64_t i, int64_t n) {
    if ((uint64_t)i >= (uint64_t)n) {
        atomicAdd(&g_bounds_violations, 1ull);
        return false;
    }
    return true;
}
#endif

constexpr int kThreads = 256;  // 8 warps
constexpr int kRows = 4;       // 3D tiles: 8 warps x 4 rows = 32 pixels along the warp axis
constexpr int kTile = 32;      // 3D tiles are 32 x 32 pixels
constexpr int kTile2D = 256;   // 2D tiles are 256 detector pixels
// Resident CTAs per SM the walk kernels are compiled for.  The plain 3D forward projection runs
// at 8 (32 registers, some set-up values spilled; the extra warps hide the gathers' latency on
// volumes larger than L2), the scatters, the 2D projection and the fused SIRT/CGLS projections at
// 6 (40 registers; at 8 the 512^3 reductions and the 2D projection slow down and the fused
// kernels spill inside the walk).
constexpr int kMinBlocksGather = 8;
constexpr int kMinBlocks = 6;

__device__ __forceinline__ float f_inf() { return __int_as_float(0x7f800000); }

// Reciprocal of a nonzero double: hardware estimate refined by one Newton-Raphson step
// r <- r + r (1 - d r), which squares the estimate's relative error (to about 2^-44).
__device__ __forceinline__ double rcp64(double d) {
    double r;
    asm("rcp.approx.ftz.f64 %0, %1;" : "=d"(r) : "d"(d));
    const double e = __fma_rn(-d, r, 1.0);
    return __fma_rn(r, e, r);
}

// Walk state of one ray.  Index 0 and 1 are the two "outer" axes, index 2 the "inner" axis,
// which is the volume axis fastest in memory.
//
// The k-th crossing of slot a lies at fmaf(k, dt[a], t0[a]).  A walk takes the crossings with
// k0[a] <= k < n[a] and runs from tstart to tend; the whole ray has k0 = 0, tstart = 0 and
// n, tend from the clip (restrict_to_slab narrows them to one slab of the inner axis).
struct Ray {
    float t0[3];   // distance (voxel units, along the ray) from entry to the first crossing
    float dt[3];   // distance between successive crossings
    int n[3];      // crossings the walk ends before (the whole ray: number of crossings)
    float k0[3];   // crossings already behind the walk's start (the whole ray: 0)
    int step[3];   // signed element stride per crossing
    int idx;       // voxel at the walk's start, linear index in the internal layout
    int entry_in;  // entry cell of the whole ray along the inner axis
    float tstart;  // where the walk starts (the whole ray: 0)
    float tend;    // where the walk ends (the whole ray: the chord length, voxel units)
    float scale;   // physical length per unit of voxel-space length along this ray
#ifdef CT_DEBUG_BOUNDS
    int64_t nvox;  // voxels of one volume (bounds-checking builds)
#endif
};

// Crossings of one axis by a walk that enters at coordinate ci, leaves at co (voxel units,
// float64) and advances the coordinate by dh per unit of its parameter: the entry cell i0 and the
// exit cell, both clamped into [0, top], the number n of planes between them, the first crossing
// t0 and the pitch dt (parameter units) and the signed element step of a crossing.  The cells and
// the distance from the entry to the first plane are taken in float64 and only that distance (at
// most one cell) is rounded to float32: a float32 entry coordinate is off by up to half an ulp of
// the coordinate (1e-6 cells near cell 30), which t0 = distance / |dh| multiplies by 1 / |dh|, so on
// an axis the ray crosses at a grazing angle it moved the crossing by 2e-4 cells.
struct AxisWalk {
    float t0, dt;
    int n, step, i0;
};

__device__ __forceinline__ AxisWalk axis_walk(double ci, double co, float dh, int top,
                                              int stride) {
    AxisWalk w;
    int i0, i1;
    if (dh > 0.0f) {
        i0 = (int)floor(ci);
        i1 = (int)ceil(co) - 1;
    } else if (dh < 0.0f) {
        i0 = (int)ceil(ci) - 1;
        i1 = (int)floor(co);
    } else {
        i0 = (int)floor(ci);
        i1 = i0;
    }
    i0 = min(max(i0, 0), top);
    i1 = min(max(i1, 0), top);
    // Crossing pitches are capped at 1e28 parameter units so that fmaf(k, dt, t0) stays finite
    // for every k < 2^31: only axes with no crossing left ever read +inf.  (An axis with
    // |dh| < 1e-28 has no crossing inside any admissible volume anyway.)
    if (dh > 0.0f) {
        const float inv = fminf(1.0f / dh, 1e28f);
        w.n = max(0, i1 - i0);
        w.dt = inv;
        w.t0 = __fmul_rn((float)((double)(i0 + 1) - ci), inv);
        w.step = stride;
    } else if (dh < 0.0f) {
        const float inv = fminf(-1.0f / dh, 1e28f);
        w.n = max(0, i0 - i1);
        w.dt = inv;
        w.t0 = __fmul_rn((float)(ci - (double)i0), inv);
        w.step = -stride;
    } else {
        w.n = 0;
        w.dt = f_inf();
        w.t0 = f_inf();
        w.step = 0;
    }
    w.i0 = i0;
    return w;
}

// Ray set-up for pixel (u, v).  Returns false when the ray misses the volume.  F is the inner
// (fast) axis; the outer axes are the other two in increasing order.
template <int F>
__device__ __forceinline__ bool setup_ray(const ViewRec& vr, const Grid& g, int u, int v,
                                          Ray& r) {
    constexpr int A = F == 0 ? 1 : 0;
    // pixel point: flat formula, or the pixel's (u, v, n) offsets on a surface detector
    double P[3];
    if (g.offsets == nullptr) {
        const double fu = (double)u, fv = (double)v;
#pragma unroll
        for (int a = 0; a < 3; ++a) P[a] = __fma_rn(fv, vr.pv[a], __fma_rn(fu, vr.pu[a], vr.pb[a]));
    } else {
        const double* off = g.offsets + ((int64_t)u * g.nv + v) * 3;
        const double ou = __ldg(off), ov = __ldg(off + 1), on = __ldg(off + 2);
#pragma unroll
        for (int a = 0; a < 3; ++a)
            P[a] = __fma_rn(on, vr.pn[a], __fma_rn(ov, vr.pv[a], __fma_rn(ou, vr.pu[a], vr.pb[a])));
    }
    double o[3], d[3];
    double amin, amax;
    if (g.parallel) {
#pragma unroll
        for (int a = 0; a < 3; ++a) {
            o[a] = P[a];
            d[a] = vr.q[a];
        }
        amin = -__longlong_as_double(0x7ff0000000000000ll);
        amax = __longlong_as_double(0x7ff0000000000000ll);
    } else {
#pragma unroll
        for (int a = 0; a < 3; ++a) {
            o[a] = vr.q[a];
            d[a] = P[a];
        }
        amin = 0.0;
        amax = 1.0;
    }
    // slab clip against [0, n_a] per axis; the sign and zero tests read the bits (integer pipe)
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        const long long bits = __double_as_longlong(d[a]);
        if ((bits & 0x7fffffffffffffffll) != 0) {
            const double ri = rcp64(d[a]);
            const double t1 = -o[a] * ri;
            const double t2 = (g.nd[a] - o[a]) * ri;
            const bool pos = bits >= 0;
            amin = fmax(amin, pos ? t1 : t2);
            amax = fmin(amax, pos ? t2 : t1);
        } else if (!(o[a] >= 0.0 && o[a] < g.nd[a])) {
            return false;  // parallel to this slab and outside it (half-open box)
        }
    }
    if (!(amax > amin)) return false;

    float df[3];
#pragma unroll
    for (int a = 0; a < 3; ++a) df[a] = (float)d[a];
    const float dl = sqrtf(__fmaf_rn(df[2], df[2], __fmaf_rn(df[1], df[1], df[0] * df[0])));
    const float inv_dl = 1.0f / dl;
    r.tend = __fmul_rn((float)(amax - amin), dl);
    if (g.iso) {
        r.scale = g.sp[0];
    } else {
        // the walk measures length in voxel units per axis; a segment of voxel-space length t
        // has physical length t |d_phys| / |d_vox|, with d_phys_a = d_vox_a * spacing_a
        const float px = __fmul_rn(df[0], g.sp[0]), py = __fmul_rn(df[1], g.sp[1]),
                    pz = __fmul_rn(df[2], g.sp[2]);
        r.scale = __fmul_rn(sqrtf(__fmaf_rn(pz, pz, __fmaf_rn(py, py, px * px))), inv_dl);
    }
    int idx = 0;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        const int slot = a == F ? 2 : (a == A ? 0 : 1);
        const AxisWalk w = axis_walk(__fma_rn(amin, d[a], o[a]), __fma_rn(amax, d[a], o[a]),
                                     __fmul_rn(df[a], inv_dl), g.n[a] - 1, g.stride[a]);
        r.n[slot] = w.n;
        r.dt[slot] = w.dt;
        r.t0[slot] = w.t0;
        r.step[slot] = w.step;
        idx += w.i0 * g.stride[a];
        if (slot == 2) r.entry_in = w.i0;
        r.k0[slot] = 0.0f;
    }
    r.idx = idx;
    r.tstart = 0.0f;
#ifdef CT_DEBUG_BOUNDS
    r.nvox = (int64_t)g.n[0] * g.n[1] * g.n[2];
#endif
    return true;
}

// Float32 copy of a view record's flat-detector vectors (slab-tiled launches).
struct ViewRecF {
    float pb[3], pu[3], pv[3], q[3];
};

__device__ __forceinline__ void load_view_f32(const ViewRec& sv, ViewRecF& sf) {
    if (threadIdx.x < 3) {
        const int a = threadIdx.x;
        sf.pb[a] = (float)sv.pb[a];
        sf.pu[a] = (float)sv.pu[a];
        sf.pv[a] = (float)sv.pv[a];
        sf.q[a] = (float)sv.q[a];
    }
    __syncthreads();
}

// Cheap float32 test, before the float64 set-up, of whether the ray of pixel (u, v) can have
// cells in the inner-axis slab [c0, c1): the ray is clipped against the box widened by one cell
// on every side and its inner-axis range widened by one more cell, far beyond float32 rounding,
// so a ray that reaches the slab is never rejected.  F is the inner axis.
template <int F>
__device__ __forceinline__ bool may_reach_slab(const ViewRecF& sf, const Grid& g, int u, int v,
                                               int c0, int c1) {
    const float fu = (float)u, fv = (float)v;
    float o[3], d[3];
    float amin = g.parallel ? -f_inf() : 0.0f, amax = g.parallel ? f_inf() : 1.0f;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        const float p = __fmaf_rn(fv, sf.pv[a], __fmaf_rn(fu, sf.pu[a], sf.pb[a]));
        o[a] = g.parallel ? p : sf.q[a];
        d[a] = g.parallel ? sf.q[a] : p;
        const float lo = -1.0f, hi = (float)g.n[a] + 1.0f;
        if (d[a] != 0.0f) {
            const float r = 1.0f / d[a];
            const float t1 = (lo - o[a]) * r, t2 = (hi - o[a]) * r;
            amin = fmaxf(amin, fminf(t1, t2));
            amax = fminf(amax, fmaxf(t1, t2));
        } else if (!(o[a] >= lo && o[a] <= hi)) {
            return false;
        }
    }
    if (!(amax >= amin)) return false;
    const float z0 = __fmaf_rn(amin, d[F], o[F]), z1 = __fmaf_rn(amax, d[F], o[F]);
    return fmaxf(z0, z1) >= (float)c0 - 1.0f && fminf(z0, z1) <= (float)c1 + 1.0f;
}

// Crossings of one axis at or before t (AT = true) or strictly before t, among the first n:
// #{k < n : fmaf(k, dt, t0) <= t} (or < t), with the walk's own crossing values.
template <bool AT>
__device__ __forceinline__ int crossings_before(float t, float t0, float dt, int n) {
    int k = 0;
    if (t >= t0) k = min(n, (int)fminf(floorf(__fdividef(__fsub_rn(t, t0), dt)) + 1.0f, (float)n));
    // the estimate can be off by one either way; settle it on the exact crossing values
    while (k > 0 && (AT ? __fmaf_rn((float)(k - 1), dt, t0) > t
                        : __fmaf_rn((float)(k - 1), dt, t0) >= t))
        --k;
    while (k < n && (AT ? __fmaf_rn((float)k, dt, t0) <= t : __fmaf_rn((float)k, dt, t0) < t)) ++k;
    return k;
}

// Narrows the walk of a whole ray to the inner-axis cells [c0, c1) (one slab): it starts at the
// crossing into the slab (or at the ray's entry) and ends at the crossing out of it (or at the
// ray's exit), and keeps the whole ray's crossing values, so every segment it takes has the bits
// the whole walk gives that segment.  Outer crossings at the slab's entry crossing belong to the
// slab's start state (the whole walk takes an outer crossing before an inner one at the same
// value), outer crossings at its exit crossing to the next slab.  Returns false when the ray has
// no segment of positive length in the slab.
__device__ __forceinline__ bool restrict_to_slab(Ray& r, int c0, int c1) {
    const int a = r.entry_in, n = r.n[2];
    float kstart = 0.0f, tstart = 0.0f, tend = r.tend;
    int nend = n;
    if (r.step[2] == 0) {
        if (a < c0 || a >= c1) return false;
    } else if (r.step[2] > 0) {  // cells a, a + 1, ..., a + n
        if (a + n < c0 || a >= c1) return false;
        if (a < c0) {
            const int k = c0 - 1 - a;  // crossing from cell c0 - 1 into c0
            kstart = (float)(k + 1);
            tstart = __fmaf_rn((float)k, r.dt[2], r.t0[2]);
        }
        if (a + n > c1 - 1) {
            nend = c1 - 1 - a;  // crossing from cell c1 - 1 into c1
            tend = __fmaf_rn((float)nend, r.dt[2], r.t0[2]);
        }
    } else {  // cells a, a - 1, ..., a - n
        if (a < c0 || a - n >= c1) return false;
        if (a > c1 - 1) {
            const int k = a - c1;  // crossing from cell c1 into c1 - 1
            kstart = (float)(k + 1);
            tstart = __fmaf_rn((float)k, r.dt[2], r.t0[2]);
        }
        if (a - n < c0) {
            nend = a - c0;  // crossing from cell c0 into c0 - 1
            tend = __fmaf_rn((float)nend, r.dt[2], r.t0[2]);
        }
    }
    if (!(tend > tstart)) return false;
    int idx = r.idx + (int)kstart * r.step[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        if (r.n[j] > 0) {
            const int k = crossings_before<true>(tstart, r.t0[j], r.dt[j], r.n[j]);
            const int e = crossings_before<false>(tend, r.t0[j], r.dt[j], r.n[j]);
            idx += k * r.step[j];
            r.k0[j] = (float)k;
            r.n[j] = e;
        }
    }
    r.k0[2] = kstart;
    r.n[2] = nend;
    r.idx = idx;
    r.tstart = tstart;
    r.tend = tend;
    return true;
}

// The walk.  GATHER returns sum_k vol[idx_k] * seg_k (voxel units); SCATTER adds val * seg_k to
// vol[idx_k] and returns 0.  Both evaluate every segment length with the same operations.
//
// Order of work: the outer loop steps through the crossings of the two outer axes; before each
// outer crossing, the inner-axis crossings that come first are taken.  A warp's lanes cover
// neighbouring pixels along the detector axis that is aligned with the inner (fast) axis, so
// they meet the same outer planes in the same order and stay in lock-step: each step's 32
// gathers or atomics land in one or two 128-byte lines.
//
// Two phases.  The main phase runs while the next outer crossing lies strictly before the
// earlier of the two outer axes' last crossings: there neither outer axis can run out, so its
// next crossing is computed without a check, and the first inner crossing of an outer step is
// handled inline (a second one is rare).  The gather issues the loads for the next outer step
// (the voxel after the outer crossing, and the one after a pending inner crossing) one step
// ahead.  The tail phase takes the remaining events with per-axis exhaustion checks.  Both
// phases visit the same events in the same order with the same arithmetic.
//
// ISIGN: 0, or the inner-axis step (+1 / -1, the inner axis has unit stride) when every ray of
// the warp that crosses inner planes moves that way.  SINGLE: every ray of the warp has at most
// one inner crossing between two outer ones, and none can run out of inner crossings in the main
// phase (see walk_dispatch), so the main phase needs neither a loop for a second inner crossing
// nor the exhaustion check.  The specialisations change no arithmetic.
template <bool SCATTER, int NB, int ISIGN, bool SINGLE, bool COUNTED>
__device__ __forceinline__ void walk(const Ray& r, const float* __restrict__ vin,
                                     float* __restrict__ vout, int64_t vstride,
                                     const float (&val)[NB], float (&acc)[NB]) {
    const int s2 = ISIGN != 0 ? ISIGN : r.step[2];
    const float INF = f_inf();
    const float na = (float)r.n[0], nb = (float)r.n[1], nf = (float)r.n[2];
    float ka = r.k0[0], kb = r.k0[1], kf = r.k0[2];
    float ta = ka < na ? __fmaf_rn(ka, r.dt[0], r.t0[0]) : INF;
    float tb = kb < nb ? __fmaf_rn(kb, r.dt[1], r.t0[1]) : INF;
    float tf = kf < nf ? __fmaf_rn(kf, r.dt[2], r.t0[2]) : INF;
    int idx = r.idx;
    float t = r.tstart;
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
    // segment [.., .. + seg) in voxel idx: gather from / scatter into every volume of the batch
    auto scatter = [&](int i, float seg) {
#ifdef CT_DEBUG_BOUNDS
        if (!in_bounds(i, r.nvox)) return;
#endif
#pragma unroll
        for (int b = 0; b < NB; ++b) atomicAdd(vout + b * vstride + i, __fmul_rn(val[b], seg));
    };
    auto load = [&](int i, float (&v)[NB]) {
#ifdef CT_DEBUG_BOUNDS
        if (!in_bounds(i, r.nvox)) {
#pragma unroll
            for (int b = 0; b < NB; ++b) v[b] = 0.0f;
            return;
        }
#endif
#pragma unroll
        for (int b = 0; b < NB; ++b) v[b] = __ldg(vin + b * vstride + i);
    };
    auto gather = [&](const float (&v)[NB], float seg) {
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b] = __fmaf_rn(v[b], seg, acc[b]);
    };
    // Main phase: outer crossings strictly before the earlier of the two outer axes' last
    // crossings, so neither outer axis can run out here and its next crossing needs no check.
    // (The last crossings use the same fmaf as the walk, so the comparison is exact.)
    const float la = na > ka ? __fmaf_rn(na - 1.0f, r.dt[0], r.t0[0]) : INF;
    const float lb = nb > kb ? __fmaf_rn(nb - 1.0f, r.dt[1], r.t0[1]) : INF;
    const float lim = fminf(la, lb);
    float tstop = fminf(ta, tb);
    bool p = tf < tstop;
    float v0[NB], v1[NB];  // gather: values of the current voxel and of the next one inward
    if (!SCATTER) {
        load(idx, v0);
        if (p) load(idx + s2, v1);
    }
    // COUNTED gathers run the main phase for an exact count of steps: the outer crossings strictly
    // before lim, counted on the walk's own crossing values, are exactly the ones the value test
    // tstop < lim admits, and with an integer count the loop unrolled by eight tests once per
    // eight steps (forward walks: cone 15.6 -> 14.4 ms, 512^3 spiral 122 -> 107 ms, tilt series
    // 46 -> 42 ms, bit-identical; by four: 14.5, 111, 42 ms).  The other walks keep the value
    // test unrolled by two: the scatter ran no faster counted (unrolled by one, four or eight) and
    // much slower counted by two, and the 2D and batched gathers were slower counted.  The
    // unrolled loops rename the loop-carried values instead of copying them.
    static_assert(!(COUNTED && SCATTER), "the scatter walks test values");
    int main_steps = 0;
    if (COUNTED && lim < INF)
        main_steps = (na > ka ? crossings_before<false>(lim, r.t0[0], r.dt[0], r.n[0]) - (int)ka : 0) +
                     (nb > kb ? crossings_before<false>(lim, r.t0[1], r.dt[1], r.n[1]) - (int)kb : 0);
    constexpr int kMainUnroll = COUNTED ? 8 : 2;
#pragma unroll kMainUnroll
    for (int step_no = 0; COUNTED ? step_no < main_steps : tstop < lim; ++step_no) {
        const float seg0 = __fsub_rn(p ? tf : tstop, t);
        if (SCATTER)
            scatter(idx, seg0);
        else
            gather(v0, seg0);
        if (p) {
            idx += s2;
            t = tf;
            kf += 1.0f;
            tf = (SINGLE || kf < nf) ? __fmaf_rn(kf, r.dt[2], r.t0[2]) : INF;
#pragma unroll 1
            while (!SINGLE && tf < tstop) {  // a second inner crossing before this outer one (rare)
                const float seg = __fsub_rn(tf, t);
                if (SCATTER) {
                    scatter(idx, seg);
                    idx += s2;
                } else {
                    gather(v1, seg);
                    idx += s2;
                    load(idx, v1);
                }
                t = tf;
                kf += 1.0f;
                tf = kf < nf ? __fmaf_rn(kf, r.dt[2], r.t0[2]) : INF;
            }
            const float seg1 = __fsub_rn(tstop, t);
            if (SCATTER)
                scatter(idx, seg1);
            else
                gather(v1, seg1);
        }
        t = tstop;
        if (ta <= tb) {
            idx += r.step[0];
            ka += 1.0f;
            ta = __fmaf_rn(ka, r.dt[0], r.t0[0]);
        } else {
            idx += r.step[1];
            kb += 1.0f;
            tb = __fmaf_rn(kb, r.dt[1], r.t0[1]);
        }
        tstop = fminf(ta, tb);
        p = tf < tstop;
        if (!SCATTER) {
            load(idx, v0);
            if (p) load(idx + s2, v1);
        }
    }
    // (SINGLE computed the crossing after the last inner one instead of +inf: restore +inf, since
    // the tail may reach past it.)
    if (SINGLE && !(kf < nf)) tf = INF;
    // Tail: the remaining events with the per-axis checks.  v0 holds the current voxel's values.
#pragma unroll 1
    for (int outer = (int)(na - ka) + (int)(nb - kb); outer > 0; --outer) {
        tstop = fminf(ta, tb);
#pragma unroll 1
        while (tf < tstop) {
            const float seg = __fsub_rn(tf, t);
            if (SCATTER) {
                scatter(idx, seg);
                idx += s2;
            } else {
                idx += s2;
                float vn[NB];
                load(idx, vn);
                gather(v0, seg);
#pragma unroll
                for (int b = 0; b < NB; ++b) v0[b] = vn[b];
            }
            t = tf;
            kf += 1.0f;
            tf = kf < nf ? __fmaf_rn(kf, r.dt[2], r.t0[2]) : INF;
        }
        const float seg = __fsub_rn(tstop, t);
        if (SCATTER) scatter(idx, seg);
        t = tstop;
        if (ta <= tb) {
            idx += r.step[0];
            ka += 1.0f;
            ta = ka < na ? __fmaf_rn(ka, r.dt[0], r.t0[0]) : INF;
        } else {
            idx += r.step[1];
            kb += 1.0f;
            tb = kb < nb ? __fmaf_rn(kb, r.dt[1], r.t0[1]) : INF;
        }
        if (!SCATTER) {
            float vn[NB];
            load(idx, vn);
            gather(v0, seg);
#pragma unroll
            for (int b = 0; b < NB; ++b) v0[b] = vn[b];
        }
    }
#pragma unroll 1
    while (tf < r.tend) {
        const float seg = __fsub_rn(tf, t);
        if (SCATTER) {
            scatter(idx, seg);
            idx += s2;
        } else {
            idx += s2;
            float vn[NB];
            load(idx, vn);
            gather(v0, seg);
#pragma unroll
            for (int b = 0; b < NB; ++b) v0[b] = vn[b];
        }
        t = tf;
        kf += 1.0f;
        tf = kf < nf ? __fmaf_rn(kf, r.dt[2], r.t0[2]) : INF;
    }
    const float seg = __fsub_rn(r.tend, t);
    if (SCATTER)
        scatter(idx, seg);
    else
        gather(v0, seg);
}

// Picks the walk's specialisation for the lanes that walk together.  At most one inner crossing
// fits between two outer ones when the inner pitch exceeds every gap between successive outer
// crossings.  Such a gap is at most min(dt_a, dt_b) plus the rounding of two crossing values, and
// successive inner crossings are at least dt_f minus that rounding apart; each crossing value is
// one fmaf below tend, so the margin 1e-5 tend (about 80 ulps of tend) covers it.
template <bool SCATTER, int NB, bool COUNTED = false>
__device__ __forceinline__ void walk_dispatch(const Ray& r, const float* __restrict__ vin,
                                              float* __restrict__ vout, int64_t vstride,
                                              const float (&val)[NB], float (&acc)[NB]) {
    const unsigned m = __activemask();
    const float INF = f_inf();
    const bool none = !((float)r.n[2] > r.k0[2]);  // no inner crossing to take
    // the crossing after the last inner one, as the walk would compute it, is not before the end
    // of the main phase (the earlier of the two outer axes' last crossings), so the main phase
    // never takes it
    const float la =
        (float)r.n[0] > r.k0[0] ? __fmaf_rn((float)r.n[0] - 1.0f, r.dt[0], r.t0[0]) : INF;
    const float lb =
        (float)r.n[1] > r.k0[1] ? __fmaf_rn((float)r.n[1] - 1.0f, r.dt[1], r.t0[1]) : INF;
    const bool single =
        none || (r.dt[2] > fminf(r.dt[0], r.dt[1]) + __fmaf_rn(r.tend, 1e-5f, 1e-6f) &&
                 __fmaf_rn((float)r.n[2], r.dt[2], r.t0[2]) >= fminf(la, lb));
    if (__all_sync(m, single && (none || r.step[2] == 1)))
        walk<SCATTER, NB, 1, true, COUNTED>(r, vin, vout, vstride, val, acc);
    else if (__all_sync(m, single && (none || r.step[2] == -1)))
        walk<SCATTER, NB, -1, true, COUNTED>(r, vin, vout, vstride, val, acc);
    else
        walk<SCATTER, NB, 0, false, COUNTED>(r, vin, vout, vstride, val, acc);
}

// Single-volume forms.
// COUNTED: the main phase runs for a counted number of steps, unrolled by eight (single-volume
// 3D gathers; the 2D and batched gathers were slower that way: 2D fan 0.42 -> 0.50 ms, four
// volumes 27.5 -> 35.3 ms).
template <bool COUNTED>
__device__ __forceinline__ float walk_gather(const Ray& r, const float* __restrict__ vin) {
    const float none[1] = {0.0f};
    float acc[1];
    walk_dispatch<false, 1, COUNTED>(r, vin, nullptr, 0, none, acc);
    return acc[0];
}
__device__ __forceinline__ void walk_scatter(const Ray& r, float* __restrict__ vout, float val) {
    const float v[1] = {val};
    float acc[1];
    walk_dispatch<true, 1>(r, nullptr, vout, 0, v, acc);
}

// Block -> (view, pixel tile).  Tiles are ordered detector-v band first, then view, then u tile,
// so that the blocks resident at one time walk one band of the volume across all views.
struct TileCoord {
    int view, ut, vt;
};
__device__ __forceinline__ TileCoord tile_of_block(const Tiling& t) {
    int b = (int)blockIdx.x;
    const int per_band = t.n_views * t.tiles_u;
    TileCoord c;
    c.vt = b / per_band;
    b -= c.vt * per_band;
    c.view = b / t.tiles_u;
    c.ut = b - c.view * t.tiles_u;
    return c;
}

__device__ __forceinline__ void load_view(const ViewRec* __restrict__ views, int view,
                                          ViewRec& sv) {
    constexpr int kWords = (int)(sizeof(ViewRec) / sizeof(double));
    if (threadIdx.x < kWords)
        reinterpret_cast<double*>(&sv)[threadIdx.x] =
            reinterpret_cast<const double*>(views + view)[threadIdx.x];
    __syncthreads();
}

// Pixel handled by this thread in row r of the tile (3D) or in the 2D tile.
template <bool TWO_D>
__device__ __forceinline__ void pixel_of(const TileCoord& c, const ViewRec& sv, int r, int& u,
                                         int& v) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (TWO_D) {
        u = c.ut * kTile2D + (int)threadIdx.x;
        v = 0;
    } else if (sv.lanes_along_v) {
        v = c.vt * kTile + lane;
        u = c.ut * kTile + r * 8 + warp;
    } else {
        u = c.ut * kTile + lane;
        v = c.vt * kTile + r * 8 + warp;
    }
}

// 3D backprojection tiles that spread a warp's lanes over every second pixel along their axis
// (two warps interleave over 64 pixels), so that neighbouring lanes' rays, which often cross the
// same voxel where a detector pixel maps to under one voxel, rarely reduce into one address in
// the same instruction: a reduction whose lanes share addresses costs about twice the L2 sectors
// of the addresses it spans (probe: 19 addresses over 32 lanes, 6.1 sectors against 3 spanned).
// Tiles are 16 lines x 64 pixels (tl.spread 1: lanes along v, 2: along u), ordered as
// tile_of_block.
__device__ __forceinline__ TileCoord tile_of_spread_block(const Tiling& t) {
    int b = (int)blockIdx.x;
    const int per_band = t.n_views * t.spread_tiles_u;
    TileCoord c;
    c.vt = b / per_band;
    b -= c.vt * per_band;
    c.view = b / t.spread_tiles_u;
    c.ut = b - c.view * t.spread_tiles_u;
    return c;
}

__device__ __forceinline__ void spread_pixel_of(const TileCoord& c, const Tiling& t, int r, int& u,
                                                int& v) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int along = 2 * lane + (warp & 1);
    if (t.spread == 1) {
        v = c.vt * 64 + along;
        u = c.ut * 16 + r * 4 + (warp >> 1);
    } else {
        u = c.ut * 64 + along;
        v = c.vt * 16 + r * 4 + (warp >> 1);
    }
}

// Resident CTAs per SM for the (batched) walks: more registers per thread for NB values.
template <bool SCATTER, bool TWO_D, int NB>
struct BatchBlocks {
    static constexpr int value = NB == 1 ? (SCATTER || TWO_D ? kMinBlocks : kMinBlocksGather)
                                         : (NB == 2 ? 5 : 4);
};

// Block -> (view, pixel tile) of a slab-tiled launch: the slab's list of (view, v-tile) entries,
// each with its row of u-tiles.
__device__ __forceinline__ TileCoord tile_of_slab_block(const SlabArgs& sl, const Tiling& t) {
    const int b = (int)blockIdx.x;
    const int i = b / t.tiles_u;
    const int e = __ldg(sl.tiles + i);
    TileCoord c;
    c.view = e / t.tiles_v;
    c.vt = e - c.view * t.tiles_v;
    c.ut = b - i * t.tiles_u;
    return c;
}

// ---- Shared-line walks ----------------------------------------------------------------------
// When the detector axis that a block's lanes run along has no component on either outer axis
// (det_v along z with the z-fastest order: every circular fan or cone orbit with an upright
// detector), the rays of one detector line (the pixels that differ only along the lane axis) have
// one projection onto the plane of the outer axes: one origin and one direction there, so one
// parameter range inside the outer-axis square and the same outer crossings.  A block then walks
// one line at a time.  Its threads first merge that line's outer crossings into a list in shared
// memory, each entry holding the crossing's position and the cell (outer-axis part of the index)
// before it; each thread then walks its own ray along the list and takes only its own inner-axis
// crossings, so a step costs a shared-memory read instead of choosing between the two outer axes
// (cone 256^3 x 360 views, forward: 25.5 -> 16.8 warp instructions per 32 updates, 14.6 -> 10.45
// ms).
//
// Positions are measured along the line's outer-plane projection from its entry into the square,
// s = (a - a_in) |d_outer| (voxel units; a is the ray parameter), so every ray of the line reads the
// same list; a segment ds of s has voxel-space length ds |d| / |d_outer| along its ray.  The list
// is the exact merge of the two outer axes' crossings fmaf(k, dt, t0), ties taken first axis
// first: an entry's rank is its index on its own axis plus the number of the other axis's
// crossings before it, counted on the same values.  Every cell it names is the line's entry cell
// moved by the crossings in order, so it lies inside the square; a ray moves along the inner axis
// at most n times from an entry cell inside the grid, so every index a walk forms is in bounds.
//
// The backprojection takes the same segments without the list: line_setup_ray gives the per-ray
// walk the line's parameters (its outer crossings in s, counted from the ray's range, and the
// ray's own inner crossings), and the per-ray walk visits the merged crossings in the list's order
// (first axis first on ties) with the same arithmetic, so A^T stays the exact transpose of A.  A
// list-reading scatter issued the same reduction sectors but ran 2.5 % slower (its list reads
// share the L1 unit that the reductions saturate); pairing the list forward walk with the
// backprojection of the per-ray parameters left adjoint gaps of 3e-5 on rays entering through
// the inner-axis faces.  Lines are used only for volumes that fit in L2: on a 512^3 volume
// (untilted helix) the forward walk took 120 ms against 107, a block's band of 128 detector pixels
// spanning four times the volume slab of the per-ray tiles.  Blocks walking two, four or eight
// lines at once (fewer pixels per line) ran slower on both sizes.

struct LineEntry {
    float s;   // crossing position
    int cell;  // outer-axis part of the index of the cell before the crossing
};

// Outer-axis walk of one detector line.
struct LineRow {
    double amin, amax;  // ray-parameter range inside the outer-axis square
    float t0[2], dt[2];  // crossings of the two outer axes: fmaf(k, dt, t0) in s, k < n
    int n[2], step[2];
    int cell;            // entry cell (outer-axis part of the index)
    float df[2];         // outer direction components (float32)
    float dl, inv_dl;    // |d_outer| and its reciprocal
    float len;           // s at the line's exit from the square
};

// Set-up of the line through pixel coordinate `line` (u for lanes along v, else v).  Returns 0
// when every ray of the line misses the volume, 2 when the line has no extent in the outer plane
// (rays along the inner axis: the per-ray walk takes them), 1 otherwise.  Every thread of a block
// computes the same result from the same inputs.
template <int F>
__device__ __forceinline__ int line_row(const ViewRec& vr, const Grid& g, bool along_v, int line,
                                        LineRow& L) {
    constexpr int A = F == 0 ? 1 : 0;
    constexpr int B = F == 2 ? 1 : 2;
    // the lane-axis vector has no outer components, so the lane coordinate (0 here) adds exactly
    // zero to the pixel point's outer coordinates, as in setup_ray
    const double fu = along_v ? (double)line : 0.0, fv = along_v ? 0.0 : (double)line;
    double o[2], d[2];
    double amin = g.parallel ? -__longlong_as_double(0x7ff0000000000000ll) : 0.0;
    double amax = g.parallel ? __longlong_as_double(0x7ff0000000000000ll) : 1.0;
    bool moves = false;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int a = j == 0 ? A : B;
        const double P = __fma_rn(fv, vr.pv[a], __fma_rn(fu, vr.pu[a], vr.pb[a]));
        o[j] = g.parallel ? P : vr.q[a];
        d[j] = g.parallel ? vr.q[a] : P;
        const long long bits = __double_as_longlong(d[j]);
        if ((bits & 0x7fffffffffffffffll) != 0) {
            moves = true;
            const double ri = rcp64(d[j]);
            const double t1 = -o[j] * ri;
            const double t2 = (g.nd[a] - o[j]) * ri;
            const bool pos = bits >= 0;
            amin = fmax(amin, pos ? t1 : t2);
            amax = fmin(amax, pos ? t2 : t1);
        } else if (!(o[j] >= 0.0 && o[j] < g.nd[a])) {
            return 0;  // parallel to this slab and outside it
        }
    }
    if (!moves) return 2;
    if (!(amax > amin)) return 0;
    L.df[0] = (float)d[0];
    L.df[1] = (float)d[1];
    L.dl = sqrtf(__fmaf_rn(L.df[1], L.df[1], L.df[0] * L.df[0]));
    if (!(L.dl >= 1e-30f)) return 2;
    L.inv_dl = 1.0f / L.dl;
    L.amin = amin;
    L.amax = amax;
    L.len = __fmul_rn((float)(amax - amin), L.dl);
    int cell = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int a = j == 0 ? A : B;
        const AxisWalk w = axis_walk(__fma_rn(amin, d[j], o[j]), __fma_rn(amax, d[j], o[j]),
                                     __fmul_rn(L.df[j], L.inv_dl), g.n[a] - 1, g.stride[a]);
        L.t0[j] = w.t0;
        L.dt[j] = w.dt;
        L.n[j] = w.n;
        L.step[j] = w.step;
        cell += w.i0 * g.stride[a];
    }
    L.cell = cell;
    return 1;
}

// Merges the line's outer crossings into list[0, n_a + n_b) and puts the exit cell after them
// (the block's `count` threads take part, `me` is this one's rank; the caller synchronises).
__device__ __forceinline__ void build_line(const LineRow& L, LineEntry* __restrict__ list, int me,
                                           int count) {
    const int na = L.n[0], nb = L.n[1], k = na + nb;
    for (int i = me; i < k; i += count) {
        int ka, kb;
        float s;
        if (i < na) {
            ka = i;
            s = __fmaf_rn((float)ka, L.dt[0], L.t0[0]);
            kb = crossings_before<false>(s, L.t0[1], L.dt[1], nb);
        } else {
            kb = i - na;
            s = __fmaf_rn((float)kb, L.dt[1], L.t0[1]);
            ka = crossings_before<true>(s, L.t0[0], L.dt[0], na);
        }
        list[ka + kb] = LineEntry{s, L.cell + ka * L.step[0] + kb * L.step[1]};
    }
    if (me == 0) list[k] = LineEntry{f_inf(), L.cell + na * L.step[0] + nb * L.step[1]};
}

// One ray of a line: its own inner-axis walk, in s.
struct LineRay {
    float t0, dt;  // inner-axis crossings fmaf(k, dt, t0) in s, k < n
    int n, step;
    int zoff;      // inner-axis part of the entry cell's index
    float s0, s1;  // the ray's range of s inside the volume
    float fac;     // physical length per unit of s
};

// Set-up of pixel (u, v) of the line L.  Returns false when the ray misses the volume.  The clip
// is setup_ray's (the same per-axis bounds, combined with exact min/max).
template <int F>
__device__ __forceinline__ bool line_ray(const ViewRec& vr, const Grid& g, const LineRow& L,
                                         int u, int v, LineRay& r) {
    constexpr int A = F == 0 ? 1 : 0;
    constexpr int B = F == 2 ? 1 : 2;
    const double P = __fma_rn((double)v, vr.pv[F], __fma_rn((double)u, vr.pu[F], vr.pb[F]));
    const double o = g.parallel ? P : vr.q[F];
    const double d = g.parallel ? vr.q[F] : P;
    double amin = L.amin, amax = L.amax;
    const long long bits = __double_as_longlong(d);
    if ((bits & 0x7fffffffffffffffll) != 0) {
        const double ri = rcp64(d);
        const double t1 = -o * ri;
        const double t2 = (g.nd[F] - o) * ri;
        const bool pos = bits >= 0;
        amin = fmax(amin, pos ? t1 : t2);
        amax = fmin(amax, pos ? t2 : t1);
    } else if (!(o >= 0.0 && o < g.nd[F])) {
        return false;
    }
    if (!(amax > amin)) return false;
    float df[3];
    df[A] = L.df[0];
    df[B] = L.df[1];
    df[F] = (float)d;
    float phys;  // |d| in physical units
    if (g.iso) {
        phys = __fmul_rn(g.sp[0],
                         sqrtf(__fmaf_rn(df[2], df[2], __fmaf_rn(df[1], df[1], df[0] * df[0]))));
    } else {
        const float px = __fmul_rn(df[0], g.sp[0]), py = __fmul_rn(df[1], g.sp[1]),
                    pz = __fmul_rn(df[2], g.sp[2]);
        phys = sqrtf(__fmaf_rn(pz, pz, __fmaf_rn(py, py, px * px)));
    }
    r.fac = __fmul_rn(phys, L.inv_dl);
    r.s0 = __fmul_rn((float)(amin - L.amin), L.dl);
    r.s1 = __fmul_rn((float)(amax - L.amin), L.dl);
    const AxisWalk w = axis_walk(__fma_rn(amin, d, o), __fma_rn(amax, d, o),
                                 __fmul_rn(df[F], L.inv_dl), g.n[F] - 1, g.stride[F]);
    r.n = w.n;
    r.dt = w.dt;
    r.step = w.step;
    r.t0 = w.n > 0 ? __fadd_rn(r.s0, w.t0) : f_inf();
    r.zoff = w.i0 * g.stride[F];
    return true;
}

// The gather of one ray along the list entries [j0, j1) (the outer crossings inside its range) and
// then to its exit: acc = sum_k vol[idx_k] * ds_k for the NB volumes at vin + b * vstride.  ISIGN
// and SINGLE as in walk (the inner axis has unit stride); with SINGLE every step takes at most
// one inner crossing and the crossing after the ray's last one lies at or after entry j1 - 1, so
// the main loop needs no exhaustion check, and it loads the next step's values (the voxel after
// the outer crossing and, when an inner crossing comes first, the one after it) one step ahead.
// Both forms take the same segments with the same operations as walk() on line_setup_ray's Ray.
template <int NB, int ISIGN, bool SINGLE>
__device__ __forceinline__ void line_walk(const LineEntry* __restrict__ E, int j0, int j1,
                                          const LineRay& r, const float* __restrict__ vin,
                                          int64_t vstride, float (&acc)[NB]
#ifdef CT_DEBUG_BOUNDS
                                          , int64_t nvox
#endif
) {
    const int s2 = ISIGN != 0 ? ISIGN : r.step;
    const float INF = f_inf();
    const float nf = (float)r.n;
    float kf = 0.0f;
    float tf = r.n > 0 ? r.t0 : INF;
    float t = r.s0;
    int zoff = r.zoff;
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
    auto load = [&](int i, float (&v)[NB]) {
#ifdef CT_DEBUG_BOUNDS
        if (!in_bounds(i, nvox)) {
#pragma unroll
            for (int b = 0; b < NB; ++b) v[b] = 0.0f;
            return;
        }
#endif
#pragma unroll
        for (int b = 0; b < NB; ++b) v[b] = __ldg(vin + b * vstride + i);
    };
    auto gather = [&](const float (&v)[NB], float seg) {
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b] = __fmaf_rn(v[b], seg, acc[b]);
    };
    auto take = [&](int i, float seg) {  // one segment, loaded where it is taken
        float v[NB];
        load(i, v);
        gather(v, seg);
    };
    if (SINGLE) {
        if (j1 > j0) {
            LineEntry e = E[j0];
            int idx = e.cell + zoff;
            bool p = tf < e.s;
            float v0[NB], v1[NB];
            load(idx, v0);
            if (p) load(idx + s2, v1);
            // unrolled by sixteen: cone 256^3 forward 12.6 (by four), 11.9 (by eight, before the
            // line set-up moved to shared memory; 10.61 after), 10.45 ms
#pragma unroll 16
            for (int j = j0 + 1; j < j1; ++j) {
                gather(v0, __fsub_rn(p ? tf : e.s, t));
                if (p) {
                    gather(v1, __fsub_rn(e.s, tf));
                    zoff += s2;
                    kf += 1.0f;
                    tf = __fmaf_rn(kf, r.dt, r.t0);
                }
                t = e.s;
                e = E[j];
                idx = e.cell + zoff;
                p = tf < e.s;
                load(idx, v0);
                if (p) load(idx + s2, v1);
            }
            gather(v0, __fsub_rn(p ? tf : e.s, t));
            if (p) {
                gather(v1, __fsub_rn(e.s, tf));
                zoff += s2;
                kf += 1.0f;
                tf = __fmaf_rn(kf, r.dt, r.t0);
            }
            t = e.s;
        }
        // (the crossing after the last inner one was computed instead of +inf: restore +inf)
        if (!(kf < nf)) tf = INF;
    } else {
#pragma unroll 1
        for (int j = j0; j < j1; ++j) {
            const LineEntry e = E[j];
            int idx = e.cell + zoff;
#pragma unroll 1
            while (tf < e.s) {
                take(idx, __fsub_rn(tf, t));
                idx += s2;
                zoff += s2;
                t = tf;
                kf += 1.0f;
                tf = kf < nf ? __fmaf_rn(kf, r.dt, r.t0) : INF;
            }
            take(idx, __fsub_rn(e.s, t));
            t = e.s;
        }
    }
    int idx = E[j1].cell + zoff;
#pragma unroll 1
    while (tf < r.s1) {
        take(idx, __fsub_rn(tf, t));
        idx += s2;
        t = tf;
        kf += 1.0f;
        tf = kf < nf ? __fmaf_rn(kf, r.dt, r.t0) : INF;
    }
    take(idx, __fsub_rn(r.s1, t));
}

// Picks the line walk's specialisation for the lanes that walk together (see walk_dispatch for
// the one-inner-crossing bound: here the gaps are those between successive list entries).
template <int NB>
__device__ __forceinline__ void line_walk_dispatch(const LineEntry* __restrict__ E, int j0,
                                                   int j1, const LineRow& L, const LineRay& r,
                                                   const float* __restrict__ vin, int64_t vstride,
                                                   float (&acc)[NB], int64_t nvox) {
    const unsigned m = __activemask();
    const bool none = r.n == 0;
    const float last = j1 > j0 ? E[j1 - 1].s : -f_inf();
    const bool single =
        none || (r.dt > fminf(L.dt[0], L.dt[1]) + __fmaf_rn(L.len, 1e-5f, 1e-6f) &&
                 __fmaf_rn((float)r.n, r.dt, r.t0) >= last);
#ifdef CT_DEBUG_BOUNDS
#define CT_LINE_NVOX , nvox
#else
#define CT_LINE_NVOX
    (void)nvox;
#endif
    if (__all_sync(m, single && (none || r.step == 1)))
        line_walk<NB, 1, true>(E, j0, j1, r, vin, vstride, acc CT_LINE_NVOX);
    else if (__all_sync(m, single && (none || r.step == -1)))
        line_walk<NB, -1, true>(E, j0, j1, r, vin, vstride, acc CT_LINE_NVOX);
    else if (__all_sync(m, single))
        line_walk<NB, 0, true>(E, j0, j1, r, vin, vstride, acc CT_LINE_NVOX);
    else
        line_walk<NB, 0, false>(E, j0, j1, r, vin, vstride, acc CT_LINE_NVOX);
#undef CT_LINE_NVOX
}

// Rays whose chord is under 1/16 of their exit position along the line take the per-ray
// parameterisation (setup_ray) in every shared-line walk: positions along the line carry absolute
// rounding errors of a few ulps of s, too coarse against a short chord far along the line, while
// setup_ray's positions start at the ray's own entry.
__device__ __forceinline__ bool short_on_line(const LineRay& r) {
    return __fsub_rn(r.s1, r.s0) < __fmul_rn(0.0625f, r.s1);
}

// List entries [j0, j1) of a ray: the line's outer crossings at or before s0 come before its
// range, those strictly before s1 inside it.
__device__ __forceinline__ void line_range(const LineRow& L, const LineRay& r, int& ka0, int& kb0,
                                           int& ka1, int& kb1) {
    ka0 = 0;
    kb0 = 0;
    if (r.s0 > 0.0f) {
        ka0 = crossings_before<true>(r.s0, L.t0[0], L.dt[0], L.n[0]);
        kb0 = crossings_before<true>(r.s0, L.t0[1], L.dt[1], L.n[1]);
    }
    ka1 = max(ka0, crossings_before<false>(r.s1, L.t0[0], L.dt[0], L.n[0]));
    kb1 = max(kb0, crossings_before<false>(r.s1, L.t0[1], L.dt[1], L.n[1]));
}

// The per-ray form of a shared-line walk for pixel (u, v): the Ray whose walk() takes the list
// walk's segments.  Its outer slots are the line's two axes with their crossings in s, restricted
// to the ray's range (k0 = crossings at or before s0, n = crossings before s1), its inner slot the
// ray's own crossings, and it runs from s0 to s1 with the line's physical length factor.  walk()
// takes the merged outer crossings in the list's order (first axis first on ties) with the same
// arithmetic, so every segment has the list walk's bits.  Returns 0 when the ray misses, 1 with r
// set, 2 when the ray takes the per-ray parameterisation (setup_ray) in the list walk as well.
template <int F>
__device__ __forceinline__ int line_setup_ray(const ViewRec& sv, const Grid& g, bool along_v,
                                              int u, int v, Ray& r) {
    LineRow L;
    const int st = line_row<F>(sv, g, along_v, along_v ? u : v, L);
    if (st != 1) return st;
    LineRay lr;
    if (!line_ray<F>(sv, g, L, u, v, lr)) return 0;
    if (short_on_line(lr)) return 2;
    int ka0, kb0, ka1, kb1;
    line_range(L, lr, ka0, kb0, ka1, kb1);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        r.t0[j] = L.t0[j];
        r.dt[j] = L.dt[j];
        r.step[j] = L.step[j];
    }
    r.n[0] = ka1;
    r.n[1] = kb1;
    r.k0[0] = (float)ka0;
    r.k0[1] = (float)kb0;
    r.t0[2] = lr.t0;
    r.dt[2] = lr.dt;
    r.n[2] = lr.n;
    r.k0[2] = 0.0f;
    r.step[2] = lr.step;
    r.idx = L.cell + ka0 * L.step[0] + kb0 * L.step[1] + lr.zoff;
    r.entry_in = lr.zoff / g.stride[F];
    r.tstart = lr.s0;
    r.tend = lr.s1;
    r.scale = lr.fac;
#ifdef CT_DEBUG_BOUNDS
    r.nvox = (int64_t)g.n[0] * g.n[1] * g.n[2];
#endif
    return 1;
}

// The per-ray forward projection of one whole pixel (lines with no extent in the outer plane,
// short chords far along their line), writing its line integrals.  Kept out of line, with no
// array crossing the call, so that it adds nothing to the register use of the line walk (an
// accumulator array passed to it by reference had kept the line walk's sums in local memory).
template <int F, int NB>
__device__ __noinline__ void ray_pixel(const ViewRec& sv, const Grid& g, int u, int v, int64_t k,
                                       const float* __restrict__ vol, int64_t vstride,
                                       float* __restrict__ sino, int64_t sstride) {
    Ray ray;
    const bool hit = setup_ray<F>(sv, g, u, v, ray);
    const float none[NB] = {};
    float acc[NB];
    if (hit) walk_dispatch<false, NB>(ray, vol, nullptr, vstride, none, acc);
#pragma unroll
    for (int c = 0; c < NB; ++c) sino[c * sstride + k] = hit ? __fmul_rn(acc[c], ray.scale) : 0.0f;
}

// Resident blocks per SM of the line kernel (kLinePixels threads each): 2048, 1280 or 1024
// threads per SM for one, two or four volumes (the batched projections take the per-ray tiles).
template <int NB>
struct LineBlocks {
    static constexpr int value = (NB == 1 ? 2048 : (NB == 2 ? 1280 : 1024)) / kLinePixels;
};

// sino[b] = A vol[b] for NB volumes over shared-line tiles: a block takes kLinePixels pixels of
// kLineRows successive lines of one view.  Blocks are ordered lane tile first, then view, then
// line tile (one band of the detector across all views at a time, as tile_of_block).
template <int F, int NB>
__global__ void __launch_bounds__(kLinePixels, LineBlocks<NB>::value)
    line_project_kernel(const ViewRec* __restrict__ views, const Grid g, const Tiling tl,
                        const float* __restrict__ vol, int64_t vstride, float* __restrict__ sino,
                        int64_t sstride) {
    extern __shared__ LineEntry line_list[];
    __shared__ ViewRec sv;
    // the line's set-up, computed once per line by one thread (it is the same for the whole
    // block; computed by every thread it cost register spills in every walk)
    __shared__ LineRow L;
    __shared__ int line_status;
    int b = (int)blockIdx.x;
    const int per_band = tl.n_views * tl.line_row_tiles;
    const int lane_tile = b / per_band;
    b -= lane_tile * per_band;
    const int view = b / tl.line_row_tiles;
    const int line_tile = b - view * tl.line_row_tiles;
    load_view(views, view, sv);
    const bool along_v = tl.line == 1;
    const int n_lane = along_v ? tl.n_v : tl.n_u, n_line = along_v ? tl.n_u : tl.n_v;
    const int lane_px = lane_tile * kLinePixels + (int)threadIdx.x;
    const bool valid = lane_px < n_lane;
    const int64_t nvox = (int64_t)g.n[0] * g.n[1] * g.n[2];
#pragma unroll 1
    for (int rr = 0; rr < kLineRows; ++rr) {
        const int line = line_tile * kLineRows + rr;
        if (line >= n_line) break;  // the same for the whole block
        const int u = along_v ? line : lane_px, v = along_v ? lane_px : line;
        if (threadIdx.x == 0) line_status = line_row<F>(sv, g, along_v, line, L);
        __syncthreads();
        const int st = line_status;
        if (st == 1) {
            build_line(L, line_list, (int)threadIdx.x, kLinePixels);
            __syncthreads();
        }
        if (valid) {
            const int64_t k = ((int64_t)view * tl.n_u + u) * tl.n_v + v;
            bool per_ray = st == 2;
            if (st == 1) {
                LineRay r;
                const bool hit = line_ray<F>(sv, g, L, u, v, r);
                per_ray = hit && short_on_line(r);
                if (hit && !per_ray) {
                    int ka0, kb0, ka1, kb1;
                    line_range(L, r, ka0, kb0, ka1, kb1);
                    float acc[NB];
                    line_walk_dispatch<NB>(line_list, ka0 + kb0, ka1 + kb1, L, r, vol, vstride,
                                           acc, nvox);
#pragma unroll
                    for (int c = 0; c < NB; ++c) sino[c * sstride + k] = __fmul_rn(acc[c], r.fac);
                } else if (!hit) {
#pragma unroll
                    for (int c = 0; c < NB; ++c) sino[c * sstride + k] = 0.0f;
                }
            } else if (st == 0) {
#pragma unroll
                for (int c = 0; c < NB; ++c) sino[c * sstride + k] = 0.0f;
            }
            if (per_ray) ray_pixel<F, NB>(sv, g, u, v, k, vol, vstride, sino, sstride);
        }
        __syncthreads();  // the next line overwrites the set-up and the list
    }
}

// sino[b] = A vol[b] for the NB volumes vol + b * vstride (internal order) and sinograms
// sino + b * sstride; one walk per ray serves all NB volumes.  SLAB: the walks are restricted to
// one slab of the inner axis and each ray's partial sum is added to its sinogram entry.  LINE:
// the rays take the shared-line parameters (line_setup_ray), which gives line_project_kernel's
// results bit for bit (the batched projections of shared-line handles).
template <bool TWO_D, int F, int NB, bool SLAB, bool LINE = false>
__global__ void __launch_bounds__(kThreads, BatchBlocks<false, TWO_D, NB>::value)
    project_kernel(const ViewRec* __restrict__ views, const Grid g, const Tiling tl,
                   const float* __restrict__ vol, int64_t vstride, float* __restrict__ sino,
                   int64_t sstride, const SlabArgs sl) {
    static_assert(!(LINE && (SLAB || TWO_D)), "shared lines are for untiled 3D walks");
    __shared__ ViewRec sv;
    __shared__ ViewRecF sf;
    const TileCoord c = SLAB ? tile_of_slab_block(sl, tl) : tile_of_block(tl);
    load_view(views, c.view, sv);
    if (SLAB) load_view_f32(sv, sf);
#pragma unroll 1
    for (int row = 0; row < (TWO_D ? 1 : kRows); ++row) {
        int u, v;
        pixel_of<TWO_D>(c, sv, row, u, v);
        if (u >= tl.n_u || v >= tl.n_v) continue;
        if (SLAB && !may_reach_slab<F>(sf, g, u, v, sl.c0, sl.c1)) continue;
        const int64_t k = ((int64_t)c.view * tl.n_u + u) * tl.n_v + v;
        Ray ray;
        bool hit;
        if (LINE) {
            const int st = line_setup_ray<F>(sv, g, tl.line == 1, u, v, ray);
            hit = st == 1 || (st == 2 && setup_ray<F>(sv, g, u, v, ray));
        } else {
            hit = setup_ray<F>(sv, g, u, v, ray);
        }
        if (SLAB) hit = hit && restrict_to_slab(ray, sl.c0, sl.c1);
        if (hit) {
            if (NB == 1) {
                const float y = __fmul_rn(walk_gather<!TWO_D>(ray, vol), ray.scale);
                sino[k] = SLAB ? __fadd_rn(sino[k], y) : y;
            } else {
                const float none[NB] = {};
                float acc[NB];
                walk_dispatch<false, NB>(ray, vol, nullptr, vstride, none, acc);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float y = __fmul_rn(acc[b], ray.scale);
                    sino[b * sstride + k] = SLAB ? __fadd_rn(sino[b * sstride + k], y) : y;
                }
            }
        } else if (!SLAB) {
#pragma unroll
            for (int b = 0; b < NB; ++b) sino[b * sstride + k] = 0.0f;
        }
    }
}

// MODE 0: scatter sino * (physical length per voxel-space length); MODE 1: the same for a sinogram
// of ones (A^T 1).  NB volumes/sinograms at strides vstride/sstride, one walk per ray.  SLAB: the
// walks are restricted to one slab of the inner axis.  LINE: the rays take the shared-line
// parameters (line_setup_ray), so that this is the exact transpose of line_project_kernel.
// SPREAD: the tiles of tile_of_spread_block (the pixel-to-lane map changes no ray's arithmetic).
template <bool TWO_D, int F, int MODE, int NB, bool SLAB, bool LINE = false, bool SPREAD = false>
__global__ void __launch_bounds__(kThreads, BatchBlocks<true, TWO_D, NB>::value)
    backproject_kernel(const ViewRec* __restrict__ views, const Grid g, const Tiling tl,
                       const float* __restrict__ sino, int64_t sstride, float* __restrict__ vol,
                       int64_t vstride, const SlabArgs sl) {
    static_assert(!(LINE && (SLAB || TWO_D)), "shared lines are for untiled 3D walks");
    static_assert(!(SPREAD && (SLAB || TWO_D)), "spread tiles are for untiled 3D walks");
    __shared__ ViewRec sv;
    __shared__ ViewRecF sf;
    const TileCoord c =
        SLAB ? tile_of_slab_block(sl, tl) : (SPREAD ? tile_of_spread_block(tl) : tile_of_block(tl));
    load_view(views, c.view, sv);
    if (SLAB) load_view_f32(sv, sf);
#pragma unroll 1
    for (int row = 0; row < (TWO_D ? 1 : kRows); ++row) {
        int u, v;
        if (SPREAD)
            spread_pixel_of(c, tl, row, u, v);
        else
            pixel_of<TWO_D>(c, sv, row, u, v);
        if (u >= tl.n_u || v >= tl.n_v) continue;
        if (SLAB && !may_reach_slab<F>(sf, g, u, v, sl.c0, sl.c1)) continue;
        const int64_t k = ((int64_t)c.view * tl.n_u + u) * tl.n_v + v;
        float y[NB];
        bool any = false;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            y[b] = MODE == 0 ? __ldg(sino + b * sstride + k) : 1.0f;
            any |= y[b] != 0.0f;
        }
        if (!any) continue;
        Ray ray;
        if (LINE) {
            // lanes along v walk detector columns (lines of fixed u), as line_project_kernel
            const int st = line_setup_ray<F>(sv, g, tl.line == 1, u, v, ray);
            if (st == 0 || (st == 2 && !setup_ray<F>(sv, g, u, v, ray))) continue;
        } else if (!setup_ray<F>(sv, g, u, v, ray)) {
            continue;
        }
        if (SLAB && !restrict_to_slab(ray, sl.c0, sl.c1)) continue;
        if (NB == 1) {
            walk_scatter(ray, vol, __fmul_rn(y[0], ray.scale));
        } else {
            float val[NB], unused[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) val[b] = __fmul_rn(y[b], ray.scale);
            walk_dispatch<true, NB>(ray, nullptr, vol, vstride, val, unused);
        }
    }
}

// r = R (y - A x) with R = 1 / (A 1) = 1 / (physical chord); 0 for rays that miss.
template <bool TWO_D, int F>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    project_residual_kernel(const ViewRec* __restrict__ views, const Grid g, const Tiling tl,
                            const float* __restrict__ x, const float* __restrict__ y,
                            float* __restrict__ res) {
    __shared__ ViewRec sv;
    const TileCoord c = tile_of_block(tl);
    load_view(views, c.view, sv);
#pragma unroll 1
    for (int row = 0; row < (TWO_D ? 1 : kRows); ++row) {
        int u, v;
        pixel_of<TWO_D>(c, sv, row, u, v);
        if (u >= tl.n_u || v >= tl.n_v) continue;
        const int64_t k = ((int64_t)c.view * tl.n_u + u) * tl.n_v + v;
        Ray ray;
        float out = 0.0f;
        if (setup_ray<F>(sv, g, u, v, ray) && ray.tend > 0.0f) {
            const float ax = __fmul_rn(walk_gather<!TWO_D>(ray, x), ray.scale);
            out = __fdiv_rn(__fsub_rn(__ldg(y + k), ax), __fmul_rn(ray.tend, ray.scale));
        }
        res[k] = out;
    }
}

// ---- CGLS ------------------------------------------------------------------------------------
// Device-side scalars of a CGLS run: gamma = |s|^2, delta = |q|^2, alpha, beta (float64).
enum { kGamma = 0, kDelta = 1, kAlpha = 2, kBeta = 3 };

// Sum of a double over the block into partials[blockIdx.x] (all threads must call it).
__device__ __forceinline__ void block_sum_to(double v, double* __restrict__ partials) {
    __shared__ double warp_sums[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_sums[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) s += warp_sums[w];
        partials[blockIdx.x] = s;
    }
}

// q = A p, and per block the float64 sum of q^2 (for delta = |q|^2).
template <bool TWO_D, int F>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    project_norm_kernel(const ViewRec* __restrict__ views, const Grid g, const Tiling tl,
                        const float* __restrict__ vol, float* __restrict__ sino,
                        double* __restrict__ partials) {
    __shared__ ViewRec sv;
    const TileCoord c = tile_of_block(tl);
    load_view(views, c.view, sv);
    double sq = 0.0;
#pragma unroll 1
    for (int row = 0; row < (TWO_D ? 1 : kRows); ++row) {
        int u, v;
        pixel_of<TWO_D>(c, sv, row, u, v);
        if (u >= tl.n_u || v >= tl.n_v) continue;
        Ray ray;
        float q = 0.0f;
        if (setup_ray<F>(sv, g, u, v, ray))
            q = __fmul_rn(walk_gather<!TWO_D>(ray, vol), ray.scale);
        sino[((int64_t)c.view * tl.n_u + u) * tl.n_v + v] = q;
        sq = __fma_rn((double)q, (double)q, sq);
    }
    block_sum_to(sq, partials);
}

// r <- r - alpha q, then scatter the new r (s = A^T r accumulates into vol).
template <bool TWO_D, int F>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    backproject_residual_kernel(const ViewRec* __restrict__ views, const Grid g, const Tiling tl,
                                float* __restrict__ r, const float* __restrict__ q,
                                const double* __restrict__ scal, float* __restrict__ vol) {
    __shared__ ViewRec sv;
    const TileCoord c = tile_of_block(tl);
    load_view(views, c.view, sv);
    const float alpha = (float)scal[kAlpha];
#pragma unroll 1
    for (int row = 0; row < (TWO_D ? 1 : kRows); ++row) {
        int u, v;
        pixel_of<TWO_D>(c, sv, row, u, v);
        if (u >= tl.n_u || v >= tl.n_v) continue;
        const int64_t k = ((int64_t)c.view * tl.n_u + u) * tl.n_v + v;
        const float y = __fmaf_rn(-alpha, __ldg(q + k), r[k]);
        r[k] = y;
        if (y == 0.0f) continue;
        Ray ray;
        if (setup_ray<F>(sv, g, u, v, ray))
            walk_scatter(ray, vol, __fmul_rn(y, ray.scale));
    }
}

// Per-block float64 sums of v^2 (grid-stride over n elements).
__global__ void __launch_bounds__(kThreads) norm_partials_kernel(const float* __restrict__ v,
                                                                  int64_t n,
                                                                  double* __restrict__ partials) {
    double s = 0.0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const double x = (double)__ldg(v + i);
        s = __fma_rn(x, x, s);
    }
    block_sum_to(s, partials);
}

// One block: total of the partials, then the CGLS scalar step `which`:
//   0: delta = total, alpha = gamma / delta      (after q = A p)
//   1: beta = total / gamma, gamma = total       (after s = A^T r)
//   2: gamma = total, alpha = beta = 0           (start)
// A zero denominator gives 0 (the run has converged).
__global__ void __launch_bounds__(kThreads) cgls_scalars_kernel(const double* __restrict__ partials,
                                                                 int32_t n, double* __restrict__ scal,
                                                                 int32_t which) {
    double s = 0.0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s += partials[i];
    __shared__ double warp_sums[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x != 0) return;
    double total = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) total += warp_sums[w];
    if (which == 0) {
        scal[kDelta] = total;
        scal[kAlpha] = total > 0.0 ? scal[kGamma] / total : 0.0;
    } else if (which == 1) {
        const double gamma = scal[kGamma];
        scal[kBeta] = gamma > 0.0 ? total / gamma : 0.0;
        scal[kGamma] = total;
    } else {
        scal[kGamma] = total;
        scal[kAlpha] = 0.0;
        scal[kBeta] = 0.0;
    }
}

// x += alpha p;  p = s + beta p;  s = 0 (ready for the next backprojection).
__global__ void cgls_update_kernel(float* __restrict__ x, float* __restrict__ p,
                                   float* __restrict__ s, const double* __restrict__ scal,
                                   int64_t n) {
    const float alpha = (float)scal[kAlpha], beta = (float)scal[kBeta];
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float pv = p[i];
        x[i] = __fmaf_rn(alpha, pv, x[i]);
        p[i] = __fmaf_rn(beta, pv, s[i]);
        s[i] = 0.0f;
    }
}

// r = y - q.
__global__ void sub_kernel(float* __restrict__ r, const float* __restrict__ y,
                           const float* __restrict__ q, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        r[i] = __fsub_rn(__ldg(y + i), __ldg(q + i));
}

__global__ void invert_kernel(float* __restrict__ c, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float v = c[i];
        c[i] = v > 0.0f ? __frcp_rn(v) : 0.0f;
    }
}

// x += relax * c * b;  b = 0 (ready for the next backprojection).
__global__ void sirt_update_kernel(float* __restrict__ x, float* __restrict__ b,
                                   const float* __restrict__ c, float relax, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        x[i] = __fmaf_rn(relax, __fmul_rn(c[i], b[i]), x[i]);
        b[i] = 0.0f;
    }
}

// out[b][c][r] = in[b][r][c]; 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) transpose_kernel(const float* __restrict__ in,
                                                        float* __restrict__ out, int64_t rows,
                                                        int64_t cols, int64_t tiles_r,
                                                        int64_t tiles_c) {
    __shared__ float tile[32][33];
    int64_t t = blockIdx.x;
    const int64_t tc = t % tiles_c;
    t /= tiles_c;
    const int64_t tr = t % tiles_r;
    const int64_t b = t / tiles_r;
    const int64_t base = b * rows * cols;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
        const int64_t r = tr * 32 + ty + k, cc = tc * 32 + tx;
        if (r < rows && cc < cols) tile[ty + k][tx] = __ldg(in + base + r * cols + cc);
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
        const int64_t cc = tc * 32 + ty + k, r = tr * 32 + tx;
        if (r < rows && cc < cols) out[base + cc * rows + r] = tile[tx][ty + k];
    }
}

}  // namespace

uint64_t siddon_bounds_violations(bool reset) {
#ifdef CT_DEBUG_BOUNDS
    unsigned long long v = 0;
    cudaMemcpyFromSymbol(&v, g_bounds_violations, sizeof(v));
    if (reset) {
        const unsigned long long zero = 0;
        cudaMemcpyToSymbol(g_bounds_violations, &zero, sizeof(zero));
    }
    return v;
#else
    (void)reset;
    return 0;
#endif
}

namespace {

int64_t grid_for(const Tiling& t) {
    return (int64_t)t.tiles_v * t.n_views * t.tiles_u;
}

int elementwise_blocks(int64_t n) {
    const int64_t most = (int64_t)device_sm_count() * 16;
    int64_t b = (n + 255) / 256;
    return (int)(b < most ? (b > 0 ? b : 1) : most);
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 148;  // a B300's count; only reached when the runtime cannot name the device
    }
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0) {
            cudaGetLastError();
            return 148;
        }
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Instantiation by (2D, inner axis).  2D grids are always walked with x inner.
#define CT_LAUNCH_BY_AXIS(KERNEL, EXTRA, ...)                                                 \
    do {                                                                                     \
        const unsigned nb_ = (unsigned)grid_for(t);                                          \
        if (nb_ == 0) return cudaSuccess;                                                    \
        if (t.two_d)                                                                         \
            KERNEL<true, 0 EXTRA><<<nb_, kThreads, 0, stream>>>(__VA_ARGS__);                \
        else if (g.fast == 2)                                                                \
            KERNEL<false, 2 EXTRA><<<nb_, kThreads, 0, stream>>>(__VA_ARGS__);               \
        else if (g.fast == 1)                                                                \
            KERNEL<false, 1 EXTRA><<<nb_, kThreads, 0, stream>>>(__VA_ARGS__);               \
        else                                                                                 \
            KERNEL<false, 0 EXTRA><<<nb_, kThreads, 0, stream>>>(__VA_ARGS__);               \
        return cudaGetLastError();                                                           \
    } while (0)

#define CT_NO_EXTRA

#define CT_NB1 , 1, false
#define CT_NB2 , 2, false
#define CT_NB4 , 4, false
#define CT_MODE0_NB1 , 0, 1, false
#define CT_MODE0_NB2 , 0, 2, false
#define CT_MODE0_NB4 , 0, 4, false
#define CT_MODE1_NB1 , 1, 1, false

// Shared-line forward projections (t.line != 0, 3D): one block per kLinePixels x kLineRows pixel
// tile, the line's crossing list in dynamic shared memory (8 bytes per outer-axis cell).
template <int NB>
cudaError_t launch_line_project(const ViewRec* views, const Grid& g, const Tiling& t,
                                const float* vol, int64_t vstride, float* sino, int64_t sstride,
                                cudaStream_t stream) {
    const int64_t nblk = (int64_t)t.line_lane_tiles * t.n_views * t.line_row_tiles;
    if (nblk == 0) return cudaSuccess;
    const int a = g.fast == 0 ? 1 : 0, b = g.fast == 2 ? 1 : 2;
    if (t.two_d || g.n[a] + g.n[b] > kLineMaxCells) return cudaErrorInvalidValue;
    const size_t smem = sizeof(LineEntry) * (size_t)(g.n[a] + g.n[b]);
    const unsigned nb = (unsigned)nblk;
    if (g.fast == 2)
        line_project_kernel<2, NB><<<nb, kLinePixels, smem, stream>>>(views, g, t, vol, vstride,
                                                                      sino, sstride);
    else if (g.fast == 1)
        line_project_kernel<1, NB><<<nb, kLinePixels, smem, stream>>>(views, g, t, vol, vstride,
                                                                      sino, sstride);
    else
        line_project_kernel<0, NB><<<nb, kLinePixels, smem, stream>>>(views, g, t, vol, vstride,
                                                                      sino, sstride);
    return cudaGetLastError();
}

// Forward projections of shared-line handles over the per-ray tiles (line parameters).
template <int NB>
cudaError_t launch_line_rays(const ViewRec* views, const Grid& g, const Tiling& t, const float* vol,
                             int64_t vstride, float* sino, int64_t sstride, cudaStream_t stream) {
    const unsigned nb = (unsigned)grid_for(t);
    if (nb == 0) return cudaSuccess;
    if (t.two_d) return cudaErrorInvalidValue;
    if (g.fast == 2)
        project_kernel<false, 2, NB, false, true><<<nb, kThreads, 0, stream>>>(
            views, g, t, vol, vstride, sino, sstride, SlabArgs{});
    else if (g.fast == 1)
        project_kernel<false, 1, NB, false, true><<<nb, kThreads, 0, stream>>>(
            views, g, t, vol, vstride, sino, sstride, SlabArgs{});
    else
        project_kernel<false, 0, NB, false, true><<<nb, kThreads, 0, stream>>>(
            views, g, t, vol, vstride, sino, sstride, SlabArgs{});
    return cudaGetLastError();
}

// 3D backprojections over spread tiles (t.spread != 0): LINE rays for shared-line handles.
template <int MODE, int NB, bool LINE>
cudaError_t launch_spread_bp(const ViewRec* views, const Grid& g, const Tiling& t,
                             const float* sino, int64_t sstride, float* vol, int64_t vstride,
                             cudaStream_t stream) {
    const int64_t nblk = (int64_t)t.spread_tiles_u * t.spread_tiles_v * t.n_views;
    if (nblk == 0) return cudaSuccess;
    const unsigned nb = (unsigned)nblk;
    if (t.two_d) return cudaErrorInvalidValue;
    if (g.fast == 2)
        backproject_kernel<false, 2, MODE, NB, false, LINE, true><<<nb, kThreads, 0, stream>>>(
            views, g, t, sino, sstride, vol, vstride, SlabArgs{});
    else if (g.fast == 1)
        backproject_kernel<false, 1, MODE, NB, false, LINE, true><<<nb, kThreads, 0, stream>>>(
            views, g, t, sino, sstride, vol, vstride, SlabArgs{});
    else
        backproject_kernel<false, 0, MODE, NB, false, LINE, true><<<nb, kThreads, 0, stream>>>(
            views, g, t, sino, sstride, vol, vstride, SlabArgs{});
    return cudaGetLastError();
}

template <int MODE, int NB>
cudaError_t launch_spread_backproject(const ViewRec* views, const Grid& g, const Tiling& t,
                                      const float* sino, int64_t sstride, float* vol,
                                      int64_t vstride, cudaStream_t stream) {
    return launch_spread_bp<MODE, NB, false>(views, g, t, sino, sstride, vol, vstride, stream);
}

// The backprojection over the same lines (line parameters; spread tiles where the handle has
// them, else the per-ray tiles).
template <int NB>
cudaError_t launch_line_backproject(const ViewRec* views, const Grid& g, const Tiling& t,
                                    const float* sino, int64_t sstride, float* vol,
                                    int64_t vstride, cudaStream_t stream) {
    if (t.two_d) return cudaErrorInvalidValue;
    if (t.spread) return launch_spread_bp<0, NB, true>(views, g, t, sino, sstride, vol, vstride, stream);
    const unsigned nb = (unsigned)grid_for(t);
    if (nb == 0) return cudaSuccess;
    if (g.fast == 2)
        backproject_kernel<false, 2, 0, NB, false, true><<<nb, kThreads, 0, stream>>>(
            views, g, t, sino, sstride, vol, vstride, SlabArgs{});
    else if (g.fast == 1)
        backproject_kernel<false, 1, 0, NB, false, true><<<nb, kThreads, 0, stream>>>(
            views, g, t, sino, sstride, vol, vstride, SlabArgs{});
    else
        backproject_kernel<false, 0, 0, NB, false, true><<<nb, kThreads, 0, stream>>>(
            views, g, t, sino, sstride, vol, vstride, SlabArgs{});
    return cudaGetLastError();
}

cudaError_t launch_project(const ViewRec* views, const Grid& g, const Tiling& t, const float* vol,
                           float* sino, cudaStream_t stream) {
    if (t.line) return launch_line_project<1>(views, g, t, vol, 0, sino, 0, stream);
    CT_LAUNCH_BY_AXIS(project_kernel, CT_NB1, views, g, t, vol, (int64_t)0, sino, (int64_t)0,
                      SlabArgs{});
}

cudaError_t launch_backproject(const ViewRec* views, const Grid& g, const Tiling& t,
                               const float* sino, float* vol, cudaStream_t stream) {
    if (t.line) return launch_line_backproject<1>(views, g, t, sino, 0, vol, 0, stream);
    if (t.spread) return launch_spread_backproject<0, 1>(views, g, t, sino, 0, vol, 0, stream);
    CT_LAUNCH_BY_AXIS(backproject_kernel, CT_MODE0_NB1, views, g, t, sino, (int64_t)0, vol,
                      (int64_t)0, SlabArgs{});
}

cudaError_t launch_backproject_ones(const ViewRec* views, const Grid& g, const Tiling& t,
                                    float* vol, cudaStream_t stream) {
    if (t.spread) return launch_spread_backproject<1, 1>(views, g, t, nullptr, 0, vol, 0, stream);
    CT_LAUNCH_BY_AXIS(backproject_kernel, CT_MODE1_NB1, views, g, t, nullptr, (int64_t)0, vol,
                      (int64_t)0, SlabArgs{});
}

cudaError_t launch_project_batch(const ViewRec* views, const Grid& g, const Tiling& t, int nb,
                                 const float* vol, int64_t vstride, float* sino, int64_t sstride,
                                 cudaStream_t stream) {
    if (t.line) {
        // several volumes: the per-ray tiles over the line parameters (the list walk's results
        // bit for bit; four volumes 39.0 -> 27.6 ms on the cone 256^3 workload against the list
        // kernel, which holds only 1024 threads per SM at that register use)
        if (nb == 4) return launch_line_rays<4>(views, g, t, vol, vstride, sino, sstride, stream);
        if (nb == 2) return launch_line_rays<2>(views, g, t, vol, vstride, sino, sstride, stream);
        if (nb == 1) return launch_line_project<1>(views, g, t, vol, vstride, sino, sstride, stream);
        return cudaErrorInvalidValue;
    }
    if (nb == 4)
        CT_LAUNCH_BY_AXIS(project_kernel, CT_NB4, views, g, t, vol, vstride, sino, sstride,
                          SlabArgs{});
    if (nb == 2)
        CT_LAUNCH_BY_AXIS(project_kernel, CT_NB2, views, g, t, vol, vstride, sino, sstride,
                          SlabArgs{});
    if (nb == 1)
        CT_LAUNCH_BY_AXIS(project_kernel, CT_NB1, views, g, t, vol, vstride, sino, sstride,
                          SlabArgs{});
    return cudaErrorInvalidValue;
}

cudaError_t launch_backproject_batch(const ViewRec* views, const Grid& g, const Tiling& t, int nb,
                                     const float* sino, int64_t sstride, float* vol,
                                     int64_t vstride, cudaStream_t stream) {
    if (t.line) {
        if (nb == 4) return launch_line_backproject<4>(views, g, t, sino, sstride, vol, vstride, stream);
        if (nb == 2) return launch_line_backproject<2>(views, g, t, sino, sstride, vol, vstride, stream);
        if (nb == 1) return launch_line_backproject<1>(views, g, t, sino, sstride, vol, vstride, stream);
        return cudaErrorInvalidValue;
    }
    if (t.spread) {
        if (nb == 4) return launch_spread_backproject<0, 4>(views, g, t, sino, sstride, vol, vstride, stream);
        if (nb == 2) return launch_spread_backproject<0, 2>(views, g, t, sino, sstride, vol, vstride, stream);
        if (nb == 1) return launch_spread_backproject<0, 1>(views, g, t, sino, sstride, vol, vstride, stream);
        return cudaErrorInvalidValue;
    }
    if (nb == 4)
        CT_LAUNCH_BY_AXIS(backproject_kernel, CT_MODE0_NB4, views, g, t, sino, sstride, vol, vstride,
                          SlabArgs{});
    if (nb == 2)
        CT_LAUNCH_BY_AXIS(backproject_kernel, CT_MODE0_NB2, views, g, t, sino, sstride, vol, vstride,
                          SlabArgs{});
    if (nb == 1)
        CT_LAUNCH_BY_AXIS(backproject_kernel, CT_MODE0_NB1, views, g, t, sino, sstride, vol, vstride,
                          SlabArgs{});
    return cudaErrorInvalidValue;
}

cudaError_t launch_project_slab(const ViewRec* views, const Grid& g, const Tiling& t, int nb,
                                const float* vol, int64_t vstride, float* sino, int64_t sstride,
                                const SlabArgs& slab, cudaStream_t stream) {
    const unsigned nblk = (unsigned)((int64_t)slab.n_tiles * t.tiles_u);
    if (nblk == 0) return cudaSuccess;
    if (t.two_d || g.fast != 2) return cudaErrorInvalidValue;
    if (nb == 4)
        project_kernel<false, 2, 4, true><<<nblk, kThreads, 0, stream>>>(views, g, t, vol, vstride,
                                                                         sino, sstride, slab);
    else if (nb == 2)
        project_kernel<false, 2, 2, true><<<nblk, kThreads, 0, stream>>>(views, g, t, vol, vstride,
                                                                         sino, sstride, slab);
    else if (nb == 1)
        project_kernel<false, 2, 1, true><<<nblk, kThreads, 0, stream>>>(views, g, t, vol, vstride,
                                                                         sino, sstride, slab);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_backproject_slab(const ViewRec* views, const Grid& g, const Tiling& t, int nb,
                                    const float* sino, int64_t sstride, float* vol,
                                    int64_t vstride, const SlabArgs& slab, cudaStream_t stream) {
    const unsigned nblk = (unsigned)((int64_t)slab.n_tiles * t.tiles_u);
    if (nblk == 0) return cudaSuccess;
    if (t.two_d || g.fast != 2) return cudaErrorInvalidValue;
    if (nb == 4)
        backproject_kernel<false, 2, 0, 4, true><<<nblk, kThreads, 0, stream>>>(
            views, g, t, sino, sstride, vol, vstride, slab);
    else if (nb == 2)
        backproject_kernel<false, 2, 0, 2, true><<<nblk, kThreads, 0, stream>>>(
            views, g, t, sino, sstride, vol, vstride, slab);
    else if (nb == 1)
        backproject_kernel<false, 2, 0, 1, true><<<nblk, kThreads, 0, stream>>>(
            views, g, t, sino, sstride, vol, vstride, slab);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_project_residual(const ViewRec* views, const Grid& g, const Tiling& t,
                                    const float* x, const float* y, float* r,
                                    cudaStream_t stream) {
    CT_LAUNCH_BY_AXIS(project_residual_kernel, CT_NO_EXTRA, views, g, t, x, y, r);
}

int64_t project_blocks(const Tiling& t) { return grid_for(t); }

cudaError_t launch_project_norm(const ViewRec* views, const Grid& g, const Tiling& t,
                                const float* vol, float* sino, double* partials,
                                cudaStream_t stream) {
    CT_LAUNCH_BY_AXIS(project_norm_kernel, CT_NO_EXTRA, views, g, t, vol, sino, partials);
}

cudaError_t launch_backproject_residual(const ViewRec* views, const Grid& g, const Tiling& t,
                                        float* r, const float* q, const double* scal, float* vol,
                                        cudaStream_t stream) {
    CT_LAUNCH_BY_AXIS(backproject_residual_kernel, CT_NO_EXTRA, views, g, t, r, q, scal, vol);
}

int norm_blocks(int sm_count) { return sm_count * 8; }

cudaError_t launch_norm_partials(const float* v, int64_t n, double* partials, int sm_count,
                                 cudaStream_t stream) {
    norm_partials_kernel<<<norm_blocks(sm_count), kThreads, 0, stream>>>(v, n, partials);
    return cudaGetLastError();
}

cudaError_t launch_cgls_scalars(const double* partials, int64_t n, double* scal, int which,
                                cudaStream_t stream) {
    cgls_scalars_kernel<<<1, kThreads, 0, stream>>>(partials, (int32_t)n, scal, which);
    return cudaGetLastError();
}

cudaError_t launch_cgls_update(float* x, float* p, float* s, const double* scal, int64_t n,
                               cudaStream_t stream) {
    cgls_update_kernel<<<elementwise_blocks(n), 256, 0, stream>>>(x, p, s, scal, n);
    return cudaGetLastError();
}

cudaError_t launch_sub(float* r, const float* y, const float* q, int64_t n, cudaStream_t stream) {
    sub_kernel<<<elementwise_blocks(n), 256, 0, stream>>>(r, y, q, n);
    return cudaGetLastError();
}

cudaError_t launch_invert(float* c, int64_t n, cudaStream_t stream) {
    invert_kernel<<<elementwise_blocks(n), 256, 0, stream>>>(c, n);
    return cudaGetLastError();
}

cudaError_t launch_sirt_update(float* x, float* b, const float* c, float relax, int64_t n,
                               cudaStream_t stream) {
    sirt_update_kernel<<<elementwise_blocks(n), 256, 0, stream>>>(x, b, c, relax, n);
    return cudaGetLastError();
}

cudaError_t launch_transpose(const float* in, float* out, int64_t rows, int64_t cols,
                             int64_t batch, cudaStream_t stream) {
    const int64_t tr = (rows + 31) / 32, tc = (cols + 31) / 32;
    const int64_t nb = tr * tc * batch;
    if (nb <= 0) return cudaSuccess;
    transpose_kernel<<<(unsigned)nb, 256, 0, stream>>>(in, out, rows, cols, tr, tc);
    return cudaGetLastError();
}

}  // namespace ct
