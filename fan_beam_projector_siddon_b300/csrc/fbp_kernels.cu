// Filtered backprojection (parallel FBP, fan FBP, cone FDK) for sm_103a.
//
// Stages (diffct "Differentiable analytical reconstruction" and its parallel/fan/cone FBP example
// pages name them; the formulas are the textbook ones):
//   1. per view: physical frame, cosine-weight constants, gather constants and the view weight
//      (fbp_prepare_kernel, float64 on the device from the raw view records);
//   2. filter taps of the band-limited ramp with the chosen window, closed forms in float64
//      (same kernel);
//   3. per detector column: cosine pre-weight and linear convolution along u with the taps,
//      columns staged in shared memory, written into a zero-padded filtered sinogram
//      (fbp_filter_blocked_kernel: 32 columns a block, 16 outputs a thread held in registers;
//      fbp_filter_kernel for 2D and very wide detectors);
//   4. voxel-driven gather: project each voxel centre onto every view's detector, interpolate
//      the filtered sinogram bilinearly (0 outside, read from the pads without branches), apply
//      the distance weight and the view weight, sum over views (fdk_gather_kernel,
//      fbp2d_gather_kernel).  Per-view constants are staged in shared memory; each thread keeps
//      several voxels along one axis so that the constants and the voxel-independent parts of
//      the projection are loaded and computed once per view.
// This operator is not the Siddon adjoint; it is a separate, approximate inverse.
#include "ct_internal.h"

#include <algorithm>

#include <cuda_runtime.h>

namespace ct {
namespace {

#ifdef CT_DEBUG_BOUNDS
__device__ unsigned long long g_bounds_violations = 0;
#endif

// True when 0 <= i < n; in bounds-checking builds a miss is counted (the caller skips the access).
__device__ __forceinline__ bool in_bounds(int64_t i, int64_t n) {
#ifdef CT_DEBUG_BOUNDS
    if ((uint64_t)i >= (uint64_t)n) {
        atomicAdd(&g_bounds_violations, 1ull);
        return false;
    }
#else
    (void)i;
    (void)n;
#endif
    return true;
}

// I(x) = int_0^F f cos(2 pi f x) df  and  J(c) = int_0^F sin(2 pi f c) df.
__device__ double ramp_I(double x, double F) {
    if (x == 0.0) return 0.5 * F * F;
    const double a = 2.0 * 3.14159265358979323846 * x;
    double s, c;
    sincos(a * F, &s, &c);
    return (c - 1.0) / (a * a) + F * s / a;
}
__device__ double ramp_J(double c0, double F) {
    if (c0 == 0.0) return 0.0;
    const double a = 2.0 * 3.14159265358979323846 * c0;
    return (1.0 - cos(a * F)) / a;
}

// h(x) = 2 int_0^F f W(f) cos(2 pi f x) df, F = 1 / (2 tau), for the windows of FbpWindow.
__device__ double ramp_tap(int window, double x, double tau) {
    const double F = 0.5 / tau;
    switch (window) {
        case FBP_SHEPP_LOGAN:  // W = sin(pi f tau) / (pi f tau)
            return (ramp_J(0.5 * tau + x, F) + ramp_J(0.5 * tau - x, F)) /
                   (3.14159265358979323846 * tau);
        case FBP_COSINE:  // W = cos(pi f tau)
            return ramp_I(x + 0.5 * tau, F) + ramp_I(x - 0.5 * tau, F);
        case FBP_HAMMING:  // W = 0.54 + 0.46 cos(2 pi f tau)
            return 2.0 * 0.54 * ramp_I(x, F) + 0.46 * (ramp_I(x + tau, F) + ramp_I(x - tau, F));
        case FBP_HANN:  // W = 0.5 + 0.5 cos(2 pi f tau)
            return ramp_I(x, F) + 0.5 * (ramp_I(x + tau, F) + ramp_I(x - tau, F));
        default:  // ram-lak: W = 1
            return 2.0 * ramp_I(x, F);
    }
}

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ int64_t qrow(const FbpParams& p, int view, int u) {
    return ((int64_t)view * p.rows + u + 1) * p.cols;
}

// Transpose scatter target: parity copies of the padded detector.  With padded indices
// U = u + 1 in [0, n_u + 2] and V = v + 1 in [0, n_v + 2], copy (pu, pv) in {0,1}^2 stores pixel
// (U, V) in the 2 x 2 block ((U + pu) / 2, (V + pv) / 2), slot ((U + pu) & 1) * 2 + ((V + pv) & 1),
// blocks of 4 floats in [copy][view][bu][bv] order.  A bilinear footprint (U0..U0+1, V0..V0+1)
// is then one aligned float4 of copy (U0 & 1, V0 & 1), added with one vector reduction; the
// pixel's value is the sum over the four copies.  2D: copies pu in {0,1} of pairs (U + pu) / 2,
// slot (U + pu) & 1, in [copy][view][bu] order (float2 reductions).
__device__ __forceinline__ float4* copy_block(const FbpParams& p, float* q, int view, int U0,
                                              int V0) {
    const int pu = U0 & 1, pv = V0 & 1;
    const int64_t blk = (((int64_t)(pu * 2 + pv) * p.n_views + view) * p.bu + ((U0 + pu) >> 1)) *
                            p.bv + ((V0 + pv) >> 1);
    if (!in_bounds(blk, 4 * (int64_t)p.n_views * p.bu * p.bv)) return nullptr;
    return reinterpret_cast<float4*>(q) + blk;
}
__device__ __forceinline__ float2* copy_pair(const FbpParams& p, float* q, int view, int U0) {
    const int pu = U0 & 1;
    const int64_t blk = ((int64_t)pu * p.n_views + view) * p.bu + ((U0 + pu) >> 1);
    if (!in_bounds(blk, 2 * (int64_t)p.n_views * p.bu)) return nullptr;
    return reinterpret_cast<float2*>(q) + blk;
}
__device__ __forceinline__ void red_add4(float4* a, float x, float y, float z, float w) {
#ifdef CT_DEBUG_BOUNDS
    if (a == nullptr) return;
#endif
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(a), "f"(x), "f"(y),
                 "f"(z), "f"(w)
                 : "memory");
}
__device__ __forceinline__ void red_add2(float2* a, float x, float y) {
#ifdef CT_DEBUG_BOUNDS
    if (a == nullptr) return;
#endif
    asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(a), "f"(x), "f"(y) : "memory");
}
// Sum of the copies at padded pixel (U, V) (2D: V ignored).
__device__ __forceinline__ float copies_at(const FbpParams& p, const float* q, int view, int U,
                                           int V) {
    if (p.two_d) {
        float s = 0.0f;
#pragma unroll
        for (int pu = 0; pu < 2; ++pu) {
            const int64_t blk = ((int64_t)pu * p.n_views + view) * p.bu + ((U + pu) >> 1);
            s += q[blk * 2 + ((U + pu) & 1)];
        }
        return s;
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int pu = c >> 1, pv = c & 1;
        const int64_t blk = (((int64_t)c * p.n_views + view) * p.bu + ((U + pu) >> 1)) * p.bv +
                            ((V + pv) >> 1);
        s += q[blk * 4 + ((U + pu) & 1) * 2 + ((V + pv) & 1)];
    }
    return s;
}

// One thread per view (its FbpView and FbpCosine) and one thread per filter tap, over one flat
// grid.
__global__ void fbp_prepare_kernel(FbpParams p, const double* __restrict__ raw,
                                   const float* __restrict__ user_weights,
                                   FbpView* __restrict__ out_views,
                                   FbpCosine* __restrict__ out_cos, float* __restrict__ taps) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int n_taps = 2 * p.n_u - 1;
    if (i < n_taps) {
        // the transpose's filter is the forward's with the taps reversed
        const int src = p.reverse_kernel ? n_taps - 1 - i : i;
        const int n = src - (p.n_u - 1);
        taps[i] = p.kernel ? p.kernel[src]
                           : (float)(ramp_tap(p.window, n * p.du, p.du) * p.du);  // tau h(n tau)
    }
    if (i >= p.n_views) return;
    const double* r = raw + (int64_t)i * (p.two_d ? 6 : 12);
    double s[3], c[3], u[3], v[3], n[3];
    if (p.two_d) {
        s[0] = r[0]; s[1] = r[1]; s[2] = 0.0;
        c[0] = r[2]; c[1] = r[3]; c[2] = 0.0;
        u[0] = r[4]; u[1] = r[5]; u[2] = 0.0;
        v[0] = 0.0; v[1] = 0.0; v[2] = 1.0;
        n[0] = u[1]; n[1] = -u[0]; n[2] = 0.0;
    } else {
        for (int a = 0; a < 3; ++a) {
            s[a] = r[a]; c[a] = r[3 + a]; u[a] = r[6 + a]; v[a] = r[9 + a];
        }
        n[0] = u[1] * v[2] - u[2] * v[1];
        n[1] = u[2] * v[0] - u[0] * v[2];
        n[2] = u[0] * v[1] - u[1] * v[0];
    }
    const double w = p.unit_weights ? 1.0
                     : user_weights ? (double)user_weights[i]
                                    : 3.14159265358979323846 / p.n_views;
    const double cu = 0.5 * (p.n_u - 1), cv = p.two_d ? 0.0 : 0.5 * (p.n_v - 1);
    const double dvv = p.two_d ? 0.0 : p.dv;
    FbpView V;
    FbpCosine C;
    double D = 0.0, Dso = 0.0, scu = 0.0, scv = 0.0, ccu = 0.0;
    for (int a = 0; a < 3; ++a) {
        D += (c[a] - s[a]) * n[a];
        Dso += (p.iso[a] - s[a]) * n[a];
        scu += (s[a] - c[a]) * u[a];
        scv += (s[a] - c[a]) * v[a];
        ccu += c[a] * u[a];
    }
    for (int a = 0; a < 3; ++a) {
        V.s[a] = (float)s[a];
        V.n[a] = (float)n[a];
        V.eu[a] = (float)(u[a] / p.du);
        V.ev[a] = p.two_d ? 0.0f : (float)(v[a] / p.dv);
        // pixel (iu, iv) minus the source = pc + iu * pdu + iv * pdv
        C.pc[a] = (float)(c[a] - cu * p.du * u[a] - cv * dvv * v[a] - s[a]);
        C.pdu[a] = (float)(p.du * u[a]);
        C.pdv[a] = (float)(dvv * v[a]);
    }
    V.D = (float)D;
    C.D = (float)fabs(D);
    C.pad[0] = C.pad[1] = 0.0f;
    if (p.parallel) {
        // u(X) = X . det_u / du - c . det_u / du + cu
        V.ku0 = (float)(cu - ccu / p.du);
        V.kv0 = 0.0f;
        V.wg = (float)w;
    } else {
        // u(X) = ku0 + D ((X - s) . det_u / du) / ((X - s) . n), likewise v
        V.ku0 = (float)(scu / p.du + cu);
        V.kv0 = (float)(p.two_d ? 0.0 : scv / p.dv + cv);
        // w (D_sd / D_so) / U^2 with U = den / D_so  =  w |D| |D_so| / den^2
        V.wg = (float)(w * fabs(D) * fabs(Dso));
    }
    out_views[i] = V;
    out_cos[i] = C;
}

// Cosine weight |(c - s) . n| / |P(iu, iv) - s| of one pixel.
__device__ __forceinline__ float cosine_weight(const FbpCosine& C, int iu, int iv) {
    const float fu = (float)iu, fv = (float)iv;
    float d2 = 0.0f;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        const float d = fmaf(fv, C.pdv[a], fmaf(fu, C.pdu[a], C.pc[a]));
        d2 = fmaf(d, d, d2);
    }
    return C.D * rsqrtf(d2);
}

// Zero pads of the filtered sinogram that belong to columns [v0, v0 + nv) of one view (rows -1,
// n_u, n_u + 1), plus the pad columns -1 and V, V + 1 over all rows when the tile touches them.
__device__ void write_pads(const FbpParams& p, int view, int v0, int nv, float* out) {
    const int V = p.two_d ? 1 : p.n_v;
    if (p.two_d) {
        if (threadIdx.x < 3) {
            const int u = threadIdx.x == 0 ? -1 : p.n_u + (int)threadIdx.x - 1;
            out[qrow(p, view, u)] = 0.0f;
        }
        return;
    }
    for (int i = threadIdx.x; i < 3 * nv; i += blockDim.x) {
        const int rr = i / nv, j = i - rr * nv;
        const int u = rr == 0 ? -1 : p.n_u + rr - 1;
        out[qrow(p, view, u) + v0 + j + 1] = 0.0f;
    }
    if (v0 == 0)
        for (int u = (int)threadIdx.x - 1; u < p.n_u + 2; u += blockDim.x)
            out[qrow(p, view, u)] = 0.0f;
    if (v0 + nv == V)
        for (int u = (int)threadIdx.x - 1; u < p.n_u + 2; u += blockDim.x) {
            out[qrow(p, view, u) + V + 1] = 0.0f;
            out[qrow(p, view, u) + V + 2] = 0.0f;
        }
}

// Cosine pre-weight and linear convolution along u for one view and a tile of tv detector
// columns (v values); one output per thread and step.  Shared memory: the pre-weighted tile
// [n_u][tv] and the taps.  Used for 2D sinograms (one column a view) and wide detectors.
// ADJ (the transpose): the input is the padded array (interior only), the convolution is the same
// (its matrix is symmetric) and the cosine weight multiplies the output instead.
template <bool ADJ>
__global__ void __launch_bounds__(256) fbp_filter_kernel(FbpParams p,
                                                        const FbpCosine* __restrict__ cosines,
                                                        const float* __restrict__ taps,
                                                        const float* __restrict__ in,
                                                        float* __restrict__ out, int tv,
                                                        int v_blocks) {
    extern __shared__ float sm[];
    const int n_u = p.n_u, V = p.two_d ? 1 : p.n_v;
    float* tile = sm;                       // [n_u][tv]
    float* stap = sm + (int64_t)n_u * tv;   // [2 n_u - 1]
    const int view = blockIdx.x / v_blocks;
    const int v0 = (blockIdx.x - view * v_blocks) * tv;
    const int nv = min(tv, V - v0);
    const int vo = p.two_d ? 0 : 1;
    const FbpCosine C = cosines[view];
    for (int i = threadIdx.x; i < 2 * n_u - 1; i += blockDim.x) stap[i] = taps[i];
    for (int i = threadIdx.x; i < n_u * tv; i += blockDim.x) {
        const int iu = i / tv, j = i - iu * tv;
        float val = 0.0f;
        if (j < nv) {
            if (ADJ) {
                val = copies_at(p, in, view, iu + 1, v0 + j + 1);
            } else {
                val = in[((int64_t)view * n_u + iu) * V + v0 + j];
                if (!p.parallel) val *= cosine_weight(C, iu, v0 + j);
                if (p.pixel_weights) val *= p.pixel_weights[(int64_t)view * n_u + iu];
            }
        }
        tile[i] = val;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_u * tv; i += blockDim.x) {
        const int iu = i / tv, j = i - iu * tv;
        if (j >= nv) continue;
        float acc = 0.0f;
        const float* h = stap + (iu + n_u - 1);  // h[iu - k] = stap[iu - k + n_u - 1]
        for (int k = 0; k < n_u; ++k) acc = fmaf(h[-k], tile[k * tv + j], acc);
        if (ADJ) {
            if (!p.parallel) acc *= cosine_weight(C, iu, v0 + j);
            if (p.pixel_weights) acc *= p.pixel_weights[(int64_t)view * n_u + iu];
            out[((int64_t)view * n_u + iu) * V + v0 + j] = acc;
        } else {
            out[qrow(p, view, iu) + v0 + j + vo] = acc;
        }
    }
    if (!ADJ) write_pads(p, view, v0, nv, out);
}

// The same filter for 3D sinograms, 32 columns a block (one per lane) and R consecutive outputs
// a thread: each step loads R tile values and 2R - 1 taps (broadcast) for R * R FMAs.  The tile
// has n_pad >= n_u rows (multiple of R, zero beyond n_u); taps are stored so that
// stap[m] = h(m - (n_pad - 1)), zero outside the filter's support.
template <int R, bool ADJ>
__global__ void __launch_bounds__(256) fbp_filter_blocked_kernel(
    FbpParams p, const FbpCosine* __restrict__ cosines, const float* __restrict__ taps,
    const float* __restrict__ in, float* __restrict__ out, int n_pad, int v_blocks) {
    extern __shared__ float sm[];
    float* tile = sm;                     // [n_pad][32]
    float* stap = sm + (int64_t)n_pad * 32;  // [2 n_pad]
    const int n_u = p.n_u, V = p.n_v;
    const int view = blockIdx.x / v_blocks;
    const int v0 = (blockIdx.x - view * v_blocks) * 32;
    const int nv = min(32, V - v0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int shift = n_pad - n_u;
    for (int m = threadIdx.x; m < 2 * n_pad; m += blockDim.x) {
        const int g = m - shift;
        stap[m] = (g >= 0 && g < 2 * n_u - 1) ? taps[g] : 0.0f;
    }
    const FbpCosine C = cosines[view];
    for (int i = threadIdx.x; i < n_pad * 32; i += blockDim.x) {
        const int k = i >> 5, j = i & 31;
        float val = 0.0f;
        if (k < n_u && j < nv) {
            if (ADJ) {
                val = copies_at(p, in, view, k + 1, v0 + j + 1);
            } else {
                val = in[((int64_t)view * n_u + k) * V + v0 + j];
                if (!p.parallel) val *= cosine_weight(C, k, v0 + j);
                if (p.pixel_weights) val *= p.pixel_weights[(int64_t)view * n_u + k];
            }
        }
        tile[i] = val;
    }
    __syncthreads();
    for (int r0 = warp * R; r0 < n_u; r0 += 8 * R) {
        float acc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] = 0.0f;
        for (int k0 = 0; k0 < n_pad; k0 += R) {
            float t[R], hh[2 * R - 1];
#pragma unroll
            for (int i = 0; i < R; ++i) t[i] = tile[(k0 + i) * 32 + lane];
            const float* hp = stap + (r0 - k0 - (R - 1) + n_pad - 1);
#pragma unroll
            for (int d = 0; d < 2 * R - 1; ++d) hh[d] = hp[d];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int i = 0; i < R; ++i) acc[r] = fmaf(hh[r - i + R - 1], t[i], acc[r]);
        }
        if (lane < nv) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r0 + r >= n_u) continue;
                if (ADJ) {
                    float a = p.parallel ? acc[r] : acc[r] * cosine_weight(C, r0 + r, v0 + lane);
                    if (p.pixel_weights) a *= p.pixel_weights[(int64_t)view * n_u + r0 + r];
                    out[((int64_t)view * n_u + r0 + r) * V + v0 + lane] = a;
                } else {
                    out[qrow(p, view, r0 + r) + v0 + lane + 1] = acc[r];
                }
            }
        }
    }
    if (!ADJ) write_pads(p, view, v0, nv, out);
}

// Cone-beam (FDK) gather.  Block: 8 warps, one x each; lane l of a warp takes the NZ voxels
// z0 + l + 32 m (m < NZ) at that x and at y = blockIdx.z, so a warp's 32 lanes read 32
// neighbouring v of the same detector rows.  Views are staged in shared memory in chunks.
template <int NZ>
__global__ void __launch_bounds__(256) fdk_gather_kernel(FbpParams p,
                                                        const FbpView* __restrict__ views,
                                                        const float* __restrict__ q,
                                                        float* __restrict__ vol, int k_begin,
                                                        int k_end) {
    constexpr int kChunk = 64;
    __shared__ float4 sv[kChunk * 4];
    __shared__ float st[8][NZ * 32 + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int z0 = blockIdx.x * (32 * NZ);
    const int ix = blockIdx.y * 8 + warp;
    const int iy = blockIdx.z;
    const float X = ((float)ix + 0.5f - 0.5f * p.nx) * p.sx;
    const float Y = ((float)iy + 0.5f - 0.5f * p.ny) * p.sy;
    float Z[NZ], acc[NZ];
#pragma unroll
    for (int m = 0; m < NZ; ++m) {
        Z[m] = ((float)(z0 + lane + 32 * m) + 0.5f - 0.5f * p.nz) * p.sz;
        acc[m] = 0.0f;
    }
    const int cols = p.cols;
    const int64_t view_stride = (int64_t)p.rows * cols;
    const float umax = (float)p.n_u, vmax = (float)p.n_v;
    for (int k0 = k_begin; k0 < k_end; k0 += kChunk) {
        __syncthreads();
        const int nk = min(kChunk, k_end - k0);
        for (int i = threadIdx.x; i < nk * 4; i += blockDim.x)
            sv[i] = reinterpret_cast<const float4*>(views + k0)[i];
        __syncthreads();
        const float* base = q + (int64_t)k0 * view_stride;
        for (int k = 0; k < nk; ++k, base += view_stride) {
            // A = (s, n.x), B = (n.y, n.z, eu.x, eu.y), C = (eu.z, ev), E = (D, ku0, kv0, wg)
            const float4 A = sv[4 * k], B = sv[4 * k + 1], C = sv[4 * k + 2], E = sv[4 * k + 3];
            const float ax = X - A.x, ay = Y - A.y;
            const float den_xy = fmaf(ay, B.x, ax * A.w);
            const float au_xy = fmaf(ay, B.w, ax * B.z);
            const float av_xy = fmaf(ay, C.z, ax * C.y);
            if (B.y == 0.0f && C.x == 0.0f) {
                // n.z = 0 and det_u.z = 0 (a detector whose v axis is the z axis, as on circular
                // and helical orbits): den, u and the weight do not depend on z.  The same
                // operations as below with the z terms exactly zero, so the results are the
                // general path's bit for bit.
                const float inv = rcp_approx(den_xy);
                const float t = E.x * inv;
                const float up = fminf(fmaxf(fmaf(t, au_xy, E.y), -1.0f), umax);
                const float fu0 = floorf(up), fu = up - fu0;
                const float g = E.w * inv * inv;
                const float* prow = base + ((int)fu0 + 1) * cols + 1;
#pragma unroll
                for (int m = 0; m < NZ; ++m) {
                    const float av = fmaf(Z[m] - A.z, C.w, av_xy);
                    const float vp = fminf(fmaxf(fmaf(t, av, E.z), -1.0f), vmax);
                    const float fv0 = floorf(vp), fv = vp - fv0;
                    const float* pq = prow + (int)fv0;
#ifdef CT_DEBUG_BOUNDS
                    if (!in_bounds(pq - q, (int64_t)p.n_views * p.rows * cols - cols - 1)) continue;
#endif
                    const float s00 = __ldg(pq), s01 = __ldg(pq + 1);
                    const float s10 = __ldg(pq + cols), s11 = __ldg(pq + cols + 1);
                    const float a0 = fmaf(fv, s01 - s00, s00);
                    const float a1 = fmaf(fv, s11 - s10, s10);
                    acc[m] = fmaf(g, fmaf(fu, a1 - a0, a0), acc[m]);
                }
                continue;
            }
#pragma unroll
            for (int m = 0; m < NZ; ++m) {
                const float az = Z[m] - A.z;
                const float den = fmaf(az, B.y, den_xy);
                const float au = fmaf(az, C.x, au_xy);
                const float av = fmaf(az, C.w, av_xy);
                const float inv = rcp_approx(den);
                const float t = E.x * inv;
                const float up = fminf(fmaxf(fmaf(t, au, E.y), -1.0f), umax);
                const float vp = fminf(fmaxf(fmaf(t, av, E.z), -1.0f), vmax);
                const float fu0 = floorf(up), fv0 = floorf(vp);
                const float fu = up - fu0, fv = vp - fv0;
                const float* pq = base + ((int)fu0 + 1) * cols + (int)fv0 + 1;
#ifdef CT_DEBUG_BOUNDS
                if (!in_bounds(pq - q, (int64_t)p.n_views * p.rows * cols - cols - 1)) continue;
#endif
                const float s00 = __ldg(pq), s01 = __ldg(pq + 1);
                const float s10 = __ldg(pq + cols), s11 = __ldg(pq + cols + 1);
                const float a0 = fmaf(fv, s01 - s00, s00);
                const float a1 = fmaf(fv, s11 - s10, s10);
                const float g = E.w * inv * inv;
                acc[m] = fmaf(g, fmaf(fu, a1 - a0, a0), acc[m]);
            }
        }
    }
    // transpose through shared memory so that the stores run along x
    __syncthreads();
#pragma unroll
    for (int m = 0; m < NZ; ++m) st[warp][lane + 32 * m] = acc[m];
    __syncthreads();
    const int x0 = blockIdx.y * 8;
    for (int i = threadIdx.x; i < 8 * 32 * NZ; i += blockDim.x) {
        const int zz = i >> 3, xx = i & 7;
        const int oz = z0 + zz, ox = x0 + xx;
        if (oz < p.nz && ox < p.nx) {
            float* o = vol + ((int64_t)oz * p.ny + iy) * p.nx + ox;
            *o = k_begin == 0 ? st[xx][zz] : *o + st[xx][zz];
        }
    }
}

// 2D gather (parallel or fan).  Block: lane = x (32 consecutive), warp w takes the NY rows
// y0 + w + 8 m.
template <bool PAR, int NY>
__global__ void __launch_bounds__(256) fbp2d_gather_kernel(FbpParams p,
                                                          const FbpView* __restrict__ views,
                                                          const float* __restrict__ q,
                                                          float* __restrict__ vol) {
    constexpr int kChunk = 64;
    __shared__ float4 sv[kChunk * 4];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ix = blockIdx.x * 32 + lane;
    const int y0 = blockIdx.y * (8 * NY) + warp;
    const float X = ((float)ix + 0.5f - 0.5f * p.nx) * p.sx;
    float Y[NY], acc[NY];
#pragma unroll
    for (int m = 0; m < NY; ++m) {
        Y[m] = ((float)(y0 + 8 * m) + 0.5f - 0.5f * p.ny) * p.sy;
        acc[m] = 0.0f;
    }
    const int rows = p.rows;
    const float umax = (float)p.n_u;
    for (int k0 = 0; k0 < p.n_views; k0 += kChunk) {
        __syncthreads();
        const int nk = min(kChunk, p.n_views - k0);
        for (int i = threadIdx.x; i < nk * 4; i += blockDim.x)
            sv[i] = reinterpret_cast<const float4*>(views + k0)[i];
        __syncthreads();
        const float* base = q + (int64_t)k0 * rows + 1;
        for (int k = 0; k < nk; ++k, base += rows) {
            const float4 A = sv[4 * k], B = sv[4 * k + 1], E = sv[4 * k + 3];
            if (PAR) {
                const float ux = fmaf(X, B.z, E.y);
#pragma unroll
                for (int m = 0; m < NY; ++m) {
                    const float up = fminf(fmaxf(fmaf(Y[m], B.w, ux), -1.0f), umax);
                    const float fu0 = floorf(up), fu = up - fu0;
                    const float* pq = base + (int)fu0;
#ifdef CT_DEBUG_BOUNDS
                    if (!in_bounds(pq - q, (int64_t)p.n_views * rows - 1)) continue;
#endif
                    const float s0 = __ldg(pq), s1 = __ldg(pq + 1);
                    acc[m] = fmaf(E.w, fmaf(fu, s1 - s0, s0), acc[m]);
                }
            } else {
                const float ax = X - A.x;
                const float den_x = ax * A.w, au_x = ax * B.z;
#pragma unroll
                for (int m = 0; m < NY; ++m) {
                    const float ay = Y[m] - A.y;
                    const float den = fmaf(ay, B.x, den_x);
                    const float au = fmaf(ay, B.w, au_x);
                    const float inv = rcp_approx(den);
                    const float up = fminf(fmaxf(fmaf(E.x * inv, au, E.y), -1.0f), umax);
                    const float fu0 = floorf(up), fu = up - fu0;
                    const float* pq = base + (int)fu0;
#ifdef CT_DEBUG_BOUNDS
                    if (!in_bounds(pq - q, (int64_t)p.n_views * rows - 1)) continue;
#endif
                    const float s0 = __ldg(pq), s1 = __ldg(pq + 1);
                    acc[m] = fmaf(E.w * inv * inv, fmaf(fu, s1 - s0, s0), acc[m]);
                }
            }
        }
    }
    if (ix < p.nx) {
#pragma unroll
        for (int m = 0; m < NY; ++m)
            if (y0 + 8 * m < p.ny) vol[(int64_t)(y0 + 8 * m) * p.nx + ix] = acc[m];
    }
}

// Transpose of the cone-beam gather: every voxel adds w g f(X) times its four bilinear
// coefficients, as one float4 reduction, to the parity copies of the padded detector
// (contributions that land in the pads are discarded later).  Same block shape, view passes and
// z-independent path as the gather.
template <int NZ>
__global__ void __launch_bounds__(256) fdk_scatter_kernel(FbpParams p,
                                                         const FbpView* __restrict__ views,
                                                         const float* __restrict__ vol,
                                                         float* __restrict__ q, int k_begin,
                                                         int k_end) {
    constexpr int kChunk = 64;
    __shared__ float4 sv[kChunk * 4];
    __shared__ float st[8][NZ * 32 + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int z0 = blockIdx.x * (32 * NZ);
    const int x0 = blockIdx.y * 8;
    const int ix = x0 + warp;
    const int iy = blockIdx.z;
    // voxel values, loaded along x and transposed through shared memory
    for (int i = threadIdx.x; i < 8 * 32 * NZ; i += blockDim.x) {
        const int zz = i >> 3, xx = i & 7;
        const int oz = z0 + zz, ox = x0 + xx;
        st[xx][zz] = (oz < p.nz && ox < p.nx) ? vol[((int64_t)oz * p.ny + iy) * p.nx + ox] : 0.0f;
    }
    __syncthreads();
    const float X = ((float)ix + 0.5f - 0.5f * p.nx) * p.sx;
    const float Y = ((float)iy + 0.5f - 0.5f * p.ny) * p.sy;
    float Z[NZ], f[NZ];
#pragma unroll
    for (int m = 0; m < NZ; ++m) {
        Z[m] = ((float)(z0 + lane + 32 * m) + 0.5f - 0.5f * p.nz) * p.sz;
        f[m] = st[warp][lane + 32 * m];
    }
    const float umax = (float)p.n_u, vmax = (float)p.n_v;
    for (int k0 = k_begin; k0 < k_end; k0 += kChunk) {
        __syncthreads();
        const int nk = min(kChunk, k_end - k0);
        for (int i = threadIdx.x; i < nk * 4; i += blockDim.x)
            sv[i] = reinterpret_cast<const float4*>(views + k0)[i];
        __syncthreads();
        for (int k = 0; k < nk; ++k) {
            const int view = k0 + k;
            const float4 A = sv[4 * k], B = sv[4 * k + 1], C = sv[4 * k + 2], E = sv[4 * k + 3];
            const float ax = X - A.x, ay = Y - A.y;
            const float den_xy = fmaf(ay, B.x, ax * A.w);
            const float au_xy = fmaf(ay, B.w, ax * B.z);
            const float av_xy = fmaf(ay, C.z, ax * C.y);
            if (B.y == 0.0f && C.x == 0.0f) {  // z-independent u and weight (see the gather)
                const float inv = rcp_approx(den_xy);
                const float t = E.x * inv;
                const float up = fminf(fmaxf(fmaf(t, au_xy, E.y), -1.0f), umax);
                const float fu0 = floorf(up), fu = up - fu0;
                const float g = E.w * inv * inv;
                const int U0 = (int)fu0 + 1;
#pragma unroll
                for (int m = 0; m < NZ; ++m) {
                    const float av = fmaf(Z[m] - A.z, C.w, av_xy);
                    const float vp = fminf(fmaxf(fmaf(t, av, E.z), -1.0f), vmax);
                    const float fv0 = floorf(vp), fv = vp - fv0;
                    const float c = g * f[m];
                    const float c1 = c * fu, c0 = c - c1;
                    const float c01 = c0 * fv, c11 = c1 * fv;
                    red_add4(copy_block(p, q, view, U0, (int)fv0 + 1), c0 - c01, c01, c1 - c11,
                             c11);
                }
                continue;
            }
#pragma unroll
            for (int m = 0; m < NZ; ++m) {
                const float az = Z[m] - A.z;
                const float den = fmaf(az, B.y, den_xy);
                const float au = fmaf(az, C.x, au_xy);
                const float av = fmaf(az, C.w, av_xy);
                const float inv = rcp_approx(den);
                const float t = E.x * inv;
                const float up = fminf(fmaxf(fmaf(t, au, E.y), -1.0f), umax);
                const float vp = fminf(fmaxf(fmaf(t, av, E.z), -1.0f), vmax);
                const float fu0 = floorf(up), fv0 = floorf(vp);
                const float fu = up - fu0, fv = vp - fv0;
                const float c = E.w * inv * inv * f[m];
                const float c1 = c * fu, c0 = c - c1;
                const float c01 = c0 * fv, c11 = c1 * fv;
                red_add4(copy_block(p, q, view, (int)fu0 + 1, (int)fv0 + 1), c0 - c01, c01,
                         c1 - c11, c11);
            }
        }
    }
}

// Transpose of the 2D gather (parallel or fan), same block shape as fbp2d_gather_kernel.
template <bool PAR, int NY>
__global__ void __launch_bounds__(256) fbp2d_scatter_kernel(FbpParams p,
                                                           const FbpView* __restrict__ views,
                                                           const float* __restrict__ vol,
                                                           float* __restrict__ q) {
    constexpr int kChunk = 64;
    __shared__ float4 sv[kChunk * 4];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ix = blockIdx.x * 32 + lane;
    const int y0 = blockIdx.y * (8 * NY) + warp;
    const float X = ((float)ix + 0.5f - 0.5f * p.nx) * p.sx;
    float Y[NY], f[NY];
#pragma unroll
    for (int m = 0; m < NY; ++m) {
        const int iy = y0 + 8 * m;
        Y[m] = ((float)iy + 0.5f - 0.5f * p.ny) * p.sy;
        f[m] = (ix < p.nx && iy < p.ny) ? vol[(int64_t)iy * p.nx + ix] : 0.0f;
    }
    const float umax = (float)p.n_u;
    for (int k0 = 0; k0 < p.n_views; k0 += kChunk) {
        __syncthreads();
        const int nk = min(kChunk, p.n_views - k0);
        for (int i = threadIdx.x; i < nk * 4; i += blockDim.x)
            sv[i] = reinterpret_cast<const float4*>(views + k0)[i];
        __syncthreads();
        for (int k = 0; k < nk; ++k) {
            const int view = k0 + k;
            const float4 A = sv[4 * k], B = sv[4 * k + 1], E = sv[4 * k + 3];
            const float ax = X - A.x;
            const float den_x = ax * A.w, au_x = ax * B.z;
            const float ux = fmaf(X, B.z, E.y);
#pragma unroll
            for (int m = 0; m < NY; ++m) {
                float up, c;
                if (PAR) {
                    up = fminf(fmaxf(fmaf(Y[m], B.w, ux), -1.0f), umax);
                    c = E.w * f[m];
                } else {
                    const float ay = Y[m] - A.y;
                    const float den = fmaf(ay, B.x, den_x);
                    const float au = fmaf(ay, B.w, au_x);
                    const float inv = rcp_approx(den);
                    up = fminf(fmaxf(fmaf(E.x * inv, au, E.y), -1.0f), umax);
                    c = E.w * inv * inv * f[m];
                }
                const float fu0 = floorf(up), fu = up - fu0;
                const float c1 = c * fu;
                red_add2(copy_pair(p, q, view, (int)fu0 + 1), c - c1, c1);
            }
        }
    }
}

constexpr int kFilterR = 16;
constexpr size_t kSmemBudget = 200u * 1024u;

// Filter stage (forward: sinogram -> padded array; ADJ: padded array -> sinogram).
template <bool ADJ>
cudaError_t launch_filter(const FbpParams& p, const FbpCosine* cosines, const float* taps,
                          const float* in, float* out, cudaStream_t stream) {
    cudaError_t e;
    const int V = p.two_d ? 1 : p.n_v;
    const int n_pad = (p.n_u + kFilterR - 1) / kFilterR * kFilterR;
    const size_t blocked_smem = sizeof(float) * ((size_t)n_pad * 32 + 2 * (size_t)n_pad);
    if (!p.two_d && blocked_smem <= kSmemBudget) {
        e = cudaFuncSetAttribute(fbp_filter_blocked_kernel<kFilterR, ADJ>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)blocked_smem);
        if (e != cudaSuccess) return e;
        const int v_blocks = (V + 31) / 32;
        if ((int64_t)v_blocks * p.n_views > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
        fbp_filter_blocked_kernel<kFilterR, ADJ>
            <<<v_blocks * p.n_views, 256, blocked_smem, stream>>>(p, cosines, taps, in, out, n_pad,
                                                                  v_blocks);
        return cudaGetLastError();
    }
    // columns per block: as many (up to 32) as fit in shared memory with the taps
    const size_t tap_bytes = sizeof(float) * (size_t)(2 * p.n_u - 1);
    int tv = 32;
    while (tv > 1 && (size_t)tv * p.n_u * sizeof(float) + tap_bytes > kSmemBudget) tv >>= 1;
    if (tv > V) tv = V;
    const size_t smem = (size_t)tv * p.n_u * sizeof(float) + tap_bytes;
    if (smem > kSmemBudget) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(fbp_filter_kernel<ADJ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    const int v_blocks = (V + tv - 1) / tv;
    if ((int64_t)v_blocks * p.n_views > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
    fbp_filter_kernel<ADJ><<<v_blocks * p.n_views, 256, smem, stream>>>(p, cosines, taps, in, out,
                                                                       tv, v_blocks);
    return cudaGetLastError();
}

// Views per gather or scatter pass: the pass's detector data (the filtered slices the gather
// reads, or the parity copies the scatter adds into, four times larger) fit in L2 together
// (about 48 MB), so that all resident blocks touch the same views and the scatter's reductions
// stay in L2.  Multiples of `step`, at least `step`.
int views_per_pass(const FbpParams& p, size_t bytes_per_view, int step) {
    int per_pass = (int)std::min<size_t>((size_t)p.n_views, (48u << 20) / bytes_per_view);
    return per_pass < step ? step : per_pass / step * step;
}
size_t gather_view_bytes(const FbpParams& p) {
    return sizeof(float) * (size_t)p.rows * (size_t)p.cols;
}
size_t scatter_view_bytes(const FbpParams& p) {
    return sizeof(float4) * 4 * (size_t)p.bu * (size_t)p.bv;  // four copies of 2 x 2 blocks
}

// The cone-beam scatter of vol into the parity copies, in view passes whose copies fit in L2.
// Every pass reads the whole volume again, which is cheap only while the volume stays in L2
// beside the copies; a larger volume takes passes of at least 16 views.
cudaError_t launch_scatter_3d(const FbpParams& p, const FbpView* views, const float* vol,
                              float* copies, cudaStream_t stream) {
    if ((p.nx + 7) / 8 > 65535 || p.ny > 65535) return cudaErrorInvalidValue;
    const size_t vol_bytes = sizeof(float) * (size_t)p.nx * (size_t)p.ny * (size_t)p.nz;
    const int per_pass = views_per_pass(p, scatter_view_bytes(p), vol_bytes > (64u << 20) ? 16 : 4);
    for (int k = 0; k < p.n_views; k += per_pass) {
        const int k_end = std::min(p.n_views, k + per_pass);
        // One voxel per thread: the reductions' latency, not the arithmetic, bounds the scatter,
        // and fewer registers hold more warps (cone 256^3 x 360 views: 8 voxels a thread
        // 27.97 ms, 4: 26.95, 2: 26.58, 1: 25.91; the 512^3 spiral's general path 320.6
        // against 322.7 ms).
        dim3 g((p.nz + 31) / 32, (p.nx + 7) / 8, p.ny);
        fdk_scatter_kernel<1><<<g, 256, 0, stream>>>(p, views, vol, copies, k, k_end);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_prepare(const FbpParams& p, const double* raw, const float* user_weights,
                           FbpView* views, FbpCosine* cosines, float* taps, cudaStream_t stream) {
    const int n_prep = p.n_views > 2 * p.n_u - 1 ? p.n_views : 2 * p.n_u - 1;
    fbp_prepare_kernel<<<(n_prep + 255) / 256, 256, 0, stream>>>(p, raw, user_weights, views,
                                                                 cosines, taps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fbp(const FbpParams& p, const double* raw, const float* user_weights,
                       FbpView* views, FbpCosine* cosines, float* taps, const float* sino,
                       float* filtered, float* vol, cudaStream_t stream) {
    cudaError_t e = launch_prepare(p, raw, user_weights, views, cosines, taps, stream);
    if (e != cudaSuccess) return e;
    if ((e = launch_filter<false>(p, cosines, taps, sino, filtered, stream)) != cudaSuccess)
        return e;
    if (p.two_d) {
        if (p.ny >= 128) {
            if ((p.ny + 31) / 32 > 65535) return cudaErrorInvalidValue;
            dim3 g((p.nx + 31) / 32, (p.ny + 31) / 32);
            if (p.parallel)
                fbp2d_gather_kernel<true, 4><<<g, 256, 0, stream>>>(p, views, filtered, vol);
            else
                fbp2d_gather_kernel<false, 4><<<g, 256, 0, stream>>>(p, views, filtered, vol);
        } else {
            dim3 g((p.nx + 31) / 32, (p.ny + 7) / 8);
            if (p.parallel)
                fbp2d_gather_kernel<true, 1><<<g, 256, 0, stream>>>(p, views, filtered, vol);
            else
                fbp2d_gather_kernel<false, 1><<<g, 256, 0, stream>>>(p, views, filtered, vol);
        }
        return cudaGetLastError();
    }
    if ((p.nx + 7) / 8 > 65535 || p.ny > 65535) return cudaErrorInvalidValue;
    const int per_pass = views_per_pass(p, gather_view_bytes(p), 16);
    for (int k = 0; k < p.n_views; k += per_pass) {
        const int k_end = std::min(p.n_views, k + per_pass);
        if (p.nz >= 192) {
            dim3 g((p.nz + 255) / 256, (p.nx + 7) / 8, p.ny);
            fdk_gather_kernel<8><<<g, 256, 0, stream>>>(p, views, filtered, vol, k, k_end);
        } else if (p.nz >= 96) {
            dim3 g((p.nz + 127) / 128, (p.nx + 7) / 8, p.ny);
            fdk_gather_kernel<4><<<g, 256, 0, stream>>>(p, views, filtered, vol, k, k_end);
        } else if (p.nz >= 48) {
            dim3 g((p.nz + 63) / 64, (p.nx + 7) / 8, p.ny);
            fdk_gather_kernel<2><<<g, 256, 0, stream>>>(p, views, filtered, vol, k, k_end);
        } else {
            dim3 g((p.nz + 31) / 32, (p.nx + 7) / 8, p.ny);
            fdk_gather_kernel<1><<<g, 256, 0, stream>>>(p, views, filtered, vol, k, k_end);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

uint64_t fbp_bounds_violations(bool reset) {
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

// dL/dw_k = sum over the detector of (G_k^T grad) * Q_k (unit-weight scatter times the filtered
// sinogram), one block per view, float64 sums in a fixed order (deterministic).
__global__ void __launch_bounds__(256) fbp_weight_grad_kernel(FbpParams p,
                                                             const float* __restrict__ copies,
                                                             const float* __restrict__ filtered,
                                                             float* __restrict__ grad_w) {
    __shared__ double part[256];
    const int view = blockIdx.x;
    const int V = p.two_d ? 1 : p.n_v;
    const int vo = p.two_d ? 0 : 1;
    double s = 0.0;
    for (int i = threadIdx.x; i < p.n_u * V; i += blockDim.x) {
        const int iu = i / V, iv = i - iu * V;
        const float g = copies_at(p, copies, view, iu + 1, iv + 1);
        const float q = filtered[((int64_t)view * p.rows + iu + 1) * p.cols + iv + vo];
        s += (double)g * (double)q;
    }
    part[threadIdx.x] = s;
    __syncthreads();
    for (int h = 128; h > 0; h >>= 1) {
        if ((int)threadIdx.x < h) part[threadIdx.x] += part[threadIdx.x + h];
        __syncthreads();
    }
    if (threadIdx.x == 0) grad_w[view] = (float)part[0];
}

// Operands of the filter-kernel gradient as row-major arrays over rows r = view * V + v (V = 1 in
// 2D): G[r][u] = w_view (G_k^T grad)[u][v], the scatter summed over the parity copies and scaled
// by the view weight; Q[r][u] = the cosine- and pixel-weighted sinogram.  Then
// dL/dk[d + n_u - 1] = sum_k w_k sum_v sum_i g[i] q[i - d] = sum_{i - j = d} M[i][j] with
// M = G^T Q: a dense contraction over the rows followed by the diagonal sums of M.
__global__ void fbp_grad_lhs_kernel(FbpParams p, const float* __restrict__ view_weights,
                                    const float* __restrict__ copies, float* __restrict__ G) {
    const int V = p.two_d ? 1 : p.n_v;
    const int64_t n = (int64_t)p.n_views * V * p.n_u;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / p.n_u;
        const int u = (int)(e - r * p.n_u);
        const int view = (int)(r / V), v = (int)(r - (int64_t)view * V);
        const float w = view_weights ? view_weights[view] : 3.14159265358979323846f / p.n_views;
        G[e] = w * copies_at(p, copies, view, u + 1, v + 1);
    }
}

__global__ void fbp_grad_rhs_kernel(FbpParams p, const FbpCosine* __restrict__ cosines,
                                    const float* __restrict__ sino, float* __restrict__ Q) {
    const int V = p.two_d ? 1 : p.n_v;
    const int64_t n = (int64_t)p.n_views * V * p.n_u;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / p.n_u;
        const int u = (int)(e - r * p.n_u);
        const int view = (int)(r / V), v = (int)(r - (int64_t)view * V);
        float val = sino[((int64_t)view * p.n_u + u) * V + v];
        if (!p.parallel) val *= cosine_weight(cosines[view], u, v);
        if (p.pixel_weights) val *= p.pixel_weights[(int64_t)view * p.n_u + u];
        Q[e] = val;
    }
}

// One 64 x 64 tile (i, j) of M = G^T Q over one chunk of rows: 16-row steps staged in shared
// memory, 4 x 4 outputs per thread in registers (float32 sums over the chunk), then the tile's
// 127 diagonals summed in shared memory and added into acc[i - j + n_u - 1] in float64.
constexpr int kGT = 64, kGK = 16;

__global__ void __launch_bounds__(256) fbp_kernel_grad_gemm_kernel(
    const float* __restrict__ G, const float* __restrict__ Q, int n_u, int64_t rows,
    int rows_per_chunk, double* __restrict__ acc) {
    __shared__ __align__(16) float As[kGK][kGT];
    __shared__ __align__(16) float Bs[kGK][kGT];
    __shared__ float diag[2 * kGT - 1];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int i0 = blockIdx.x * kGT, j0 = blockIdx.y * kGT;
    const int64_t r_begin = (int64_t)blockIdx.z * rows_per_chunk;
    const int64_t r_end = r_begin + rows_per_chunk < rows ? r_begin + rows_per_chunk : rows;
    float c[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) c[x][y] = 0.0f;
    for (int64_t r0 = r_begin; r0 < r_end; r0 += kGK) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int idx = tid + 256 * e;
            const int k = idx >> 6, col = idx & (kGT - 1);
            const int64_t r = r0 + k;
            const bool ok = r < r_end;
            As[k][col] = (ok && i0 + col < n_u) ? __ldg(G + r * n_u + i0 + col) : 0.0f;
            Bs[k][col] = (ok && j0 + col < n_u) ? __ldg(Q + r * n_u + j0 + col) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kGK; ++k) {
            const float4 a = *reinterpret_cast<const float4*>(&As[k][ty * 4]);
            const float4 b = *reinterpret_cast<const float4*>(&Bs[k][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) c[x][y] = fmaf(av[x], bv[y], c[x][y]);
        }
        __syncthreads();
    }
    for (int t = tid; t < 2 * kGT - 1; t += 256) diag[t] = 0.0f;
    __syncthreads();
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int li = ty * 4 + x, lj = tx * 4 + y;
            if (i0 + li < n_u && j0 + lj < n_u) atomicAdd(&diag[li - lj + kGT - 1], c[x][y]);
        }
    __syncthreads();
    for (int t = tid; t < 2 * kGT - 1; t += 256) {
        const int d = i0 - j0 + t - (kGT - 1);  // i - j
        if (d > -n_u && d < n_u && diag[t] != 0.0f)
            atomicAdd(acc + d + n_u - 1, (double)diag[t]);
    }
}

__global__ void fbp_finish_kernel_grad(const double* __restrict__ acc, float* __restrict__ out,
                                       int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = (float)acc[i];
}

}  // namespace

size_t fbp_copies_floats(const FbpParams& p) {
    return p.two_d ? 2 * 2 * (size_t)p.n_views * (size_t)p.bu
                   : 4 * 4 * (size_t)p.n_views * (size_t)p.bu * (size_t)p.bv;
}

cudaError_t launch_fbp_transpose(const FbpParams& p_in, const double* raw,
                                 const float* user_weights, FbpView* views, FbpCosine* cosines,
                                 float* taps, const float* vol, float* scattered, float* sino,
                                 cudaStream_t stream) {
    FbpParams p = p_in;
    p.reverse_kernel = 1;  // the filter's transpose: the kernel reversed
    cudaError_t e = launch_prepare(p, raw, user_weights, views, cosines, taps, stream);
    if (e != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(scattered, 0, sizeof(float) * fbp_copies_floats(p), stream)) !=
        cudaSuccess)
        return e;
    if (p.two_d) {
        if (p.ny >= 128) {
            if ((p.ny + 31) / 32 > 65535) return cudaErrorInvalidValue;
            dim3 g((p.nx + 31) / 32, (p.ny + 31) / 32);
            if (p.parallel)
                fbp2d_scatter_kernel<true, 4><<<g, 256, 0, stream>>>(p, views, vol, scattered);
            else
                fbp2d_scatter_kernel<false, 4><<<g, 256, 0, stream>>>(p, views, vol, scattered);
        } else {
            dim3 g((p.nx + 31) / 32, (p.ny + 7) / 8);
            if (p.parallel)
                fbp2d_scatter_kernel<true, 1><<<g, 256, 0, stream>>>(p, views, vol, scattered);
            else
                fbp2d_scatter_kernel<false, 1><<<g, 256, 0, stream>>>(p, views, vol, scattered);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    } else if ((e = launch_scatter_3d(p, views, vol, scattered, stream)) != cudaSuccess) {
        return e;
    }
    return launch_filter<true>(p, cosines, taps, scattered, sino, stream);
}

cudaError_t launch_fbp_gradients(const FbpParams& p_in, const double* raw,
                                 const float* user_weights, FbpView* views, FbpCosine* cosines,
                                 float* taps, const float* sino, const float* grad_vol,
                                 float* copies, float* filtered, double* acc, float* grad_kernel,
                                 float* grad_view_weights, cudaStream_t stream) {
    cudaError_t e;
    // (1) the scatter of dL/df with unit view weights: G_k^T grad in the parity copies
    FbpParams pu = p_in;
    pu.unit_weights = 1;
    pu.reverse_kernel = 0;
    if ((e = launch_prepare(pu, raw, user_weights, views, cosines, taps, stream)) != cudaSuccess)
        return e;
    if ((e = cudaMemsetAsync(copies, 0, sizeof(float) * fbp_copies_floats(pu), stream)) !=
        cudaSuccess)
        return e;
    if (pu.two_d) {
        if ((pu.ny + 31) / 32 > 65535) return cudaErrorInvalidValue;
        dim3 g((pu.nx + 31) / 32, (pu.ny + 7) / 8);
        if (pu.parallel)
            fbp2d_scatter_kernel<true, 1><<<g, 256, 0, stream>>>(pu, views, grad_vol, copies);
        else
            fbp2d_scatter_kernel<false, 1><<<g, 256, 0, stream>>>(pu, views, grad_vol, copies);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    } else if ((e = launch_scatter_3d(pu, views, grad_vol, copies, stream)) != cudaSuccess) {
        return e;
    }
    // (2) dL/dw: the filtered sinogram (forward filter) against the scatter
    if (grad_view_weights != nullptr) {
        if ((e = launch_filter<false>(pu, cosines, taps, sino, filtered, stream)) != cudaSuccess)
            return e;
        fbp_weight_grad_kernel<<<pu.n_views, 256, 0, stream>>>(pu, copies, filtered,
                                                                grad_view_weights);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // (3) dL/dkernel: the diagonal sums of G^T Q.  G goes into the filtered buffer (free after
    // step 2), Q into the parity copies (free once G is built); same stream, so in order.
    if (grad_kernel != nullptr) {
        const int n_u = pu.n_u, V = pu.two_d ? 1 : pu.n_v;
        const int64_t rows = (int64_t)pu.n_views * V;
        float* G = filtered;
        float* Q = copies;
        const int64_t n = rows * n_u;
        const int eb = (int)std::min<int64_t>((n + 255) / 256, (int64_t)device_sm_count() * 32);
        fbp_grad_lhs_kernel<<<eb, 256, 0, stream>>>(pu, user_weights, copies, G);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        fbp_grad_rhs_kernel<<<eb, 256, 0, stream>>>(pu, cosines, sino, Q);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(acc, 0, sizeof(double) * (size_t)(2 * n_u - 1), stream)) !=
            cudaSuccess)
            return e;
        // enough row chunks for ~4096 blocks, each at least 256 rows, at most 65535 chunks
        const int64_t tiles = (int64_t)((n_u + kGT - 1) / kGT) * ((n_u + kGT - 1) / kGT);
        int64_t chunk = rows * tiles / 4096;
        chunk = std::max<int64_t>(chunk, 256);
        chunk = std::max<int64_t>(chunk, (rows + 65534) / 65535);
        chunk = (chunk + kGK - 1) / kGK * kGK;
        if (chunk > INT32_MAX) return cudaErrorInvalidValue;
        const dim3 g((n_u + kGT - 1) / kGT, (n_u + kGT - 1) / kGT,
                     (unsigned)((rows + chunk - 1) / chunk));
        if (g.y > 65535) return cudaErrorInvalidValue;
        fbp_kernel_grad_gemm_kernel<<<g, 256, 0, stream>>>(G, Q, n_u, rows, (int)chunk, acc);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        fbp_finish_kernel_grad<<<(2 * n_u - 1 + 255) / 256, 256, 0, stream>>>(acc, grad_kernel,
                                                                              2 * n_u - 1);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace ct
