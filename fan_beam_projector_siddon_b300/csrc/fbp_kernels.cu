// Filtered backprojection (parallel FBP, fan FBP, cone FDK) for sm_103a.
//
// Stages (diffct "Differentiable analytical reconstruction" and its parallel/fan/cone FBP example
// pages name them; the formulas are the textbook ones):
//   1. per view: physical frame, cosine-weight constants, gather constants and the view weight
//      (fbp_prepare_kernel, float64 on the device from the raw view records);
//   2. filter taps of the band-limited ramp with the chosen window, closed forms in float64
//      (same kernel);
//   3. per detector column: cosine pre-weight and linear convolution along u with the taps,
//      columns staged in shared memory (fbp_filter_kernel);
//   4. voxel-driven gather: project each voxel centre onto every view's detector, interpolate
//      the filtered sinogram bilinearly (0 outside), apply the distance weight and the view
//      weight, sum over views (fbp_gather_kernel).
// This operator is not the Siddon adjoint; it is a separate, approximate inverse.
#include "ct_internal.h"

#include <cuda_runtime.h>

namespace ct {
namespace {

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

// One thread per view (its FbpView) and one thread per filter tap, over one flat grid.
__global__ void fbp_prepare_kernel(FbpParams p, const double* __restrict__ raw,
                                   const float* __restrict__ user_weights,
                                   FbpView* __restrict__ out_views, float* __restrict__ taps) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int n_taps = 2 * p.n_u - 1;
    if (i < n_taps) {
        const int n = i - (p.n_u - 1);
        taps[i] = (float)(ramp_tap(p.window, n * p.du, p.du) * p.du);  // tau * h(n tau)
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
        for (int a = 0; a < 3; ++a) { s[a] = r[a]; c[a] = r[3 + a]; u[a] = r[6 + a]; v[a] = r[9 + a]; }
        n[0] = u[1] * v[2] - u[2] * v[1];
        n[1] = u[2] * v[0] - u[0] * v[2];
        n[2] = u[0] * v[1] - u[1] * v[0];
    }
    const double w = user_weights ? (double)user_weights[i] : 3.14159265358979323846 / p.n_views;
    const double cu = 0.5 * (p.n_u - 1), cv = p.two_d ? 0.0 : 0.5 * (p.n_v - 1);
    FbpView V;
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
        // pixel (iu, iv) = pc + iu * pdu + iv * pdv   (for the cosine weights)
        V.pc[a] = (float)(c[a] - cu * p.du * u[a] - cv * (p.two_d ? 0.0 : p.dv * v[a]) - s[a]);
        V.pdu[a] = (float)(p.du * u[a]);
        V.pdv[a] = p.two_d ? 0.0f : (float)(p.dv * v[a]);
    }
    V.D = (float)D;
    if (p.parallel) {
        // u(X) = X . eu - c . eu / du + cu
        V.ku0 = (float)(cu - ccu / p.du);
        V.kv0 = 0.0f;
        V.wg = (float)w;
    } else {
        V.ku0 = (float)(scu / p.du + cu);
        V.kv0 = (float)(p.two_d ? 0.0 : scv / p.dv + cv);
        // weight w * (D_sd / D_so) / U^2 with U = den / D_so  ->  w * |D| * |D_so| / den^2
        V.wg = (float)(w * fabs(D) * fabs(Dso));
    }
    out_views[i] = V;
}

// Cosine pre-weight and linear convolution along u for one view and a tile of tv detector
// columns (v values).  Shared memory: the pre-weighted tile [n_u][tv] and the taps.
__global__ void __launch_bounds__(256) fbp_filter_kernel(FbpParams p,
                                                        const FbpView* __restrict__ views,
                                                        const float* __restrict__ taps,
                                                        const float* __restrict__ sino,
                                                        float* __restrict__ out, int tv,
                                                        int v_blocks) {
    extern __shared__ float sm[];
    const int n_u = p.n_u, V = p.two_d ? 1 : p.n_v;
    float* tile = sm;                       // [n_u][tv]
    float* stap = sm + (int64_t)n_u * tv;   // [2 n_u - 1]
    const int view = blockIdx.x / v_blocks;
    const int v0 = (blockIdx.x - view * v_blocks) * tv;
    const int nv = min(tv, V - v0);
    const FbpView& W = views[view];
    for (int i = threadIdx.x; i < 2 * n_u - 1; i += blockDim.x) stap[i] = taps[i];
    for (int i = threadIdx.x; i < n_u * tv; i += blockDim.x) {
        const int iu = i / tv, j = i - iu * tv;
        float val = 0.0f;
        if (j < nv) {
            val = sino[((int64_t)view * n_u + iu) * V + v0 + j];
            if (!p.parallel) {  // |(c - s) . n| / |pixel - s|
                const float fu = (float)iu, fv = (float)(v0 + j);
                float d2 = 0.0f;
#pragma unroll
                for (int a = 0; a < 3; ++a) {
                    const float d = fmaf(fv, W.pdv[a], fmaf(fu, W.pdu[a], W.pc[a]));
                    d2 = fmaf(d, d, d2);
                }
                val *= fabsf(W.D) * rsqrtf(d2);
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
        out[((int64_t)view * n_u + iu) * V + v0 + j] = acc;
    }
}

// Voxel-driven gather.  Block: 32 lanes along the volume's fastest gathered axis (z for 3D, x for
// 2D) x 8 along x (3D) or y (2D); views staged in shared memory in chunks.
template <int MODE>  // 0 parallel 2D, 1 fan 2D, 2 cone
__global__ void __launch_bounds__(256) fbp_gather_kernel(FbpParams p,
                                                        const FbpView* __restrict__ views,
                                                        const float* __restrict__ q,
                                                        float* __restrict__ vol) {
    constexpr int kChunk = 32;
    __shared__ FbpView sv[kChunk];
    __shared__ float st[8][33];
    const int lane = threadIdx.x & 31, row = threadIdx.x >> 5;
    int ix, iy, iz;
    if (MODE == 2) {  // blocks: (z tiles of 32) x (x tiles of 8) x y
        iz = blockIdx.x * 32 + lane;
        ix = blockIdx.y * 8 + row;
        iy = blockIdx.z;
    } else {          // blocks: (x tiles of 32) x (y tiles of 8)
        ix = blockIdx.x * 32 + lane;
        iy = blockIdx.y * 8 + row;
        iz = 0;
    }
    const bool inside = ix < p.nx && iy < p.ny && iz < p.nz;
    const float X = ((float)ix + 0.5f - 0.5f * p.nx) * p.sx;
    const float Y = ((float)iy + 0.5f - 0.5f * p.ny) * p.sy;
    const float Z = MODE == 2 ? ((float)iz + 0.5f - 0.5f * p.nz) * p.sz : 0.0f;
    const int n_u = p.n_u, V = MODE == 2 ? p.n_v : 1;
    float acc = 0.0f;
    for (int k0 = 0; k0 < p.n_views; k0 += kChunk) {
        __syncthreads();
        const int nk = min(kChunk, p.n_views - k0);
        constexpr int kWords = (int)(sizeof(FbpView) / sizeof(float));
        for (int i = threadIdx.x; i < nk * kWords; i += blockDim.x)
            reinterpret_cast<float*>(sv)[i] = reinterpret_cast<const float*>(views + k0)[i];
        __syncthreads();
        if (!inside) continue;
        for (int k = 0; k < nk; ++k) {
            const FbpView& W = sv[k];
            float up, vp = 0.0f, g;
            if (MODE == 0) {
                up = fmaf(Y, W.eu[1], fmaf(X, W.eu[0], W.ku0));
                g = W.wg;
            } else {
                const float ax = X - W.s[0], ay = Y - W.s[1], az = Z - W.s[2];
                const float den = fmaf(az, W.n[2], fmaf(ay, W.n[1], ax * W.n[0]));
                const float inv = 1.0f / den;
                const float t = W.D * inv;
                up = fmaf(t, fmaf(az, W.eu[2], fmaf(ay, W.eu[1], ax * W.eu[0])), W.ku0);
                if (MODE == 2) vp = fmaf(t, fmaf(az, W.ev[2], fmaf(ay, W.ev[1], ax * W.ev[0])), W.kv0);
                g = W.wg * inv * inv;
            }
            // keep the indices in int range (a voxel in the source's plane gives inf or NaN,
            // which lands off the detector and contributes 0)
            up = fminf(fmaxf(up, -2.0f), (float)n_u + 1.0f);
            vp = fminf(fmaxf(vp, -2.0f), (float)V + 1.0f);
            const float fu0 = floorf(up), fv0 = floorf(vp);
            const int u0 = (int)fu0, v0 = (int)fv0;
            const float fu = up - fu0, fv = vp - fv0;
            const float* base = q + (int64_t)(k0 + k) * n_u * V;
            float s00 = 0.f, s10 = 0.f, s01 = 0.f, s11 = 0.f;
            const bool u0ok = u0 >= 0 && u0 < n_u, u1ok = u0 + 1 >= 0 && u0 + 1 < n_u;
            const bool v0ok = v0 >= 0 && v0 < V, v1ok = v0 + 1 >= 0 && v0 + 1 < V;
            if (u0ok && v0ok) s00 = __ldg(base + (int64_t)u0 * V + v0);
            if (u1ok && v0ok) s10 = __ldg(base + (int64_t)(u0 + 1) * V + v0);
            if (MODE == 2) {
                if (u0ok && v1ok) s01 = __ldg(base + (int64_t)u0 * V + v0 + 1);
                if (u1ok && v1ok) s11 = __ldg(base + (int64_t)(u0 + 1) * V + v0 + 1);
            }
            const float a0 = fmaf(fu, s10 - s00, s00);
            const float val = MODE == 2 ? fmaf(fv, fmaf(fu, s11 - s01, s01) - a0, a0) : a0;
            acc = fmaf(g, val, acc);
        }
    }
    if (MODE == 2) {  // transpose through shared memory so that the stores run along x
        __syncthreads();
        st[row][lane] = acc;
        __syncthreads();
        // 256 threads store the 8 (x) x 32 (z) tile: thread -> (z = t / 8, x = t % 8)
        const int t = threadIdx.x, zz = t >> 3, xx = t & 7;
        const int oz = blockIdx.x * 32 + zz, ox = blockIdx.y * 8 + xx;
        if (oz < p.nz && ox < p.nx)
            vol[((int64_t)oz * p.ny + iy) * p.nx + ox] = st[xx][zz];
    } else if (inside) {
        vol[(int64_t)iy * p.nx + ix] = acc;
    }
}

}  // namespace

cudaError_t launch_fbp(const FbpParams& p, const double* raw, const float* user_weights,
                       FbpView* views, float* taps, const float* sino, float* filtered,
                       float* vol, cudaStream_t stream) {
    const int n_prep = p.n_views > 2 * p.n_u - 1 ? p.n_views : 2 * p.n_u - 1;
    fbp_prepare_kernel<<<(n_prep + 255) / 256, 256, 0, stream>>>(p, raw, user_weights, views,
                                                                 taps);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int V = p.two_d ? 1 : p.n_v;
    // columns per filter block: as many (up to 32) as fit in shared memory with the taps
    const size_t tap_bytes = sizeof(float) * (size_t)(2 * p.n_u - 1);
    const size_t budget = 200u * 1024u;
    int tv = 32;
    while (tv > 1 && (size_t)tv * p.n_u * sizeof(float) + tap_bytes > budget) tv >>= 1;
    if (tv > V) tv = V;
    const size_t smem = (size_t)tv * p.n_u * sizeof(float) + tap_bytes;
    if (smem > budget) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(fbp_filter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    const int v_blocks = (V + tv - 1) / tv;
    if ((int64_t)v_blocks * p.n_views > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
    fbp_filter_kernel<<<v_blocks * p.n_views, 256, smem, stream>>>(p, views, taps, sino, filtered,
                                                                  tv, v_blocks);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (p.two_d) {
        if ((p.ny + 7) / 8 > 65535) return cudaErrorInvalidValue;
        dim3 g((p.nx + 31) / 32, (p.ny + 7) / 8);
        if (p.parallel)
            fbp_gather_kernel<0><<<g, 256, 0, stream>>>(p, views, filtered, vol);
        else
            fbp_gather_kernel<1><<<g, 256, 0, stream>>>(p, views, filtered, vol);
    } else {
        if ((p.nx + 7) / 8 > 65535 || p.ny > 65535) return cudaErrorInvalidValue;
        dim3 g((p.nz + 31) / 32, (p.nx + 7) / 8, p.ny);
        fbp_gather_kernel<2><<<g, 256, 0, stream>>>(p, views, filtered, vol);
    }
    return cudaGetLastError();
}

}  // namespace ct
