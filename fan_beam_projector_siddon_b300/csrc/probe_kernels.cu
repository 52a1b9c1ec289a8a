// Roofline probes: the access patterns the projector's kernels press on, run over buffers that
// stay resident in L2 (or L1), so that the benchmark can time them with CUDA events and use the
// rates as measured denominators (the on-chip counterpart of a STREAM copy for HBM).
//
//   read:   every thread streams 16-byte loads that bypass L1 (ld.global.cg) over the buffer,
//           `passes` times; the forward walk's gathers are 4-byte loads served by L1 and L2.
//   L1:     every block re-reads the same few KB with loads that allocate in L1, so that after
//           the first pass every load hits (the FDK gather's bilinear reads are L1-served).
//   reduce: every warp issues red.global.add.f32 of 1.0 to 32 floats `stride` elements apart,
//           sweeping the buffer `passes` times; stride 1 puts 8 updates in each 32-byte sector
//           (the best case), stride 2 puts 4 (about what the backprojection achieves).
#include "ct_internal.h"

#include <cuda_runtime.h>

namespace ct {
namespace {

constexpr int kProbeThreads = 512;

__global__ void __launch_bounds__(kProbeThreads)
    l2_read_kernel(const float4* __restrict__ buf, int64_t n4, int32_t passes,
                   float* __restrict__ sink) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a, c = a, d = a;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int32_t p = 0; p < passes; ++p) {
        int64_t i = first;
        // four loads in flight per thread and iteration
        for (; i + 3 * stride < n4; i += 4 * stride) {
            const float4 x = __ldcg(buf + i), y = __ldcg(buf + i + stride),
                         z = __ldcg(buf + i + 2 * stride), w = __ldcg(buf + i + 3 * stride);
            a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
            b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
            c.x += z.x; c.y += z.y; c.z += z.z; c.w += z.w;
            d.x += w.x; d.y += w.y; d.z += w.z; d.w += w.w;
        }
        for (; i < n4; i += stride) {
            const float4 x = __ldcg(buf + i);
            a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
        }
    }
    const float s = a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w + c.x + c.y + c.z + c.w + d.x +
                    d.y + d.z + d.w;
    if (s == -1.0f) sink[0] = s;  // keeps the loads; the caller's buffer holds no such sums
}

// Every block reads the same n4 float4s (a few KB: resident in every SM's L1) `passes` times
// with loads that allocate in L1 (ld.global.ca).
__global__ void __launch_bounds__(kProbeThreads)
    l1_read_kernel(const float4* __restrict__ buf, int64_t n4, int32_t passes,
                   float* __restrict__ sink) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    for (int32_t p = 0; p < passes; ++p) {
        int64_t i = threadIdx.x;
        for (; i + blockDim.x < n4; i += 2 * blockDim.x) {
            const float4 x = __ldca(buf + i), y = __ldca(buf + i + blockDim.x);
            a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
            b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
        }
        if (i < n4) {
            const float4 x = __ldca(buf + i);
            a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
        }
    }
    const float s = a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w;
    if (s == -1.0f) sink[0] = s;
}

__global__ void __launch_bounds__(kProbeThreads)
    l2_reduce_kernel(float* __restrict__ buf, int64_t n, int32_t passes, int32_t stride) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t span = 32 * (int64_t)stride;  // elements one warp instruction covers
    const int64_t groups = n / span;
    float* const base = buf + (int64_t)lane * stride;
    for (int32_t p = 0; p < passes; ++p) {
        int64_t gi = warp;
        // four reductions per warp and iteration, to distant groups
        for (; gi + 3 * warps < groups; gi += 4 * warps) {
            atomicAdd(base + gi * span, 1.0f);
            atomicAdd(base + (gi + warps) * span, 1.0f);
            atomicAdd(base + (gi + 2 * warps) * span, 1.0f);
            atomicAdd(base + (gi + 3 * warps) * span, 1.0f);
        }
        for (; gi < groups; gi += warps) atomicAdd(base + gi * span, 1.0f);
    }
}

}  // namespace

int probe_blocks() { return device_sm_count() * (2048 / kProbeThreads); }

cudaError_t launch_l2_read(const float* buf, int64_t n_floats, int32_t passes, float* sink,
                           cudaStream_t stream) {
    l2_read_kernel<<<probe_blocks(), kProbeThreads, 0, stream>>>(
        reinterpret_cast<const float4*>(buf), n_floats / 4, passes, sink);
    return cudaGetLastError();
}

cudaError_t launch_l1_read(const float* buf, int64_t n_floats, int32_t passes, float* sink,
                           cudaStream_t stream) {
    l1_read_kernel<<<probe_blocks(), kProbeThreads, 0, stream>>>(
        reinterpret_cast<const float4*>(buf), n_floats / 4, passes, sink);
    return cudaGetLastError();
}

cudaError_t launch_l2_reduce(float* buf, int64_t n_floats, int32_t passes, int32_t stride,
                             cudaStream_t stream) {
    l2_reduce_kernel<<<probe_blocks(), kProbeThreads, 0, stream>>>(buf, n_floats, passes, stride);
    return cudaGetLastError();
}

}  // namespace ct
