/*
 * Test program (plain C99): drives libctproj through include/ct.h with raw device pointers, the
 * way a C or C++ caller would, and writes the forward and back projections of a seeded volume to
 * a binary file for the Python test to compare with the ctypes binding.
 *
 *   abi_check OUT_FILE      exit 0 on success, 2 on an unexpected status
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ct.h"

#define CHECK(call, want)                                                                  \
    do {                                                                                   \
        ct_status s_ = (call);                                                             \
        if (s_ != (want)) {                                                                \
            fprintf(stderr, "%s:%d %s -> %s (want %s)\n", __FILE__, __LINE__, #call,       \
                    ct_status_string(s_), ct_status_string(want));                         \
            return 2;                                                                      \
        }                                                                                  \
    } while (0)

static uint64_t lcg = 12345u;
static float next_uniform(void) {
    lcg = lcg * 6364136223846793005ull + 1442695040888963407ull;
    return (float)((lcg >> 40) & 0xffffff) / 16777216.0f;
}

int main(int argc, char** argv) {
    if (argc != 2) return 1;
    enum { NV = 12, NZ = 20, NY = 24, NX = 28, NU = 40, NVV = 30 };
    double views[NV * 12];
    for (int k = 0; k < NV; ++k) {
        const double th = 6.283185307179586 * k / NV, c = cos(th), s = sin(th);
        double* r = views + 12 * k;
        r[0] = 60.0 * c; r[1] = 60.0 * s; r[2] = 0.0;          /* source */
        r[3] = -40.0 * c; r[4] = -40.0 * s; r[5] = 0.0;        /* detector centre */
        r[6] = -s; r[7] = c; r[8] = 0.0;                       /* det_u */
        r[9] = 0.0; r[10] = 0.0; r[11] = 1.0;                  /* det_v */
    }
    ct_geometry* g = NULL;
    CHECK(ct_geometry_create(CT_CONE, NV, views, NZ, NY, NX, 1.0, NU, NVV, 1.5, 1.5, &g), CT_OK);
    ct_geometry_info info;
    CHECK(ct_geometry_get_info(g, &info), CT_OK);
    const size_t nvox = (size_t)info.n_voxels, nray = (size_t)info.n_rays;
    float* h_vol = (float*)malloc(nvox * sizeof(float));
    float* h_out = (float*)malloc((nray + nvox) * sizeof(float));
    for (size_t i = 0; i < nvox; ++i) h_vol[i] = next_uniform();
    float *d_vol = NULL, *d_sino = NULL, *d_back = NULL;
    void* d_ws = NULL;
    if (cudaMalloc((void**)&d_vol, nvox * sizeof(float)) != cudaSuccess ||
        cudaMalloc((void**)&d_sino, nray * sizeof(float)) != cudaSuccess ||
        cudaMalloc((void**)&d_back, nvox * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&d_ws, info.workspace_bytes ? info.workspace_bytes : 1) != cudaSuccess)
        return 3;
    cudaMemcpy(d_vol, h_vol, nvox * sizeof(float), cudaMemcpyHostToDevice);
    cudaStream_t stream;
    cudaStreamCreate(&stream);
    /* error paths: NULL handle, host pointer, aliasing, short workspace */
    CHECK(ct_project(NULL, d_vol, d_sino, d_ws, info.workspace_bytes, stream),
          CT_ERR_INVALID_ARGUMENT);
    CHECK(ct_project(g, h_vol, d_sino, d_ws, info.workspace_bytes, stream),
          CT_ERR_NOT_DEVICE_POINTER);
    CHECK(ct_project(g, d_vol, (float*)d_vol, d_ws, info.workspace_bytes, stream),
          CT_ERR_ALIASING);
    if (info.workspace_bytes)
        CHECK(ct_project(g, d_vol, d_sino, d_ws, info.workspace_bytes - 1, stream),
              CT_ERR_WORKSPACE);
    /* the path */
    CHECK(ct_project(g, d_vol, d_sino, d_ws, info.workspace_bytes, stream), CT_OK);
    CHECK(ct_backproject(g, d_sino, d_back, d_ws, info.workspace_bytes, stream), CT_OK);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return 4;
    cudaMemcpy(h_out, d_sino, nray * sizeof(float), cudaMemcpyDeviceToHost);
    cudaMemcpy(h_out + nray, d_back, nvox * sizeof(float), cudaMemcpyDeviceToHost);
    FILE* f = fopen(argv[1], "wb");
    if (!f) return 5;
    fwrite(views, sizeof(double), NV * 12, f);
    fwrite(h_vol, sizeof(float), nvox, f);
    fwrite(h_out, sizeof(float), nray + nvox, f);
    fclose(f);
    cudaStreamDestroy(stream);
    cudaFree(d_vol); cudaFree(d_sino); cudaFree(d_back); cudaFree(d_ws);
    CHECK(ct_geometry_destroy(g), CT_OK);
    free(h_vol); free(h_out);
    printf("abi_check ok: %zu rays, %zu voxels\n", nray, nvox);
    return 0;
}
