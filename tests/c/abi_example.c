/*
 * A C caller of libvce.so: the logits-form forward and backward on the
 * hand-derived worked example of tests/golden/worked_examples.json (case
 * "three_rows_one_ignored_mean": z row 0 = (ln1, ln2, ln3, ln4) with y = 3,
 * row 1 ignored, row 2 all zeros with y = 1, mean reduction, g = 1).
 * FP32 logits.  Exit code 0 when every value matches.
 */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "vce.h"

#define CHECK(x)                                                              \
    do {                                                                      \
        if (!(x)) {                                                           \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #x);   \
            return 1;                                                         \
        }                                                                     \
    } while (0)

static int close_to(double a, double b, double tol) { return fabs(a - b) <= tol; }

int main(void) {
    const int64_t n = 3, v = 4;
    const float z[12] = {0.0f, 0.6931471805599453f, 1.0986122886681098f, 1.3862943611198906f,
                         5.0f, -3.0f,  2.0f,  7.0f,
                         0.0f,  0.0f,  0.0f,  0.0f};
    const int64_t y[3] = {3, -100, 1};
    const float g = 1.0f;
    /* expected values (derivation in the golden file) */
    const double loss_ref = 1.151292546497023;
    const double dz_ref[12] = {0.05, 0.1, 0.15, -0.3, 0, 0, 0, 0, 0.125, -0.375, 0.125, 0.125};

    float *dz_dev, *z_dev, *loss_dev, *stats_dev, *g_dev;
    int64_t *y_dev, *nv_dev;
    int* status_dev;
    void* ws;
    const size_t ws_bytes = ce_workspace_size(n, v, VCE_REDUCE_MEAN);
    CHECK(cudaMalloc((void**)&z_dev, sizeof z) == cudaSuccess);
    CHECK(cudaMalloc((void**)&dz_dev, sizeof z) == cudaSuccess);
    CHECK(cudaMalloc((void**)&y_dev, sizeof y) == cudaSuccess);
    CHECK(cudaMalloc((void**)&loss_dev, sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc((void**)&stats_dev, 2 * n * sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc((void**)&g_dev, sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc((void**)&nv_dev, sizeof(int64_t)) == cudaSuccess);
    CHECK(cudaMalloc((void**)&status_dev, sizeof(int)) == cudaSuccess);
    CHECK(cudaMalloc(&ws, ws_bytes) == cudaSuccess);
    CHECK(cudaMemcpy(z_dev, z, sizeof z, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(y_dev, y, sizeof y, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(g_dev, &g, sizeof g, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemset(status_dev, 0, sizeof(int)) == cudaSuccess);

    vce_status st = ce_forward(z_dev, VCE_F32, n, v, v, y_dev, 0.0f, VCE_REDUCE_MEAN, -100, loss_dev, stats_dev,
                               nv_dev, ws, ws_bytes, status_dev, NULL);
    CHECK(st == VCE_OK);
    st = ce_backward(z_dev, VCE_F32, n, v, v, y_dev, stats_dev, nv_dev, g_dev, 0.0f, VCE_REDUCE_MEAN, -100, dz_dev,
                     status_dev, NULL);
    CHECK(st == VCE_OK);
    /* host-side validation happens before any launch */
    CHECK(ce_forward(z_dev, 7, n, v, v, y_dev, 0.0f, 1, -100, loss_dev, stats_dev, nv_dev, ws, ws_bytes, NULL,
                     NULL) == VCE_ERR_DTYPE);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);

    float loss, stats[6], dz[12];
    int64_t nv;
    int status;
    CHECK(cudaMemcpy(&loss, loss_dev, sizeof loss, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(stats, stats_dev, sizeof stats, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(dz, dz_dev, sizeof dz, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(&nv, nv_dev, sizeof nv, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(&status, status_dev, sizeof status, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(status == 0);
    CHECK(nv == 2);
    CHECK(close_to(loss, loss_ref, 1e-5 * loss_ref));
    CHECK(close_to(stats[1], 2.302585092994046, 1e-5 * 2.3) && stats[2] == 0.0f && stats[3] == 0.0f);
    for (int i = 0; i < 12; ++i) CHECK(close_to(dz[i], dz_ref[i], 1e-6));
    printf("abi_example ok: loss %.7f n_valid %lld\n", loss, (long long)nv);
    return 0;
}
