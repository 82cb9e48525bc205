/*
 * A C caller of libvce.so.
 *
 * Logits form: ce_forward + ce_backward, then the fused ce_forward_backward,
 * on the hand-derived worked example of tests/golden/worked_examples.json (case
 * "three_rows_one_ignored_mean": z row 0 = (ln1, ln2, ln3, ln4) with y = 3,
 * row 1 ignored, row 2 all zeros with y = 1, mean reduction, g = 1), FP32
 * logits.
 *
 * Linear form (when a case file is given as argv[1]): lce_forward +
 * lce_backward on BF16 X [n, h] and W [v, h], checked against FP64 values of
 * the oracle.  The file is plain whitespace-separated text:
 *     n h v label_smoothing reduce_loss ignore_idx grad_output n_valid loss
 *     target[n]  X bits[n*h]  W bits[v*h]  (BF16 bit patterns)
 *     lse[n]  dX[n*h]  dW[v*h]
 *
 * Exit code 0 when every value matches.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

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

static double bf16_value(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ||got - ref|| / ||ref|| for BF16 results against FP64 references */
static double rel_err_bf16(const uint16_t* got, const double* ref, long long count) {
    double num = 0.0, den = 0.0;
    for (long long i = 0; i < count; ++i) {
        const double d = bf16_value(got[i]) - ref[i];
        num += d * d;
        den += ref[i] * ref[i];
    }
    return sqrt(num) / sqrt(den);
}

static int run_linear(const char* path) {
    FILE* f = fopen(path, "r");
    CHECK(f != NULL);
    long long n, h, v, red, ign, nv_ref;
    double eps, g, loss_ref;
    CHECK(fscanf(f, "%lld %lld %lld %lf %lld %lld %lf %lld %lf", &n, &h, &v, &eps, &red, &ign, &g, &nv_ref,
                 &loss_ref) == 9);
    int64_t* y = malloc(n * sizeof *y);
    uint16_t* x = malloc(n * h * sizeof *x);
    uint16_t* w = malloc(v * h * sizeof *w);
    double* lse_ref = malloc(n * sizeof *lse_ref);
    double* dx_ref = malloc(n * h * sizeof *dx_ref);
    double* dw_ref = malloc(v * h * sizeof *dw_ref);
    CHECK(y && x && w && lse_ref && dx_ref && dw_ref);
    for (long long i = 0; i < n; ++i) {
        long long t;
        CHECK(fscanf(f, "%lld", &t) == 1);
        y[i] = t;
    }
    for (long long i = 0; i < n * h; ++i) {
        unsigned b;
        CHECK(fscanf(f, "%u", &b) == 1);
        x[i] = (uint16_t)b;
    }
    for (long long i = 0; i < v * h; ++i) {
        unsigned b;
        CHECK(fscanf(f, "%u", &b) == 1);
        w[i] = (uint16_t)b;
    }
    for (long long i = 0; i < n; ++i) CHECK(fscanf(f, "%lf", &lse_ref[i]) == 1);
    for (long long i = 0; i < n * h; ++i) CHECK(fscanf(f, "%lf", &dx_ref[i]) == 1);
    for (long long i = 0; i < v * h; ++i) CHECK(fscanf(f, "%lf", &dw_ref[i]) == 1);
    fclose(f);

    void *x_dev, *w_dev, *dx_dev, *dw_dev, *ws;
    int64_t *y_dev, *nv_dev;
    float *loss_dev, *lse_dev, *g_dev;
    int* status_dev;
    const float gf = (float)g;
    const size_t ws_bytes = lce_workspace_size(n, h, v, (int)red, 0);
    CHECK(ws_bytes > 0);
    CHECK(cudaMalloc(&x_dev, n * h * 2) == cudaSuccess);
    CHECK(cudaMalloc(&w_dev, v * h * 2) == cudaSuccess);
    CHECK(cudaMalloc(&dx_dev, n * h * 2) == cudaSuccess);
    CHECK(cudaMalloc(&dw_dev, v * h * 2) == cudaSuccess);
    CHECK(cudaMalloc(&ws, ws_bytes) == cudaSuccess);
    CHECK(cudaMalloc((void**)&y_dev, n * sizeof *y) == cudaSuccess);
    CHECK(cudaMalloc((void**)&nv_dev, sizeof(int64_t)) == cudaSuccess);
    CHECK(cudaMalloc((void**)&loss_dev, sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc((void**)&lse_dev, n * sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc((void**)&g_dev, sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc((void**)&status_dev, sizeof(int)) == cudaSuccess);
    CHECK(cudaMemcpy(x_dev, x, n * h * 2, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(w_dev, w, v * h * 2, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(y_dev, y, n * sizeof *y, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(g_dev, &gf, sizeof gf, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemset(status_dev, 0, sizeof(int)) == cudaSuccess);

    CHECK(lce_forward(x_dev, w_dev, n, h, v, y_dev, (float)eps, (int)red, ign, loss_dev, lse_dev, NULL, nv_dev,
                      ws, ws_bytes, status_dev, NULL) == VCE_OK);
    CHECK(lce_backward(x_dev, w_dev, n, h, v, y_dev, lse_dev, nv_dev, g_dev, (float)eps, (int)red, ign, dx_dev,
                       dw_dev, ws, ws_bytes, status_dev, NULL) == VCE_OK);
    /* host-side validation: H must be a multiple of 8 */
    CHECK(lce_forward(x_dev, w_dev, n, h - 1, v, y_dev, (float)eps, (int)red, ign, loss_dev, lse_dev, NULL,
                      nv_dev, ws, ws_bytes, status_dev, NULL) == VCE_ERR_ALIGN);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);

    float loss;
    int64_t nv;
    int status;
    float* lse = malloc(n * sizeof *lse);
    uint16_t* dx = malloc(n * h * 2);
    uint16_t* dw = malloc(v * h * 2);
    CHECK(lse && dx && dw);
    CHECK(cudaMemcpy(&loss, loss_dev, sizeof loss, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(&nv, nv_dev, sizeof nv, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(&status, status_dev, sizeof status, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(lse, lse_dev, n * sizeof *lse, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(dx, dx_dev, n * h * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(dw, dw_dev, v * h * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(status == 0);
    CHECK(nv == nv_ref);
    /* BF16 inputs: loss and lse within 2e-3, dX and dW within 1e-2 norm-wise */
    CHECK(close_to(loss, loss_ref, 2e-3));
    for (long long i = 0; i < n; ++i) CHECK(close_to(lse[i], lse_ref[i], 2e-3));
    const double ex = rel_err_bf16(dx, dx_ref, n * h), ew = rel_err_bf16(dw, dw_ref, v * h);
    CHECK(ex <= 1e-2 && ew <= 1e-2);
    for (long long i = 0; i < n; ++i)
        if (y[i] == ign)
            for (long long j = 0; j < h; ++j) CHECK(dx[i * h + j] == 0); /* ignored token: zero gradient */
    printf("abi_example linear ok: loss %.7f n_valid %lld dX err %.2e dW err %.2e\n", loss, (long long)nv, ex, ew);
    cudaFree(x_dev); cudaFree(w_dev); cudaFree(dx_dev); cudaFree(dw_dev); cudaFree(ws); cudaFree(y_dev);
    cudaFree(nv_dev); cudaFree(loss_dev); cudaFree(lse_dev); cudaFree(g_dev); cudaFree(status_dev);
    free(y); free(x); free(w); free(lse_ref); free(dx_ref); free(dw_ref); free(lse); free(dx); free(dw);
    return 0;
}

int main(int argc, char** argv) {
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

    /* the fused call: the same results from one pass over the logits */
    CHECK(cudaMemset(dz_dev, 0, sizeof z) == cudaSuccess);
    CHECK(ce_forward_backward(z_dev, VCE_F32, n, v, v, y_dev, 0.0f, VCE_REDUCE_MEAN, -100, g_dev, loss_dev,
                              stats_dev, nv_dev, dz_dev, ws, ws_bytes, status_dev, NULL) == VCE_OK);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    CHECK(cudaMemcpy(&loss, loss_dev, sizeof loss, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(dz, dz_dev, sizeof dz, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(&nv, nv_dev, sizeof nv, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(&status, status_dev, sizeof status, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(status == 0 && nv == 2);
    CHECK(close_to(loss, loss_ref, 1e-5 * loss_ref));
    for (int i = 0; i < 12; ++i) CHECK(close_to(dz[i], dz_ref[i], 1e-6));
    printf("abi_example ok: loss %.7f n_valid %lld\n", loss, (long long)nv);
    cudaFree(z_dev); cudaFree(dz_dev); cudaFree(y_dev); cudaFree(loss_dev); cudaFree(stats_dev);
    cudaFree(g_dev); cudaFree(nv_dev); cudaFree(status_dev); cudaFree(ws);

    if (argc > 1 && run_linear(argv[1]) != 0) return 1;
    return 0;
}
