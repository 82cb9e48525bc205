/*
 * FP64 CPU oracle in plain C -- TEST INFRASTRUCTURE ONLY.
 *
 * A second, independent restatement of the cross entropy that the NumPy oracle
 * (oracle/__init__.py) also computes; tests check that the two agree.  Nothing
 * in the product links or calls this file.  Plain loops, one row at a time,
 * in the order the definitions state them:
 *
 *   Transformer Engine parallel_cross_entropy (API card "Description",
 *   "I/O Contract"; pull request #3273 "Changes"):
 *     m_n    = max_v z[n, v]
 *     lse_n  = m_n + log sum_v exp(z[n, v] - m_n)
 *     loss_n = (1 - eps)(lse_n - z[n, y_n]) + eps (lse_n - (1/V) sum_v z[n, v])
 *     dz[n, v] = g_n (exp(z[n, v] - lse_n) - (1 - eps)[v = y_n] - eps / V)
 *   rows with y_n == ignore_idx: loss 0, gradient 0, statistics (0, 0);
 *   y_n outside [0, V) and not ignore_idx: loss NaN, gradient 0, flagged.
 *
 *   Linear form (Cut Cross-Entropy card "what_it_does"): z = X W^T, a naive
 *   triple loop; its gradients (Liger SM100 pull request "Summary": backward =
 *   logits recomputation, dX, dW) dX = dZ W and dW = dZ^T X, naive loops.
 *   Per-token entropy of the softmax (Liger pull request, optional entropy):
 *     H_n = -sum_v p_v log p_v = lse_n - sum_v p_v z[n, v],  p_v = exp(z[n, v] - lse_n).
 *
 * Build: gcc -O2 -fPIC -shared -fopenmp (see oracle/c_oracle.py).
 */
#include <math.h>
#include <stdint.h>

/* Forward of the logits form.  z: [n, ld] doubles (first V used per row).
 * Outputs: loss_rows[n], m[n], lse[n], bad[n] (0/1); returns N_v. */
int64_t oracle_ce_forward(const double* z, int64_t n, int64_t V, int64_t ld, const int64_t* y, double eps,
                          int64_t ignore_idx, double* loss_rows, double* m, double* lse, int32_t* bad) {
    int64_t n_valid = 0;
    for (int64_t r = 0; r < n; ++r) n_valid += (y[r] != ignore_idx);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        const double* row = z + r * ld;
        bad[r] = 0;
        if (y[r] == ignore_idx) {
            loss_rows[r] = 0.0;
            m[r] = 0.0;
            lse[r] = 0.0;
            continue;
        }
        double mx = row[0];
        for (int64_t v = 1; v < V; ++v)
            if (row[v] > mx) mx = row[v];
        double s = 0.0;
        for (int64_t v = 0; v < V; ++v) s += exp(row[v] - mx);
        const double l = mx + log(s);
        m[r] = mx;
        lse[r] = l;
        if (y[r] < 0 || y[r] >= V) {
            bad[r] = 1;
            loss_rows[r] = NAN;
            continue;
        }
        double loss = (1.0 - eps) * (l - row[y[r]]);
        if (eps != 0.0) {
            double sum = 0.0;
            for (int64_t v = 0; v < V; ++v) sum += row[v];
            loss += eps * (l - sum / (double)V);
        }
        loss_rows[r] = loss;
    }
    return n_valid;
}

/* Backward of the logits form from the saved lse.  g_rows[n] is the upstream
 * gradient of each row (the caller applies the reduction).  dz: [n, V]. */
void oracle_ce_backward(const double* z, int64_t n, int64_t V, int64_t ld, const int64_t* y, const double* lse,
                        const double* g_rows, double eps, int64_t ignore_idx, double* dz) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        const double* row = z + r * ld;
        double* out = dz + r * V;
        const int zero = (y[r] == ignore_idx) || y[r] < 0 || y[r] >= V;
        for (int64_t v = 0; v < V; ++v) {
            if (zero) {
                out[v] = 0.0;
                continue;
            }
            double d = g_rows[r] * (exp(row[v] - lse[r]) - eps / (double)V);
            if (v == y[r]) d -= g_rows[r] * (1.0 - eps);
            out[v] = d;
        }
    }
}

/* z[n, V] = X[n, H] W[V, H]^T, naive. */
void oracle_linear_logits(const double* X, const double* W, int64_t n, int64_t H, int64_t V, double* z) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r)
        for (int64_t v = 0; v < V; ++v) {
            double acc = 0.0;
            for (int64_t k = 0; k < H; ++k) acc += X[r * H + k] * W[v * H + k];
            z[r * V + v] = acc;
        }
}

/* dX[n, H] = dZ[n, V] W[V, H] and dW[V, H] = dZ^T X, naive. */
void oracle_linear_grads(const double* dz, const double* X, const double* W, int64_t n, int64_t H, int64_t V,
                         double* dX, double* dW) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r)
        for (int64_t k = 0; k < H; ++k) {
            double acc = 0.0;
            for (int64_t v = 0; v < V; ++v) acc += dz[r * V + v] * W[v * H + k];
            dX[r * H + k] = acc;
        }
#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < V; ++v)
        for (int64_t k = 0; k < H; ++k) {
            double acc = 0.0;
            for (int64_t r = 0; r < n; ++r) acc += dz[r * V + v] * X[r * H + k];
            dW[v * H + k] = acc;
        }
}

/* Entropy of each row's softmax from its logits and lse: ent[n]. */
void oracle_entropy(const double* z, int64_t n, int64_t V, const double* lse, double* ent) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        double pz = 0.0;
        for (int64_t v = 0; v < V; ++v) pz += exp(z[r * V + v] - lse[r]) * z[r * V + v];
        ent[r] = lse[r] - pz;
    }
}
