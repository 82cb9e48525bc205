// Internal declarations shared by the translation units of libvce.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/vce.h"

namespace vce {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Hardware base-2 exponential (MUFU.EX2 through the PTX instruction); relative
// error of a few ulp, well inside the loss/gradient tolerances.
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The exp2 offset -lse * log2(e) of a row rounded to FP32, and the factor
// 1 + r ln 2 that puts back its rounding residual r (computed exactly with an
// FMA).  Every exponent of the row shares the residual, so the factor scales the
// row's softmax term once instead of changing each element's arithmetic; without
// it the rounding reaches |lse| * 2^-24 relative (4e-5 for logits near 1000).
struct Exp2Offset {
    float neg;  // -lse * log2(e), rounded
    float fix;  // multiply exp2(z * log2(e) + neg) by this
};
__device__ __forceinline__ Exp2Offset exp2_offset(float lse) {
    const float neg = -lse * kLog2e;
    const float r = fmaf(-lse, kLog2e, -neg);
    return {neg, fmaf(r, kLn2, 1.f)};
}

// Upstream gradient of row ``row``: grad_output[row] (no reduction),
// grad_output[0] / N_v (mean) or grad_output[0] (sum).
__device__ __forceinline__ float upstream_grad(int reduce, const float* grad_output, const int64_t* n_valid,
                                               int64_t row) {
    if (reduce == VCE_REDUCE_MEAN) return grad_output[0] / float(n_valid[0]);
    if (reduce == VCE_REDUCE_SUM) return grad_output[0];
    return grad_output[row];
}

__device__ __forceinline__ void report(int* dev_status, int bits) {
    if (dev_status) atomicOr(dev_status, bits);
}

// Bounds checks of the debugging build (-DVCE_BOUNDS_CHECK): VCE_BOUNDS(cond,
// status) is ``cond``, and a false one reports VCE_DEVSTATUS_BOUNDS; callers
// skip the access it guards.  In the normal build it is the constant true.
#ifdef VCE_BOUNDS_CHECK
__device__ __forceinline__ bool bounds_ok(bool ok, int* dev_status) {
    if (!ok) report(dev_status, VCE_DEVSTATUS_BOUNDS);
    return ok;
}
#define VCE_BOUNDS(cond, status) ::vce::bounds_ok(bool(cond), (status))
#else
#define VCE_BOUNDS(cond, status) true
#endif

__device__ __forceinline__ bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Host-side count of the kernels this library has launched (diagnostics).
void count_launch();

// Limits of the bounded mbarrier waits in the pipelined kernels (the GEMM and
// the fused ring kernel).  A wait for work or data gives up after
// kPipeTimeoutNs, sets the CTA's abort flag and the kernel reports
// VCE_DEVSTATUS_TIMEOUT.  A drain wait (for copies or MMAs that were already
// issued, which complete on their own) ignores the abort flag and has a much
// longer limit, so that a CTA gives up its shared and tensor memory only once
// nothing issued into them is still running.
constexpr uint64_t kPipeTimeoutNs = 2000000000ull;    // 2 s
constexpr uint64_t kDrainTimeoutNs = 10000000000ull;  // 10 s

// Settings of one pipelined launch.  The library's own calls use the defaults;
// the failure-detection self-tests shorten the wait limit and set ``hold``: the
// GEMM's scheduler then publishes no work unit and the ring kernel's producer
// issues no copy, so every role's first wait runs out with no copy or MMA in
// flight.
struct PipeDiag {
    uint64_t timeout_ns = kPipeTimeoutNs;
    int hold = 0;
};

// Round up to a multiple of 256 bytes (workspace carving).
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Device properties cached per device ordinal.
struct DeviceInfo {
    int ordinal = -1;
    int cc_major = 0, cc_minor = 0;
    int num_sms = 0;
    size_t max_smem_optin = 0;
    size_t l2_bytes = 0;
};

// Returns VCE_OK and fills ``info`` for the current device, VCE_ERR_CUDA if the
// runtime cannot be queried, VCE_ERR_ARCH if the device is not CC 10.3.
vce_status current_device(DeviceInfo& info);

// ---- logits form launchers (ce_rows.cu) ----
vce_status launch_ce_forward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                             int64_t row_stride, const int64_t* target, float eps,
                             int reduce_loss, int64_t ignore_idx, float* loss, float* stats,
                             int64_t* n_valid, void* ws, int* dev_status, cudaStream_t s,
                             const DeviceInfo& dev);
vce_status launch_ce_backward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                              int64_t row_stride, const int64_t* target, const float* stats,
                              const int64_t* n_valid, const float* grad_output, float eps,
                              int reduce_loss, int64_t ignore_idx, void* dlogits,
                              int* dev_status, cudaStream_t s, const DeviceInfo& dev);
vce_status launch_ce_forward_backward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                                      int64_t row_stride, const int64_t* target, float eps, int reduce_loss,
                                      int64_t ignore_idx, const float* grad_output, float* loss, float* stats,
                                      int64_t* n_valid, void* dlogits, void* ws, int* dev_status,
                                      cudaStream_t s, const DeviceInfo& dev, const PipeDiag& diag = PipeDiag());
// whether ce_forward_backward runs rows of this length through the ring kernel
bool ce_fused_uses_ring(int dtype, int64_t vocab);
vce_status launch_shift_targets(const int64_t* target, int64_t n, int64_t seq_len, int64_t ignore_idx,
                                int64_t* shifted, cudaStream_t s);
// mean of per-row losses over rows whose target is not ignore_idx, and the count
vce_status launch_mean_loss(const float* loss_rows, const int64_t* target, int64_t n_rows,
                            int64_t ignore_idx, int reduce, float* loss_out, int64_t* n_valid,
                            cudaStream_t s);

// ---- linear form (lce_tc.cu) ----
size_t lce_forward_ws_bytes(int64_t n, int64_t v, int reduce_loss);
int64_t lce_slab_for_ws(int64_t n, int64_t h, int64_t v, size_t ws_bytes);
size_t lce_backward_ws_bytes(int64_t n, int64_t h, int64_t v, int64_t slab);
vce_status launch_lce_forward(const void* X, const void* W, int64_t n, int64_t h, int64_t v,
                              const int64_t* target, float eps, int reduce_loss,
                              int64_t ignore_idx, float* loss, float* lse, float* entropy, int64_t* n_valid,
                              void* ws, int* dev_status, cudaStream_t s, const DeviceInfo& dev,
                              const PipeDiag& diag = PipeDiag());
vce_status launch_lce_backward(const void* X, const void* W, int64_t n, int64_t h, int64_t v,
                               const int64_t* target, const float* lse, const int64_t* n_valid,
                               const float* grad_output, float eps, int reduce_loss,
                               int64_t ignore_idx, void* dX, void* dW, void* ws, int64_t slab,
                               int* dev_status, cudaStream_t s, const DeviceInfo& dev);

}  // namespace vce
