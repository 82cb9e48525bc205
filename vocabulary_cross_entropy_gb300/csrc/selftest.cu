// Diagnostics: failure detection of the bounded waits, exercised without a
// GPU fault.
//
// vce_selftest_wait_timeout runs the bounded mbarrier wait that every pipeline
// wait in this library uses, on a barrier that nothing ever arrives on.
//
// vce_selftest_lce_forward_timeout and vce_selftest_ce_fused_timeout run the
// real pipelined kernels (the tensor-core GEMM of lce_forward, the TMA-fed
// ring kernel of ce_forward_backward) with a short wait limit and their work
// held back: the GEMM's scheduler publishes no work unit, the ring's producer
// issues no copy.  Every role's first wait then runs out with no copy or MMA in
// flight, and the kernels take their timeout exits (abort flag, drain, tensor
// memory released) and report VCE_DEVSTATUS_TIMEOUT.  The context stays
// usable; the outputs of such a call are undefined.

#include "vce_internal.cuh"
#include "sm100_ptx.cuh"

namespace vce {
namespace {

__global__ void wait_timeout_kernel(uint64_t timeout_ns, int* dev_status, unsigned long long* waited_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    sm100::mbar_init(&bar, 1);  // expects one arrival; none comes
    sm100::fence_mbar_init();
    abort_flag = 0;
    const uint64_t t0 = sm100::globaltimer();
    const bool ok = sm100::mbar_wait(&bar, 0, reinterpret_cast<volatile int*>(&abort_flag), timeout_ns);
    if (waited_ns) *waited_ns = sm100::globaltimer() - t0;
    if (!ok) report(dev_status, VCE_DEVSTATUS_TIMEOUT);
}

constexpr uint64_t kMinSelftestNs = 1000;  // 1 us

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace vce

using namespace vce;

extern "C" vce_status vce_selftest_wait_timeout(uint64_t timeout_ns, int* dev_status,
                                                unsigned long long* waited_ns, void* stream) {
    if (!dev_status || timeout_ns == 0 || timeout_ns > kPipeTimeoutNs) return VCE_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (vce_status st = current_device(dev)) return st;
    count_launch();
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns, dev_status, waited_ns);
    return cudaGetLastError() == cudaSuccess ? VCE_OK : VCE_ERR_CUDA;
}

extern "C" vce_status vce_selftest_lce_forward_timeout(const void* X, const void* W, int64_t n, int64_t h,
                                                       int64_t v, const int64_t* target, uint64_t timeout_ns,
                                                       float* loss, float* lse, void* ws, size_t ws_bytes,
                                                       int* dev_status, void* stream) {
    if (!dev_status || timeout_ns < kMinSelftestNs || timeout_ns > kPipeTimeoutNs) return VCE_ERR_INVALID_ARG;
    if (n < 1 || h < 1 || v < 1 || !X || !W || !target || !loss || !lse) return VCE_ERR_INVALID_ARG;
    if (h % 8 != 0 || !aligned(X, 16) || !aligned(W, 16)) return VCE_ERR_ALIGN;
    if (!ws || ws_bytes < lce_forward_ws_bytes(n, v, VCE_REDUCE_NONE)) return VCE_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return VCE_ERR_ALIGN;
    DeviceInfo dev;
    if (vce_status st = current_device(dev)) return st;
    PipeDiag diag;
    diag.timeout_ns = timeout_ns;
    diag.hold = 1;
    return launch_lce_forward(X, W, n, h, v, target, 0.f, VCE_REDUCE_NONE, -100, loss, lse, nullptr, nullptr, ws,
                              dev_status, static_cast<cudaStream_t>(stream), dev, diag);
}

extern "C" vce_status vce_selftest_ce_fused_timeout(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                                                    int64_t row_stride, const int64_t* target,
                                                    const float* grad_output, uint64_t timeout_ns, float* loss,
                                                    float* stats, void* dlogits, int* dev_status, void* stream) {
    if (dtype != VCE_BF16 && dtype != VCE_F32) return VCE_ERR_DTYPE;
    if (!dev_status || timeout_ns < kMinSelftestNs || timeout_ns > kPipeTimeoutNs) return VCE_ERR_INVALID_ARG;
    if (n_rows < 1 || vocab < 1 || row_stride < vocab || !logits || !target || !grad_output || !loss || !stats ||
        !dlogits)
        return VCE_ERR_INVALID_ARG;
    if (!ce_fused_uses_ring(dtype, vocab)) return VCE_ERR_INVALID_ARG;  // short rows have no pipeline
    const size_t es = dtype == VCE_BF16 ? 2 : 4;
    if (!aligned(logits, es) || !aligned(dlogits, es) || !aligned(stats, 8)) return VCE_ERR_ALIGN;
    if (((reinterpret_cast<uintptr_t>(logits) ^ reinterpret_cast<uintptr_t>(dlogits)) & 15) != 0)
        return VCE_ERR_ALIGN;
    DeviceInfo dev;
    if (vce_status st = current_device(dev)) return st;
    PipeDiag diag;
    diag.timeout_ns = timeout_ns;
    diag.hold = 1;
    return launch_ce_forward_backward(logits, dtype, n_rows, vocab, row_stride, target, 0.f, VCE_REDUCE_NONE, -100,
                                      grad_output, loss, stats, nullptr, dlogits, nullptr, dev_status,
                                      static_cast<cudaStream_t>(stream), dev, diag);
}
