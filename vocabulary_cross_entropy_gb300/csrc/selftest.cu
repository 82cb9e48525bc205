// Diagnostics: exercises the bounded mbarrier wait that every tensor-core
// pipeline wait in this library uses, on a barrier that nothing ever arrives
// on.  The wait must give up after its limit and report VCE_DEVSTATUS_TIMEOUT,
// leaving the context usable.  No copy, MMA or tensor memory is involved.

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

}  // namespace
}  // namespace vce

using namespace vce;

extern "C" vce_status vce_selftest_wait_timeout(uint64_t timeout_ns, int* dev_status,
                                                unsigned long long* waited_ns, void* stream) {
    if (!dev_status || timeout_ns == 0 || timeout_ns > 2000000000ull) return VCE_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (vce_status st = current_device(dev)) return st;
    count_launch();
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns, dev_status, waited_ns);
    return cudaGetLastError() == cudaSuccess ? VCE_OK : VCE_ERR_CUDA;
}
