// ce_forward_noalloc: the logits-form forward for callers that cannot allocate
// device memory.
//
// ce_forward with reduce_loss needs a workspace of n_rows floats for the
// per-row losses it sums afterwards.  Some callers are handed only their
// inputs and outputs and have no way to obtain that buffer: a plugin running
// inside another runtime's execution plan, or a deployment that forbids
// device allocation once it has started.  This entry point keeps that scratch
// in a fixed array compiled into the library instead.
//
// The array below lives in global memory on every GPU that loads the library
// and is held until the process exits (4 MiB per GPU).  Host code only knows
// the array's name as a host-side stand-in, so the device address is fetched
// with cudaGetSymbolAddress, with the device current, on the first call made on
// that device; make that first call before any stream capture.  The address
// is cached per device together with the id of the context it belongs to; a
// call that finds another context current (after cudaDeviceReset, which
// destroys the context and unloads the array with it) looks the address up
// again, so that call, too, should come before any capture.  Every call uses
// the same array: each call writes every row slot it reads, so no clearing is
// needed, but calls that overlap on the GPU (two streams, or two host threads)
// race on it.

#include "vce_internal.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace {

constexpr int64_t kNoAllocMaxRows = VCE_NOALLOC_MAX_ROWS;  // 1,048,576 rows = 4 MiB of FP32

static __device__ __align__(256) float g_row_loss_scratch[kNoAllocMaxRows];

struct ScratchEntry {
    void* addr = nullptr;
    unsigned long long ctx_id = 0;  // context the address belongs to (0: unknown)
};

std::mutex g_scratch_mu;
ScratchEntry g_scratch[64];

// Id of the calling thread's current context, or 0 when there is none or the
// driver cannot say (the address is then looked up on every call).
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_row_loss_scratch on the current device, cached per
// device ordinal and context.
vce_status scratch_address(int ordinal, void** out) {
    if (ordinal < 0 || ordinal >= 64) return VCE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry& e = g_scratch[ordinal];
    const unsigned long long ctx = current_context_id();
    if (!e.addr || ctx == 0 || ctx != e.ctx_id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_row_loss_scratch) != cudaSuccess || p == nullptr) return VCE_ERR_CUDA;
        e.addr = p;
        e.ctx_id = current_context_id();  // the lookup makes the device's context current if it was not
    }
    *out = e.addr;
    return VCE_OK;
}

}  // namespace

extern "C" vce_status ce_forward_noalloc(const void* logits, int dtype, int64_t n_rows,
                                         int64_t vocab, int64_t row_stride,
                                         const int64_t* target, float label_smoothing,
                                         int reduce_loss, int64_t ignore_idx, float* loss,
                                         float* stats, int64_t* n_valid, int* dev_status,
                                         void* stream) {
    if (reduce_loss && n_rows > kNoAllocMaxRows) return VCE_ERR_WORKSPACE;
    vce::DeviceInfo dev;
    if (vce_status st = vce::current_device(dev)) return st;
    void* scratch = nullptr;
    size_t scratch_bytes = 0;
    if (reduce_loss) {
        if (vce_status st = scratch_address(dev.ordinal, &scratch)) return st;
        scratch_bytes = size_t(kNoAllocMaxRows) * sizeof(float);
    }
    return ce_forward(logits, dtype, n_rows, vocab, row_stride, target, label_smoothing,
                      reduce_loss, ignore_idx, loss, stats, n_valid, scratch, scratch_bytes,
                      dev_status, stream);
}
