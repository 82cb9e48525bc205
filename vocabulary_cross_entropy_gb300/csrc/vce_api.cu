// The C ABI of libvce.so: argument validation, workspace carving and dispatch.
// Every host-detectable error returns before any launch; nothing here
// allocates, frees or synchronises.

#include "vce_internal.cuh"

#include <atomic>
#include <mutex>

namespace vce {

namespace {
std::atomic<unsigned long long> g_launches{0};
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

vce_status current_device(DeviceInfo& info) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return VCE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return VCE_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (cache[dev].ordinal != dev) {
            DeviceInfo d;
            d.ordinal = dev;
            int v = 0, l2 = 0;
            if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
                return VCE_ERR_CUDA;
            d.max_smem_optin = size_t(v);
            d.l2_bytes = size_t(l2);
            cache[dev] = d;
        }
        info = cache[dev];
    }
    if (info.cc_major != 10 || info.cc_minor != 3) return VCE_ERR_ARCH;
    return VCE_OK;
}

}  // namespace vce

using namespace vce;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool eps_ok(float eps) { return eps >= 0.f && eps <= 1.f; }  // false for NaN too

bool reduce_ok(int r) { return r == VCE_REDUCE_NONE || r == VCE_REDUCE_MEAN || r == VCE_REDUCE_SUM; }

size_t elem_size(int dtype) { return dtype == VCE_BF16 ? 2 : 4; }

}  // namespace

extern "C" {

const char* vce_status_string(int status) {
    switch (status) {
        case VCE_OK: return "VCE_OK";
        case VCE_ERR_INVALID_ARG: return "VCE_ERR_INVALID_ARG";
        case VCE_ERR_DTYPE: return "VCE_ERR_DTYPE";
        case VCE_ERR_ALIGN: return "VCE_ERR_ALIGN";
        case VCE_ERR_WORKSPACE: return "VCE_ERR_WORKSPACE";
        case VCE_ERR_ARCH: return "VCE_ERR_ARCH";
        case VCE_ERR_CUDA: return "VCE_ERR_CUDA";
        default: return "VCE_UNKNOWN_STATUS";
    }
}

int vce_version(void) { return 100; }

unsigned long long vce_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int vce_bounds_check_build(void) {
#ifdef VCE_BOUNDS_CHECK
    return 1;
#else
    return 0;
#endif
}

size_t ce_workspace_size(int64_t n_rows, int64_t vocab, int reduce_loss) {
    (void)vocab;
    if (!reduce_loss || n_rows <= 0) return 0;
    return align256(size_t(n_rows) * sizeof(float));
}

vce_status ce_forward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                      int64_t row_stride, const int64_t* target, float label_smoothing,
                      int reduce_loss, int64_t ignore_idx, float* loss, float* stats,
                      int64_t* n_valid, void* ws, size_t ws_bytes, int* dev_status,
                      void* stream) {
    if (dtype != VCE_BF16 && dtype != VCE_F32) return VCE_ERR_DTYPE;
    if (n_rows < 0 || vocab < 1 || row_stride < vocab || !eps_ok(label_smoothing) || !reduce_ok(reduce_loss))
        return VCE_ERR_INVALID_ARG;
    if (!loss || (n_rows > 0 && (!logits || !target || !stats))) return VCE_ERR_INVALID_ARG;
    if (reduce_loss == VCE_REDUCE_MEAN && !n_valid) return VCE_ERR_INVALID_ARG;
    if (!aligned(logits, elem_size(dtype)) || !aligned(stats, 8)) return VCE_ERR_ALIGN;
    const size_t need = ce_workspace_size(n_rows, vocab, reduce_loss);
    if (need > 0 && (!ws || ws_bytes < need)) return VCE_ERR_WORKSPACE;
    if (ws && !aligned(ws, 256)) return VCE_ERR_ALIGN;
    DeviceInfo dev;
    if (vce_status st = current_device(dev)) return st;
    return launch_ce_forward(logits, dtype, n_rows, vocab, row_stride, target, label_smoothing,
                             reduce_loss, ignore_idx, loss, stats, n_valid, ws, dev_status,
                             static_cast<cudaStream_t>(stream), dev);
}

vce_status ce_backward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                       int64_t row_stride, const int64_t* target, const float* stats,
                       const int64_t* n_valid, const float* grad_output,
                       float label_smoothing, int reduce_loss, int64_t ignore_idx,
                       void* dlogits, int* dev_status, void* stream) {
    if (dtype != VCE_BF16 && dtype != VCE_F32) return VCE_ERR_DTYPE;
    if (n_rows < 0 || vocab < 1 || row_stride < vocab || !eps_ok(label_smoothing) || !reduce_ok(reduce_loss))
        return VCE_ERR_INVALID_ARG;
    if (n_rows > 0 && (!logits || !target || !stats || !grad_output || !dlogits))
        return VCE_ERR_INVALID_ARG;
    if (n_rows > 0 && reduce_loss == VCE_REDUCE_MEAN && !n_valid) return VCE_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (!aligned(logits, es) || !aligned(dlogits, es) || !aligned(stats, 8)) return VCE_ERR_ALIGN;
    // logits and dlogits rows must share their offset within 16 bytes (vector path)
    if (((reinterpret_cast<uintptr_t>(logits) ^ reinterpret_cast<uintptr_t>(dlogits)) & 15) != 0)
        return VCE_ERR_ALIGN;
    DeviceInfo dev;
    if (vce_status st = current_device(dev)) return st;
    return launch_ce_backward(logits, dtype, n_rows, vocab, row_stride, target, stats, n_valid,
                              grad_output, label_smoothing, reduce_loss, ignore_idx, dlogits,
                              dev_status, static_cast<cudaStream_t>(stream), dev);
}

vce_status ce_forward_backward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                               int64_t row_stride, const int64_t* target, float label_smoothing,
                               int reduce_loss, int64_t ignore_idx, const float* grad_output,
                               float* loss, float* stats, int64_t* n_valid, void* dlogits, void* ws,
                               size_t ws_bytes, int* dev_status, void* stream) {
    if (dtype != VCE_BF16 && dtype != VCE_F32) return VCE_ERR_DTYPE;
    if (n_rows < 0 || vocab < 1 || row_stride < vocab || !eps_ok(label_smoothing) || !reduce_ok(reduce_loss))
        return VCE_ERR_INVALID_ARG;
    if (!loss || (n_rows > 0 && (!logits || !target || !stats || !grad_output || !dlogits)))
        return VCE_ERR_INVALID_ARG;
    if (reduce_loss == VCE_REDUCE_MEAN && !n_valid) return VCE_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (!aligned(logits, es) || !aligned(dlogits, es) || !aligned(stats, 8)) return VCE_ERR_ALIGN;
    if (((reinterpret_cast<uintptr_t>(logits) ^ reinterpret_cast<uintptr_t>(dlogits)) & 15) != 0)
        return VCE_ERR_ALIGN;
    const size_t need = ce_workspace_size(n_rows, vocab, reduce_loss);
    if (need > 0 && (!ws || ws_bytes < need)) return VCE_ERR_WORKSPACE;
    if (ws && !aligned(ws, 256)) return VCE_ERR_ALIGN;
    DeviceInfo dev;
    if (vce_status st = current_device(dev)) return st;
    return launch_ce_forward_backward(logits, dtype, n_rows, vocab, row_stride, target, label_smoothing,
                                      reduce_loss, ignore_idx, grad_output, loss, stats, n_valid, dlogits, ws,
                                      dev_status, static_cast<cudaStream_t>(stream), dev);
}

vce_status shift_targets(const int64_t* target, int64_t n, int64_t seq_len, int64_t ignore_idx,
                         int64_t* shifted, void* stream) {
    if (n < 0 || seq_len < 1 || (n > 0 && (!target || !shifted))) return VCE_ERR_INVALID_ARG;
    if (n > 0 && target == shifted) return VCE_ERR_INVALID_ARG;  // the kernel reads target[i + 1]
    DeviceInfo dev;
    if (vce_status st = current_device(dev)) return st;
    return launch_shift_targets(target, n, seq_len, ignore_idx, shifted, static_cast<cudaStream_t>(stream));
}

size_t lce_workspace_size(int64_t n, int64_t h, int64_t v, int reduce_loss,
                          size_t max_slab_bytes) {
    if (n <= 0 || h <= 0 || v <= 0) return 0;
    const size_t fwd = lce_forward_ws_bytes(n, v, reduce_loss);
    if (max_slab_bytes == 0) max_slab_bytes = VCE_DEFAULT_SLAB_BYTES;
    const int64_t cap = int64_t(max_slab_bytes / (size_t(n) * 2)) / 256 * 256;  // at most 2^63 - 1
    const int64_t slab = cap < 256 ? 256 : (cap < v ? cap : v);
    const size_t bwd = lce_backward_ws_bytes(n, h, v, slab);
    return fwd > bwd ? fwd : bwd;
}

vce_status lce_forward(const void* X, const void* W, int64_t n, int64_t h, int64_t v,
                       const int64_t* target, float label_smoothing, int reduce_loss,
                       int64_t ignore_idx, float* loss, float* lse, float* entropy,
                       int64_t* n_valid, void* ws, size_t ws_bytes, int* dev_status,
                       void* stream) {
    if (n < 0 || h < 1 || v < 1 || !eps_ok(label_smoothing) || !reduce_ok(reduce_loss)) return VCE_ERR_INVALID_ARG;
    if (!loss || (n > 0 && (!X || !W || !target || !lse))) return VCE_ERR_INVALID_ARG;
    if (reduce_loss == VCE_REDUCE_MEAN && !n_valid) return VCE_ERR_INVALID_ARG;
    if (h % 8 != 0 || !aligned(X, 16) || !aligned(W, 16)) return VCE_ERR_ALIGN;
    if (n > 0) {
        const size_t need = lce_forward_ws_bytes(n, v, reduce_loss);
        if (!ws || ws_bytes < need) return VCE_ERR_WORKSPACE;
        if (!aligned(ws, 256)) return VCE_ERR_ALIGN;
    }
    DeviceInfo dev;
    if (vce_status st = current_device(dev)) return st;
    return launch_lce_forward(X, W, n, h, v, target, label_smoothing, reduce_loss, ignore_idx,
                              loss, lse, entropy, n_valid, ws, dev_status,
                              static_cast<cudaStream_t>(stream), dev);
}

vce_status lce_backward(const void* X, const void* W, int64_t n, int64_t h, int64_t v,
                        const int64_t* target, const float* lse, const int64_t* n_valid,
                        const float* grad_output, float label_smoothing, int reduce_loss,
                        int64_t ignore_idx, void* dX, void* dW, void* ws, size_t ws_bytes,
                        int* dev_status, void* stream) {
    if (n < 0 || h < 1 || v < 1 || !eps_ok(label_smoothing) || !reduce_ok(reduce_loss)) return VCE_ERR_INVALID_ARG;
    if (!dW || (n > 0 && (!X || !W || !target || !lse || !grad_output || !dX)))
        return VCE_ERR_INVALID_ARG;
    if (n > 0 && reduce_loss == VCE_REDUCE_MEAN && !n_valid) return VCE_ERR_INVALID_ARG;
    if (h % 8 != 0 || !aligned(X, 16) || !aligned(W, 16) || !aligned(dX, 16) || !aligned(dW, 16))
        return VCE_ERR_ALIGN;
    int64_t slab = 0;
    if (n > 0) {
        slab = lce_slab_for_ws(n, h, v, ws ? ws_bytes : 0);
        if (slab <= 0) return VCE_ERR_WORKSPACE;
        if (!aligned(ws, 256)) return VCE_ERR_ALIGN;
    }
    DeviceInfo dev;
    if (vce_status st = current_device(dev)) return st;
    return launch_lce_backward(X, W, n, h, v, target, lse, n_valid, grad_output, label_smoothing,
                               reduce_loss, ignore_idx, dX, dW, ws, slab, dev_status,
                               static_cast<cudaStream_t>(stream), dev);
}

}  // extern "C"
