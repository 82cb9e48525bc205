// Linear-form cross entropy on tcgen05 tensor cores (sm_103a).
#include "vce_internal.cuh"

namespace vce {

size_t lce_forward_ws_bytes(int64_t n, int64_t v, int reduce_loss) {
    const int64_t nb = (v + 255) / 256;
    size_t b = align256(size_t(nb) * size_t(n) * 12) + align256(size_t(n) * 4);
    if (reduce_loss) b += align256(size_t(n) * 4);
    return b;
}

size_t lce_backward_ws_bytes(int64_t n, int64_t h, int64_t v, int64_t slab) {
    const int64_t ld = (slab + 7) / 8 * 8;
    size_t b = align256(size_t(n) * size_t(ld) * 2);
    if (slab < v) b += align256(size_t(n) * size_t(h) * 4);
    return b;
}

int64_t lce_slab_for_ws(int64_t n, int64_t h, int64_t v, size_t ws_bytes) {
    if (ws_bytes >= lce_backward_ws_bytes(n, h, v, v)) return v;
    const size_t acc = align256(size_t(n) * size_t(h) * 4);
    if (ws_bytes <= acc) return 0;
    const int64_t cap = int64_t((ws_bytes - acc) / (size_t(n) * 2)) / 256 * 256;
    if (cap < 256) return 0;
    return cap < v ? cap : v;
}

vce_status launch_lce_forward(const void*, const void*, int64_t, int64_t, int64_t,
                              const int64_t*, float, int, int64_t, float*, float*, int64_t*,
                              void*, int*, cudaStream_t, const DeviceInfo&) {
    return VCE_ERR_INVALID_ARG;
}

vce_status launch_lce_backward(const void*, const void*, int64_t, int64_t, int64_t,
                               const int64_t*, const float*, const int64_t*, const float*, float,
                               int, int64_t, void*, void*, void*, int64_t, int*, cudaStream_t,
                               const DeviceInfo&) {
    return VCE_ERR_INVALID_ARG;
}

}  // namespace vce
