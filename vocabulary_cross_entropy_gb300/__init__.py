"""GB300-native vocabulary cross entropy: a thin Python binding over libvce.so.

The functions here carry the names of the C ABI in ``include/vce.h`` and do
argument marshalling only: torch tensors supply device memory and the current
CUDA stream, every step of the computation runs in the library's sm_103a
kernels.  There is no CPU or PyTorch fallback: if libvce.so is missing or the
device is not a GB300 the calls raise.

Build the library with ``python -m vocabulary_cross_entropy_gb300.build``.
"""
from ._binding import (  # noqa: F401
    VceError,
    BF16,
    F32,
    DEVSTATUS_BAD_TARGET,
    DEVSTATUS_TIMEOUT,
    DEVSTATUS_BOUNDS,
    DEFAULT_SLAB_BYTES,
    SLAB_UNCAPPED,
    REDUCE_NONE,
    REDUCE_MEAN,
    REDUCE_SUM,
    library,
    library_path,
    vce_status_string,
    vce_version,
    vce_kernel_launches,
    vce_bounds_check_build,
    ce_workspace_size,
    ce_forward,
    ce_forward_noalloc,
    ce_backward,
    ce_forward_backward,
    shift_targets,
    lce_workspace_size,
    lce_forward,
    lce_backward,
    selftest_lce_forward_timeout,
    selftest_ce_fused_timeout,
)
from .autograd import parallel_cross_entropy, linear_cross_entropy  # noqa: F401,E402
