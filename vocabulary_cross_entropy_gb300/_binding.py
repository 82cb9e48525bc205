"""ctypes marshalling between torch tensors and the C ABI of libvce.so."""
from __future__ import annotations

import ctypes
import os
from collections import namedtuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# VCE_LIBRARY selects another build of the library (the bounds-checking
# variant, libvce_bounds.so); by default the one built beside this file
library_path = os.environ.get("VCE_LIBRARY") or os.path.join(_HERE, "libvce.so")

BF16 = 0
F32 = 1
DEVSTATUS_BAD_TARGET = 1
DEVSTATUS_TIMEOUT = 2
DEVSTATUS_BOUNDS = 4
# max_slab_bytes: 0 selects the library's default cap (VCE_DEFAULT_SLAB_BYTES);
# SLAB_UNCAPPED lets one dZ slab cover the whole vocabulary
DEFAULT_SLAB_BYTES = 256 << 20
SLAB_UNCAPPED = (1 << 64) - 1
REDUCE_NONE, REDUCE_MEAN, REDUCE_SUM = 0, 1, 2

_c_i64 = ctypes.c_int64
_c_int = ctypes.c_int
_c_f32 = ctypes.c_float
_c_p = ctypes.c_void_p
_c_size = ctypes.c_size_t

_lib = None


class VceError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} failed: {vce_status_string(status)} ({status})")


def library() -> ctypes.CDLL:
    """Load libvce.so (raises if it has not been built: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise ImportError(f"{library_path} is missing; build it with "
                          "`python -m vocabulary_cross_entropy_gb300.build`")
    lib = ctypes.CDLL(library_path)
    lib.vce_status_string.argtypes = [_c_int]
    lib.vce_status_string.restype = ctypes.c_char_p
    lib.vce_version.argtypes = []
    lib.vce_version.restype = _c_int
    lib.vce_kernel_launches.argtypes = []
    lib.vce_kernel_launches.restype = ctypes.c_ulonglong
    lib.vce_bounds_check_build.argtypes = []
    lib.vce_bounds_check_build.restype = _c_int
    lib.ce_workspace_size.argtypes = [_c_i64, _c_i64, _c_int]
    lib.ce_workspace_size.restype = _c_size
    lib.ce_forward.argtypes = [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_p, _c_f32, _c_int, _c_i64,
                               _c_p, _c_p, _c_p, _c_p, _c_size, _c_p, _c_p]
    lib.ce_forward.restype = _c_int
    lib.ce_forward_noalloc.argtypes = [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_p, _c_f32, _c_int,
                                       _c_i64, _c_p, _c_p, _c_p, _c_p, _c_p]
    lib.ce_forward_noalloc.restype = _c_int
    lib.ce_backward.argtypes = [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_f32,
                                _c_int, _c_i64, _c_p, _c_p, _c_p]
    lib.ce_backward.restype = _c_int
    lib.ce_forward_backward.argtypes = [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_p, _c_f32, _c_int,
                                        _c_i64, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_size, _c_p, _c_p]
    lib.ce_forward_backward.restype = _c_int
    lib.shift_targets.argtypes = [_c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p]
    lib.shift_targets.restype = _c_int
    lib.lce_workspace_size.argtypes = [_c_i64, _c_i64, _c_i64, _c_int, _c_size]
    lib.lce_workspace_size.restype = _c_size
    lib.lce_forward.argtypes = [_c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_f32, _c_int, _c_i64,
                                _c_p, _c_p, _c_p, _c_p, _c_p, _c_size, _c_p, _c_p]
    lib.lce_forward.restype = _c_int
    lib.lce_backward.argtypes = [_c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_f32,
                                 _c_int, _c_i64, _c_p, _c_p, _c_p, _c_size, _c_p, _c_p]
    lib.lce_backward.restype = _c_int
    lib.vce_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _c_p, _c_p, _c_p]
    lib.vce_selftest_wait_timeout.restype = _c_int
    lib.vce_selftest_lce_forward_timeout.argtypes = [_c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_p, ctypes.c_uint64,
                                                     _c_p, _c_p, _c_p, _c_size, _c_p, _c_p]
    lib.vce_selftest_lce_forward_timeout.restype = _c_int
    lib.vce_selftest_ce_fused_timeout.argtypes = [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_p, _c_p,
                                                  ctypes.c_uint64, _c_p, _c_p, _c_p, _c_p, _c_p]
    lib.vce_selftest_ce_fused_timeout.restype = _c_int
    _lib = lib
    return lib


def vce_status_string(status: int) -> str:
    return library().vce_status_string(int(status)).decode()


def vce_version() -> int:
    return int(library().vce_version())


def vce_kernel_launches() -> int:
    """Kernels the library has launched in this process (host-side count)."""
    return int(library().vce_kernel_launches())


def vce_bounds_check_build() -> bool:
    """Whether the loaded library is the bounds-checking variant."""
    return bool(library().vce_bounds_check_build())


def _check(func: str, status: int):
    if status != 0:
        raise VceError(func, status)


def _ptr(t):
    # a plain int: the argtypes bound in library() convert it to a pointer
    return None if t is None else t.data_ptr()


# torch's raw current-stream and current-device queries: the public
# torch.cuda.current_stream() builds a Stream object on every call, which was
# most of the host time of a small call; the public forms are the fallback
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_raw_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(device, stream):
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and device.index is not None:
        return _raw_stream(device.index)
    return torch.cuda.current_stream(device).cuda_stream


def _on(device, fn, *args):
    """fn(*args) with ``device`` current (switching only when another device is)."""
    cur = _raw_device() if _raw_device is not None else torch.cuda.current_device()
    if device.index is None or device.index == cur:
        return fn(*args)
    with torch.cuda.device(device):
        return fn(*args)


def _f32_on(t, device):
    """``t`` as a contiguous FP32 tensor on ``device`` (no copy when it already is)."""
    if t.dtype is torch.float32 and t.device == device and t.is_contiguous():
        return t
    return t.to(device=device, dtype=torch.float32).contiguous()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _rows_view(logits: torch.Tensor):
    """(n_rows, vocab, row_stride) of a [..., V] tensor whose rows have one stride."""
    if logits.dim() < 1 or logits.stride(-1) != 1:
        raise ValueError("logits must be contiguous along the vocabulary dimension")
    vocab = logits.shape[-1]
    if logits.dim() == 1:
        return 1, vocab, vocab
    if logits.dim() == 2:  # the common case, read without building a view
        n = logits.shape[0]
        return n, vocab, logits.stride(0) if n > 1 else vocab
    flat = logits.view(-1, vocab) if logits.is_contiguous() else None
    if flat is None:
        try:
            flat = logits.view(-1, vocab)
        except RuntimeError:
            raise ValueError("the leading dimensions of logits must flatten to one row stride")
    return flat.shape[0], vocab, flat.stride(0) if flat.shape[0] > 1 else vocab


def _reduce(reduce_loss) -> int:
    """reduce_loss as the ABI code: False/0/'none', True/1/'mean', 2/'sum'."""
    if isinstance(reduce_loss, str):
        codes = {"none": REDUCE_NONE, "mean": REDUCE_MEAN, "sum": REDUCE_SUM}
        if reduce_loss not in codes:
            raise ValueError(f"reduce_loss must be one of {sorted(codes)}")
        return codes[reduce_loss]
    return int(reduce_loss)


def _target(target: torch.Tensor, n: int):
    if target.dtype != torch.int64 or not target.is_contiguous() or target.numel() != n:
        raise ValueError("target must be a contiguous int64 tensor with one entry per row")
    return target


CEForward = namedtuple("CEForward", "loss stats n_valid dev_status")
LCEForward = namedtuple("LCEForward", "loss lse n_valid dev_status entropy")
LCEBackward = namedtuple("LCEBackward", "dX dW dev_status")


def ce_workspace_size(n_rows: int, vocab: int, reduce_loss: bool) -> int:
    return int(library().ce_workspace_size(n_rows, vocab, _reduce(reduce_loss)))


def ce_forward(logits, target, label_smoothing=0.0, reduce_loss=False, ignore_idx=-100, *,
               loss=None, stats=None, n_valid=None, workspace=None, dev_status=None, stream=None):
    """Logits-form forward.  Returns (loss, stats [N, 2] = (max, lse), n_valid, dev_status)."""
    lib = library()
    dev = logits.device
    n, vocab, stride = _rows_view(logits)
    target = _target(target, n)
    red = _reduce(reduce_loss)
    if loss is None:
        loss = torch.empty(1 if red else n, dtype=torch.float32, device=dev)
    if stats is None:
        stats = torch.empty(n, 2, dtype=torch.float32, device=dev)
    if n_valid is None:
        n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    if workspace is None:
        ws_bytes = ce_workspace_size(n, vocab, red)
        if ws_bytes:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    st = _on(dev, lib.ce_forward, _ptr(logits), _dtype_code(logits), n, vocab, stride, _ptr(target),
             float(label_smoothing), red, int(ignore_idx), _ptr(loss), _ptr(stats), _ptr(n_valid),
             _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
             _ptr(dev_status), _stream(dev, stream))
    _check("ce_forward", st)
    return CEForward(loss if red else loss.view(logits.shape[:-1]), stats, n_valid, dev_status)


def ce_forward_noalloc(logits, target, label_smoothing=0.0, reduce_loss=False, ignore_idx=-100, *,
                       loss=None, stats=None, n_valid=None, dev_status=None, stream=None):
    """ce_forward without a workspace argument: the library's fixed scratch array holds
    the per-row losses (for callers that cannot allocate; see include/vce.h).  Outputs
    not passed in are allocated here by torch, before the call."""
    lib = library()
    dev = logits.device
    n, vocab, stride = _rows_view(logits)
    target = _target(target, n)
    if loss is None:
        loss = torch.empty(1 if _reduce(reduce_loss) else n, dtype=torch.float32, device=dev)
    if stats is None:
        stats = torch.empty(n, 2, dtype=torch.float32, device=dev)
    if n_valid is None:
        n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = _on(dev, lib.ce_forward_noalloc, _ptr(logits), _dtype_code(logits), n, vocab, stride, _ptr(target),
             float(label_smoothing), _reduce(reduce_loss), int(ignore_idx), _ptr(loss), _ptr(stats),
             _ptr(n_valid), _ptr(dev_status), _stream(dev, stream))
    _check("ce_forward_noalloc", st)
    return CEForward(loss if _reduce(reduce_loss) else loss.view(logits.shape[:-1]), stats, n_valid, dev_status)


def ce_backward(logits, target, stats, n_valid, grad_output, label_smoothing=0.0, reduce_loss=False,
                ignore_idx=-100, *, dlogits=None, inplace=False, dev_status=None, stream=None):
    """Logits-form backward: dlogits (written over ``logits`` when ``inplace``)."""
    lib = library()
    dev = logits.device
    n, vocab, stride = _rows_view(logits)
    target = _target(target, n)
    if inplace:
        dlogits = logits
    elif dlogits is None:
        dlogits = torch.empty_like(logits)
    if dlogits.stride() != logits.stride() or dlogits.dtype != logits.dtype:
        raise ValueError("dlogits must have the dtype and strides of logits")
    grad_output = _f32_on(grad_output, dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = _on(dev, lib.ce_backward, _ptr(logits), _dtype_code(logits), n, vocab, stride, _ptr(target),
             _ptr(stats), _ptr(n_valid), _ptr(grad_output), float(label_smoothing), _reduce(reduce_loss),
             int(ignore_idx), _ptr(dlogits), _ptr(dev_status), _stream(dev, stream))
    _check("ce_backward", st)
    return dlogits


CEForwardBackward = namedtuple("CEForwardBackward", "loss stats n_valid dlogits dev_status")


def ce_forward_backward(logits, target, grad_output, label_smoothing=0.0, reduce_loss=False,
                        ignore_idx=-100, *, inplace=False, dlogits=None, loss=None, stats=None,
                        n_valid=None, workspace=None, dev_status=None, stream=None):
    """Fused logits-form forward + backward (one HBM read and one write per logit).
    Returns (loss, stats, n_valid, dlogits, dev_status); dlogits is ``logits`` when ``inplace``."""
    lib = library()
    dev = logits.device
    n, vocab, stride = _rows_view(logits)
    target = _target(target, n)
    if inplace:
        dlogits = logits
    elif dlogits is None:
        dlogits = torch.empty_like(logits)
    if dlogits.stride() != logits.stride() or dlogits.dtype != logits.dtype:
        raise ValueError("dlogits must have the dtype and strides of logits")
    grad_output = _f32_on(grad_output, dev)
    red = _reduce(reduce_loss)
    if loss is None:
        loss = torch.empty(1 if red else n, dtype=torch.float32, device=dev)
    if stats is None:
        stats = torch.empty(n, 2, dtype=torch.float32, device=dev)
    if n_valid is None:
        n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    if workspace is None:
        ws_bytes = ce_workspace_size(n, vocab, red)
        if ws_bytes:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    st = _on(dev, lib.ce_forward_backward, _ptr(logits), _dtype_code(logits), n, vocab, stride, _ptr(target),
             float(label_smoothing), red, int(ignore_idx), _ptr(grad_output), _ptr(loss), _ptr(stats),
             _ptr(n_valid), _ptr(dlogits), _ptr(workspace), 0 if workspace is None else workspace.numel(),
             _ptr(dev_status), _stream(dev, stream))
    _check("ce_forward_backward", st)
    return CEForwardBackward(loss if red else loss.view(logits.shape[:-1]), stats, n_valid, dlogits, dev_status)


def shift_targets(target, seq_len, ignore_idx=-100, *, out=None, stream=None):
    """Targets for token-shifted causal LM loss: out[i] = target[i + 1], ignore_idx at the
    last position of every ``seq_len``-long sequence.  ``target`` may be [B, SQ] or flat."""
    lib = library()
    flat = target.reshape(-1)
    if flat.dtype != torch.int64 or not flat.is_contiguous():
        raise ValueError("target must be a contiguous int64 tensor")
    if out is None:
        out = torch.empty_like(flat)
    dev = flat.device
    st = _on(dev, lib.shift_targets, _ptr(flat), flat.numel(), int(seq_len), int(ignore_idx), _ptr(out),
             _stream(dev, stream))
    _check("shift_targets", st)
    return out.view(target.shape)


def _bf16_2d(t, name):
    if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D bfloat16 tensor")
    return t


def lce_workspace_size(n: int, h: int, v: int, reduce_loss: bool, max_slab_bytes: int = 0) -> int:
    return int(library().lce_workspace_size(n, h, v, _reduce(reduce_loss), int(max_slab_bytes)))


def lce_forward(X, W, target, label_smoothing=0.0, reduce_loss=False, ignore_idx=-100, *,
                loss=None, lse=None, n_valid=None, entropy=None, workspace=None, max_slab_bytes=0,
                dev_status=None, stream=None):
    """Linear-form forward.  Returns (loss, lse [N], n_valid, dev_status, entropy).

    ``entropy``: None (not computed), True (allocate [N] FP32) or an [N] FP32 tensor.

    A workspace not passed in is allocated with lce_workspace_size(..., max_slab_bytes), the
    size one workspace shared by lce_forward and lce_backward needs."""
    lib = library()
    X = _bf16_2d(X, "X")
    W = _bf16_2d(W, "W")
    n, h = X.shape
    v = W.shape[0]
    if W.shape[1] != h:
        raise ValueError("X and W must share the hidden dimension")
    dev = X.device
    target = _target(target, n)
    if loss is None:
        loss = torch.empty(1 if _reduce(reduce_loss) else n, dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty(n, dtype=torch.float32, device=dev)
    if n_valid is None:
        n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    if entropy is True:
        entropy = torch.empty(n, dtype=torch.float32, device=dev)
    elif entropy is False:
        entropy = None
    if workspace is None:
        workspace = torch.empty(max(1, lce_workspace_size(n, h, v, reduce_loss, max_slab_bytes)),
                                dtype=torch.uint8, device=dev)
    st = _on(dev, lib.lce_forward, _ptr(X), _ptr(W), n, h, v, _ptr(target), float(label_smoothing),
             _reduce(reduce_loss), int(ignore_idx), _ptr(loss), _ptr(lse), _ptr(entropy), _ptr(n_valid),
             _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(dev, stream))
    _check("lce_forward", st)
    return LCEForward(loss, lse, n_valid, dev_status, entropy)


def lce_backward(X, W, target, lse, n_valid, grad_output, label_smoothing=0.0, reduce_loss=False,
                 ignore_idx=-100, *, dX=None, dW=None, workspace=None, max_slab_bytes=0,
                 dev_status=None, stream=None):
    """Linear-form backward.  Returns (dX [N, H], dW [V, H], dev_status), both bfloat16."""
    lib = library()
    X = _bf16_2d(X, "X")
    W = _bf16_2d(W, "W")
    n, h = X.shape
    v = W.shape[0]
    dev = X.device
    target = _target(target, n)
    if dX is None:
        dX = torch.empty_like(X)
    if dW is None:
        dW = torch.empty_like(W)
    grad_output = _f32_on(grad_output, dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, lce_workspace_size(n, h, v, reduce_loss, max_slab_bytes)),
                                dtype=torch.uint8, device=dev)
    st = _on(dev, lib.lce_backward, _ptr(X), _ptr(W), n, h, v, _ptr(target), _ptr(lse), _ptr(n_valid),
             _ptr(grad_output), float(label_smoothing), _reduce(reduce_loss), int(ignore_idx), _ptr(dX),
             _ptr(dW), _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(dev, stream))
    _check("lce_backward", st)
    return LCEBackward(dX, dW, dev_status)


# ---------------------------------------------------------------------------
# failure-detection self-tests (diagnostics; see include/vce.h)
# ---------------------------------------------------------------------------

def selftest_lce_forward_timeout(X, W, target, timeout_ns, *, dev_status=None, stream=None):
    """Runs lce_forward's GEMM with its work held back so that every wait runs out after
    ``timeout_ns``; returns the device status word (VCE_DEVSTATUS_TIMEOUT expected)."""
    lib = library()
    X = _bf16_2d(X, "X")
    W = _bf16_2d(W, "W")
    n, h = X.shape
    v = W.shape[0]
    dev = X.device
    target = _target(target, n)
    loss = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, lce_workspace_size(n, h, v, REDUCE_NONE)), dtype=torch.uint8, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = _on(dev, lib.vce_selftest_lce_forward_timeout, _ptr(X), _ptr(W), n, h, v, _ptr(target),
             int(timeout_ns), _ptr(loss), _ptr(lse), _ptr(ws), ws.numel(), _ptr(dev_status), _stream(dev, stream))
    _check("vce_selftest_lce_forward_timeout", st)
    return dev_status


def selftest_ce_fused_timeout(logits, target, grad_output, timeout_ns, *, dev_status=None, stream=None):
    """Runs ce_forward_backward's ring kernel with its copies held back so that every wait
    runs out after ``timeout_ns``; returns the device status word."""
    lib = library()
    dev = logits.device
    n, vocab, stride = _rows_view(logits)
    target = _target(target, n)
    grad_output = _f32_on(grad_output, dev)
    loss = torch.empty(n, dtype=torch.float32, device=dev)
    stats = torch.empty(n, 2, dtype=torch.float32, device=dev)
    dlogits = torch.empty_like(logits)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = _on(dev, lib.vce_selftest_ce_fused_timeout, _ptr(logits), _dtype_code(logits), n, vocab, stride,
             _ptr(target), _ptr(grad_output), int(timeout_ns), _ptr(loss), _ptr(stats), _ptr(dlogits),
             _ptr(dev_status), _stream(dev, stream))
    _check("vce_selftest_ce_fused_timeout", st)
    return dev_status
