"""The C ABI without a GPU: libvce.so builds, loads, exports every entry point
include/vce.h declares, and rejects bad arguments on the host before touching
the device."""
import ctypes
import os
import re

import pytest

from vocabulary_cross_entropy_gb300 import build as vbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vce.h")

OK, INVALID, DTYPE, ALIGN, WORKSPACE, ARCH, CUDA = range(7)
FAKE = 0x10000  # never dereferenced: host validation fails first


@pytest.fixture(scope="module")
def lib():
    path = vbuild.build()
    lib = ctypes.CDLL(path)
    return lib


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("ce_forward", "ce_backward", "lce_forward", "lce_backward",
              "ce_workspace_size", "lce_workspace_size", "vce_status_string", "vce_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    lib.vce_status_string.restype = ctypes.c_char_p
    assert lib.vce_status_string(0) == b"VCE_OK"
    assert lib.vce_status_string(4) == b"VCE_ERR_WORKSPACE"
    assert lib.vce_status_string(99) == b"VCE_UNKNOWN_STATUS"


def _ce_forward(lib, logits=FAKE, dtype=0, n=4, v=8, stride=8, target=FAKE, eps=0.0, red=0,
                loss=FAKE, stats=FAKE, n_valid=FAKE, ws=None, ws_bytes=0):
    f = lib.ce_forward
    f.restype = ctypes.c_int
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    return f(P(logits), ctypes.c_int(dtype), I64(n), I64(v), I64(stride), P(target),
             ctypes.c_float(eps), ctypes.c_int(red), I64(-100), P(loss), P(stats), P(n_valid),
             P(ws), ctypes.c_size_t(ws_bytes), P(None), P(None))


def test_ce_forward_host_validation(lib):
    assert _ce_forward(lib, dtype=7) == DTYPE
    assert _ce_forward(lib, v=0) == INVALID
    assert _ce_forward(lib, stride=7) == INVALID
    assert _ce_forward(lib, eps=1.5) == INVALID
    assert _ce_forward(lib, eps=float("nan")) == INVALID
    assert _ce_forward(lib, logits=None) == INVALID
    assert _ce_forward(lib, red=1, n_valid=None) == INVALID
    assert _ce_forward(lib, logits=FAKE + 1) == ALIGN
    assert _ce_forward(lib, red=1) == WORKSPACE                       # needs n*4 bytes
    assert _ce_forward(lib, red=1, ws=FAKE, ws_bytes=8) == WORKSPACE
    lib.ce_workspace_size.restype = ctypes.c_size_t
    assert lib.ce_workspace_size(ctypes.c_int64(1000), ctypes.c_int64(5), 1) == 4096
    assert lib.ce_workspace_size(ctypes.c_int64(1000), ctypes.c_int64(5), 0) == 0


def test_valid_call_without_gpu_reports_cuda_or_arch(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _ce_forward(lib) in (CUDA, ARCH)


def test_lce_host_validation(lib):
    f = lib.lce_forward
    f.restype = ctypes.c_int
    P, I64 = ctypes.c_void_p, ctypes.c_int64

    def call(x=FAKE, w=FAKE, n=16, h=64, v=100, ws=FAKE, ws_bytes=1 << 30):
        return f(P(x), P(w), I64(n), I64(h), I64(v), P(FAKE), ctypes.c_float(0.0), 0, I64(-100),
                 P(FAKE), P(FAKE), P(None), P(FAKE), P(ws), ctypes.c_size_t(ws_bytes), P(None), P(None))

    assert call(h=60) == ALIGN         # h must be a multiple of 8 (16-byte TMA strides)
    assert call(x=FAKE + 8) == ALIGN
    assert call(ws=None, ws_bytes=0) == WORKSPACE
    assert call(ws_bytes=16) == WORKSPACE
    assert call(v=0) == INVALID
    lib.lce_workspace_size.restype = ctypes.c_size_t
    ws = lambda cap: lib.lce_workspace_size(I64(4096), I64(4096), I64(131072), 1, ctypes.c_size_t(cap))
    # SIZE_MAX (VCE_SLAB_UNCAPPED): one dZ slab over the whole vocabulary; 0: the
    # default 256 MiB cap; an explicit cap below it is smaller still
    full, default, capped = ws((1 << 64) - 1), ws(0), ws(64 << 20)
    assert full >= 4096 * 131072 * 2
    assert default == ws(256 << 20) and default < full and capped < default
