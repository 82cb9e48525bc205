"""ce_forward_noalloc: the logits-form forward for callers that cannot allocate
device memory (for example a plugin inside another runtime's execution plan,
which is handed only its inputs and outputs).  It keeps its per-row loss
scratch in a fixed array inside libvce.so instead of a caller workspace.

Called here through the C ABI with preallocated outputs; its results must
match ce_forward's (which takes a workspace) on two calls in a row, so the
second call runs over scratch left behind by the first.  This file is
collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wk
import vocabulary_cross_entropy_gb300 as vce

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _noalloc(lib, logits, dtype, target, eps, red, loss, stats, n_valid, status):
    n, vocab = logits.shape
    P = ctypes.c_void_p
    return lib.ce_forward_noalloc(P(logits.data_ptr()), dtype, n, vocab, logits.stride(0),
                                  P(target.data_ptr()), ctypes.c_float(eps), int(red),
                                  ctypes.c_int64(-100), P(loss.data_ptr()), P(stats.data_ptr()),
                                  P(n_valid.data_ptr()), P(status.data_ptr()),
                                  P(torch.cuda.current_stream().cuda_stream))


CASES = [
    # n, vocab, dtype, eps, std, loss tolerance (absolute)
    (3000, 50000, "bf16", 0.1, 3.0, 2e-3),
    (777, 32001, "f32", 0.0, 2.0, None),
]


def test_noalloc_matches_ce_forward_on_two_calls():
    from vocabulary_cross_entropy_gb300 import build
    build.build()
    lib = vce.library()
    for n, vocab, dtype, eps, std, tol in CASES:
        z = wk.normal_matrix(n + vocab, wk.TID_LOGITS, n, vocab, std, dtype == "bf16")
        y = wk.uniform_targets(n, n, vocab, 0.1)
        if dtype == "bf16":
            logits = torch.from_numpy(z.view(np.int16)).to(DEV).view(torch.bfloat16)
            code = vce.BF16
        else:
            logits = torch.from_numpy(z).to(DEV)
            code = vce.F32
        target = torch.from_numpy(y).to(DEV)
        ref = vce.ce_forward(logits, target, eps, True)
        loss = torch.full((1,), float("nan"), device=DEV)
        stats = torch.zeros(n, 2, device=DEV)
        n_valid = torch.zeros(1, dtype=torch.int64, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        st = _noalloc(lib, logits, code, target, eps, True, loss, stats, n_valid, status)
        torch.cuda.synchronize()
        assert st == 0, vce.vce_status_string(st)
        assert torch.cuda.memory_allocated() == before
        assert int(status.item()) == 0
        assert int(n_valid.item()) == int(ref.n_valid.item())
        a, b = loss.item(), ref.loss.item()
        limit = tol if tol is not None else 1e-5 * abs(b)
        assert abs(a - b) <= limit, (a, b)
        assert torch.allclose(stats, ref.stats, rtol=1e-6, atol=0)


def test_noalloc_rejects_rows_beyond_its_scratch():
    lib = vce.library()
    n = 1048576 + 1
    logits = torch.empty(1, 8, device=DEV)  # never read: the size check comes first
    target = torch.empty(1, dtype=torch.int64, device=DEV)
    loss = torch.empty(1, device=DEV)
    stats = torch.empty(1, 2, device=DEV)
    n_valid = torch.empty(1, dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    P = ctypes.c_void_p
    st = lib.ce_forward_noalloc(P(logits.data_ptr()), vce.F32, n, 8, 8, P(target.data_ptr()),
                                ctypes.c_float(0.0), 1, ctypes.c_int64(-100), P(loss.data_ptr()),
                                P(stats.data_ptr()), P(n_valid.data_ptr()), P(status.data_ptr()),
                                P(None))
    assert st == 4  # VCE_ERR_WORKSPACE
