"""CUDA-graph capture of every entry point (the API card's CUDA-graph-capturable
mode: no host synchronisation or allocation inside a call) and the bounded-wait
failure detection of the pipelined kernels, exercised without a GPU fault: the
waits run out because work is held back, never because a copy or MMA hangs."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wk
import vocabulary_cross_entropy_gb300 as vce

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from vocabulary_cross_entropy_gb300 import build
    build.build()


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def test_all_entry_points_replay_in_a_cuda_graph():
    n, v, h, vl = 300, 5003, 256, 3001
    z = _bf16(wk.normal_matrix(1, wk.TID_LOGITS, n, v, 3.0, True))
    y = torch.from_numpy(wk.uniform_targets(1, n, v, 0.1)).to(DEV)
    x = _bf16(wk.normal_matrix(1, wk.TID_X, n, h, 1.0, True))
    w = _bf16(wk.normal_matrix(1, wk.TID_W, vl, h, h ** -0.5, True))
    yl = torch.from_numpy(wk.uniform_targets(2, n, vl, 0.05)).to(DEV)
    g = torch.ones(1, device=DEV)
    # every buffer allocated up front; the graph holds only library launches
    loss, stats, nv = torch.empty(1, device=DEV), torch.empty(n, 2, device=DEV), torch.empty(1, dtype=torch.int64, device=DEV)
    ws = torch.empty(vce.ce_workspace_size(n, v, True), dtype=torch.uint8, device=DEV)
    dz = torch.empty_like(z)
    lloss, lse, lnv = torch.empty(1, device=DEV), torch.empty(n, device=DEV), torch.empty(1, dtype=torch.int64, device=DEV)
    lws = torch.empty(vce.lce_workspace_size(n, h, vl, True), dtype=torch.uint8, device=DEV)
    dx, dw = torch.empty_like(x), torch.empty_like(w)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    # ce_forward_backward on the short-row kernel (v = 5003) and on every BF16 ring
    # shape: four CTAs per SM (24 KiB rows), two with 112 KiB rings (59 KiB) and with
    # 96 KiB rings (98 KiB), one with a 224 KiB ring (137 KiB) and with a 192 KiB
    # ring (254 KiB, 4 vectors per thread; 293 KiB, 8), and rows split over a
    # cluster pair (469 KiB)
    fused = []
    for vf in (5003, 12000, 30000, 50257, 70001, 130001, 150001, 240000):
        zf = _bf16(wk.normal_matrix(7, wk.TID_LOGITS, n, vf, 3.0, True))
        yf = torch.from_numpy(wk.uniform_targets(7, n, vf, 0.1)).to(DEV)
        fused.append((zf, yf, torch.empty(1, device=DEV), torch.empty(n, 2, device=DEV),
                      torch.empty(1, dtype=torch.int64, device=DEV),
                      torch.empty(vce.ce_workspace_size(n, vf, True), dtype=torch.uint8, device=DEV),
                      torch.empty_like(zf)))

    def step():
        vce.ce_forward(z, y, 0.1, True, loss=loss, stats=stats, n_valid=nv, workspace=ws, dev_status=status)
        vce.ce_backward(z, y, stats, nv, g, 0.1, True, dlogits=dz, dev_status=status)
        vce.lce_forward(x, w, yl, 0.0, True, loss=lloss, lse=lse, n_valid=lnv, workspace=lws, dev_status=status)
        vce.lce_backward(x, w, yl, lse, lnv, g, 0.0, True, dX=dx, dW=dw, workspace=lws, dev_status=status)
        for zf, yf, fl, fs, fn, fw, fd in fused:
            vce.ce_forward_backward(zf, yf, g, 0.1, True, dlogits=fd, loss=fl, stats=fs, n_valid=fn,
                                    workspace=fw, dev_status=status)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # eager run first: per-kernel attributes are set outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    outs = [loss, stats, dz, lloss, lse, dx, dw] + [t for f in fused for t in (f[2], f[3], f[6])]
    eager = [t.clone() for t in outs]
    for t in outs:
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)
    assert int(status.item()) == 0


def test_concurrent_streams_match_sequential():
    # Two linear-form forward + backward calls with separate workspaces on two
    # streams at once: each GEMM takes its work units from the counter in its own
    # workspace, so the results equal those of running the calls one after another.
    n, h, v = 2048, 512, 9000
    cases = []
    for seed in (5, 6):
        x = _bf16(wk.normal_matrix(seed, wk.TID_X, n, h, 1.0, True))
        w = _bf16(wk.normal_matrix(seed, wk.TID_W, v, h, h ** -0.5, True))
        y = torch.from_numpy(wk.uniform_targets(seed, n, v, 0.05)).to(DEV)
        cases.append((x, w, y))
    g = torch.ones(1, device=DEV)

    def run(stream, x, w, y):
        with torch.cuda.stream(stream):
            ws = torch.empty(vce.lce_workspace_size(n, h, v, True, 8 << 20), dtype=torch.uint8, device=DEV)
            f = vce.lce_forward(x, w, y, 0.1, True, workspace=ws)
            b = vce.lce_backward(x, w, y, f.lse, f.n_valid, g, 0.1, True, workspace=ws)
        return f, b

    main = torch.cuda.current_stream()
    seq = [run(main, *c) for c in cases]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for st in streams:
        st.wait_stream(main)
    for _ in range(3):
        par = [run(st, *c) for st, c in zip(streams, cases)]
        torch.cuda.synchronize()
        for (fs, bs), (fp, bp) in zip(seq, par):
            assert torch.equal(fs.loss, fp.loss) and torch.equal(fs.lse, fp.lse)
            assert torch.equal(bs.dX.view(torch.int16), bp.dX.view(torch.int16))
            assert torch.equal(bs.dW.view(torch.int16), bp.dW.view(torch.int16))
            assert int(fp.dev_status.item()) == 0 and int(bp.dev_status.item()) == 0


@pytest.mark.parametrize("timeout_ns", [1000, 2_000_000])
def test_bounded_wait_times_out_and_reports(timeout_ns):
    lib = vce.library()
    f = lib.vce_selftest_wait_timeout
    f.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    waited = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = f(timeout_ns, ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(waited.data_ptr()),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert int(status.item()) == vce.DEVSTATUS_TIMEOUT
    assert timeout_ns <= int(waited.item()) < timeout_ns + 1_000_000_000
    # the context is still usable afterwards
    a = torch.arange(10, device=DEV)
    assert int(a.sum().item()) == 45


def _f64(t):
    return oracle.widen(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), "bf16")


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def test_gemm_timeout_exit_then_normal_call():
    # The forward GEMM with its scheduler holding back every work unit: the MMA
    # issuer, the epilogue warps and the odd CTA's producer each give up on their
    # first wait for a unit after 1 ms, with no copy or MMA issued; the kernel
    # takes its timeout exit (drain, tensor memory released) and reports it.
    n, h, v = 700, 256, 3001
    x = wk.normal_matrix(11, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(11, wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(11, n, v, 0.05)
    xt, wt, yt = _bf16(x), _bf16(w), torch.from_numpy(y).to(DEV)
    for _ in range(2):
        status = vce.selftest_lce_forward_timeout(xt, wt, yt, 1_000_000)
        torch.cuda.synchronize()
        assert int(status.item()) == vce.DEVSTATUS_TIMEOUT
    # the context and every SM's tensor memory are usable again: a normal
    # forward + backward on the same device matches the oracle
    f = vce.lce_forward(xt, wt, yt, 0.1, True)
    b = vce.lce_backward(xt, wt, yt, f.lse, f.n_valid, torch.ones(1, device=DEV), 0.1, True)
    torch.cuda.synchronize()
    assert int(f.dev_status.item()) == 0 and int(b.dev_status.item()) == 0
    ref = oracle.lce_forward(x, w, y, 0.1, True)
    dx, dw, _ = oracle.lce_backward(x, w, y, ref["lse"], ref["n_valid"], [1.0], 0.1, True, z=ref["z"])
    assert abs(f.loss.item() - ref["loss"]) <= 2e-3
    assert np.max(np.abs(f.lse.double().cpu().numpy() - ref["lse"])) <= 2e-3
    assert _rel(_f64(b.dX), dx) <= 1e-2 and _rel(_f64(b.dW), dw) <= 1e-2


# every ring shape: BF16 four CTAs per SM (24 KiB rows), two with 112 KiB rings (59
# KiB) and with 96 KiB rings (98 KiB), one with a 224 KiB ring (137 KiB) and with a
# 192 KiB ring (254 KiB, 4 vectors per thread; 293 KiB, 8); FP32 two CTAs per SM
# with 96 KiB rings (23 KiB rows) and one with a 192 KiB ring (117 KiB, 4 vectors
# per thread; 234 KiB, 8); rows split over a cluster pair (BF16 469 KiB)
@pytest.mark.parametrize("dtype,vocab", [("bf16", 12000), ("bf16", 30000), ("bf16", 50257), ("bf16", 70001),
                                         ("bf16", 130001), ("bf16", 150001), ("f32", 6000), ("f32", 30000),
                                         ("f32", 60001), ("bf16", 240000)])
def test_ring_timeout_exit_then_normal_call(dtype, vocab):
    # The fused ring kernel with its producer issuing no copy: the compute warps'
    # first wait for a chunk runs out after 1 ms with nothing in flight, the
    # CTA's roles stop and the timeout is reported.
    n = 400
    z = wk.normal_matrix(13, wk.TID_LOGITS, n, vocab, 3.0, dtype == "bf16")
    y = wk.uniform_targets(13, n, vocab, 0.1)
    g = wk.grad_rows(13, n)
    zt = _bf16(z) if dtype == "bf16" else torch.from_numpy(z).to(DEV)
    yt, gt = torch.from_numpy(y).to(DEV), torch.from_numpy(g).to(DEV)
    status = vce.selftest_ce_fused_timeout(zt, yt, gt, 1_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) == vce.DEVSTATUS_TIMEOUT
    # then the normal fused call on the same context matches the oracle
    r = vce.ce_forward_backward(zt, yt, gt, 0.1, False)
    torch.cuda.synchronize()
    assert int(r.dev_status.item()) == 0
    ref = oracle.ce_forward(z, y, 0.1, False, dtype=dtype)
    ref_dz = oracle.ce_backward(z, y, ref["lse"], ref["n_valid"], g, 0.1, False, dtype=dtype)
    rel, ab = (1e-5, 0.0) if dtype == "f32" else (0.0, 2e-3)
    loss = r.loss.double().cpu().numpy()
    assert np.all(np.abs(loss - ref["loss_rows"]) <= ab + rel * np.maximum(np.abs(ref["loss_rows"]), 1.0))
    got = (oracle.widen(r.dlogits.view(torch.int16).cpu().numpy().view(np.uint16), "bf16") if dtype == "bf16"
           else r.dlogits.double().cpu().numpy())
    lim = 1e-5 if dtype == "f32" else 1e-2
    assert np.linalg.norm(got - ref_dz) <= lim * np.linalg.norm(ref_dz)


def test_timeout_selftests_reject_bad_arguments():
    x = torch.zeros(4, 16, dtype=torch.bfloat16, device=DEV)
    y = torch.zeros(4, dtype=torch.int64, device=DEV)
    with pytest.raises(vce.VceError):  # below the 1 us floor
        vce.selftest_lce_forward_timeout(x, x, y, 10)
    with pytest.raises(vce.VceError):  # 16-element rows never reach the ring kernel
        vce.selftest_ce_fused_timeout(x, y, torch.ones(4, device=DEV), 1_000_000)
