"""GPU results checked against the plain-C FP64 oracle (oracle/vce_oracle.c)
instead of the NumPy one: the tiny FP32 logits workload in full, a ragged BF16
logits case, and a small linear-form case.  The two oracles are independent
restatements of the same definitions (TE card "Description"; TE PR "Changes";
CCE card "what_it_does"; Liger PR "Summary"), so a mistake shared by the NumPy
oracle and the kernels would show here."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wk
from oracle import c_oracle
import vocabulary_cross_entropy_gb300 as vce

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from vocabulary_cross_entropy_gb300 import build
    build.build()
    c_oracle.build()


def _dev(a, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _host(t, dtype):
    if dtype == "bf16":
        return oracle.widen(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
    return t.double().cpu().numpy()


@pytest.mark.parametrize("n,vocab,dtype,eps,red", [
    (128, 1024, "f32", 0.0, 0), (128, 1024, "f32", 0.1, 1),   # the tiny workload
    (64, 32001, "bf16", 0.1, 0), (40, 70001, "bf16", 0.0, 1),
])
def test_logits_form_against_c_oracle(n, vocab, dtype, eps, red):
    seed = 17 + n + vocab
    z = wk.normal_matrix(seed, wk.TID_LOGITS, n, vocab, 2.0 if dtype == "f32" else 3.0, dtype == "bf16")
    y = wk.uniform_targets(seed, n, vocab, 0.1)
    g = np.ones(1, np.float32) if red else wk.grad_rows(seed, n)
    zt, yt, gt = _dev(z, dtype), torch.from_numpy(y).to(DEV), torch.from_numpy(g).to(DEV)
    f = vce.ce_forward(zt, yt, eps, red)
    dz = vce.ce_backward(zt, yt, f.stats, f.n_valid, gt, eps, red)
    r = vce.ce_forward_backward(zt, yt, gt, eps, red)
    torch.cuda.synchronize()
    z64 = oracle.widen(z, "bf16") if dtype == "bf16" else z.astype(np.float64)
    ref = c_oracle.ce_forward(z64, y, eps)
    n_valid = ref["n_valid"]
    g_rows = np.full(n, g[0] / n_valid) if red else g.astype(np.float64)
    ref_dz = c_oracle.ce_backward(z64, y, ref["lse"], g_rows, eps)
    rel, ab = (1e-5, 0.0) if dtype == "f32" else (0.0, 2e-3)
    ok = y != -100
    for loss, stats, grad in ((f.loss, f.stats, dz), (r.loss, r.stats, r.dlogits)):
        assert int(f.n_valid.item()) == n_valid and int(r.n_valid.item()) == n_valid
        if red:
            ref_loss = ref["loss_rows"].sum() / n_valid
            assert abs(loss.item() - ref_loss) <= ab + rel * max(1.0, abs(ref_loss))
        else:
            got = loss.double().cpu().numpy()
            assert np.all(np.abs(got - ref["loss_rows"]) <= ab + rel * np.maximum(np.abs(ref["loss_rows"]), 1.0))
        st = stats.double().cpu().numpy()
        np.testing.assert_array_equal(st[ok, 0], ref["m"][ok])
        assert np.all(np.abs(st[ok, 1] - ref["lse"][ok]) <= ab + rel * np.maximum(np.abs(ref["lse"][ok]), 1.0))
        got_dz = _host(grad, dtype)
        lim = 1e-5 if dtype == "f32" else 1e-2
        assert np.all(got_dz[~ok] == 0.0)
        assert np.linalg.norm(got_dz - ref_dz) <= lim * np.linalg.norm(ref_dz)


def test_linear_form_against_c_oracle():
    n, h, v, eps = 257, 520, 2309, 0.1
    x = wk.normal_matrix(23, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(23, wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(23, n, v, 0.1)
    xt, wt, yt = _dev(x, "bf16"), _dev(w, "bf16"), torch.from_numpy(y).to(DEV)
    fw = vce.lce_forward(xt, wt, yt, eps, 1, entropy=True)
    bw = vce.lce_backward(xt, wt, yt, fw.lse, fw.n_valid, torch.ones(1, device=DEV), eps, 1)
    torch.cuda.synchronize()
    x64, w64 = oracle.widen(x, "bf16"), oracle.widen(w, "bf16")
    z = c_oracle.linear_logits(x64, w64)
    ref = c_oracle.ce_forward(z, y, eps)
    dzr = c_oracle.ce_backward(z, y, ref["lse"], np.full(n, 1.0 / ref["n_valid"]), eps)
    dx, dw = c_oracle.linear_grads(dzr, x64, w64)
    # the linear form computes the logits, lse and entropy of ignored rows too; the
    # C oracle's logits-form forward skips them, so take every row's lse from a call
    # with no row ignored
    lse_all = c_oracle.ce_forward(z, np.zeros(n, np.int64), 0.0)["lse"]
    ent = c_oracle.entropy(z, lse_all)
    assert int(fw.n_valid.item()) == ref["n_valid"]
    assert abs(fw.loss.item() - ref["loss_rows"].sum() / ref["n_valid"]) <= 2e-3
    assert np.max(np.abs(fw.lse.double().cpu().numpy() - lse_all)) <= 2e-3
    assert np.max(np.abs(fw.entropy.double().cpu().numpy() - ent)) <= 2e-3
    gx, gw = _host(bw.dX, "bf16"), _host(bw.dW, "bf16")
    assert np.linalg.norm(gx - dx) <= 1e-2 * np.linalg.norm(dx)
    assert np.linalg.norm(gw - dw) <= 1e-2 * np.linalg.norm(dw)
