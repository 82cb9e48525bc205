"""The autograd front ends: losses and gradients through torch.autograd equal the
direct C-ABI calls, and match the FP64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wk
import vocabulary_cross_entropy_gb300 as vce

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def _f64(t):
    return oracle.widen(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), "bf16")


@pytest.mark.parametrize("reduce_loss", [True, False])
@pytest.mark.parametrize("overwrite", [False, True])
def test_parallel_cross_entropy_autograd(reduce_loss, overwrite):
    b, sq, v = 2, 64, 3001
    z = wk.normal_matrix(8, wk.TID_LOGITS, b * sq, v, 2.0, True)
    y = wk.uniform_targets(8, b * sq, v, 0.1)
    inp = _bf16(z).view(b, sq, v).requires_grad_(True)
    tgt = torch.from_numpy(y).to(DEV).view(b, sq)
    loss = vce.parallel_cross_entropy(inp, tgt, 0.1, reduce_loss, ignore_idx=-100, overwrite_input=overwrite)
    g = torch.full((), 1.5, device=DEV) if reduce_loss else torch.from_numpy(wk.grad_rows(8, b * sq)).to(DEV).view(b, sq)
    loss.backward(g)
    torch.cuda.synchronize()
    ref = oracle.ce_forward(z, y, 0.1, reduce_loss, dtype="bf16")
    gnp = np.array([1.5]) if reduce_loss else wk.grad_rows(8, b * sq)
    ref_dz = oracle.ce_backward(z, y, ref["lse"], ref["n_valid"], gnp, 0.1, reduce_loss, dtype="bf16")
    if reduce_loss:
        assert loss.shape == () or loss.numel() == 1
        assert abs(loss.item() - ref["loss"]) <= 2e-3
    else:
        assert loss.shape == (b, sq)
        assert np.max(np.abs(loss.detach().double().cpu().numpy().reshape(-1) - ref["loss"])) <= 2e-3
    got = _f64(inp.grad.reshape(-1, v))
    assert np.linalg.norm(got - ref_dz) <= 1e-2 * np.linalg.norm(ref_dz)


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_linear_cross_entropy_autograd(reduction):
    b, sq, h, v = 2, 150, 256, 2000
    x = wk.normal_matrix(9, wk.TID_X, b * sq, h, 1.0, True)
    w = wk.normal_matrix(9, wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(9, b * sq, v, 0.05)
    xt = _bf16(x).view(b, sq, h).requires_grad_(True)
    wt = _bf16(w).requires_grad_(True)
    yt = torch.from_numpy(y).to(DEV).view(b, sq)
    loss, ent = vce.linear_cross_entropy(xt, wt, yt, reduction=reduction, label_smoothing=0.05, shift=True,
                                         return_entropy=True)
    (loss.sum() if reduction == "none" else loss).backward()
    torch.cuda.synchronize()
    ys = oracle.shift_targets(y, sq)
    red = {"none": 0, "mean": 1, "sum": 2}[reduction]
    ref = oracle.lce_forward(x, w, ys, 0.05, red)
    g = np.ones(b * sq) if red == 0 else np.ones(1)
    dx, dw, _ = oracle.lce_backward(x, w, ys, ref["lse"], ref["n_valid"], g, 0.05, red, z=ref["z"])
    if red == 0:
        assert loss.shape == (b, sq)
        assert np.max(np.abs(loss.detach().double().cpu().numpy().reshape(-1) - ref["loss"])) <= 2e-3
    else:
        assert abs(loss.item() - ref["loss"]) <= 2e-3 * (ref["n_valid"] if red == 2 else 1)
    assert ent.shape == (b, sq)
    assert np.max(np.abs(ent.double().cpu().numpy().reshape(-1) - ref["entropy"])) <= 2e-3
    gx, gw = _f64(xt.grad.reshape(-1, h)), _f64(wt.grad)
    assert np.linalg.norm(gx - dx) <= 1e-2 * np.linalg.norm(dx)
    assert np.linalg.norm(gw - dw) <= 1e-2 * np.linalg.norm(dw)
