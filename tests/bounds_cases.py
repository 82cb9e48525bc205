"""Cases run against the bounds-checking build of the library (libvce_bounds.so,
selected with VCE_LIBRARY by tests/test_bounds_check_gpu.py in a child process).

Every entry point runs on small, ragged and padded inputs that reach each kernel
shape: the short-row, 128/256/512-thread row kernels, every ring shape of the
fused kernel (with rows off 16-byte alignment and padding between rows, in
place and not), the linear form's GEMMs with ragged M/N/K, several vocabulary
slabs and the 512-wide dX and dW tiles, the no-alloc forward and the token shift.  Each
result is checked against the FP64 oracle at the stated tolerances, and the
device status word must stay 0: no address failed a check.  Exit status 0 when
everything passes.
"""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads as wk  # noqa: E402
import vocabulary_cross_entropy_gb300 as vce  # noqa: E402

DEV = "cuda:0"


def bf16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def host64(t, dtype):
    if dtype == "bf16":
        return oracle.widen(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
    return t.double().cpu().numpy()


def check_logits(n, vocab, pad, offset, dtype, eps, red, fused, inplace):
    """Logits form on rows of ``vocab`` elements inside rows of ``vocab + pad``, the
    first ``offset`` columns skipped (rows start off 16-byte alignment)."""
    seed = n + vocab + pad
    full = wk.normal_matrix(seed, wk.TID_LOGITS, n, vocab + pad + offset, 3.0, dtype == "bf16")
    z = full[:, offset:offset + vocab]
    y = wk.uniform_targets(seed, n, vocab, 0.1)
    g = np.ones(1, np.float32) if red else wk.grad_rows(seed, n)
    dfull = bf16_dev(full) if dtype == "bf16" else torch.from_numpy(full).to(DEV)
    logits = dfull[:, offset:offset + vocab]
    yt, gt = torch.from_numpy(y).to(DEV), torch.from_numpy(g).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    if fused:
        out = dfull.clone() if not inplace else dfull
        r = vce.ce_forward_backward(logits, yt, gt, eps, red, dlogits=out[:, offset:offset + vocab],
                                    dev_status=status)
        loss, stats, dz = r.loss, r.stats, r.dlogits
    else:
        f = vce.ce_forward(logits, yt, eps, red, dev_status=status)
        out = dfull.clone() if not inplace else dfull
        dz = vce.ce_backward(logits, yt, f.stats, f.n_valid, gt, eps, red, dlogits=out[:, offset:offset + vocab],
                             dev_status=status)
        loss, stats = f.loss, f.stats
    torch.cuda.synchronize()
    assert int(status.item()) == 0, ("status", int(status.item()), n, vocab, dtype, fused)
    ref = oracle.ce_forward(z, y, eps, red, dtype=dtype)
    ref_dz = oracle.ce_backward(z, y, ref["lse"], ref["n_valid"], g, eps, red, dtype=dtype)
    rel, ab = (1e-5, 0.0) if dtype == "f32" else (0.0, 2e-3)
    if red:
        assert abs(loss.item() - ref["loss"]) <= ab * (ref["n_valid"] if red == 2 else 1) + rel * max(
            1.0, abs(ref["loss"]))
    else:
        got = loss.double().cpu().numpy().reshape(-1)
        assert np.all(np.abs(got - ref["loss_rows"]) <= ab + rel * np.maximum(np.abs(ref["loss_rows"]), 1.0))
    ok = y != -100
    assert np.all(np.abs(stats.double().cpu().numpy()[ok, 1] - ref["lse"][ok]) <= ab + rel * np.maximum(
        np.abs(ref["lse"][ok]), 1.0))
    gz = host64(dz, dtype)
    lim = 1e-5 if dtype == "f32" else 1e-2
    assert np.linalg.norm(gz - ref_dz) <= lim * np.linalg.norm(ref_dz) + 1e-6
    # the padding on both sides of every row is untouched
    whole = host64(out, dtype)
    src = oracle.widen(full, "bf16") if dtype == "bf16" else full.astype(np.float64)
    if not inplace:
        assert np.array_equal(whole[:, :offset], src[:, :offset])
        assert np.array_equal(whole[:, offset + vocab:], src[:, offset + vocab:])


def check_linear(n, h, v, eps, red, slab_ids):
    seed = n + h + v
    x = wk.normal_matrix(seed, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(seed, wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(seed, n, v, 0.05)
    g = np.ones(1, np.float32) if red else wk.grad_rows(seed, n)
    xt, wt, yt = bf16_dev(x), bf16_dev(w), torch.from_numpy(y).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    cap = n * 2 * slab_ids
    f = vce.lce_forward(xt, wt, yt, eps, red, entropy=True, max_slab_bytes=cap, dev_status=status)
    b = vce.lce_backward(xt, wt, yt, f.lse, f.n_valid, torch.from_numpy(g).to(DEV), eps, red, max_slab_bytes=cap,
                         dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, ("status", int(status.item()), n, h, v)
    ref = oracle.lce_forward(x, w, y, eps, red)
    dx, dw, _ = oracle.lce_backward(x, w, y, ref["lse"], ref["n_valid"], g, eps, red, z=ref["z"])
    assert np.max(np.abs(f.lse.double().cpu().numpy() - ref["lse"])) <= 2e-3
    assert np.max(np.abs(f.entropy.double().cpu().numpy() - ref["entropy"])) <= 2e-3
    gx, gw = host64(b.dX, "bf16"), host64(b.dW, "bf16")
    assert np.linalg.norm(gx - dx) <= 1e-2 * np.linalg.norm(dx)
    assert np.linalg.norm(gw - dw) <= 1e-2 * np.linalg.norm(dw)


def main():
    assert vce.vce_bounds_check_build(), "VCE_LIBRARY does not point at the bounds-checking build"
    logits_cases = [
        # n, vocab, pad, offset, dtype, eps, reduce, fused, in place
        (5, 7, 3, 1, "bf16", 0.1, 1, False, False),        # shorter than one vector
        (64, 1000, 5, 3, "f32", 0.0, 0, False, False),     # 128-thread forward, misaligned rows
        (33, 32001, 7, 1, "bf16", 0.1, 2, False, True),    # 256/512-thread forward, in place
        (40, 5003, 2, 5, "bf16", 0.1, 1, True, False),     # fused, short rows
        (300, 12000, 1, 1, "bf16", 0.0, 0, True, False),   # fused ring: four CTAs per SM
        (300, 40000, 9, 3, "bf16", 0.1, 1, True, True),    # two CTAs per SM, 112 KiB rings, in place
        (100, 52001, 2, 1, "bf16", 0.1, 1, True, False),   # two CTAs per SM, 96 KiB rings
        (200, 70001, 4, 2, "bf16", 0.1, 2, True, False),   # one CTA per SM, 224 KiB ring
        (40, 130001, 5, 3, "bf16", 0.1, 1, True, False),   # one CTA per SM, 192 KiB ring, 4 vectors per thread
        (60, 150001, 3, 1, "bf16", 0.0, 0, True, True),    # 192 KiB ring, 8 vectors per thread, in place
        (50, 9001, 3, 1, "f32", 0.1, 1, True, False),      # FP32, two CTAs per SM, 96 KiB rings
        (20, 50257, 3, 1, "f32", 0.0, 0, True, False),     # FP32, 192 KiB ring
        (40, 210000, 8, 7, "bf16", 0.1, 1, True, False),   # 192 KiB ring, 8 vectors per thread, 410 KiB rows
        (40, 240000, 8, 7, "bf16", 0.1, 1, True, False),   # rows split over a cluster pair
    ]
    for c in logits_cases:
        check_logits(*c)
    linear_cases = [
        # n, h, v, eps, reduce, slab ids (0: one slab)
        (5, 8, 40, 0.1, 0, 0),
        (129, 72, 300, 0.1, 1, 0),
        (384, 256, 1800, 0.1, 1, 256),     # several slabs, FP32 dX across them
        (300, 1032, 70000, 0.0, 2, 0),     # 512-wide dX tile, ragged H
        (8200, 1032, 600, 0.1, 1, 0),      # 512-wide dW tile (8192 tokens or more), ragged M, N and K
    ]
    for c in linear_cases:
        check_linear(*c)
    # the allocation-free forward and the token shift
    z = wk.normal_matrix(9, wk.TID_LOGITS, 77, 3001, 3.0, True)
    y = wk.uniform_targets(9, 77, 3001, 0.1)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    f = vce.ce_forward_noalloc(bf16_dev(z), torch.from_numpy(y).to(DEV), 0.1, True, dev_status=st)
    sh = vce.shift_targets(torch.from_numpy(y).to(DEV), 10)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert abs(f.loss.item() - oracle.ce_forward(z, y, 0.1, True, dtype="bf16")["loss"]) <= 2e-3
    assert np.array_equal(sh.cpu().numpy(), oracle.shift_targets(y, 10))
    print("bounds cases ok", flush=True)


if __name__ == "__main__":
    main()
