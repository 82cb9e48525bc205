"""Seeded random sweep of small ragged shapes, both forms, against the FP64 oracle:
row counts that are not tile multiples, vocabularies that end mid-tile or
mid-vector, hidden sizes that end mid-K-block, every reduction, smoothing on and
off, ignored and out-of-range targets, slab caps that force several slabs."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wk
import vocabulary_cross_entropy_gb300 as vce

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
N_CASES = 24


@pytest.fixture(scope="module", autouse=True)
def _built():
    from vocabulary_cross_entropy_gb300 import build
    build.build()


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def _f64(t):
    return oracle.widen(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), "bf16")


def _rel(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / nb if nb > 0 else np.linalg.norm(a)


def _case(i):
    r = np.random.default_rng(1000 + i)
    return dict(n=int(r.integers(1, 700)), h=int(8 * r.integers(1, 80)), v=int(r.integers(1, 5000)),
                eps=float(r.choice([0.0, 0.05, 0.3])), red=int(r.integers(0, 3)),
                ign=float(r.choice([0.0, 0.1, 0.5])), slab=int(r.choice([0, 256, 512])), seed=i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_linear_random_shape(i):
    c = _case(i)
    n, h, v = c["n"], c["h"], c["v"]
    x = wk.normal_matrix(c["seed"], wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(c["seed"], wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(c["seed"], n, v, c["ign"])
    g = np.full(1, 1.25, np.float32) if c["red"] else wk.grad_rows(c["seed"], n)
    yt = torch.from_numpy(y).to(DEV)
    f = vce.lce_forward(_bf16(x), _bf16(w), yt, c["eps"], c["red"], entropy=True,
                        max_slab_bytes=n * 2 * c["slab"])
    b = vce.lce_backward(_bf16(x), _bf16(w), yt, f.lse, f.n_valid, torch.from_numpy(g).to(DEV), c["eps"],
                         c["red"], max_slab_bytes=n * 2 * c["slab"])
    torch.cuda.synchronize()
    ref = oracle.lce_forward(x, w, y, c["eps"], c["red"])
    dx, dw, _ = oracle.lce_backward(x, w, y, ref["lse"], ref["n_valid"], g, c["eps"], c["red"], z=ref["z"])
    assert int(f.n_valid.item()) == ref["n_valid"] and int(f.dev_status.item()) == 0
    assert np.max(np.abs(f.lse.double().cpu().numpy() - ref["lse"])) <= 2e-3
    assert np.max(np.abs(f.entropy.double().cpu().numpy() - ref["entropy"])) <= 2e-3
    if c["red"] == 0:
        assert np.max(np.abs(f.loss.double().cpu().numpy() - ref["loss"])) <= 2e-3
    elif ref["n_valid"] > 0:
        scale = ref["n_valid"] if c["red"] == 2 else 1
        assert abs(f.loss.item() - ref["loss"]) <= 2e-3 * scale
    gx, gw = _f64(b.dX), _f64(b.dW)
    assert np.all(gx[y == -100] == 0.0)
    assert _rel(gx, dx) <= 1e-2 and _rel(gw, dw) <= 1e-2


def test_last_slab_narrower_than_one_k_block():
    # three full 256-wide slabs and a 40-wide last one: the dX GEMM of the last
    # slab has a single K block, fewer than the K chunks the first slab set up
    n, h, v = 640, 256, 3 * 256 + 40
    x = wk.normal_matrix(5, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(5, wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(5, n, v, 0.05)
    yt = torch.from_numpy(y).to(DEV)
    f = vce.lce_forward(_bf16(x), _bf16(w), yt, 0.1, True, max_slab_bytes=n * 2 * 256)
    b = vce.lce_backward(_bf16(x), _bf16(w), yt, f.lse, f.n_valid, torch.ones(1, device=DEV), 0.1, True,
                         max_slab_bytes=n * 2 * 256)
    torch.cuda.synchronize()
    ref = oracle.lce_forward(x, w, y, 0.1, True)
    dx, dw, _ = oracle.lce_backward(x, w, y, ref["lse"], ref["n_valid"], [1.0], 0.1, True, z=ref["z"])
    assert _rel(_f64(b.dX), dx) <= 1e-2 and _rel(_f64(b.dW), dw) <= 1e-2


@pytest.mark.parametrize("i", range(N_CASES))
def test_logits_random_shape(i):
    r = np.random.default_rng(2000 + i)
    n, v = int(r.integers(1, 300)), int(r.integers(1, 70000))
    pad = int(r.integers(0, 9))
    dtype = "bf16" if r.random() < 0.6 else "f32"
    eps = float(r.choice([0.0, 0.1]))
    red = int(r.integers(0, 3))
    fused = bool(r.random() < 0.5)
    z = wk.normal_matrix(3000 + i, wk.TID_LOGITS, n, v + pad, 3.0, dtype == "bf16")
    y = wk.uniform_targets(3000 + i, n, v, 0.1)
    if n > 3:
        y[2] = v + 5  # an out-of-range target
    g = np.full(1, 0.5, np.float32) if red else wk.grad_rows(i, n)
    if dtype == "bf16":
        full = torch.from_numpy(z.view(np.int16)).to(DEV).view(torch.bfloat16)
    else:
        full = torch.from_numpy(z).to(DEV)
    logits = full[:, :v]
    dz_full = torch.zeros_like(full)
    tgt = torch.from_numpy(y).to(DEV)
    gt = torch.from_numpy(g).to(DEV)
    if fused:
        res = vce.ce_forward_backward(logits, tgt, gt, eps, red, dlogits=dz_full[:, :v])
        loss, stats, nv, status = res.loss, res.stats, res.n_valid, res.dev_status
    else:
        fw = vce.ce_forward(logits, tgt, eps, red)
        vce.ce_backward(logits, tgt, fw.stats, fw.n_valid, gt, eps, red, dlogits=dz_full[:, :v],
                        dev_status=fw.dev_status)
        loss, stats, nv, status = fw.loss, fw.stats, fw.n_valid, fw.dev_status
    torch.cuda.synchronize()
    zz = z[:, :v]
    ref = oracle.ce_forward(zz, y, eps, red, dtype=dtype)
    ref_dz = oracle.ce_backward(zz, y, ref["lse"], ref["n_valid"], g, eps, red, dtype=dtype)
    assert int(nv.item()) == ref["n_valid"]
    assert bool(int(status.item()) & vce.DEVSTATUS_BAD_TARGET) == bool(ref["bad"].any())
    ok = ~ref["bad"] & (y != -100)
    st = stats.double().cpu().numpy()
    np.testing.assert_array_equal(st[ok, 0], ref["m"][ok])
    # the stated bounds: FP32 1e-5 relative (floor of 1 nat), BF16 2e-3 absolute
    rel, ab = (1e-5, 0.0) if dtype == "f32" else (0.0, 2e-3)
    lse_err = np.abs(st[ok, 1] - ref["lse"][ok])
    assert np.all(lse_err <= ab + rel * np.maximum(np.abs(ref["lse"][ok]), 1.0)), lse_err.max()
    if red == 0:
        got = loss.double().cpu().numpy().reshape(-1)
        assert np.all(np.isnan(got[ref["bad"]]))
        good = ~ref["bad"]
        err = np.abs(got[good] - ref["loss"][good])
        assert np.all(err <= ab + rel * np.maximum(np.abs(ref["loss"][good]), 1.0)), err.max(initial=0.0)
    else:
        got = float(loss.item())
        if np.isnan(ref["loss"]):  # a bad target counted in the reduction, or N_v = 0 for the mean
            assert np.isnan(got)
        else:
            # mean: the per-row bound; sum: the per-row bound times N_v (FP32 stays relative)
            lim = rel * max(abs(ref["loss"]), 1.0) + ab * (ref["n_valid"] if red == 2 else 1)
            assert abs(got - ref["loss"]) <= lim, (got, ref["loss"])
    dzh = (oracle.widen(dz_full.view(torch.int16).cpu().numpy().view(np.uint16), "bf16") if dtype == "bf16"
           else dz_full.double().cpu().numpy())
    assert np.all(dzh[:, v:] == 0.0)  # padding untouched
    got = dzh[:, :v]
    assert np.all(got[~ok] == 0.0)
    lim = 1e-5 if dtype == "f32" else 1e-2
    assert np.linalg.norm(got - ref_dz) <= lim * np.linalg.norm(ref_dz) + 1e-6
