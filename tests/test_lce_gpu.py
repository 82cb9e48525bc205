"""Linear form on the GPU against the FP64 oracle (Cut Cross-Entropy /
Liger fused linear cross entropy semantics).  Tolerances (BF16 inputs, FP32
accumulation, BF16 gradients):

* loss and lse: |d| <= 2e-3 per row and for the mean;
* dX, dW: norm-wise ||d|| / ||ref|| <= 1e-2;
* N_v and the zero rows of ignored tokens in dX: bit-exact.
"""
import math

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


def dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def host_f64(t):
    return oracle.widen(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), "bf16")


def rel(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / nb if nb > 0 else np.linalg.norm(a)


def run(x, w, target, eps, red, grad, max_slab_bytes=0, entropy=True):
    xt, wt = dev_bf16(x), dev_bf16(w)
    yt = torch.from_numpy(target).to(DEV)
    f = vce.lce_forward(xt, wt, yt, eps, red, entropy=entropy)
    g = torch.from_numpy(np.asarray(grad, np.float32)).to(DEV)
    b = vce.lce_backward(xt, wt, yt, f.lse, f.n_valid, g, eps, red, max_slab_bytes=max_slab_bytes)
    torch.cuda.synchronize()
    return f, b


def check_full(x, w, target, eps, red, grad, max_slab_bytes=0):
    f, b = run(x, w, target, eps, red, grad, max_slab_bytes)
    ref = oracle.lce_forward(x, w, target, eps, red)
    dx, dw, _ = oracle.lce_backward(x, w, target, ref["lse"], ref["n_valid"], grad, eps, red, z=ref["z"])
    assert int(f.dev_status.item()) == 0 and int(b.dev_status.item()) == 0
    assert int(f.n_valid.item()) == ref["n_valid"]
    lse = f.lse.double().cpu().numpy()
    assert np.max(np.abs(lse - ref["lse"])) <= 2e-3
    ent = f.entropy.double().cpu().numpy()
    assert np.max(np.abs(ent - ref["entropy"])) <= 2e-3
    if red == 2:
        # a sum over N rows: 2e-3 per row
        assert abs(f.loss.item() - ref["loss"]) <= 2e-3 * max(1, ref["n_valid"]), (f.loss.item(), ref["loss"])
    elif red:
        assert abs(f.loss.item() - ref["loss"]) <= 2e-3, (f.loss.item(), ref["loss"])
    else:
        assert np.max(np.abs(f.loss.double().cpu().numpy() - ref["loss"])) <= 2e-3
    gx, gw = host_f64(b.dX), host_f64(b.dW)
    ign = target == -100
    assert np.all(gx[ign] == 0.0)
    assert rel(gx, dx) <= 1e-2, rel(gx, dx)
    assert rel(gw, dw) <= 1e-2, rel(gw, dw)


SMALL = [
    # n, h, v, eps, reduce, ignore fraction
    (200, 128, 1000, 0.0, True, 0.05),
    (1, 64, 7, 0.1, False, 0.0),
    (129, 72, 300, 0.1, True, 0.1),
    (300, 256, 513, 0.0, False, 0.02),
    (257, 520, 2309, 0.1, True, 0.1),
    (1000, 512, 4099, 0.0, True, 0.0),
    (333, 128, 3000, 0.1, 2, 0.1),     # reduction='sum'
    (5, 8, 40, 0.1, False, 0.0),        # the smallest hidden size (one 16-byte row)
]


@pytest.mark.parametrize("n,h,v,eps,red,ign", SMALL)
def test_small_shapes_full(n, h, v, eps, red, ign):
    seed = n + h + v
    x = wk.normal_matrix(seed, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(seed, wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(seed, n, v, ign)
    g = np.full(1, 0.75, np.float32) if red else wk.grad_rows(seed, n)
    check_full(x, w, y, eps, red, g)


@pytest.mark.parametrize("slab_rows", [256, 512])
def test_vocab_slabs_accumulate_dx(slab_rows):
    # a workspace cap that forces several vocabulary slabs (FP32 dX accumulation)
    n, h, v = 384, 256, 1800
    x = wk.normal_matrix(11, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(11, wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(11, n, v, 0.05)
    check_full(x, w, y, 0.1, True, np.ones(1, np.float32), max_slab_bytes=n * 2 * slab_rows)


@pytest.mark.parametrize("n,h,v,slab_ids", [
    # dX on 256 x 512 pair tiles (H >= 1024 and K chunks of at least 16384 ids):
    (700, 1032, 70000, 0),        # a hidden size that ends 8 columns into its last 512-wide tile
    (512, 1024, 100000, 65536),   # two slabs, the second narrower, FP32 dX summed across them
])
def test_dx_wide_tiles(n, h, v, slab_ids):
    x = wk.normal_matrix(31, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(31, wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(31, n, v, 0.05)
    check_full(x, w, y, 0.1, True, np.ones(1, np.float32), max_slab_bytes=n * 2 * slab_ids)


@pytest.mark.parametrize("n,h,v,slab_ids", [
    (8200, 1032, 600, 0),         # 512-wide dW tiles (8192 tokens or more); ragged M, N and K
    (8192, 1024, 1800, 512),      # several slabs, each with its own wide dW launch
])
def test_dw_wide_tiles(n, h, v, slab_ids):
    x = wk.normal_matrix(37, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(37, wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(37, n, v, 0.05)
    check_full(x, w, y, 0.1, True, np.ones(1, np.float32), max_slab_bytes=n * 2 * slab_ids)


def test_token_wave_boundaries():
    # 4097- and 5000-token shapes (one token past a 4K wave; a two-wave tail)
    for n in (4097, 5000):
        h, v = 128, 700
        x = wk.normal_matrix(n, wk.TID_X, n, h, 1.0, True)
        w = wk.normal_matrix(n, wk.TID_W, v, h, h ** -0.5, True)
        y = wk.uniform_targets(n, n, v, 0.02)
        check_full(x, w, y, 0.0, True, np.ones(1, np.float32))


def test_many_short_units_repeatable():
    # H = 64: every forward work unit is a single K block, so each CTA pair takes
    # about 27 units from the in-order ticket counter in quick succession, and
    # the per-launch counter reset is exercised by three calls in a row; the
    # results must not depend on which pair computed which tile.
    n, h, v = 4096, 64, 32768
    x = wk.normal_matrix(21, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(21, wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(21, n, v, 0.05)
    g = np.ones(1, np.float32)
    runs = [run(x, w, y, 0.1, True, g) for _ in range(3)]
    for f, b in runs[1:]:
        assert torch.equal(f.lse, runs[0][0].lse) and torch.equal(f.loss, runs[0][0].loss)
        assert torch.equal(b.dX.view(torch.int16), runs[0][1].dX.view(torch.int16))
        assert torch.equal(b.dW.view(torch.int16), runs[0][1].dW.view(torch.int16))
    check_full(x, w, y, 0.1, True, g)


def test_bad_target_status():
    n, h, v = 64, 64, 300
    x = wk.normal_matrix(1, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(1, wk.TID_W, v, h, 0.125, True)
    y = wk.uniform_targets(1, n, v, 0.0)
    y[5] = v
    f, b = run(x, w, y, 0.0, False, np.ones(n, np.float32))
    assert int(f.dev_status.item()) & vce.DEVSTATUS_BAD_TARGET
    loss = f.loss.cpu().numpy()
    assert math.isnan(loss[5]) and np.isfinite(np.delete(loss, 5)).all()
    assert torch.count_nonzero(b.dX[5]).item() == 0


def test_all_ignored():
    n, h, v = 50, 64, 333
    x = wk.normal_matrix(2, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(2, wk.TID_W, v, h, 0.125, True)
    y = np.full(n, -100, np.int64)
    f, b = run(x, w, y, 0.1, True, np.ones(1, np.float32))
    assert int(f.n_valid.item()) == 0 and math.isnan(f.loss.item())
    assert torch.count_nonzero(b.dX).item() == 0 and torch.count_nonzero(b.dW).item() == 0


def test_zero_tokens():
    h, v = 64, 300
    x = torch.empty(0, h, dtype=torch.bfloat16, device=DEV)
    w = dev_bf16(wk.normal_matrix(3, wk.TID_W, v, h, 0.125, True))
    y = torch.empty(0, dtype=torch.int64, device=DEV)
    f = vce.lce_forward(x, w, y, 0.0, True)
    dW = torch.full_like(w, 3.0)
    b = vce.lce_backward(x, w, y, f.lse, f.n_valid, torch.ones(1, device=DEV), 0.0, True, dW=dW)
    torch.cuda.synchronize()
    assert int(f.n_valid.item()) == 0 and math.isnan(f.loss.item())
    assert b.dX.shape == (0, h) and torch.count_nonzero(b.dW).item() == 0


def test_small_linear_workload_full():
    wl = wk.LINEAR_SMALL
    inp = wk.make_linear_inputs(wl)
    check_full(inp.x, inp.w, inp.target, wl.label_smoothing, wl.reduce_loss, inp.grad)


# ---------------------------------------------------------------------------
# full-size workloads, run as the benchmark runs them; sampled rows against
# the oracle (dW rows need the oracle's lse of every token: one FP64 forward)
# ---------------------------------------------------------------------------

def _sampled_check(wl, inp, f, b, entropy):
    assert int(f.dev_status.item()) == 0 and int(b.dev_status.item()) == 0
    n_valid = int((inp.target != -100).sum())
    assert int(f.n_valid.item()) == n_valid
    lse_all, loss_all, ent_all = oracle.lce_lse_all(inp.x, inp.w, inp.target, wl.label_smoothing,
                                                    entropy=entropy)
    lse_gpu = f.lse.double().cpu().numpy()
    assert np.max(np.abs(lse_gpu - lse_all)) <= 2e-3
    if entropy:
        assert np.max(np.abs(f.entropy.double().cpu().numpy() - ent_all)) <= 2e-3
    assert abs(f.loss.item() - oracle.reduce(loss_all, n_valid, wl.reduce_loss)) <= 2e-3
    g_all = oracle.upstream(inp.grad, wl.n, n_valid, wl.reduce_loss)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(wl.n, min(wl.n, 24), replace=False), [0, wl.n - 1]]))
    dx_ref = oracle.lce_dx_rows(inp.x[rows], inp.w, inp.target[rows], lse_all[rows], g_all[rows],
                                wl.label_smoothing)
    gx = host_f64(b.dX[torch.from_numpy(rows).to(DEV)])
    assert rel(gx, dx_ref) <= 1e-2, rel(gx, dx_ref)
    ign = np.nonzero(inp.target == -100)[0]
    if len(ign):
        assert torch.count_nonzero(b.dX[torch.from_numpy(ign).to(DEV)]).item() == 0
    vids = np.unique(np.concatenate([rng.choice(wl.vocab, 24, replace=False), [0, wl.vocab - 1],
                                     inp.target[:4][inp.target[:4] >= 0]]))
    dw_ref = oracle.lce_dw_rows(inp.x, inp.w, vids, inp.target, lse_all, g_all, wl.label_smoothing)
    gw = host_f64(b.dW[torch.from_numpy(vids).to(DEV)])
    assert rel(gw, dw_ref) <= 1e-2, rel(gw, dw_ref)


# production classifier shapes (H, V) of the model-shape sweep, at 512 tokens so the
# oracle's FP64 forward over every token stays short; V = 151936 ends in a half tile
@pytest.mark.parametrize("shape", wk.MODEL_SHAPES, ids=lambda w: w.name)
def test_model_shapes_sampled(shape):
    import dataclasses
    wl = dataclasses.replace(shape, n=512, name=shape.name + "_512tok", ignore_frac=0.05,
                             label_smoothing=0.1)
    inp = wk.make_linear_inputs(wl)
    f, b = run(inp.x, inp.w, inp.target, wl.label_smoothing, wl.reduce_loss, inp.grad, 0, True)
    _sampled_check(wl, inp, f, b, True)


# the benchmark's launch configurations: the headline in one vocabulary slab, the
# large workload with its dZ slab capped at 1 GiB (4 slabs, FP32 dX accumulation)
@pytest.mark.parametrize("wl,slab_cap,entropy", [(wk.LINEAR_HEADLINE, 0, False),
                                                 (wk.LINEAR_LARGE, 1 << 30, True)],
                         ids=["headline", "large_slab1GiB_entropy"])
def test_full_size_sampled(wl, slab_cap, entropy):
    inp = wk.make_linear_inputs(wl)
    f, b = run(inp.x, inp.w, inp.target, wl.label_smoothing, wl.reduce_loss, inp.grad, slab_cap, entropy)
    _sampled_check(wl, inp, f, b, entropy)


def test_dz_slab_beyond_2_31_elements_sampled():
    # One uncapped dZ slab of 16384 x 131080 (the leading dimension of V = 131073
    # rounded up to 8): 2.1476e9 elements, past 2^31, so the dZ epilogue's stores,
    # the tensor maps over dZ and the dX/dW reads of it need 64-bit offsets.
    # H = 1024 keeps the oracle's FP64 forward to 4.4e12 flop; the wide dX tile runs.
    wl = wk.LinearWorkload("linear_16384x1024x131073", 16384, 1024, 131073, ignore_frac=0.02,
                           label_smoothing=0.1, reduce_loss=True)
    assert wl.n * ((wl.vocab + 7) // 8 * 8) > 2 ** 31
    inp = wk.make_linear_inputs(wl)
    f, b = run(inp.x, inp.w, inp.target, wl.label_smoothing, wl.reduce_loss, inp.grad, vce.SLAB_UNCAPPED, False)
    _sampled_check(wl, inp, f, b, False)


def test_token_shifted_causal_lm_loss():
    # (B, SQ) = (3, 100) sequences: shifted targets from the library, losses and
    # gradients against the oracle's own shift of the same targets
    b, sq, h, v = 3, 100, 128, 1000
    n = b * sq
    x = wk.normal_matrix(21, wk.TID_X, n, h, 1.0, True)
    w = wk.normal_matrix(21, wk.TID_W, v, h, h ** -0.5, True)
    y = wk.uniform_targets(21, n, v, 0.05)
    yt = torch.from_numpy(y).to(DEV).view(b, sq)
    shifted = vce.shift_targets(yt, sq)
    torch.cuda.synchronize()
    ref_shift = oracle.shift_targets(y, sq)
    assert np.array_equal(shifted.reshape(-1).cpu().numpy(), ref_shift)
    check_full(x, w, ref_shift, 0.1, True, np.ones(1, np.float32))
