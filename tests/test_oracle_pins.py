"""Pins for the FP64 oracle: closed forms, worked examples, brute force, finite
differences and torch's float64 CPU cross entropy.  No GPU is needed.

Each test fixes something the definitions of the pages determine (Transformer
Engine parallel_cross_entropy API card and pull request #3273 for the logits
form; the Cut Cross-Entropy card and the Liger SM100 pull request for the
linear form), chosen so that a dropped term, a wrong sign, a wrong index or a
transposed operand anywhere in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
rng = np.random.default_rng(1234)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("vocab", [1, 2, 7, 1000])
@pytest.mark.parametrize("eps", [0.0, 0.1, 0.5])
@pytest.mark.parametrize("c", [-3.0, 0.0, 5.5])
def test_uniform_logits_give_log_v(vocab, eps, c):
    n = 6
    z = np.full((n, vocab), c)
    y = rng.integers(0, vocab, n)
    out = oracle.ce_forward(z, y, eps)
    np.testing.assert_allclose(out["loss"], math.log(vocab), rtol=0, atol=1e-13)
    np.testing.assert_allclose(out["lse"], c + math.log(vocab), rtol=0, atol=1e-13)
    np.testing.assert_array_equal(out["m"], np.full(n, c))
    g = rng.standard_normal(n)
    dz = oracle.ce_backward(z, y, out["lse"], out["n_valid"], g, eps)
    expect = np.repeat(g[:, None], vocab, 1) * (1.0 / vocab - eps / vocab)
    expect[np.arange(n), y] -= g * (1.0 - eps)
    np.testing.assert_allclose(dz, expect, rtol=0, atol=1e-14)


def test_single_class_vocab_gives_zero():
    z = rng.standard_normal((5, 1)) * 10
    y = np.zeros(5, np.int64)
    for eps in (0.0, 0.3):
        out = oracle.ce_forward(z, y, eps)
        np.testing.assert_allclose(out["loss"], 0.0, atol=1e-14)
        dz = oracle.ce_backward(z, y, out["lse"], out["n_valid"], np.ones(5), eps)
        np.testing.assert_allclose(dz, 0.0, atol=1e-14)


@pytest.mark.parametrize("vocab", [2, 50, 128256])
@pytest.mark.parametrize("eps", [0.0, 0.1])
def test_dominant_logit_closed_form(vocab, eps):
    # z_y = 40, every other logit 0: lse = log(e^40 + V - 1), mean z = 40 / V
    y = vocab // 3
    z = np.zeros((1, vocab))
    z[0, y] = 40.0
    out = oracle.ce_forward(z, [y], eps)
    lse = 40.0 + math.log1p((vocab - 1) * math.exp(-40.0))
    nll = math.log1p((vocab - 1) * math.exp(-40.0))
    expect = (1 - eps) * nll + eps * (lse - 40.0 / vocab)
    assert abs(out["loss"][0] - expect) <= 1e-12 * max(1.0, abs(expect))
    assert out["m"][0] == 40.0


def test_shift_invariance():
    z = rng.standard_normal((9, 33)) * 3
    y = rng.integers(0, 33, 9)
    g = rng.standard_normal(9)
    for eps in (0.0, 0.2):
        a = oracle.ce_forward(z, y, eps)
        b = oracle.ce_forward(z + 64.0, y, eps)
        np.testing.assert_allclose(a["loss"], b["loss"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(b["lse"] - a["lse"], 64.0, rtol=0, atol=1e-12)
        da = oracle.ce_backward(z, y, a["lse"], a["n_valid"], g, eps)
        db = oracle.ce_backward(z + 64.0, y, b["lse"], b["n_valid"], g, eps)
        np.testing.assert_allclose(da, db, rtol=1e-10, atol=1e-14)


def test_smoothing_equals_cross_entropy_against_smoothed_targets():
    # second way: -sum_v q_v log p_v with q = (1-eps) onehot + eps/V, log p from scipy
    from scipy.special import log_softmax
    n, vocab = 7, 29
    z = rng.standard_normal((n, vocab)) * 2
    y = rng.integers(0, vocab, n)
    for eps in (0.0, 0.1, 0.7):
        q = np.full((n, vocab), eps / vocab)
        q[np.arange(n), y] += 1 - eps
        expect = -(q * log_softmax(z, axis=1)).sum(axis=1)
        np.testing.assert_allclose(oracle.ce_forward(z, y, eps)["loss"], expect, rtol=1e-13)


def test_gradient_rows_sum_to_zero():
    n, vocab = 11, 301
    z = rng.standard_normal((n, vocab)) * 4
    y = rng.integers(0, vocab, n)
    y[3] = -100
    g = rng.standard_normal(n)
    for eps in (0.0, 0.1):
        out = oracle.ce_forward(z, y, eps)
        dz = oracle.ce_backward(z, y, out["lse"], out["n_valid"], g, eps)
        np.testing.assert_allclose(dz.sum(axis=1), 0.0, atol=1e-14)
        assert np.all(dz[3] == 0.0)


# ---------------------------------------------------------------------------
# worked examples (tests/golden)
# ---------------------------------------------------------------------------

def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_worked_examples(case):
    z = np.array(case["z"])
    y = np.array(case["target"])
    eps, red = case["label_smoothing"], case["reduce_loss"]
    out = oracle.ce_forward(z, y, eps, red)
    np.testing.assert_allclose(out["loss"], case["loss"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(out["lse"], case["lse"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(out["m"], case["m"], rtol=0, atol=0)
    if "n_valid" in case:
        assert out["n_valid"] == case["n_valid"]
    dz = oracle.ce_backward(z, y, out["lse"], out["n_valid"], case["grad_output"], eps, red)
    np.testing.assert_allclose(dz, case["dz"], rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------
# ignore / bad targets / reduction
# ---------------------------------------------------------------------------

def test_ignored_rows_and_mean_denominator():
    n, vocab = 10, 17
    z = rng.standard_normal((n, vocab))
    y = rng.integers(0, vocab, n)
    y[[1, 4, 5]] = -100
    out_none = oracle.ce_forward(z, y, 0.1, False)
    out_mean = oracle.ce_forward(z, y, 0.1, True)
    assert out_mean["n_valid"] == 7
    assert np.all(out_none["loss"][[1, 4, 5]] == 0.0)
    assert np.all(out_none["lse"][[1, 4, 5]] == 0.0) and np.all(out_none["m"][[1, 4, 5]] == 0.0)
    assert abs(out_mean["loss"] - out_none["loss"].sum() / 7) < 1e-15
    dz = oracle.ce_backward(z, y, out_mean["lse"], 7, [2.0], 0.1, True)
    dz1 = oracle.ce_backward(z, y, out_none["lse"], 7, np.full(n, 2.0 / 7), 0.1, False)
    np.testing.assert_allclose(dz, dz1, rtol=1e-15, atol=0)
    assert np.all(dz[[1, 4, 5]] == 0.0)


def test_custom_ignore_index():
    z = rng.standard_normal((4, 5))
    y = np.array([0, 3, 3, 1])
    out = oracle.ce_forward(z, y, 0.0, True, ignore_idx=3)
    assert out["n_valid"] == 2
    assert out["loss_rows"][1] == 0.0 and out["loss_rows"][2] == 0.0


def test_all_ignored_is_nan_with_zero_gradient():
    z = rng.standard_normal((3, 8))
    y = np.full(3, -100)
    out = oracle.ce_forward(z, y, 0.1, True)
    assert out["n_valid"] == 0 and math.isnan(out["loss"])
    dz = oracle.ce_backward(z, y, out["lse"], 0, [1.0], 0.1, True)
    assert np.all(dz == 0.0)


def test_out_of_range_target_is_flagged():
    z = rng.standard_normal((4, 8))
    y = np.array([1, 8, -1, -100])
    out = oracle.ce_forward(z, y, 0.0, False)
    assert list(out["bad"]) == [False, True, True, False]
    assert math.isnan(out["loss"][1]) and math.isnan(out["loss"][2])
    assert out["n_valid"] == 3
    dz = oracle.ce_backward(z, y, out["lse"], 3, np.ones(4), 0.0, False)
    assert np.all(dz[1:] == 0.0) and np.any(dz[0] != 0.0)


# ---------------------------------------------------------------------------
# brute force and library special case
# ---------------------------------------------------------------------------

def _brute_loss(zrow, y, eps):
    vocab = len(zrow)
    s = 0.0
    for v in range(vocab):
        s += math.exp(zrow[v])
    lse = math.log(s)
    loss = 0.0
    for v in range(vocab):
        q = eps / vocab + ((1.0 - eps) if v == y else 0.0)
        loss -= q * (zrow[v] - lse)
    return loss


def test_brute_force_python_loops():
    n, vocab = 6, 13
    z = rng.standard_normal((n, vocab)) * 2
    y = rng.integers(0, vocab, n)
    for eps in (0.0, 0.25):
        got = oracle.ce_forward(z, y, eps)["loss"]
        for i in range(n):
            assert abs(got[i] - _brute_loss(list(z[i]), int(y[i]), eps)) < 1e-13


@pytest.mark.parametrize("reduction", ["none", "mean"])
@pytest.mark.parametrize("eps", [0.0, 0.1])
def test_matches_torch_float64_cross_entropy(reduction, eps):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    n, vocab = 37, 211
    z = rng.standard_normal((n, vocab)) * 3
    y = rng.integers(0, vocab, n)
    y[rng.random(n) < 0.2] = -100
    zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    ref = F.cross_entropy(zt, torch.tensor(y), ignore_index=-100, label_smoothing=eps,
                          reduction=reduction)
    red = reduction == "mean"
    out = oracle.ce_forward(z, y, eps, red)
    np.testing.assert_allclose(out["loss"], ref.detach().numpy(), rtol=1e-12, atol=1e-14)
    g = rng.standard_normal(n) if not red else np.array([1.7])
    ref.backward(torch.tensor(g if not red else g[0], dtype=torch.float64))
    dz = oracle.ce_backward(z, y, out["lse"], out["n_valid"], g, eps, red)
    np.testing.assert_allclose(dz, zt.grad.numpy(), rtol=1e-11, atol=1e-15)


# ---------------------------------------------------------------------------
# finite differences
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("red", [False, True])
@pytest.mark.parametrize("eps", [0.0, 0.15])
def test_logits_gradient_matches_central_differences(red, eps):
    n, vocab = 5, 11
    z = rng.standard_normal((n, vocab)) * 1.5
    y = rng.integers(0, vocab, n)
    y[2] = -100
    g = rng.standard_normal(n) if not red else np.array([0.8])

    def objective(zz):
        out = oracle.ce_forward(zz, y, eps, red)
        return float(out["loss"] * g[0]) if red else float((out["loss"] * g).sum())

    out = oracle.ce_forward(z, y, eps, red)
    dz = oracle.ce_backward(z, y, out["lse"], out["n_valid"], g, eps, red)
    h = 1e-5
    fd = np.zeros_like(z)
    for i in range(n):
        for j in range(vocab):
            zp, zm = z.copy(), z.copy()
            zp[i, j] += h
            zm[i, j] -= h
            fd[i, j] = (objective(zp) - objective(zm)) / (2 * h)
    np.testing.assert_allclose(dz, fd, rtol=1e-6, atol=1e-9)


def test_linear_gradients_match_central_differences():
    n, hidden, vocab = 4, 8, 13
    x = rng.standard_normal((n, hidden))
    w = rng.standard_normal((vocab, hidden)) / math.sqrt(hidden)
    y = rng.integers(0, vocab, n)
    y[1] = -100
    eps = 0.1
    g = np.array([1.3])

    def objective(xx, ww):
        return oracle.lce_forward(xx, ww, y, eps, True)["loss"] * g[0]

    f = oracle.lce_forward(x, w, y, eps, True)
    dx, dw, _ = oracle.lce_backward(x, w, y, f["lse"], f["n_valid"], g, eps, True)
    h = 1e-6
    fdx = np.zeros_like(x)
    for i in range(n):
        for k in range(hidden):
            xp, xm = x.copy(), x.copy()
            xp[i, k] += h
            xm[i, k] -= h
            fdx[i, k] = (objective(xp, w) - objective(xm, w)) / (2 * h)
    fdw = np.zeros_like(w)
    for v in range(vocab):
        for k in range(hidden):
            wp, wm = w.copy(), w.copy()
            wp[v, k] += h
            wm[v, k] -= h
            fdw[v, k] = (objective(x, wp) - objective(x, wm)) / (2 * h)
    np.testing.assert_allclose(dx, fdx, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(dw, fdw, rtol=1e-6, atol=1e-9)
    assert np.all(dx[1] == 0.0)


# ---------------------------------------------------------------------------
# linear form = logits form on X W^T
# ---------------------------------------------------------------------------

def test_linear_equals_logits_of_brute_force_product():
    n, hidden, vocab = 3, 5, 7
    x = rng.standard_normal((n, hidden))
    w = rng.standard_normal((vocab, hidden))
    z = np.zeros((n, vocab))
    for i in range(n):
        for v in range(vocab):
            acc = 0.0
            for k in range(hidden):
                acc += x[i, k] * w[v, k]
            z[i, v] = acc
    y = np.array([0, 6, -100])
    for eps, red in ((0.0, False), (0.2, True)):
        a = oracle.lce_forward(x, w, y, eps, red)
        b = oracle.ce_forward(z, y, eps, red)
        np.testing.assert_allclose(a["loss"], b["loss"], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(a["lse"][:2], b["lse"][:2], rtol=1e-13)


def test_linear_logit_row_sum_identity():
    # sum_v z[n, v] = x_n . (sum_v w_v)
    x = rng.standard_normal((6, 16))
    w = rng.standard_normal((40, 16))
    z = oracle.lce_logits(x, w)
    np.testing.assert_allclose(z.sum(axis=1), x @ w.sum(axis=0), rtol=1e-12, atol=1e-12)


def test_bf16_widening_is_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4040, 0x0000, 0x8000, 0x7F7F, 0x0001], np.uint16)
    expect = [1.0, -1.0, 3.0, 0.0, -0.0, 3.3895313892515355e38, 9.183549615799121e-41]
    np.testing.assert_array_equal(oracle.widen(bits), expect)


def test_sampled_forms_agree_with_full_forms():
    n, hidden, vocab = 40, 24, 300
    x = (rng.standard_normal((n, hidden))).astype(np.float32)
    w = (rng.standard_normal((vocab, hidden)) / 5).astype(np.float32)
    y = rng.integers(0, vocab, n)
    y[::7] = -100
    eps = 0.1
    g = rng.standard_normal(n)
    f = oracle.lce_forward(x, w, y, eps, False)
    dx, dw, _ = oracle.lce_backward(x, w, y, f["lse"], f["n_valid"], g, eps, False)
    rows = np.array([0, 3, 7, 39])
    lse_r, loss_r = oracle.lce_forward_rows(x[rows], w, y[rows], eps)
    np.testing.assert_allclose(lse_r, f["lse"][rows], rtol=1e-14)
    np.testing.assert_allclose(loss_r, f["loss_rows"][rows], rtol=1e-13, atol=1e-15)
    lse_all, loss_all, _ = oracle.lce_lse_all(x, w, y, eps, rows_per_chunk=7)
    np.testing.assert_allclose(lse_all, f["lse"], rtol=1e-14)
    np.testing.assert_allclose(loss_all, f["loss_rows"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(oracle.lce_dx_rows(x[rows], w, y[rows], f["lse"][rows], g[rows], eps),
                               dx[rows], rtol=1e-12, atol=1e-15)
    vids = np.array([0, 5, 299])
    np.testing.assert_allclose(oracle.lce_dw_rows(x, w, vids, y, f["lse"], g, eps),
                               dw[vids], rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------------------
# reduction='sum' and the per-token entropy
# ---------------------------------------------------------------------------

def test_sum_reduction_and_its_gradient():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    n, vocab = 23, 57
    z = rng.standard_normal((n, vocab)) * 2
    y = rng.integers(0, vocab, n)
    y[::5] = -100
    for eps in (0.0, 0.1):
        out = oracle.ce_forward(z, y, eps, 2)
        zt = torch.tensor(z, requires_grad=True)
        ref = F.cross_entropy(zt, torch.tensor(y), ignore_index=-100, label_smoothing=eps, reduction="sum")
        assert abs(out["loss"] - ref.item()) <= 1e-12 * abs(ref.item())
        ref.backward(torch.tensor(0.7, dtype=torch.float64))
        dz = oracle.ce_backward(z, y, out["lse"], out["n_valid"], [0.7], eps, 2)
        np.testing.assert_allclose(dz, zt.grad.numpy(), rtol=1e-11, atol=1e-15)


@pytest.mark.parametrize("vocab", [1, 2, 13, 1000])
def test_entropy_closed_forms(vocab):
    # uniform logits: H = log V; one dominant logit: H -> 0
    z = np.full((3, vocab), 1.5)
    _, lse = oracle.row_stats(z)
    np.testing.assert_allclose(oracle.row_entropy(z, lse), math.log(vocab), atol=1e-13)
    z2 = np.zeros((1, vocab))
    z2[0, 0] = 60.0
    _, lse2 = oracle.row_stats(z2)
    assert abs(oracle.row_entropy(z2, lse2)[0]) < 1e-20 * vocab + 1e-22 or vocab == 1


def test_entropy_matches_scipy():
    from scipy.stats import entropy
    from scipy.special import softmax
    z = rng.standard_normal((9, 77)) * 3
    _, lse = oracle.row_stats(z)
    expect = entropy(softmax(z, axis=1), axis=1)
    np.testing.assert_allclose(oracle.row_entropy(z, lse), expect, rtol=1e-12)


def test_linear_forward_entropy_equals_logits_entropy():
    x = rng.standard_normal((5, 12))
    w = rng.standard_normal((31, 12))
    out = oracle.lce_forward(x, w, np.zeros(5, np.int64), 0.0, False)
    z = oracle.lce_logits(x, w)
    _, lse = oracle.row_stats(z)
    np.testing.assert_allclose(out["entropy"], oracle.row_entropy(z, lse), rtol=1e-13)
    _, _, ent = oracle.lce_lse_all(x, w, np.zeros(5, np.int64), entropy=True, rows_per_chunk=2)
    np.testing.assert_allclose(ent, out["entropy"], rtol=1e-13)


# ---------------------------------------------------------------------------
# token shift (causal language modelling)
# ---------------------------------------------------------------------------

def test_shift_targets_small_example():
    # two sequences of length 4: labels move one to the left, each sequence's last is ignored
    t = np.array([10, 11, 12, 13, 20, 21, 22, 23])
    assert list(oracle.shift_targets(t, 4)) == [11, 12, 13, -100, 21, 22, 23, -100]
    # a trailing partial sequence ends with an ignored position too
    assert list(oracle.shift_targets(np.arange(6), 4)) == [1, 2, 3, -100, 5, -100]
    # one long sequence: the plain one-step shift
    assert list(oracle.shift_targets(np.arange(5), 5, ignore_idx=-1)) == [1, 2, 3, 4, -1]


def test_shifted_loss_equals_unshifted_loss_on_sliced_logits():
    # CCE's shift: logits[:, :-1] scored against labels[:, 1:]
    b, t, vocab = 3, 7, 19
    z = rng.standard_normal((b, t, vocab))
    y = rng.integers(0, vocab, (b, t))
    shifted = oracle.shift_targets(y.reshape(-1), t)
    full = oracle.ce_forward(z.reshape(-1, vocab), shifted, 0.1, True)
    ref = oracle.ce_forward(z[:, :-1].reshape(-1, vocab), y[:, 1:].reshape(-1), 0.1, True)
    assert full["n_valid"] == b * (t - 1)
    assert abs(full["loss"] - ref["loss"]) < 1e-13
