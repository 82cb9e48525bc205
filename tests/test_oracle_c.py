"""The plain-C FP64 oracle (oracle/vce_oracle.c) against the NumPy FP64 oracle and
the closed forms: two independent restatements of the same definitions must agree
to FP64 rounding.  No GPU."""
import math

import numpy as np
import pytest

import oracle
from oracle import c_oracle

rng = np.random.default_rng(77)


@pytest.mark.parametrize("eps", [0.0, 0.1])
@pytest.mark.parametrize("n,vocab", [(1, 1), (7, 13), (64, 1000), (5, 32001)])
def test_c_oracle_matches_numpy_oracle(n, vocab, eps):
    z = rng.standard_normal((n, vocab)) * 3
    y = rng.integers(0, vocab, n)
    y[rng.random(n) < 0.2] = -100
    if n > 2:
        y[1] = vocab  # an out-of-range target
    c = c_oracle.ce_forward(z, y, eps)
    p = oracle.ce_forward(z, y, eps, False)
    assert c["n_valid"] == p["n_valid"]
    np.testing.assert_array_equal(c["bad"], p["bad"])
    np.testing.assert_allclose(c["loss_rows"], p["loss_rows"], rtol=1e-12, atol=1e-13, equal_nan=True)
    np.testing.assert_array_equal(c["m"], p["m"])
    np.testing.assert_allclose(c["lse"], p["lse"], rtol=1e-13, atol=1e-13)
    g = rng.standard_normal(n)
    dc = c_oracle.ce_backward(z, y, c["lse"], g, eps)
    dp = oracle.ce_backward(z, y, p["lse"], p["n_valid"], g, eps, False)
    np.testing.assert_allclose(dc, dp, rtol=1e-11, atol=1e-15)


def test_c_oracle_uniform_logits_closed_form():
    vocab = 777
    z = np.full((4, vocab), -2.5)
    c = c_oracle.ce_forward(z, np.array([0, 5, 776, -100]), 0.3)
    np.testing.assert_allclose(c["loss_rows"][:3], math.log(vocab), atol=1e-12)
    assert c["loss_rows"][3] == 0.0 and c["lse"][3] == 0.0


def test_c_linear_logits_matches_numpy_product():
    x = rng.standard_normal((9, 33))
    w = rng.standard_normal((57, 33))
    np.testing.assert_allclose(c_oracle.linear_logits(x, w), oracle.lce_logits(x, w), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("eps", [0.0, 0.1])
def test_c_linear_backward_matches_numpy_oracle(eps):
    # the whole linear backward restated in C: its own product, lse, gradient and
    # dX / dW loops, against the NumPy oracle's lce_forward / lce_backward
    n, h, vocab = 11, 24, 37
    x = rng.standard_normal((n, h))
    w = rng.standard_normal((vocab, h)) * h ** -0.5
    y = rng.integers(0, vocab, n)
    y[3] = -100
    g = rng.standard_normal(n)
    zc = c_oracle.linear_logits(x, w)
    fc = c_oracle.ce_forward(zc, y, eps)
    dzc = c_oracle.ce_backward(zc, y, fc["lse"], g, eps)
    dxc, dwc = c_oracle.linear_grads(dzc, x, w)
    fp = oracle.lce_forward(x, w, y, eps, False)
    dxp, dwp, _ = oracle.lce_backward(x, w, y, fp["lse"], fp["n_valid"], g, eps, False)
    np.testing.assert_allclose(dxc, dxp, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dwc, dwp, rtol=1e-11, atol=1e-13)
    assert np.all(dxc[3] == 0.0)  # an ignored token contributes nothing


def test_c_entropy_matches_numpy_oracle_and_uniform_closed_form():
    z = rng.standard_normal((6, 50)) * 2
    fc = c_oracle.ce_forward(z, np.zeros(6, np.int64))
    np.testing.assert_allclose(c_oracle.entropy(z, fc["lse"]), oracle.row_entropy(z, fc["lse"]),
                               rtol=1e-12, atol=1e-13)
    u = np.full((2, 300), 1.5)  # uniform softmax: entropy log V
    fu = c_oracle.ce_forward(u, np.zeros(2, np.int64))
    np.testing.assert_allclose(c_oracle.entropy(u, fu["lse"]), math.log(300), atol=1e-12)
