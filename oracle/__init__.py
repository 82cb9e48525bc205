"""FP64 CPU oracle for large-vocabulary softmax cross-entropy.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
Python binding) imports, links or calls this module; only the tests, the smoke
check and the benchmark's CPU-baseline leg do.  It shares no code with the CUDA
path: it is a plain, slow, obviously correct restatement of what the loss is,
written out in NumPy float64.

What it computes, with the passages it follows
-----------------------------------------------
Logits form -- Transformer Engine ``parallel_cross_entropy`` (API card,
"Description" and "I/O Contract"; pull request #3273, "Changes"):

* every row n of logits z[n, :] (length V) with target y_n:
    m_n   = max_v z[n, v]
    lse_n = m_n + log sum_v exp(z[n, v] - m_n)
    loss_n = (1 - eps) * (lse_n - z[n, y_n]) + eps * (lse_n - (1/V) sum_v z[n, v])
  i.e. the cross-entropy against the smoothed target distribution
  q = (1 - eps) * onehot(y_n) + eps / V (smoothing spread over all V classes,
  target included, the convention of torch.nn.functional.cross_entropy, of
  which the API card calls the op a drop-in replacement);
* rows whose target equals ``ignore_idx`` give loss 0 and gradient 0, and their
  row is never read: their saved statistics are written as (0, 0);
* a target that is neither ``ignore_idx`` nor in [0, V) is an error: that row's
  loss is NaN, its gradient row is 0, and ``bad`` flags it;
* ``reduce_loss`` = 1 (mean) returns sum_n loss_n / N_v with N_v the number of
  rows whose target is not ``ignore_idx`` (NaN when N_v = 0), and then the
  per-row upstream gradient is g / N_v; ``reduce_loss`` = 2 (sum, the Cut
  Cross-Entropy card's reduction modes beside 'none') returns sum_n loss_n with
  upstream gradient g for every row; 0 (none) returns the per-row losses;
* the saved state is the per-row statistics (m_n, lse_n) instead of the full
  derivative (pull request #3273, "Changes"); backward rebuilds
    dz[n, v] = g_n * (exp(z[n, v] - lse_n) - (1 - eps) [v = y_n] - eps / V).

Linear form -- Cut Cross-Entropy package card ("what_it_does": logits of
embeddings x classifier computed on the fly, only the target logit and the
log-sum-exp over the vocabulary kept) and the Liger SM100 pull request
("Summary"; backward = logits recomputation, dX, dW):

* z = X @ W^T  (X [N, H], W [V, H]); loss and lse as above, lse kept for every
  row (the logits of ignored rows are computed anyway);
* dZ by the formula above, dX = dZ @ W, dW = dZ^T @ X;
* optional per-token entropy of the softmax (Liger pull request, "Summary":
  optional entropy): H_n = -sum_v p_v log p_v = lse_n - sum_v p_v z[n, v];
* token shift for causal language modelling (Cut Cross-Entropy card,
  "what_it_does": optional token shifting): with sequences of length T laid
  out one after another, position t of a sequence is scored against the label
  at t + 1 of the same sequence, and the last position of each sequence is
  ignored.

Inputs are the exact stored values (bfloat16 or float32) widened to float64.
The matrix products use NumPy's float64 matmul as a library step; every other
step is written out here.  Rows are independent, so large inputs are processed
in row chunks; no reduction is reordered or blocked.

Parity pins: every function here is checked in tests/test_oracle_pins.py
against closed forms, a hand-derived worked example (tests/golden/), central
finite differences, brute-force loops and torch's float64 CPU cross entropy.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "widen", "row_stats", "row_loss", "grad_columns",
    "ce_forward", "ce_backward", "lce_logits", "lce_forward", "lce_backward",
    "lce_forward_rows", "lce_dx_rows", "lce_lse_all", "lce_dw_rows",
    "mean_loss", "reduce", "row_entropy", "upstream", "shift_targets",
]


def widen(a, dtype: str | None = None) -> np.ndarray:
    """Exact float64 value of stored logits/weights.

    ``dtype='bf16'`` (or a uint16 array) means bfloat16 bit patterns: the value
    is the pattern shifted into the high half of an IEEE float32.
    """
    a = np.asarray(a)
    if dtype == "bf16" or a.dtype == np.uint16:
        f32 = (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
        return f32.astype(np.float64)
    return a.astype(np.float64)


# ---------------------------------------------------------------------------
# per-row pieces (z is float64 [rows, V])
# ---------------------------------------------------------------------------

def row_stats(z: np.ndarray):
    """(m, lse) per row: m = max_v z, lse = m + log(sum_v exp(z - m))."""
    m = z.max(axis=1)
    with np.errstate(invalid="ignore", over="ignore"):
        lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    return m, lse


def _row_classes(target: np.ndarray, vocab: int, ignore_idx: int):
    target = np.asarray(target, dtype=np.int64)
    ignored = target == ignore_idx
    bad = ~ignored & ((target < 0) | (target >= vocab))
    return ignored, bad


def row_loss(z: np.ndarray, target: np.ndarray, lse: np.ndarray, eps: float,
             ignore_idx: int) -> np.ndarray:
    """loss_n = (1-eps)(lse_n - z[n, y_n]) + eps (lse_n - mean_v z[n, v]); 0 if ignored, NaN if bad."""
    n, vocab = z.shape
    ignored, bad = _row_classes(target, vocab, ignore_idx)
    ok = ~ignored & ~bad
    loss = np.zeros(n, dtype=np.float64)
    rows = np.nonzero(ok)[0]
    zy = z[rows, np.asarray(target)[rows]]
    loss[rows] = (1.0 - eps) * (lse[rows] - zy)
    if eps != 0.0:
        loss[rows] += eps * (lse[rows] - z[rows].sum(axis=1) / vocab)
    loss[bad] = np.nan
    return loss


def grad_columns(z_cols: np.ndarray, cols: np.ndarray, vocab: int, target: np.ndarray,
                 lse: np.ndarray, g_rows: np.ndarray, eps: float, ignore_idx: int) -> np.ndarray:
    """dz[n, c] for the vocabulary ids ``cols`` (z_cols = z[:, cols]).

    dz[n, v] = g_n * (exp(z[n, v] - lse_n) - (1-eps)[v = y_n] - eps/V); rows that
    are ignored or have a bad target are 0.
    """
    target = np.asarray(target, dtype=np.int64)
    ignored, bad = _row_classes(target, vocab, ignore_idx)
    ok = ~ignored & ~bad
    g = np.where(ok, np.asarray(g_rows, dtype=np.float64), 0.0)
    lse_safe = np.where(ok, lse, 0.0)
    with np.errstate(invalid="ignore", over="ignore"):
        p = np.exp(z_cols - lse_safe[:, None])
    dz = g[:, None] * (p - eps / vocab)
    hit = np.asarray(cols)[None, :] == target[:, None]
    dz -= np.where(hit, g[:, None] * (1.0 - eps), 0.0)
    dz[~ok] = 0.0
    return dz


def _upstream(grad_output, n: int, n_valid: int, reduce_loss) -> np.ndarray:
    grad_output = np.asarray(grad_output, dtype=np.float64).reshape(-1)
    if int(reduce_loss) == 2:
        return np.full(n, grad_output[0])
    if reduce_loss:
        if n_valid == 0:
            return np.zeros(n)
        return np.full(n, grad_output[0] / n_valid)
    return grad_output[:n]


def mean_loss(loss_rows: np.ndarray, n_valid: int) -> float:
    """sum_n loss_n / N_v (0/0 = NaN when every row is ignored)."""
    with np.errstate(invalid="ignore", divide="ignore"):
        return float(np.float64(loss_rows.sum()) / np.float64(n_valid))


def reduce(loss_rows: np.ndarray, n_valid: int, reduce_loss):
    """The loss a call returns: per-row (0), mean over non-ignored rows (1) or sum (2)."""
    if int(reduce_loss) == 2:
        return float(loss_rows.sum())
    return mean_loss(loss_rows, n_valid) if reduce_loss else loss_rows


def shift_targets(target, seq_len: int, ignore_idx: int = -100) -> np.ndarray:
    """shifted[b*T + t] = target[b*T + t + 1] for t < T - 1, ignore_idx for t = T - 1
    (a final partial sequence of length n mod T follows the same rule)."""
    target = np.asarray(target, dtype=np.int64)
    n = len(target)
    out = np.full(n, ignore_idx, dtype=np.int64)
    for i in range(n):
        last_in_sequence = (i % seq_len == seq_len - 1) or (i == n - 1)
        if not last_in_sequence:
            out[i] = target[i + 1]
    return out


def row_entropy(z: np.ndarray, lse: np.ndarray) -> np.ndarray:
    """H_n = lse_n - sum_v p_v z[n, v] with p_v = exp(z[n, v] - lse_n)."""
    with np.errstate(invalid="ignore", over="ignore"):
        p = np.exp(z - lse[:, None])
    return lse - (p * z).sum(axis=1)


# ---------------------------------------------------------------------------
# logits form
# ---------------------------------------------------------------------------

def ce_forward(z, target, label_smoothing: float = 0.0, reduce_loss: bool = False,
               ignore_idx: int = -100, dtype: str | None = None):
    """Logits-form forward.  Returns dict(loss, loss_rows, m, lse, n_valid, bad)."""
    z = widen(z, dtype)
    n, vocab = z.shape
    target = np.asarray(target, dtype=np.int64)
    ignored, bad = _row_classes(target, vocab, ignore_idx)
    m, lse = row_stats(z)
    loss_rows = row_loss(z, target, lse, label_smoothing, ignore_idx)
    m = np.where(ignored, 0.0, m)
    lse = np.where(ignored, 0.0, lse)
    n_valid = int((~ignored).sum())
    loss = reduce(loss_rows, n_valid, reduce_loss)
    return dict(loss=loss, loss_rows=loss_rows, m=m, lse=lse, n_valid=n_valid, bad=bad)


def ce_backward(z, target, lse, n_valid: int, grad_output, label_smoothing: float = 0.0,
                reduce_loss: bool = False, ignore_idx: int = -100, dtype: str | None = None):
    """Logits-form backward from the saved lse: dz [N, V] float64."""
    z = widen(z, dtype)
    n, vocab = z.shape
    g = _upstream(grad_output, n, n_valid, reduce_loss)
    return grad_columns(z, np.arange(vocab), vocab, target, np.asarray(lse, np.float64), g,
                        label_smoothing, ignore_idx)


# ---------------------------------------------------------------------------
# linear form
# ---------------------------------------------------------------------------

def lce_logits(x, w) -> np.ndarray:
    """z = X @ W^T in float64."""
    return widen(x) @ widen(w).T


def lce_forward(x, w, target, label_smoothing: float = 0.0, reduce_loss: bool = False,
                ignore_idx: int = -100):
    """Linear-form forward on full inputs.  Returns dict(loss, loss_rows, lse, n_valid, bad, z)."""
    z = lce_logits(x, w)
    vocab = z.shape[1]
    target = np.asarray(target, dtype=np.int64)
    ignored, bad = _row_classes(target, vocab, ignore_idx)
    _, lse = row_stats(z)
    loss_rows = row_loss(z, target, lse, label_smoothing, ignore_idx)
    n_valid = int((~ignored).sum())
    loss = reduce(loss_rows, n_valid, reduce_loss)
    return dict(loss=loss, loss_rows=loss_rows, lse=lse, n_valid=n_valid, bad=bad, z=z,
                entropy=row_entropy(z, lse))


def lce_backward(x, w, target, lse, n_valid: int, grad_output, label_smoothing: float = 0.0,
                 reduce_loss: bool = False, ignore_idx: int = -100, z=None):
    """Linear-form backward on full inputs: (dX [N, H], dW [V, H], dZ [N, V]) in float64."""
    xd, wd = widen(x), widen(w)
    if z is None:
        z = xd @ wd.T
    n, vocab = z.shape
    g = _upstream(grad_output, n, n_valid, reduce_loss)
    dz = grad_columns(z, np.arange(vocab), vocab, target, np.asarray(lse, np.float64), g,
                      label_smoothing, ignore_idx)
    return dz @ wd, dz.T @ xd, dz


# --- sampled forms for inputs too large to hold as float64 ------------------

def lce_forward_rows(x_rows, w, target_rows, label_smoothing: float = 0.0,
                     ignore_idx: int = -100):
    """Per-row lse and loss for a subset of tokens (x_rows [S, H]); returns (lse [S], loss [S])."""
    z = lce_logits(x_rows, w)
    _, lse = row_stats(z)
    return lse, row_loss(z, np.asarray(target_rows), lse, label_smoothing, ignore_idx)


def lce_lse_all(x, w, target, label_smoothing: float = 0.0, ignore_idx: int = -100,
                rows_per_chunk: int = 512, entropy: bool = False):
    """lse and loss (and optionally the entropy) for every token, rows processed in
    independent chunks (each row whole)."""
    n = x.shape[0]
    wd = widen(w)
    target = np.asarray(target, dtype=np.int64)
    lse = np.empty(n)
    loss = np.empty(n)
    ent = np.empty(n)
    for r0 in range(0, n, rows_per_chunk):
        r1 = min(n, r0 + rows_per_chunk)
        z = widen(x[r0:r1]) @ wd.T
        _, l = row_stats(z)
        lse[r0:r1] = l
        loss[r0:r1] = row_loss(z, target[r0:r1], l, label_smoothing, ignore_idx)
        if entropy:
            ent[r0:r1] = row_entropy(z, l)
    return lse, loss, (ent if entropy else None)


def lce_dx_rows(x_rows, w, target_rows, lse_rows, g_rows, label_smoothing: float = 0.0,
                ignore_idx: int = -100):
    """dX rows for a subset of tokens: dX[n] = sum_v dz[n, v] W[v]."""
    wd = widen(w)
    z = widen(x_rows) @ wd.T
    vocab = z.shape[1]
    dz = grad_columns(z, np.arange(vocab), vocab, target_rows, np.asarray(lse_rows, np.float64),
                      g_rows, label_smoothing, ignore_idx)
    return dz @ wd


def lce_dw_rows(x, w, vocab_ids, target, lse_all, g_all, label_smoothing: float = 0.0,
                ignore_idx: int = -100):
    """dW rows for a subset of vocabulary ids: dW[v] = sum_n dz[n, v] X[n] (needs lse of every token)."""
    xd = widen(x)
    vocab = w.shape[0]
    vocab_ids = np.asarray(vocab_ids, dtype=np.int64)
    z_cols = xd @ widen(w[vocab_ids]).T                     # [N, S]
    dz = grad_columns(z_cols, vocab_ids, vocab, target, np.asarray(lse_all, np.float64),
                      g_all, label_smoothing, ignore_idx)
    return dz.T @ xd


def upstream(grad_output, n: int, n_valid: int, reduce_loss: bool) -> np.ndarray:
    """Per-row upstream gradient g_n: grad_output[n], or grad_output[0] / N_v when reduced."""
    return _upstream(grad_output, n, n_valid, reduce_loss)
