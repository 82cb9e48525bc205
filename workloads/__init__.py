"""Seeded synthetic inputs for the vocabulary cross-entropy workloads.

This module is shared by the tests, the benchmark and the oracle's callers.  It
draws random numbers and rounds them to the storage dtype; it holds none of the
loss arithmetic (no softmax, no log-sum-exp, no gradient), so neither the CUDA
library nor the oracle depends on the other through it.

Every tensor is produced in independent row blocks.  Block ``b`` of tensor
``tensor_id`` is drawn from ``SFC64(SeedSequence([seed, tensor_id, b]))``, so any
row can be regenerated on its own (the oracle checks sampled rows of tensors
that are too large to hold in FP64) and blocks can be generated in parallel.

Workload shapes and value distributions follow the configurations the pages
benchmark: Transformer Engine's ``parallel_cross_entropy`` logits form
(I/O contract: logits (B, SQ, V), targets (B, SQ), ignore_idx = -100) and the
fused linear cross-entropy form of the Liger SM100 pull request ("Performance
methodology": BF16 inputs, H = 4096, V = 131072, M = 4096 tokens).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

IGNORE_IDX = -100

# tensor ids: one independent stream family per logical tensor
TID_LOGITS = 1
TID_TARGET = 2
TID_IGNORE = 3
TID_GRAD = 4
TID_X = 5
TID_W = 6

_BLOCK_ELEMS = 1 << 20


def _rng(seed: int, tensor_id: int, block: int) -> np.random.Generator:
    return np.random.Generator(np.random.SFC64(np.random.SeedSequence([seed, tensor_id, block])))


def _rows_per_block(ncols: int) -> int:
    return max(1, _BLOCK_ELEMS // max(1, ncols))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float32 exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_block(seed, tid, block, rows_in_block, ncols, std, bf16):
    g = _rng(seed, tid, block)
    v = g.standard_normal(rows_in_block * ncols, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    v = v.reshape(rows_in_block, ncols)
    return f32_to_bf16_bits(v) if bf16 else v


def normal_matrix(seed: int, tensor_id: int, nrows: int, ncols: int, std: float,
                  bf16: bool, threads: int | None = None) -> np.ndarray:
    """A [nrows, ncols] matrix of N(0, std^2) values (bf16 bit patterns when ``bf16``)."""
    rpb = _rows_per_block(ncols)
    nblocks = (nrows + rpb - 1) // rpb
    out = np.empty((nrows, ncols), dtype=np.uint16 if bf16 else np.float32)

    def fill(b):
        r0 = b * rpb
        r1 = min(nrows, r0 + rpb)
        blk = _normal_block(seed, tensor_id, b, rpb, ncols, std, bf16)
        out[r0:r1] = blk[: r1 - r0]

    threads = threads or min(32, os.cpu_count() or 1)
    if nblocks == 1 or threads == 1:
        for b in range(nblocks):
            fill(b)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(nblocks)))
    return out


def normal_rows(seed: int, tensor_id: int, rows, ncols: int, std: float, bf16: bool) -> np.ndarray:
    """Regenerate only the given rows of ``normal_matrix(seed, tensor_id, *, ncols, std, bf16)``.

    Rows past the end of the full matrix are not checked here: the caller passes
    row ids of the matrix it generated.
    """
    rows = np.asarray(rows, dtype=np.int64)
    rpb = _rows_per_block(ncols)
    out = np.empty((len(rows), ncols), dtype=np.uint16 if bf16 else np.float32)
    cache = {}
    for i, r in enumerate(rows):
        b = int(r) // rpb
        if b not in cache:
            cache[b] = _normal_block(seed, tensor_id, b, rpb, ncols, std, bf16)
        out[i] = cache[b][int(r) - b * rpb]
    return out


def uniform_targets(seed: int, n: int, vocab: int, ignore_frac: float) -> np.ndarray:
    """Targets uniform in [0, vocab); each token independently set to IGNORE_IDX with prob ignore_frac."""
    t = _rng(seed, TID_TARGET, 0).integers(0, vocab, size=n, dtype=np.int64)
    if ignore_frac > 0.0:
        drop = _rng(seed, TID_IGNORE, 0).random(n) < ignore_frac
        t[drop] = IGNORE_IDX
    return t


def zipf_targets(seed: int, n: int, vocab: int, s: float) -> np.ndarray:
    """Targets with P(id = k - 1) proportional to k^-s for k = 1..vocab (rank k maps to id k - 1).

    Sampled by inverse CDF: a uniform draw is located in the FP64 prefix sum of the
    unnormalised weights by binary search.
    """
    k = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(k ** (-s))
    u = _rng(seed, TID_TARGET, 0).random(n) * cdf[-1]
    t = np.searchsorted(cdf, u, side="right").astype(np.int64)
    return np.minimum(t, vocab - 1)


def grad_rows(seed: int, n: int) -> np.ndarray:
    """Per-token upstream gradient g ~ N(0, 1) (FP32), for reduction='none'."""
    return _rng(seed, TID_GRAD, 0).standard_normal(n, dtype=np.float32)


# ---------------------------------------------------------------------------
# workload table
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class LogitsWorkload:
    name: str
    n_rows: int
    vocab: int
    dtype: str            # "f32" or "bf16"
    std: float
    ignore_frac: float
    label_smoothing: float
    reduce_loss: bool
    seed: int = 0


@dataclass(frozen=True)
class LinearWorkload:
    name: str
    n: int
    hidden: int
    vocab: int
    ignore_frac: float = 0.0
    ignore_tail: int = 0            # last ``ignore_tail`` tokens are ignored (padding)
    zipf_s: float | None = None     # Zipf targets instead of uniform
    label_smoothing: float = 0.0
    reduce_loss: bool = True
    seed: int = 0
    w_std: float | None = None      # default 1/sqrt(H): W ~ N(0, 1/H)


LOGITS_TINY = [
    LogitsWorkload(f"logits_tiny_eps{eps}_reduce{int(red)}", 128, 1024, "f32", 2.0, 0.10, eps, red)
    for eps in (0.0, 0.1) for red in (False, True)
]
LOGITS_MEMBOUND = LogitsWorkload("logits_membound_4x4096x128256", 4 * 4096, 128256, "bf16",
                                 3.0, 0.05, 0.1, True)
LINEAR_SMALL = LinearWorkload("linear_4096x2048x32000", 4096, 2048, 32000, ignore_frac=0.02,
                              label_smoothing=0.0, reduce_loss=False)
LINEAR_HEADLINE = LinearWorkload("linear_headline_4096x4096x131072", 4096, 4096, 131072,
                                 label_smoothing=0.0, reduce_loss=True)
LINEAR_LARGE = LinearWorkload("linear_large_16384x4096x128256", 16384, 4096, 128256,
                              ignore_tail=903, zipf_s=1.1, label_smoothing=0.1, reduce_loss=True)


@dataclass
class LogitsInputs:
    logits: np.ndarray        # [N, V] float32, or uint16 bf16 bit patterns
    target: np.ndarray        # [N] int64
    grad: np.ndarray          # [N] float32 (reduction='none') or [1] (mean)
    wl: LogitsWorkload = field(repr=False)


def make_logits_inputs(wl: LogitsWorkload, threads: int | None = None) -> LogitsInputs:
    logits = normal_matrix(wl.seed, TID_LOGITS, wl.n_rows, wl.vocab, wl.std, wl.dtype == "bf16", threads)
    target = uniform_targets(wl.seed, wl.n_rows, wl.vocab, wl.ignore_frac)
    grad = np.ones(1, np.float32) if wl.reduce_loss else grad_rows(wl.seed, wl.n_rows)
    return LogitsInputs(logits, target, grad, wl)


def logits_rows(wl: LogitsWorkload, rows) -> np.ndarray:
    return normal_rows(wl.seed, TID_LOGITS, rows, wl.vocab, wl.std, wl.dtype == "bf16")


# classifier shapes of production models at M = 8192 tokens (the Liger SM100 pull
# request's "Model-shape campaign": random BF16 inputs)
MODEL_SHAPES = [
    LinearWorkload("qwen3_30b_a3b_8192x2048x151936", 8192, 2048, 151936),
    LinearWorkload("llama4_8192x5120x202048", 8192, 5120, 202048),
    LinearWorkload("deepseek_v3_8192x7168x129280", 8192, 7168, 129280),
]


@dataclass
class LinearInputs:
    x: np.ndarray             # [N, H] uint16 bf16 bits
    w: np.ndarray             # [V, H] uint16 bf16 bits
    target: np.ndarray        # [N] int64
    grad: np.ndarray          # [N] float32 or [1]
    wl: LinearWorkload = field(repr=False)


def linear_w_std(wl: LinearWorkload) -> float:
    return wl.w_std if wl.w_std is not None else float(1.0 / np.sqrt(wl.hidden))


def linear_targets(wl: LinearWorkload) -> np.ndarray:
    if wl.zipf_s is not None:
        t = zipf_targets(wl.seed, wl.n, wl.vocab, wl.zipf_s)
    else:
        t = uniform_targets(wl.seed, wl.n, wl.vocab, wl.ignore_frac)
    if wl.ignore_tail:
        t[wl.n - wl.ignore_tail:] = IGNORE_IDX
    return t


def make_linear_inputs(wl: LinearWorkload, threads: int | None = None) -> LinearInputs:
    x = normal_matrix(wl.seed, TID_X, wl.n, wl.hidden, 1.0, True, threads)
    w = normal_matrix(wl.seed, TID_W, wl.vocab, wl.hidden, linear_w_std(wl), True, threads)
    grad = np.ones(1, np.float32) if wl.reduce_loss else grad_rows(wl.seed, wl.n)
    return LinearInputs(x, w, linear_targets(wl), grad, wl)
