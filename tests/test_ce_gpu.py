"""Logits form on the GPU against the FP64 oracle (Transformer Engine
parallel_cross_entropy semantics).  Tolerances:

* FP32 logits: per-row loss |d| <= 1e-5 max(|ref|, 1), dlogits tensor-wise
  ||d|| <= 1e-5 ||ref||;
* BF16 logits: loss |d| <= 2e-3 (per row and the mean), dlogits norm-wise
  ||d|| / ||ref|| <= 1e-2 (BF16 output rounding is 2^-9 relative);
* ignore masks (zero loss, zero gradient rows) and N_v: bit-exact.
"""
import math
from concurrent.futures import ThreadPoolExecutor

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


def to_dev(logits_np, dtype):
    if dtype == "bf16":
        return torch.from_numpy(logits_np.view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(logits_np).to(DEV)


def bf16_np(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_gpu(logits, target, eps, red, grad, ignore_idx=-100, inplace=False, dlogits=None):
    tgt = torch.from_numpy(target).to(DEV)
    f = vce.ce_forward(logits, tgt, eps, red, ignore_idx)
    g = torch.from_numpy(np.asarray(grad, np.float32)).to(DEV)
    dz = vce.ce_backward(logits, tgt, f.stats, f.n_valid, g, eps, red, ignore_idx, inplace=inplace,
                         dlogits=dlogits)
    torch.cuda.synchronize()
    return f, dz


def dz_np(dz, dtype):
    return oracle.widen(bf16_np(dz), "bf16") if dtype == "bf16" else dz.double().cpu().numpy()


def check_rows(f, dz, ref_f, ref_dz, rows, dtype, red, target):
    loss_tol_rel = 1e-5 if dtype == "f32" else 0.0
    loss_tol_abs = 0.0 if dtype == "f32" else 2e-3
    stats = f.stats.double().cpu().numpy()
    valid = target[rows] != -100
    if not red:
        got = f.loss.double().cpu().numpy().reshape(-1)[rows]
        ref = ref_f["loss_rows"]
        assert np.all(got[~valid] == 0.0)
        err = np.abs(got - ref)
        # relative with a floor of 1 nat: a near-zero loss has no meaningful relative error
        assert np.all(err <= loss_tol_abs + loss_tol_rel * np.maximum(np.abs(ref), 1.0)), err.max()
    # statistics: max is an exact max of stored values; lse within loss tolerance
    np.testing.assert_array_equal(stats[rows][valid, 0], ref_f["m"][valid])
    np.testing.assert_allclose(stats[rows][valid, 1], ref_f["lse"][valid],
                               rtol=loss_tol_rel, atol=loss_tol_abs + 1e-30)
    assert np.all(stats[rows][~valid] == 0.0)
    got_dz = dz_np(dz, dtype)[rows] if dz.shape[0] != len(rows) else dz_np(dz, dtype)
    assert np.all(got_dz[~valid] == 0.0)
    if dtype == "f32":
        # tensor-wise relative error: a single row can be nearly zero (prediction
        # close to the smoothed target) and there FP32 lse rounding alone exceeds 1e-5
        err = np.linalg.norm(got_dz - ref_dz)
        assert err <= 1e-5 * np.linalg.norm(ref_dz) + 1e-12, err / np.linalg.norm(ref_dz)
    else:
        # norm-wise; the absolute floor covers an all-zero reference (V = 1), where
        # only FP32 rounding of the exponent argument z*log2(e) - lse*log2(e) remains
        err = np.linalg.norm(got_dz - ref_dz)
        assert err <= 1e-2 * np.linalg.norm(ref_dz) + 1e-6, (err, np.linalg.norm(ref_dz))


# ---------------------------------------------------------------------------
# tiny FP32 workload: N=128, V=1024, z ~ N(0, 2^2), 10% ignored
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("wl", wk.LOGITS_TINY, ids=lambda w: w.name)
def test_tiny_fp32_full(wl):
    inp = wk.make_logits_inputs(wl)
    logits = to_dev(inp.logits, wl.dtype)
    f, dz = run_gpu(logits, inp.target, wl.label_smoothing, wl.reduce_loss, inp.grad)
    ref = oracle.ce_forward(inp.logits, inp.target, wl.label_smoothing, wl.reduce_loss)
    ref_dz = oracle.ce_backward(inp.logits, inp.target, ref["lse"], ref["n_valid"], inp.grad,
                                wl.label_smoothing, wl.reduce_loss)
    assert int(f.n_valid.item()) == ref["n_valid"]
    assert int(f.dev_status.item()) == 0
    if wl.reduce_loss:
        assert abs(f.loss.item() - ref["loss"]) <= 1e-5 * abs(ref["loss"])
    rows = np.arange(wl.n_rows)
    check_rows(f, dz, ref, ref_dz, rows, wl.dtype, wl.reduce_loss, inp.target)


# ---------------------------------------------------------------------------
# edge shapes: ragged / odd V, padded and misaligned rows, N = 1, both dtypes
# ---------------------------------------------------------------------------

EDGE = [
    # (n, vocab, pad, dtype, eps, reduce: 0 none, 1 mean, 2 sum)
    (1, 1, 0, "f32", 0.0, False),
    (3, 1, 0, "bf16", 0.1, True),
    (5, 7, 0, "f32", 0.1, False),
    (127, 7, 3, "bf16", 0.0, True),
    (64, 1000, 0, "bf16", 0.1, False),
    (33, 32001, 0, "bf16", 0.1, True),
    (17, 32001, 5, "f32", 0.0, False),
    (9, 128257, 0, "bf16", 0.1, True),
    (4097, 129, 0, "f32", 0.1, True),
    (6, 262144, 0, "bf16", 0.0, False),
    (77, 5000, 0, "f32", 0.1, 2),
    (200, 32001, 0, "bf16", 0.0, 2),
]


@pytest.mark.parametrize("n,vocab,pad,dtype,eps,red", EDGE)
def test_edge_shapes(n, vocab, pad, dtype, eps, red):
    seed = n * 7 + vocab
    stride = vocab + pad
    full = wk.normal_matrix(seed, wk.TID_LOGITS, n, stride, 3.0, dtype == "bf16")
    target = wk.uniform_targets(seed, n, vocab, 0.1)
    grad = np.ones(1, np.float32) if red else wk.grad_rows(seed, n)
    dev_full = to_dev(full, dtype)
    logits = dev_full[:, :vocab]
    dz_full = torch.full_like(dev_full, 7.0)
    f, dz = run_gpu(logits, target, eps, red, grad, dlogits=dz_full[:, :vocab])
    z = full[:, :vocab]
    ref = oracle.ce_forward(z, target, eps, red, dtype=dtype)
    ref_dz = oracle.ce_backward(z, target, ref["lse"], ref["n_valid"], grad, eps, red, dtype=dtype)
    assert int(f.n_valid.item()) == ref["n_valid"]
    assert int(f.dev_status.item()) == 0
    if red and ref["n_valid"] > 0:
        tol = 1e-5 * abs(ref["loss"]) if dtype == "f32" else 2e-3 * (ref["n_valid"] if red == 2 else 1)
        assert abs(f.loss.item() - ref["loss"]) <= tol
    check_rows(f, dz, ref, ref_dz, np.arange(n), dtype, red, target)
    # the padding columns between rows are untouched by backward
    if pad:
        assert torch.all(dz_full[:, vocab:] == 7.0).item()


@pytest.mark.parametrize("dtype,offset", [("f32", 200.0), ("f32", 1000.0), ("bf16", 1000.0)])
def test_large_logit_offset(dtype, offset):
    # Logits far from zero.  The softmax works relative to the row maximum, and the
    # rounding of -lse * log2(e) in the exponent is put back per row, so what is
    # left is lse itself being an FP32 value: its rounding, |lse| * 2^-24, moves
    # every probability of the row by that relative amount.  At +200 that stays
    # inside the usual FP32 tolerance; at +1000 the FP32 gradient is checked
    # against that bound instead.
    n, vocab = 64, 5000
    z = wk.normal_matrix(77, wk.TID_LOGITS, n, vocab, 3.0, False) + np.float32(offset)
    if dtype == "bf16":
        z = wk.f32_to_bf16_bits(z)  # BF16 spacing is 4 near 1000: few distinct values per row
    target = wk.uniform_targets(77, n, vocab, 0.1)
    grad = wk.grad_rows(77, n)
    ref = oracle.ce_forward(z, target, 0.1, False, dtype=dtype)
    with np.errstate(over="ignore", invalid="ignore"):  # ignored rows: lse 0 in the oracle, zeroed after
        ref_dz = oracle.ce_backward(z, target, ref["lse"], ref["n_valid"], grad, 0.1, False, dtype=dtype)
    for f, dz in (run_gpu(to_dev(z, dtype), target, 0.1, False, grad),
                  (lambda r: (r, r.dlogits))(run_fused(to_dev(z, dtype), target, 0.1, False, grad))):
        assert int(f.dev_status.item()) == 0
        if dtype == "f32" and offset > 500:
            lse_max = float(np.max(np.abs(ref["lse"])))
            got = dz_np(dz, dtype)
            assert np.linalg.norm(got - ref_dz) <= 2.0 ** -23 * lse_max * np.linalg.norm(ref_dz)
            loss = f.loss.double().cpu().numpy()
            assert np.all(np.abs(loss - ref["loss_rows"]) <= 2.0 ** -22 * lse_max + 1e-5)
        else:
            check_rows(f, dz, ref, ref_dz, np.arange(n), dtype, False, target)


def test_inplace_backward_matches_out_of_place():
    n, vocab = 300, 50257
    z = wk.normal_matrix(5, wk.TID_LOGITS, n, vocab, 3.0, True)
    target = wk.uniform_targets(5, n, vocab, 0.05)
    a = to_dev(z, "bf16")
    b = a.clone()
    fa, dza = run_gpu(a, target, 0.1, True, np.ones(1, np.float32))
    fb, dzb = run_gpu(b, target, 0.1, True, np.ones(1, np.float32), inplace=True)
    assert dzb.data_ptr() == b.data_ptr()
    assert torch.equal(dza.view(torch.int16), dzb.view(torch.int16))
    assert torch.equal(fa.stats, fb.stats)


def test_all_ignored_gives_nan_and_zero_gradient():
    n, vocab = 8, 333
    z = wk.normal_matrix(1, wk.TID_LOGITS, n, vocab, 1.0, False)
    target = np.full(n, -100, np.int64)
    f, dz = run_gpu(to_dev(z, "f32"), target, 0.1, True, np.ones(1, np.float32))
    assert int(f.n_valid.item()) == 0
    assert math.isnan(f.loss.item())
    assert torch.count_nonzero(dz).item() == 0


def test_custom_ignore_index():
    n, vocab = 40, 999
    z = wk.normal_matrix(2, wk.TID_LOGITS, n, vocab, 2.0, True)
    target = wk.uniform_targets(2, n, vocab, 0.0)
    target[::3] = 5
    f, dz = run_gpu(to_dev(z, "bf16"), target, 0.0, True, np.ones(1, np.float32), ignore_idx=5)
    ref = oracle.ce_forward(z, target, 0.0, True, ignore_idx=5, dtype="bf16")
    assert int(f.n_valid.item()) == ref["n_valid"]
    assert abs(f.loss.item() - ref["loss"]) <= 2e-3
    assert torch.count_nonzero(dz[::3].float()).item() == 0


def test_bad_target_sets_status_and_nan():
    n, vocab = 6, 100
    z = wk.normal_matrix(3, wk.TID_LOGITS, n, vocab, 1.0, False)
    target = np.array([1, 100, -1, -100, 99, 0], np.int64)
    f, dz = run_gpu(to_dev(z, "f32"), target, 0.0, False, np.ones(n, np.float32))
    loss = f.loss.cpu().numpy()
    assert int(f.dev_status.item()) & vce.DEVSTATUS_BAD_TARGET
    assert math.isnan(loss[1]) and math.isnan(loss[2]) and loss[3] == 0.0
    assert np.isfinite(loss[[0, 4, 5]]).all()
    assert torch.count_nonzero(dz[1:4]).item() == 0
    assert int(f.n_valid.item()) == 5


def test_zero_rows_reduce():
    z = torch.empty(0, 10, device=DEV, dtype=torch.float32)
    t = torch.empty(0, dtype=torch.int64, device=DEV)
    f = vce.ce_forward(z, t, 0.0, True)
    torch.cuda.synchronize()
    assert int(f.n_valid.item()) == 0 and math.isnan(f.loss.item())


def test_layout_sq_b_v_matches_flattened():
    sq, b, vocab = 16, 3, 4099
    z = wk.normal_matrix(4, wk.TID_LOGITS, sq * b, vocab, 3.0, True)
    target = wk.uniform_targets(4, sq * b, vocab, 0.1)
    t3 = to_dev(z, "bf16").view(sq, b, vocab)
    tt = torch.from_numpy(target).to(DEV).view(sq, b)
    f3 = vce.ce_forward(t3, tt.reshape(-1), 0.1, False)
    f2 = vce.ce_forward(t3.view(-1, vocab), tt.reshape(-1), 0.1, False)
    torch.cuda.synchronize()
    assert f3.loss.shape == (sq, b)
    assert torch.equal(f3.loss.reshape(-1), f2.loss)


# ---------------------------------------------------------------------------
# full-size memory-bound workload: B=4, SQ=4096, V=128256 BF16, 5% ignored
# (the launch configuration the benchmark times); sampled rows + exact mean
# ---------------------------------------------------------------------------

def _oracle_rows_chunked(wl, target, rows_per_chunk=128):
    """Per-row FP64 oracle loss for every row of the workload (rows regenerated in chunks)."""
    n = wl.n_rows

    def chunk(r0):
        r1 = min(n, r0 + rows_per_chunk)
        z = wk.logits_rows(wl, np.arange(r0, r1))
        return oracle.ce_forward(z, target[r0:r1], wl.label_smoothing, False, dtype=wl.dtype)["loss_rows"]

    with ThreadPoolExecutor(16) as ex:
        parts = list(ex.map(chunk, range(0, n, rows_per_chunk)))
    return np.concatenate(parts)


def test_membound_full_size_sampled():
    wl = wk.LOGITS_MEMBOUND
    inp = wk.make_logits_inputs(wl)
    logits = to_dev(inp.logits, wl.dtype)
    del inp.logits
    f, dz = run_gpu(logits, inp.target, wl.label_smoothing, wl.reduce_loss, inp.grad)
    n_valid_ref = int((inp.target != -100).sum())
    assert int(f.n_valid.item()) == n_valid_ref
    assert int(f.dev_status.item()) == 0
    # mean over every row, in FP64
    loss_rows = _oracle_rows_chunked(wl, inp.target)
    mean_ref = oracle.mean_loss(loss_rows, n_valid_ref)
    assert abs(f.loss.item() - mean_ref) <= 2e-3
    # ignore mask of the gradient: every ignored row is exactly zero
    ign = torch.from_numpy(inp.target == -100).to(DEV)
    assert torch.count_nonzero(dz[ign]).item() == 0
    # sampled rows, compared element by element
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(wl.n_rows, 48, replace=False),
                                     np.nonzero(inp.target == -100)[0][:4], [0, wl.n_rows - 1]]))
    z = wk.logits_rows(wl, rows)
    ref = oracle.ce_forward(z, inp.target[rows], wl.label_smoothing, False, dtype=wl.dtype)
    ref_dz = oracle.ce_backward(z, inp.target[rows], ref["lse"], n_valid_ref, inp.grad,
                                wl.label_smoothing, True, dtype=wl.dtype)
    sel = torch.from_numpy(rows).to(DEV)
    check_rows(f._replace(stats=f.stats), dz[sel], ref, ref_dz, rows, wl.dtype, True, inp.target)


def test_logits_beyond_2_31_elements_sampled():
    # 17000 x 128257 BF16 logits: 2.18e9 elements, so the rows from 16744 on start
    # past element 2^31 (every row offset is 64-bit).  ce_forward + ce_backward into a
    # separate buffer, then the fused call in place over the logits; sampled rows
    # element by element, the mean over every row, N_v exactly.
    import dataclasses
    wl = dataclasses.replace(wk.LOGITS_MEMBOUND, name="logits_17000x128257", n_rows=17000, vocab=128257)
    assert wl.n_rows * wl.vocab > 2 ** 31
    inp = wk.make_logits_inputs(wl)
    logits = to_dev(inp.logits, wl.dtype)
    del inp.logits
    f, dz = run_gpu(logits, inp.target, wl.label_smoothing, wl.reduce_loss, inp.grad)
    n_valid_ref = int((inp.target != -100).sum())
    assert int(f.n_valid.item()) == n_valid_ref and int(f.dev_status.item()) == 0
    loss_rows = _oracle_rows_chunked(wl, inp.target)
    mean_ref = oracle.mean_loss(loss_rows, n_valid_ref)
    assert abs(f.loss.item() - mean_ref) <= 2e-3
    rng = np.random.default_rng(1)
    first_far = -(-(2 ** 31) // wl.vocab)  # the first row that starts past element 2^31
    rows = np.unique(np.concatenate([rng.choice(wl.n_rows, 16, replace=False),
                                     rng.choice(np.arange(first_far, wl.n_rows), 16, replace=False),
                                     [0, first_far - 1, first_far, wl.n_rows - 1]]))
    z = wk.logits_rows(wl, rows)
    ref = oracle.ce_forward(z, inp.target[rows], wl.label_smoothing, False, dtype=wl.dtype)
    ref_dz = oracle.ce_backward(z, inp.target[rows], ref["lse"], n_valid_ref, inp.grad,
                                wl.label_smoothing, True, dtype=wl.dtype)
    sel = torch.from_numpy(rows).to(DEV)
    check_rows(f, dz[sel], ref, ref_dz, rows, wl.dtype, True, inp.target)
    del dz
    r = run_fused(logits, inp.target, wl.label_smoothing, wl.reduce_loss, inp.grad, inplace=True)
    assert int(r.n_valid.item()) == n_valid_ref and int(r.dev_status.item()) == 0
    assert abs(r.loss.item() - mean_ref) <= 2e-3
    check_rows(r, r.dlogits[sel], ref, ref_dz, rows, wl.dtype, True, inp.target)


# ---------------------------------------------------------------------------
# fused forward + backward (ce_forward_backward)
# ---------------------------------------------------------------------------

def run_fused(logits, target, eps, red, grad, ignore_idx=-100, inplace=False):
    tgt = torch.from_numpy(target).to(DEV)
    g = torch.from_numpy(np.asarray(grad, np.float32)).to(DEV)
    r = vce.ce_forward_backward(logits, tgt, g, eps, red, ignore_idx, inplace=inplace)
    torch.cuda.synchronize()
    return r


def assert_fused_matches_separate(r, sep_f, sep_dz, target, dtype):
    """The fused call against ce_forward + ce_backward on the same data.  Where
    both use the same threads per row the results are bit-identical; for long
    rows the fused kernel may split a row's sum differently, so lse and the loss
    may differ by FP32 rounding, and the gradient by what that does to
    exp(z - lse) - eps/V (tensor-wise; single elements near p = eps/V cancel).
    Counts, row maxima and ignored rows are exact either way."""
    assert int(r.n_valid.item()) == int(sep_f.n_valid.item())
    st, ss = r.stats.double().cpu().numpy(), sep_f.stats.double().cpu().numpy()
    np.testing.assert_array_equal(st[:, 0], ss[:, 0])
    np.testing.assert_allclose(st[:, 1], ss[:, 1], rtol=2e-6, atol=1e-6)
    lf, ls = r.loss.double().cpu().numpy().reshape(-1), sep_f.loss.double().cpu().numpy().reshape(-1)
    np.testing.assert_allclose(lf, ls, rtol=2e-6, atol=2e-6)
    a = r.dlogits.float().cpu().numpy()
    b = sep_dz.float().cpu().numpy()
    ign = target == -100
    assert np.all(a[ign] == 0.0) and np.all(b[ign] == 0.0)
    tol = 1e-3 if dtype == "bf16" else 1e-5
    assert np.linalg.norm(a - b) <= tol * np.linalg.norm(b) + 1e-30


@pytest.mark.parametrize("vocab,dtype", [(5003, "bf16"), (30000, "bf16"), (100000, "bf16"), (130001, "bf16"),
                                         (190000, "bf16"), (210000, "bf16"), (9001, "f32"), (25000, "f32"),
                                         (60001, "f32")])
def test_fused_bit_identical_where_threads_match(vocab, dtype):
    # Rows the fused call gives the forward kernel's own thread count: up to
    # 16 KiB (128 threads), BF16 48-64 KiB and FP32 16-56 KiB (8 ring warps = 256
    # threads), BF16 112-448 KiB and FP32 64-400 KiB (16 ring warps = 512
    # threads).  Each thread then takes the same elements in the same order as
    # in ce_forward, and the second pass is ce_backward's arithmetic: every
    # output bit matches.
    n = 300
    z = wk.normal_matrix(vocab, wk.TID_LOGITS, n, vocab, 3.0, dtype == "bf16")
    target = wk.uniform_targets(vocab, n, vocab, 0.1)
    # targets in the first and last columns too: on rows off 16-byte alignment
    # they fall among the scalar head and tail elements
    target[1::9], target[2::9], target[3::9] = 0, 1, vocab - 1
    logits = to_dev(z, dtype)
    grad = np.ones(1, np.float32)
    f, dz = run_gpu(logits, target, 0.1, True, grad)
    r = run_fused(logits, target, 0.1, True, grad)
    assert torch.equal(r.stats, f.stats) and torch.equal(r.loss, f.loss)
    assert int(r.n_valid.item()) == int(f.n_valid.item())
    assert torch.equal(r.dlogits.view(torch.int16), dz.view(torch.int16))


@pytest.mark.parametrize("n,vocab,dtype", [(20000, 2000, "bf16"), (17000, 9001, "f32")])
def test_fused_mean_bit_identical_many_rows(n, vocab, dtype):
    # More rows than the mean kernel's 1024 threads x 8 rows per step: the fused
    # call's mean (N_v counted before its pass) groups and compensates each
    # thread's rows exactly as ce_forward's mean does, so the loss matches bit for
    # bit where the rows do (short rows here; FP32 16-56 KiB rows on the ring)
    z = wk.normal_matrix(n + vocab, wk.TID_LOGITS, n, vocab, 3.0, dtype == "bf16")
    target = wk.uniform_targets(n + vocab, n, vocab, 0.1)
    logits = to_dev(z, dtype)
    grad = np.ones(1, np.float32)
    f, dz = run_gpu(logits, target, 0.1, True, grad)
    r = run_fused(logits, target, 0.1, True, grad)
    assert int(r.n_valid.item()) == int(f.n_valid.item())
    assert torch.equal(r.stats, f.stats)
    assert torch.equal(r.loss.view(torch.int32), f.loss.view(torch.int32))


FUSED = [
    # n, vocab, dtype, eps, reduce, inplace
    (128, 1024, "f32", 0.0, False, False),
    (128, 1024, "f32", 0.1, True, True),
    (5, 7, "bf16", 0.1, True, False),
    (300, 50257, "bf16", 0.1, True, True),
    (33, 32001, "f32", 0.0, False, True),
    (6, 262144, "bf16", 0.0, True, False),
    (64, 4099, "bf16", 0.1, 2, True),
    (40, 49152, "bf16", 0.1, True, False),
    (25, 98304, "f32", 0.0, 2, True),
    (130, 128256, "bf16", 0.0, False, True),
    # several rows per persistent CTA on every shape of the TMA-fed ring kernel
    # (rows above 16 KiB): one CTA per SM with a 224 KiB ring (bf16 128 KiB rows) or
    # a 192 KiB ring (bf16 293 KiB rows, f32 196 and 78 KiB rows), longer rows
    # split over the two CTAs of a cluster (f32 512 KiB rows), two CTAs per SM with
    # 112 KiB rings (bf16 78 and 59 KiB rows) or 96 KiB rings (bf16 102 KiB rows,
    # f32 35 KiB rows), and four with 48 KiB rings (bf16 39 and 23 KiB rows)
    (500, 65536, "bf16", 0.0, 2, True),
    (400, 150001, "bf16", 0.1, True, False),
    (300, 50257, "f32", 0.1, True, True),
    (400, 131072, "f32", 0.1, True, False),
    (700, 40000, "bf16", 0.1, True, True),
    (400, 30000, "bf16", 0.1, True, False),
    (900, 52000, "bf16", 0.0, 2, False),
    (600, 9001, "f32", 0.1, True, True),
    (333, 20001, "f32", 0.0, False, False),
    (1000, 20000, "bf16", 0.1, True, False),
    (1500, 12000, "bf16", 0.0, 2, True),
    # several rows per CTA with the next-row prefetch on the 128-thread path
    (3000, 1000, "bf16", 0.0, 2, True),
]


@pytest.mark.parametrize("n,vocab,dtype,eps,red,inplace", FUSED)
def test_fused_matches_oracle_and_separate_path(n, vocab, dtype, eps, red, inplace):
    seed = 3 * n + vocab
    z = wk.normal_matrix(seed, wk.TID_LOGITS, n, vocab, 3.0, dtype == "bf16")
    target = wk.uniform_targets(seed, n, vocab, 0.1)
    grad = np.full(1, 1.5, np.float32) if red else wk.grad_rows(seed, n)
    a = to_dev(z, dtype)
    sep_f, sep_dz = run_gpu(a, target, eps, red, grad)
    b = to_dev(z, dtype)
    r = run_fused(b, target, eps, red, grad, inplace=inplace)
    if inplace:
        assert r.dlogits.data_ptr() == b.data_ptr()
    assert_fused_matches_separate(r, sep_f, sep_dz, target, dtype)
    ref = oracle.ce_forward(z, target, eps, red, dtype=dtype)
    ref_dz = oracle.ce_backward(z, target, ref["lse"], ref["n_valid"], grad, eps, red, dtype=dtype)
    check_rows(r, r.dlogits, ref, ref_dz, np.arange(n), dtype, red, target)


@pytest.mark.parametrize("n,vocab,pad,dtype,eps,red", [
    (200, 50001, 3, "bf16", 0.1, True),   # ring kernel, two CTAs per SM, 96 KiB rings, rows off 16-byte alignment
    (300, 40001, 5, "bf16", 0.1, True),   # ring kernel, two CTAs per SM, 112 KiB rings
    (400, 70001, 7, "bf16", 0.0, 2),      # ring kernel, one CTA per SM, 224 KiB ring, rows off 16-byte alignment
    (100, 150001, 3, "bf16", 0.0, False), # ring kernel, one CTA per SM, 192 KiB ring
    (160, 240003, 3, "bf16", 0.1, True),  # rows split over a cluster pair, rows off alignment
    (400, 12001, 1, "bf16", 0.0, 2),      # ring kernel, four CTAs per SM
    (150, 9001, 5, "f32", 0.0, False),    # ring kernel, FP32, two CTAs per SM, 96 KiB rings
    (300, 129, 1, "bf16", 0.1, 2),        # 128 threads per row
])
def test_fused_padded_rows(n, vocab, pad, dtype, eps, red):
    seed = 5 * n + vocab
    stride = vocab + pad
    full = wk.normal_matrix(seed, wk.TID_LOGITS, n, stride, 3.0, dtype == "bf16")
    target = wk.uniform_targets(seed, n, vocab, 0.1)
    grad = np.full(1, 0.5, np.float32) if red else wk.grad_rows(seed, n)
    dev_full = to_dev(full, dtype)
    sep_f, sep_dz = run_gpu(dev_full[:, :vocab], target, eps, red, grad,
                            dlogits=torch.empty_like(dev_full)[:, :vocab])
    dz_full = torch.full_like(dev_full, 7.0)
    tgt = torch.from_numpy(target).to(DEV)
    g = torch.from_numpy(np.asarray(grad, np.float32)).to(DEV)
    r = vce.ce_forward_backward(dev_full[:, :vocab], tgt, g, eps, red, dlogits=dz_full[:, :vocab])
    torch.cuda.synchronize()
    assert_fused_matches_separate(r, sep_f, sep_dz, target, dtype)
    assert torch.all(dz_full[:, vocab:] == 7.0).item()
    z = full[:, :vocab]
    ref = oracle.ce_forward(z, target, eps, red, dtype=dtype)
    ref_dz = oracle.ce_backward(z, target, ref["lse"], ref["n_valid"], grad, eps, red, dtype=dtype)
    check_rows(r, r.dlogits, ref, ref_dz, np.arange(n), dtype, red, target)


@pytest.mark.parametrize("vocab,dtype,n", [(40000, "bf16", 1000), (70001, "bf16", 1000), (33000, "f32", 1000),
                                           (20003, "bf16", 1000), (210001, "bf16", 400)])
def test_fused_ring_bad_and_ignored_rows(vocab, dtype, n):
    """Rows whose target is out of range get one pass through the ring kernel (their
    statistics) and a zero gradient, ignored rows none; the producer and the compute
    warps must agree on that sequence for every later row to be right (for the
    longest rows also the two CTAs of a cluster pair, which exchange the partials
    of every row that is not ignored, bad rows included)."""
    seed = 11 + vocab
    z = wk.normal_matrix(seed, wk.TID_LOGITS, n, vocab, 3.0, dtype == "bf16")
    target = wk.uniform_targets(seed, n, vocab, 0.1)
    target[5::97] = vocab          # out of range above
    target[50::131] = -7           # out of range below
    grad = wk.grad_rows(seed, n)
    r = run_fused(to_dev(z, dtype), target, 0.1, False, grad)
    bad = (target == vocab) | (target == -7)
    assert int(r.dev_status.item()) & vce.DEVSTATUS_BAD_TARGET
    loss = r.loss.double().cpu().numpy()
    assert np.all(np.isnan(loss[bad])) and np.all(np.isfinite(loss[~bad]))
    dz = r.dlogits.float().cpu().numpy()
    assert np.all(dz[bad] == 0.0)
    good = ~bad
    ref = oracle.ce_forward(z[good], target[good], 0.1, False, dtype=dtype)
    ref_dz = oracle.ce_backward(z[good], target[good], ref["lse"], ref["n_valid"], grad[good], 0.1, False,
                                dtype=dtype)
    rows = np.nonzero(good)[0]
    sub = r._replace(loss=r.loss[torch.from_numpy(rows).to(DEV)], stats=r.stats[torch.from_numpy(rows).to(DEV)])
    check_rows(sub, r.dlogits[torch.from_numpy(rows).to(DEV)], ref, ref_dz, np.arange(len(rows)), dtype, False,
               target[good])
    # the statistics of a bad row are still those of its logits
    bad_rows = np.nonzero(bad)[0]
    ref_bad = oracle.ce_forward(z[bad_rows], np.zeros(len(bad_rows), np.int64), 0.1, False, dtype=dtype)
    st = r.stats.double().cpu().numpy()[bad_rows]
    np.testing.assert_array_equal(st[:, 0], ref_bad["m"])
    np.testing.assert_allclose(st[:, 1], ref_bad["lse"], rtol=1e-5 if dtype == "f32" else 0.0,
                               atol=0.0 if dtype == "f32" else 2e-3)


def test_fused_membound_full_size_inplace():
    wl = wk.LOGITS_MEMBOUND
    inp = wk.make_logits_inputs(wl)
    logits = to_dev(inp.logits, wl.dtype)
    del inp.logits
    r = run_fused(logits, inp.target, wl.label_smoothing, wl.reduce_loss, inp.grad, inplace=True)
    n_valid_ref = int((inp.target != -100).sum())
    assert int(r.n_valid.item()) == n_valid_ref and int(r.dev_status.item()) == 0
    loss_rows = _oracle_rows_chunked(wl, inp.target)
    assert abs(r.loss.item() - oracle.mean_loss(loss_rows, n_valid_ref)) <= 2e-3
    ign = torch.from_numpy(inp.target == -100).to(DEV)
    assert torch.count_nonzero(r.dlogits[ign]).item() == 0
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([rng.choice(wl.n_rows, 32, replace=False), [0, wl.n_rows - 1]]))
    z = wk.logits_rows(wl, rows)
    ref = oracle.ce_forward(z, inp.target[rows], wl.label_smoothing, False, dtype=wl.dtype)
    ref_dz = oracle.ce_backward(z, inp.target[rows], ref["lse"], n_valid_ref, inp.grad,
                                wl.label_smoothing, True, dtype=wl.dtype)
    sel = torch.from_numpy(rows).to(DEV)
    check_rows(r, r.dlogits[sel], ref, ref_dz, rows, wl.dtype, True, inp.target)
