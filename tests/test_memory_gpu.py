"""Peak device memory of one forward + backward: the caller-visible workspace, the
saved statistics and a few words, never an N x V FP32 logits or gradient buffer
(Liger PR "Memory" tables; TE PR "Changes": the backward rebuilds the gradient
from saved statistics and may write it over the logits).

Measured as the rise of torch.cuda.max_memory_allocated around the calls, with the
inputs, weights and final outputs allocated beforehand, as bench.py reports it."""
import pytest
import torch

import vocabulary_cross_entropy_gb300 as vce

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
MiB = 1 << 20


def _peak_rise(fn):
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    fn()
    torch.cuda.synchronize()
    return torch.cuda.max_memory_allocated() - base


@pytest.mark.parametrize("max_slab_bytes", [vce.SLAB_UNCAPPED, 0, 64 * MiB])
def test_linear_headline_extra_memory(max_slab_bytes):
    # one slab over the whole vocabulary, the default 256 MiB cap, a 64 MiB cap
    n, h, v = 4096, 4096, 131072
    g = torch.Generator(device=DEV).manual_seed(7)
    x = torch.randn(n, h, device=DEV, generator=g).to(torch.bfloat16)
    w = (torch.randn(v, h, device=DEV, generator=g) * h ** -0.5).to(torch.bfloat16)
    y = torch.randint(0, v, (n,), device=DEV, generator=g)
    dx, dw = torch.empty_like(x), torch.empty_like(w)
    loss, grad = torch.empty(1, device=DEV), torch.ones(1, device=DEV)
    ws_bytes = vce.lce_workspace_size(n, h, v, True, max_slab_bytes)

    def step():
        f = vce.lce_forward(x, w, y, 0.0, True, loss=loss, max_slab_bytes=max_slab_bytes)
        r = vce.lce_backward(x, w, y, f.lse, f.n_valid, grad, 0.0, True, dX=dx, dW=dw,
                             max_slab_bytes=max_slab_bytes)
        assert int(f.dev_status.item()) == 0 and int(r.dev_status.item()) == 0

    rise = _peak_rise(step)
    # one workspace per call (forward and backward each allocate theirs on demand),
    # plus lse [N] and a few words; the caching allocator rounds each block up
    assert rise <= 2 * ws_bytes + n * 4 + 4 * MiB, (rise, ws_bytes)
    assert rise < n * v * 4
    if max_slab_bytes != vce.SLAB_UNCAPPED:
        # the dZ slab cap bounds the workspace (slab + at most four FP32 dX partials),
        # and with it the extra memory: below even one BF16 copy of the logits
        cap = max_slab_bytes or vce.DEFAULT_SLAB_BYTES
        assert ws_bytes <= cap + 4 * n * h * 4
        assert rise < n * v * 2
    assert torch.isfinite(loss).all()


def test_logits_inplace_backward_extra_memory():
    n, v = 4096, 128256
    g = torch.Generator(device=DEV).manual_seed(8)
    z = (torch.randn(n, v, device=DEV, generator=g) * 3).to(torch.bfloat16)
    y = torch.randint(0, v, (n,), device=DEV, generator=g)
    grad = torch.ones(1, device=DEV)
    loss = torch.empty(1, device=DEV)

    def separate():
        f = vce.ce_forward(z, y, 0.1, True, loss=loss)
        dz = vce.ce_backward(z, y, f.stats, f.n_valid, grad, 0.1, True, inplace=True)
        assert dz.data_ptr() == z.data_ptr()

    rise = _peak_rise(separate)
    small = vce.ce_workspace_size(n, v, True) + n * 2 * 4 + 2 * MiB
    assert rise <= small, rise

    z2 = (torch.randn(n, v, device=DEV, generator=g) * 3).to(torch.bfloat16)

    def fused():
        r = vce.ce_forward_backward(z2, y, grad, 0.1, True, inplace=True, loss=loss)
        assert r.dlogits.data_ptr() == z2.data_ptr()

    rise = _peak_rise(fused)
    assert rise <= small, rise
    assert torch.isfinite(loss).all()
