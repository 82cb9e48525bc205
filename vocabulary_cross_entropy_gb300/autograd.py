"""torch.autograd front ends over the C ABI (marshalling only: every step runs in
libvce.so's kernels).

parallel_cross_entropy  the logits form, with the call shape of Transformer
                        Engine's parallel_cross_entropy (API card "Signature")
                        minus the process group; ``overwrite_input`` is the
                        pull request's destructive mode (backward writes the
                        gradient over the saved logits).
linear_cross_entropy    the linear form, loss from embeddings [..., H] and the
                        classifier [V, H] (Cut Cross-Entropy card
                        "what_it_does"), with optional token shifting and
                        per-token entropy.
"""
from __future__ import annotations

import torch

from . import _binding as b


def _grad_tensor(grad, reduce_code, n, device):
    if reduce_code:
        return grad.reshape(1).to(device=device, dtype=torch.float32)
    return grad.reshape(n).to(device=device, dtype=torch.float32).contiguous()


class _LogitsCE(torch.autograd.Function):
    @staticmethod
    def forward(ctx, inp, target, label_smoothing, reduce_code, ignore_idx, overwrite_input):
        flat_t = target.reshape(-1).contiguous()
        f = b.ce_forward(inp, flat_t, label_smoothing, reduce_code, ignore_idx)
        ctx.save_for_backward(inp, flat_t, f.stats, f.n_valid)
        ctx.args = (label_smoothing, reduce_code, ignore_idx, overwrite_input)
        return f.loss.reshape(()) if reduce_code else f.loss.reshape(target.shape)

    @staticmethod
    def backward(ctx, grad):
        inp, flat_t, stats, n_valid = ctx.saved_tensors
        eps, reduce_code, ignore_idx, overwrite = ctx.args
        g = _grad_tensor(grad, reduce_code, flat_t.numel(), inp.device)
        dz = b.ce_backward(inp, flat_t, stats, n_valid, g, eps, reduce_code, ignore_idx, inplace=overwrite)
        return dz.detach(), None, None, None, None, None


def parallel_cross_entropy(inp, target, label_smoothing: float = 0.0, reduce_loss: bool = False,
                           dist_process_group=None, ignore_idx: int = -100, is_cg_capturable: bool = False,
                           overwrite_input: bool = False):
    """Cross entropy of logits ``inp`` (B, SQ, V) or (SQ, B, V) against ``target``.

    Returns the mean over non-ignored tokens when ``reduce_loss``, else the per-token
    loss shaped like ``target``.  Every call is CUDA-graph capturable, so
    ``is_cg_capturable`` has no effect.  With ``overwrite_input`` the backward writes
    the gradient over ``inp`` (no extra buffer); ``inp`` must not be used afterwards.
    """
    if dist_process_group is not None:
        raise NotImplementedError("vocabulary-parallel process groups are not supported: one GPU")
    del is_cg_capturable
    code = b._reduce(reduce_loss)
    return _LogitsCE.apply(inp, target, float(label_smoothing), code, int(ignore_idx), bool(overwrite_input))


class _LinearCE(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w, target, label_smoothing, reduce_code, ignore_idx, want_entropy):
        f = b.lce_forward(x, w, target, label_smoothing, reduce_code, ignore_idx, entropy=want_entropy)
        ctx.save_for_backward(x, w, target, f.lse, f.n_valid)
        ctx.args = (label_smoothing, reduce_code, ignore_idx)
        loss = f.loss.reshape(()) if reduce_code else f.loss
        if want_entropy:
            ctx.mark_non_differentiable(f.entropy)
            return loss, f.entropy
        return loss

    @staticmethod
    def backward(ctx, grad, *unused):
        x, w, target, lse, n_valid = ctx.saved_tensors
        eps, reduce_code, ignore_idx = ctx.args
        g = _grad_tensor(grad, reduce_code, target.numel(), x.device)
        r = b.lce_backward(x, w, target, lse, n_valid, g, eps, reduce_code, ignore_idx)
        return r.dX, r.dW, None, None, None, None, None


def linear_cross_entropy(embeddings, classifier, labels, ignore_index: int = -100, reduction: str = "mean",
                         label_smoothing: float = 0.0, shift: bool = False, return_entropy: bool = False):
    """Cross entropy of ``embeddings @ classifier.T`` against ``labels`` without the logits.

    embeddings [..., H] and classifier [V, H] are BF16; labels [...] int64.  ``reduction``
    is 'mean' (over non-ignored tokens), 'sum' or 'none'.  ``shift`` scores position t
    of each sequence (the last dimension of ``labels``) against label t + 1.  With
    ``return_entropy`` the per-token entropy of the softmax is returned as well.
    """
    lead = embeddings.shape[:-1]
    h = embeddings.shape[-1]
    x = embeddings.reshape(-1, h)
    if not x.is_contiguous():
        x = x.contiguous()
    flat = labels.reshape(-1).contiguous()
    if shift:
        flat = b.shift_targets(flat, labels.shape[-1], ignore_index)
    code = b._reduce(reduction)
    out = _LinearCE.apply(x, classifier, flat, float(label_smoothing), code, int(ignore_index),
                          bool(return_entropy))
    loss, ent = (out if return_entropy else (out, None))
    if code == b.REDUCE_NONE:
        loss = loss.reshape(lead)
    if return_entropy:
        return loss, ent.reshape(lead)
    return loss
