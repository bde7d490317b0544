"""PyTorch autograd wrapper over the general C entry points.

`linear_cross_entropy(hidden, weight, target, bias=None, ignore_index=-100,
reduction="mean")` mirrors the functional form of the PyTorch 2.13 chapter
(F.linear_cross_entropy with linear_bias, ignore_index and reduction), with
the fused GB300 kernels underneath:
  forward   flce_forward_ex: per-row LSE and the reduced (or per-row) loss;
            the LSE is saved, no logits are kept;
  backward  flce_backward_ex with the upstream gradient as a device tensor:
            recomputes the logits and returns dH, dW and d(bias).
Forward plus backward cost the same 8*N*V*D FLOPs as the one-call
flce_forward_backward. Because nothing is precomputed, the backward may run
more than once (retain_graph) and works for every reduction, "none"
included. Gradients come out in fp32; autograd casts them to the dtype of a
bf16 leaf. Every call of a device shares one cached workspace, so calls that
overlap on different streams must be serialised by the caller.
"""

from __future__ import annotations

import torch

from . import _binding as B
from .api import Workspace, _check_inputs

_WORKSPACES: dict = {}


def _workspace(device: torch.device) -> Workspace:
    key = (device.type, device.index if device.index is not None else torch.cuda.current_device())
    ws = _WORKSPACES.get(key)
    if ws is None:
        ws = _WORKSPACES[key] = Workspace(torch.device("cuda", key[1]))
    return ws


class _LinearCrossEntropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden, weight, bias, target, ignore_index, reduction, filter_eps, flags):
        _check_inputs(hidden, weight, target)
        if bias is not None:
            if bias.dtype != torch.float32 or not bias.is_cuda or bias.shape != (weight.shape[0],):
                raise ValueError("bias must be a CUDA float32 tensor of shape [V]")
            bias = bias.contiguous()
        red = B.REDUCTIONS[reduction]
        n, d, v = hidden.shape[0], hidden.shape[1], weight.shape[0]
        prob = B.make_problem(n, d, v, ignore_index, filter_eps, flags)
        ws = _workspace(hidden.device)
        buf = ws.get(prob)
        lse = torch.empty(n, dtype=torch.float32, device=hidden.device)
        loss = torch.empty((n,) if red == B.REDUCTIONS["none"] else (), dtype=torch.float32, device=hidden.device)
        st = B.flce_forward_ex(prob, red, hidden, weight, bias, target, lse, loss, buf)
        if st != B.Status.OK:
            raise B.FlceError(st, "flce_forward_ex")
        ctx.save_for_backward(hidden, weight, bias, target, lse)
        ctx.red, ctx.ignore_index, ctx.filter_eps, ctx.flags = red, ignore_index, filter_eps, flags
        ctx.mark_non_differentiable(lse)
        return loss, lse

    @staticmethod
    def backward(ctx, grad_loss, grad_lse):
        hidden, weight, bias, target, lse = ctx.saved_tensors
        n, d, v = hidden.shape[0], hidden.shape[1], weight.shape[0]
        prob = B.make_problem(n, d, v, ctx.ignore_index, ctx.filter_eps, ctx.flags)
        buf = _workspace(hidden.device).get(prob)
        grad = grad_loss.to(torch.float32).contiguous().reshape(-1)
        dH = torch.empty(hidden.shape, dtype=torch.float32, device=hidden.device)
        dW = torch.empty(weight.shape, dtype=torch.float32, device=hidden.device)
        db = torch.empty(v, dtype=torch.float32, device=hidden.device) if bias is not None else None
        st = B.flce_backward_ex(prob, ctx.red, hidden, weight, bias, target, lse, grad, dH, dW, db, buf)
        if st != B.Status.OK:
            raise B.FlceError(st, "flce_backward_ex")
        return dH, dW, db, None, None, None, None, None


def linear_cross_entropy(hidden: torch.Tensor, weight: torch.Tensor, target: torch.Tensor,
                         bias: torch.Tensor | None = None, ignore_index: int = -100, reduction: str = "mean",
                         filter_eps: float = 0.0, return_lse: bool = False, sort_vocab: bool = False):
    """Cross-entropy of the logits hidden @ weight.T (+ bias) against target.

    hidden [N,D] and weight [V,D] are CUDA bf16; target [N] is int64; bias is
    an optional CUDA fp32 [V]. reduction is "mean" (over non-ignored rows,
    the count clamped to one), "sum" or "none" (a loss per row, 0 on ignored
    rows). With filter_eps > 0 the backward leaves out 128x256 gradient tiles
    whose every |softmax - onehot| is below it; sort_vocab = True makes the
    backward visit the vocabulary by decreasing average logit, which groups
    the negligible columns into tiles the filter can leave out (Cut
    Cross-Entropy, Sec. 4.3 "Vocabulary sorting").
    """
    if reduction not in B.REDUCTIONS:
        raise ValueError(f"reduction must be one of {sorted(B.REDUCTIONS)}")
    flags = B.FLAG_SORT_VOCAB if sort_vocab else 0
    loss, lse = _LinearCrossEntropy.apply(hidden, weight, bias, target, ignore_index, reduction, filter_eps, flags)
    return (loss, lse) if return_lse else loss


class FusedLinearCrossEntropy(torch.nn.Module):
    """Module form: holds the reduction options; the LM-head weight (and
    bias) are passed in, so a tied embedding or an existing lm_head keeps its
    parameter."""

    def __init__(self, ignore_index: int = -100, reduction: str = "mean", filter_eps: float = 0.0,
                 sort_vocab: bool = False):
        super().__init__()
        if reduction not in B.REDUCTIONS:
            raise ValueError(f"reduction must be one of {sorted(B.REDUCTIONS)}")
        self.ignore_index, self.reduction, self.filter_eps = ignore_index, reduction, filter_eps
        self.sort_vocab = sort_vocab

    def forward(self, hidden, weight, target, bias=None):
        return linear_cross_entropy(hidden, weight, target, bias, self.ignore_index, self.reduction,
                                    self.filter_eps, sort_vocab=self.sort_vocab)
