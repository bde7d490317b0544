"""Convenience layer over the C-ABI for PyTorch users.

PyTorch only provides device memory and the stream here: outputs and the
workspace are torch tensors, and every step of the loss and its gradient runs
in libflce.so. Status codes other than FLCE_OK raise FlceError.
"""

from __future__ import annotations

import torch

from . import _binding as B


def _check_inputs(H: torch.Tensor, W: torch.Tensor, y: torch.Tensor):
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("H and W must be torch.bfloat16")
    if y.dtype != torch.int64:
        raise TypeError("targets must be torch.int64")
    if not (H.is_cuda and W.is_cuda and y.is_cuda):
        raise ValueError("H, W and y must be CUDA tensors: the library has no CPU path")
    if H.dim() != 2 or W.dim() != 2 or y.dim() != 1:
        raise ValueError("expected H [N,D], W [V,D], y [N]")
    if H.shape[1] != W.shape[1] or H.shape[0] != y.shape[0]:
        raise ValueError("shape mismatch between H, W and y")
    if not (H.is_contiguous() and W.is_contiguous() and y.is_contiguous()):
        raise ValueError("H, W and y must be contiguous")


class Workspace:
    """A reusable device workspace (a torch uint8 buffer) grown on demand."""

    def __init__(self, device=None):
        self.device = torch.device(device if device is not None else "cuda")
        self.buf: torch.Tensor | None = None

    def get(self, problem: B.FlceProblem, forward_only: bool = False) -> torch.Tensor:
        need = B.flce_forward_workspace_bytes(problem) if forward_only else B.flce_workspace_bytes(problem)
        if need == 0:
            raise B.FlceError(B.Status.ERR_INVALID_ARGUMENT, "flce_workspace_bytes")
        if self.buf is None or self.buf.numel() < need:
            self.buf = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self.buf


def _problem(H, W, ignore_index, filter_eps, flags):
    return B.make_problem(H.shape[0], H.shape[1], W.shape[0], ignore_index, filter_eps, flags)


def forward(H, W, y, ignore_index: int = -100, workspace: Workspace | None = None, stream=None):
    """Mean loss (fp32 scalar tensor) and per-row LSE [N] (fp32)."""
    _check_inputs(H, W, y)
    prob = _problem(H, W, ignore_index, 0.0, 0)
    ws = (workspace or Workspace(H.device)).get(prob, forward_only=True)
    lse = torch.empty(H.shape[0], dtype=torch.float32, device=H.device)
    loss = torch.empty((), dtype=torch.float32, device=H.device)
    st = B.flce_forward(prob, H, W, y, lse, loss, ws, stream=stream)
    if st != B.Status.OK:
        raise B.FlceError(st, "flce_forward")
    return loss, lse


def forward_backward(H, W, y, grad_loss: float = 1.0, ignore_index: int = -100, filter_eps: float = 0.0,
                     workspace: Workspace | None = None, out=None, flags: int = 0, stream=None):
    """Loss, LSE [N], dH [N,D] and dW [V,D] (fp32) of the mean cross-entropy."""
    _check_inputs(H, W, y)
    prob = _problem(H, W, ignore_index, filter_eps, flags)
    ws = (workspace or Workspace(H.device)).get(prob)
    if out is None:
        lse = torch.empty(H.shape[0], dtype=torch.float32, device=H.device)
        loss = torch.empty((), dtype=torch.float32, device=H.device)
        dH = torch.empty(H.shape, dtype=torch.float32, device=H.device)
        dW = torch.empty(W.shape, dtype=torch.float32, device=H.device)
    else:
        loss, lse, dH, dW = out
    st = B.flce_forward_backward(prob, H, W, y, grad_loss, lse, loss, dH, dW, ws, stream=stream)
    if st != B.Status.OK:
        raise B.FlceError(st, "flce_forward_backward")
    return loss, lse, dH, dW


def device_status(workspace: Workspace, stream=None) -> B.Status:
    """Synchronise and return (and clear) the device status of the last call."""
    return B.flce_get_device_status(workspace.buf, stream)
