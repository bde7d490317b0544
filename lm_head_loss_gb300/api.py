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


def _check_out(out, H: torch.Tensor, W: torch.Tensor):
    """`out` = (loss, lse, dH, dW) written by the kernels: fp32, contiguous, on
    H's device, with the shapes the call writes (the library sees only
    pointers, so a smaller buffer would be written past its end)."""
    if len(out) != 4:
        raise ValueError("out must be (loss, lse, dH, dW)")
    n, d, v = H.shape[0], H.shape[1], W.shape[0]
    for t, shape, name in zip(out, ((), (n,), (n, d), (v, d)), ("loss", "lse", "dH", "dW")):
        ok_shape = t.numel() == 1 if name == "loss" else tuple(t.shape) == shape
        if (not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not ok_shape or t.device != H.device
                or not t.is_contiguous()):
            raise ValueError(f"out {name} must be a contiguous fp32 tensor of shape {shape} on {H.device}")


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
        _check_out(out, H, W)
        loss, lse, dH, dW = out
    st = B.flce_forward_backward(prob, H, W, y, grad_loss, lse, loss, dH, dW, ws, stream=stream)
    if st != B.Status.OK:
        raise B.FlceError(st, "flce_forward_backward")
    return loss, lse, dH, dW


def adamw_hparams(lr: float, step: int, betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 0.01,
                  device=None) -> torch.Tensor:
    """One step's flce_adamw_hparams in device memory (a uint8 tensor)."""
    raw = B.adamw_hparams_bytes(lr, betas[0], betas[1], eps, weight_decay, step)
    return torch.frombuffer(bytearray(raw), dtype=torch.uint8).to(device if device is not None else "cuda")


def forward_backward_adamw(H, W, y, w_master, adam_m, adam_v, w_out, hparams: torch.Tensor, grad_loss: float = 1.0,
                           ignore_index: int = -100, filter_eps: float = 0.0, flags: int = 0,
                           workspace: Workspace | None = None, stream=None):
    """Loss, LSE [N] and dH [N,D]; W's AdamW step is applied on the way.

    w_master, adam_m and adam_v (fp32 [V,D]) are updated in place and w_out
    (bf16 [V,D], not W itself) receives the new weights; dW is never formed.
    hparams comes from adamw_hparams."""
    _check_inputs(H, W, y)
    for t, dt in ((w_master, torch.float32), (adam_m, torch.float32), (adam_v, torch.float32),
                  (w_out, torch.bfloat16)):
        if t.dtype != dt or t.shape != W.shape or not t.is_cuda or not t.is_contiguous():
            raise ValueError("w_master, adam_m, adam_v must be fp32 and w_out bf16, all contiguous [V,D] on the GPU")
    prob = _problem(H, W, ignore_index, filter_eps, flags)
    ws = (workspace or Workspace(H.device)).get(prob)
    lse = torch.empty(H.shape[0], dtype=torch.float32, device=H.device)
    loss = torch.empty((), dtype=torch.float32, device=H.device)
    dH = torch.empty(H.shape, dtype=torch.float32, device=H.device)
    st = B.flce_forward_backward_adamw(prob, H, W, y, grad_loss, lse, loss, dH, w_master, adam_m, adam_v, w_out,
                                       hparams, ws, stream=stream)
    if st != B.Status.OK:
        raise B.FlceError(st, "flce_forward_backward_adamw")
    return loss, lse, dH


class FusedAdamWHead:
    """An LM-head weight trained with AdamW fused into its gradient.

    Keeps the fp32 master weights, the two moments and two bf16 copies of
    the weights: each step reads one copy and writes the other (the call may
    not update the W it is reading), and `weight` is the current one."""

    def __init__(self, weight: torch.Tensor, lr: float = 1e-3, betas=(0.9, 0.999), eps: float = 1e-8,
                 weight_decay: float = 0.01):
        if weight.dim() != 2 or not weight.is_cuda:
            raise ValueError("weight must be a CUDA [V,D] tensor")
        self.master = weight.detach().to(torch.float32).contiguous().clone()
        self.m = torch.zeros_like(self.master)
        self.v = torch.zeros_like(self.master)
        self._w = [self.master.to(torch.bfloat16), torch.empty_like(self.master, dtype=torch.bfloat16)]
        self._cur = 0
        self.lr, self.betas, self.eps, self.weight_decay = lr, betas, eps, weight_decay
        self.steps = 0
        self.workspace = Workspace(weight.device)

    @property
    def weight(self) -> torch.Tensor:
        return self._w[self._cur]

    def step(self, H, y, grad_loss: float = 1.0, ignore_index: int = -100, filter_eps: float = 0.0, flags: int = 0):
        """One forward + backward + AdamW step on a batch; returns loss, LSE and dH."""
        self.steps += 1
        hp = adamw_hparams(self.lr, self.steps, self.betas, self.eps, self.weight_decay, self.master.device)
        out = forward_backward_adamw(H, self._w[self._cur], y, self.master, self.m, self.v, self._w[1 - self._cur],
                                     hp, grad_loss, ignore_index, filter_eps, flags, self.workspace)
        self._cur = 1 - self._cur
        return out


def device_status(workspace: Workspace, stream=None) -> B.Status:
    """Synchronise and return (and clear) the device status of the last call."""
    return B.flce_get_device_status(workspace.buf, stream)
