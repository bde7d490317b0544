"""Data parallelism over rows: one process per GPU, each holding its own token
rows (H, y) and the whole LM-head weight W.

The mean loss runs over the valid rows of every rank, so the count is global
and has to be known before a rank scales its gradient. One step exchanges
three sums over the ranks (all-reduce). The FORGE explainer states the first
of these needs, an all-reduce of the weight gradient under data parallelism.
The PyTorch 2.13 chapter lists sharding the LM head across devices as an open
item.

  1. count   each rank counts its valid rows (flce_count_valid); summed
  2. step    each rank runs flce_forward_backward_global with the summed
             count: its loss is its share of the global mean and its dW its
             contribution to the gradient of that mean
  3. loss, dW  summed; dH and the per-row LSE stay with the rank that owns
             the rows

`exchange_step` is that sequence with the local work and the all-reduce
passed in, so the same host logic runs over NCCL on GPUs and over gloo on
CPU ranks in the tests. `DataParallelStep` binds it to the library and
torch.distributed; every step of the loss itself runs in libflce.so.
"""

from __future__ import annotations

from typing import Callable

import torch

from . import _binding as B
from .api import _check_inputs


def exchange_step(local_count: Callable[[], torch.Tensor],
                  local_step: Callable[[torch.Tensor], tuple],
                  all_reduce_sum: Callable[[torch.Tensor], None]):
    """One data-parallel step on this rank.

    local_count() returns this rank's valid count (an int64 tensor [1]);
    local_step(count) runs the forward and backward with the mean over
    `count` and returns (loss share, lse, dH, dW); all_reduce_sum(t) sums t
    over the ranks in place. Returns (loss, lse, dH, dW, count) with loss,
    dW and count summed over the ranks."""
    count = local_count()
    all_reduce_sum(count)
    loss, lse, dH, dW = local_step(count)
    all_reduce_sum(loss)
    all_reduce_sum(dW)
    return loss, lse, dH, dW, count


def _all_reduce_sum(group):
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return lambda t: None

    def reduce(t: torch.Tensor) -> None:
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return reduce


class DataParallelStep:
    """The LM-head forward and backward of this rank's rows, with the mean
    and W's gradient taken over every rank of `group` (the default process
    group when None; a single process needs none).

    The output buffers and the workspace are allocated once, for batches of
    n_rows rows; each call returns views of them: the global mean loss ([1]),
    this rank's LSE [N] and dH [N,D], and the summed dW [V,D] (fp32)."""

    def __init__(self, n_rows: int, hidden: int, vocab: int, device=None, group=None, ignore_index: int = -100,
                 filter_eps: float = 0.0, flags: int = 0):
        self.device = torch.device(device if device is not None else "cuda")
        self.group = group
        self.problem = B.make_problem(n_rows, hidden, vocab, ignore_index, filter_eps, flags)
        nb = B.flce_workspace_bytes(self.problem)
        if nb == 0:
            raise B.FlceError(B.Status.ERR_INVALID_ARGUMENT, "flce_workspace_bytes")
        f32 = dict(dtype=torch.float32, device=self.device)
        self.ws = torch.empty(nb, dtype=torch.uint8, device=self.device)
        self.count = torch.zeros(1, dtype=torch.int64, device=self.device)
        self.loss = torch.zeros(1, **f32)
        self.lse = torch.empty(n_rows, **f32)
        self.dH = torch.empty(n_rows, hidden, **f32)
        self.dW = torch.empty(vocab, hidden, **f32)
        self._reduce = _all_reduce_sum(group)

    def __call__(self, H: torch.Tensor, W: torch.Tensor, y: torch.Tensor, grad_loss: float = 1.0):
        """Runs on torch's current stream, the stream torch.distributed's
        NCCL all-reduces order themselves with."""
        p = self.problem
        _check_inputs(H, W, y)
        if H.shape != (p.n_rows, p.hidden) or W.shape != (p.vocab, p.hidden) or y.shape != (p.n_rows,):
            raise ValueError("H, W, y do not match the shapes this step was built for")
        if not (H.device == W.device == y.device == self.ws.device):
            raise ValueError(f"H, W and y must be on {self.ws.device}, the device of this step's buffers")
        stream = torch.cuda.current_stream(self.device)

        def local_count():
            st = B.flce_count_valid(p, y, self.count, stream)
            if st != B.Status.OK:
                raise B.FlceError(st, "flce_count_valid")
            return self.count

        def local_step(count):
            st = B.flce_forward_backward_global(p, H, W, y, count, grad_loss, self.lse, self.loss, self.dH, self.dW,
                                                self.ws, stream=stream)
            if st != B.Status.OK:
                raise B.FlceError(st, "flce_forward_backward_global")
            return self.loss, self.lse, self.dH, self.dW

        return exchange_step(local_count, local_step, self._reduce)

    def device_status(self) -> B.Status:
        """Synchronise and return (and clear) the device status of the last step."""
        return B.flce_get_device_status(self.ws, torch.cuda.current_stream(self.device))
