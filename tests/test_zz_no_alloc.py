"""flce_forward_static_scratch: the forward for callers that cannot allocate.

Some callers have no way to give the library a workspace when they need the
loss: a plugin of an inference or training engine whose execute step is not
allowed to allocate device memory, or code that fixed its memory budget at
start-up. This entry point serves them by keeping its scratch in a fixed
16 MiB array inside the library instead of asking for one. These tests call
it through the C-ABI and check it against flce_forward, the entry point with
a caller-provided workspace, on two calls in a row, with the tolerances the
other GPU tests use. The file is named to be collected last.
"""

import numpy as np
import pytest
import torch

import lm_head_loss_gb300 as flce
from gpu_common import LOSS_REL, LSE_ABS, small_inputs, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _with_workspace(prob, H, W, y):
    ws = torch.empty(flce.flce_workspace_bytes(prob), dtype=torch.uint8, device="cuda")
    lse = torch.empty(prob.n_rows, device="cuda")
    loss = torch.empty((), device="cuda")
    assert flce.flce_forward(prob, H, W, y, lse, loss, ws) == flce.Status.OK
    assert flce.flce_get_device_status(ws) == flce.Status.OK
    return loss.item(), lse.cpu().numpy()


def _static(prob, H, W, y):
    lse = torch.full((prob.n_rows,), float("nan"), device="cuda")
    loss = torch.full((), float("nan"), device="cuda")
    assert flce.flce_forward_static_scratch(prob, H, W, y, lse, loss) == flce.Status.OK
    torch.cuda.synchronize()
    return loss.item(), lse.cpu().numpy()


@pytest.mark.parametrize("n,d,v", [(1000, 256, 50000), (20000, 128, 151552)])
def test_static_scratch_matches_workspace_forward_twice(n, d, v):
    # The second shape needs several row chunks to fit the 16 MiB scratch.
    inp = small_inputs(n, d, v, seed=21 + n, targets="zipf", ignore=0.05)
    H, W, y = to_device(inp)
    prob = flce.make_problem(n, d, v)
    ref_loss, ref_lse = _with_workspace(prob, H, W, y)
    for _ in range(2):
        loss, lse = _static(prob, H, W, y)
        assert abs(loss - ref_loss) <= LOSS_REL * abs(ref_loss)
        assert np.max(np.abs(lse - ref_lse)) <= LSE_ABS


def test_static_scratch_rejects_problems_beyond_its_size():
    H = torch.zeros(16, 8, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(1, 8, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(16, dtype=torch.int64, device="cuda")
    lse = torch.empty(16, device="cuda")
    loss = torch.empty((), device="cuda")
    too_big = flce.make_problem(16, 8, 4_000_000)   # never launched: rejected on the host
    assert flce.flce_forward_static_scratch(too_big, H, W, y, lse, loss) == flce.Status.ERR_UNSUPPORTED


def test_static_scratch_matches_the_oracle():
    import oracle
    inp = small_inputs(700, 128, 9000, seed=5, targets="zipf", ignore=0.05)
    H, W, y = to_device(inp)
    loss, lse = _static(flce.make_problem(700, 128, 9000), H, W, y)
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    r_lse, r_loss, _ = oracle.forward(H64, W64, inp["y"])
    assert abs(loss - r_loss) <= LOSS_REL * abs(r_loss)
    assert np.max(np.abs(lse - r_lse)) <= LSE_ABS


def test_static_scratch_reports_a_timed_out_forward_as_nan_loss():
    # With every bounded wait cut to about a microsecond the forward GEMM
    # gives up: with D = 4096 each tile's accumulator takes 64 k-blocks (over
    # 30,000 SM cycles) of MMAs, so the epilogue's first wait cannot end in
    # time. With no workspace to query, the NaN loss is the report. The next
    # call starts from a clean scratch and matches flce_forward.
    inp = small_inputs(512, 4096, 4096, seed=11)
    H, W, y = to_device(inp)
    loss, _ = _static(flce.make_problem(512, 4096, 4096, flags=flce.FLAG_TEST_SHORT_WAITS), H, W, y)
    assert np.isnan(loss)
    prob = flce.make_problem(512, 4096, 4096)
    ref_loss, ref_lse = _with_workspace(prob, H, W, y)
    loss, lse = _static(prob, H, W, y)
    assert abs(loss - ref_loss) <= LOSS_REL * abs(ref_loss)
    assert np.max(np.abs(lse - ref_lse)) <= LSE_ABS
