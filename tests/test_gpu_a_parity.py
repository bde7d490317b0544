"""GPU parity of the C-ABI against the fp64 oracle on seeded inputs: the small
oracle workload, ragged tails in every dimension, several row and vocabulary
chunks, and the method's degenerate cases."""

import math

import numpy as np
import pytest
import torch

import lm_head_loss_gb300 as flce
import oracle
import synth
from gpu_common import (assert_parity, dh_filter_rows, errors, gpu_fwd, gpu_fwd_bwd, oracle_full, small_inputs,
                        to_device)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def test_tiny_workload_full_parity():
    inp = synth.make_inputs(synth.WORKLOADS["tiny"], seed=0)
    ref = oracle_full(inp)
    got = gpu_fwd_bwd(inp)
    assert got["status"] == flce.Status.OK
    e = assert_parity(got, ref)
    print("tiny", e)


def test_forward_only_matches():
    inp = synth.make_inputs(synth.WORKLOADS["tiny"], seed=1)
    ref = oracle_full(inp)
    got = gpu_fwd(inp)
    assert got["status"] == flce.Status.OK
    assert_parity(got, ref)


@pytest.mark.parametrize("n,d,v", [(1, 8, 1), (5, 8, 3), (129, 72, 257), (300, 136, 1000), (640, 264, 4099),
                                   (1000, 512, 2500)])
def test_ragged_shapes(n, d, v):
    inp = small_inputs(n, d, v, seed=n + d + v)
    ref = oracle_full(inp)
    got = gpu_fwd_bwd(inp)
    assert got["status"] == flce.Status.OK
    e = assert_parity(got, ref)
    print((n, d, v), e)


@pytest.mark.parametrize("n,d,v", [(200, 64, 1_000_003), (300, 16384, 3000)])
def test_extreme_shapes(n, d, v):
    # A vocabulary of a million ids (3907 logit tiles, over a hundred
    # vocabulary chunks) and a hidden size of 16384 (256 k-blocks per tile).
    inp = small_inputs(n, d, v, seed=n + v, targets="zipf", ignore=0.05)
    ref = oracle_full(inp)
    got = gpu_fwd_bwd(inp)
    assert got["status"] == flce.Status.OK
    e = assert_parity(got, ref)
    print((n, d, v), e)


def test_several_row_and_vocab_chunks():
    # 2 row chunks (8192 + 384 rows) x 3 vocabulary chunks (8192 + 8192 + 100).
    inp = small_inputs(8192 + 384, 64, 2 * 8192 + 100, seed=3, targets="zipf", ignore=0.1)
    ref = oracle_full(inp)
    got = gpu_fwd_bwd(inp)
    e = assert_parity(got, ref)
    print("chunks", e)


def test_bitwise_deterministic():
    inp = small_inputs(8192 + 384, 64, 2 * 8192 + 100, seed=4, targets="zipf")
    ws = flce.Workspace()
    a = gpu_fwd_bwd(inp, ws=ws)
    b = gpu_fwd_bwd(inp, ws=ws)
    assert a["loss"] == b["loss"]
    for k in ("lse", "dH", "dW"):
        assert np.array_equal(a[k], b[k]), k


def test_zero_weight_gives_log_v():
    inp = small_inputs(300, 64, 5000, seed=5)
    inp["W"] = np.zeros_like(inp["W"])
    got = gpu_fwd_bwd(inp)
    assert np.max(np.abs(got["lse"] - math.log(5000))) < 1e-5
    assert abs(got["loss"] - math.log(5000)) < 1e-5
    assert np.all(got["dH"] == 0.0)
    ref = oracle_full(inp)
    assert_parity(got, ref)


def test_all_rows_ignored():
    inp = small_inputs(200, 64, 700, seed=6)
    inp["y"][:] = -100
    got = gpu_fwd_bwd(inp)
    assert got["loss"] == 0.0
    assert np.all(got["dH"] == 0.0) and np.all(got["dW"] == 0.0)
    ref = oracle_full(inp)
    assert np.max(np.abs(got["lse"] - ref["lse"])) < 2e-3


def test_no_rows():
    H = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.ones(100, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(0, dtype=torch.int64, device="cuda")
    dW = torch.full((100, 64), 7.0, device="cuda")
    ws = flce.Workspace()
    loss, lse, dH, dW = flce.forward_backward(H, W, y, workspace=ws,
                                              out=(torch.empty((), device="cuda"), torch.empty(0, device="cuda"),
                                                   torch.empty(0, 64, device="cuda"), dW))
    assert loss.item() == 0.0 and torch.all(dW == 0).item()


def test_bad_target_is_reported_and_row_ignored():
    inp = small_inputs(256, 64, 1000, seed=7)
    inp["y"][3] = 1005
    inp["y"][10] = -7
    got = gpu_fwd_bwd(inp)
    assert got["status"] == flce.Status.ERR_BAD_TARGET
    assert np.isfinite(got["loss"]) and np.all(np.isfinite(got["dH"])) and np.all(np.isfinite(got["dW"]))
    fixed = dict(inp)
    fixed["y"] = inp["y"].copy()
    fixed["y"][[3, 10]] = -100
    ref = oracle_full(fixed)
    assert_parity(got, ref)
    # The status word is cleared once read.
    ws = flce.Workspace()
    gpu_fwd_bwd(fixed, ws=ws)
    assert flce.device_status(ws) == flce.Status.OK


def test_grad_loss_scales_gradients():
    inp = small_inputs(256, 64, 1000, seed=8)
    ref = oracle_full(inp, grad_loss=-2.5)
    got = gpu_fwd_bwd(inp, grad_loss=-2.5)
    assert_parity(got, ref)


def test_lse_buffer_optional():
    inp = small_inputs(256, 64, 1000, seed=9)
    a = gpu_fwd_bwd(inp, lse_out=True)
    b = gpu_fwd_bwd(inp, lse_out=False)
    assert a["loss"] == b["loss"]
    assert np.array_equal(a["dH"], b["dH"]) and np.array_equal(a["dW"], b["dW"])


def test_ignore_index_inside_vocab_range():
    inp = small_inputs(256, 64, 1000, seed=10, ignore=0.0)
    H, W, y = to_device(inp)
    loss, lse, dH, dW = flce.forward_backward(H, W, y, ignore_index=5)
    yy = inp["y"].copy()
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    r = oracle.forward_backward(H64, W64, yy, ignore_index=5)
    got = {"loss": loss.item(), "lse": lse.cpu().numpy(), "dH": dH.cpu().numpy(), "dW": dW.cpu().numpy()}
    assert_parity(got, {"loss": r[1], "lse": r[0], "dH": r[2], "dW": r[3]})


def test_short_wait_flag_reports_timeout_and_context_survives():
    inp = small_inputs(512, 256, 4096, seed=11)
    H, W, y = to_device(inp)
    ws = flce.Workspace()
    prob = flce.make_problem(512, 256, 4096, flags=flce.FLAG_TEST_SHORT_WAITS)
    buf = ws.get(prob)
    lse = torch.empty(512, device="cuda")
    loss = torch.empty((), device="cuda")
    dH = torch.empty(512, 256, device="cuda")
    dW = torch.empty(4096, 256, device="cuda")
    st = flce.flce_forward_backward(prob, H, W, y, 1.0, lse, loss, dH, dW, buf)
    assert st == flce.Status.OK
    assert flce.flce_get_device_status(buf) == flce.Status.ERR_TIMEOUT
    # A normal call afterwards works and matches the oracle.
    got = gpu_fwd_bwd(inp)
    assert got["status"] == flce.Status.OK
    assert_parity(got, oracle_full(inp))


def test_filtered_gradient_matches_tile_mask_oracle():
    # A softmax peaky enough that whole 128x256 tiles of the gradient fall
    # below 2^-12 (logit std ~ 30, targets among each row's top 16): with
    # Gaussian logits of std ~ 3 no tile would be skipped at this granularity.
    wl = synth.Workload("peaky_filter", 512, 64, 262144, 900.0, "top16", 0.0)
    inp = synth.make_inputs(wl, seed=12)
    eps = 2.0 ** -12
    got = gpu_fwd_bwd(inp, filter_eps=eps)
    assert got["status"] == flce.Status.OK
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    lse, loss, dH, dW, _, frac = oracle.forward_backward_filtered(H64, W64, inp["y"], eps, 128, 256,
                                                                  dH_tile_rows=dh_filter_rows())
    full = oracle_full(inp)
    e_filt = errors(got, {"loss": loss, "lse": lse, "dH": dH, "dW": dW})
    e_full = errors(got, full)
    print("filtered vs tile-mask oracle", e_filt, "vs unfiltered", e_full, "skipped", got["skipped"], frac)
    assert frac > 0.5
    assert abs(got["skipped"] - frac) <= 0.02
    assert e_filt["dH_rel"] <= 1e-2 and e_filt["dW_rel"] <= 1e-2
    assert e_full["loss_rel"] <= 1e-3 and e_full["lse_abs"] <= 2e-3


def test_cuda_graph_capture_and_replay():
    # The call allocates nothing and only enqueues work on the given stream, so
    # it can be captured once and replayed; replays match the eager call bit
    # for bit (the path is deterministic). The eager call comes first: it sets
    # up the device (kernel attributes), which is not a stream operation.
    inp = small_inputs(2000, 256, 9000, seed=77, targets="zipf")
    H, W, y = to_device(inp)
    prob = flce.make_problem(2000, 256, 9000)
    ws = torch.empty(flce.flce_workspace_bytes(prob), dtype=torch.uint8, device="cuda")
    outs = [torch.empty((), device="cuda"), torch.empty(2000, device="cuda"),
            torch.empty(2000, 256, device="cuda"), torch.empty(9000, 256, device="cuda")]
    loss, lse, dH, dW = outs
    assert flce.flce_forward_backward(prob, H, W, y, 1.0, lse, loss, dH, dW, ws) == flce.Status.OK
    torch.cuda.synchronize()
    eager = [t.clone() for t in outs]
    for t in outs:
        t.zero_()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        st = flce.flce_forward_backward(prob, H, W, y, 1.0, lse, loss, dH, dW, ws, stream=side)
    assert st == flce.Status.OK
    for _ in range(2):
        for t in outs:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip(outs, eager):
            assert torch.equal(a, b)


def test_calls_allocate_no_device_memory():
    # After a first call has set the device up, further calls of every entry
    # point leave the device's free memory exactly where it was: the caller's
    # workspace is the only scratch the library uses.
    n, d, v = 3000, 256, 20000
    inp = small_inputs(n, d, v, seed=91, targets="zipf")
    H, W, y = to_device(inp)
    prob = flce.make_problem(n, d, v)
    ws = torch.empty(flce.flce_workspace_bytes(prob), dtype=torch.uint8, device="cuda")
    fws = torch.empty(flce.flce_forward_workspace_bytes(prob), dtype=torch.uint8, device="cuda")
    loss, lse = torch.empty((), device="cuda"), torch.empty(n, device="cuda")
    dH, dW = torch.empty(n, d, device="cuda"), torch.empty(v, d, device="cuda")

    def calls():
        assert flce.flce_forward_backward(prob, H, W, y, 1.0, lse, loss, dH, dW, ws) == flce.Status.OK
        assert flce.flce_forward(prob, H, W, y, lse, loss, fws) == flce.Status.OK

    calls()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        calls()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert flce.flce_get_device_status(fws) == flce.Status.OK
    ref = oracle_full(inp)
    assert abs(loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
