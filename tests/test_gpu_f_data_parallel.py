"""Data parallelism over rows on one GPU: two row shards run one after the
other through the C-ABI, as two ranks would, with the valid count summed
over both before either step. Their summed loss shares and dW, and their
dH and LSE rows side by side, must match the fp64 oracle on the whole batch
at the parity tolerances."""

import numpy as np
import pytest
import torch

import lm_head_loss_gb300 as flce
from gpu_common import assert_parity, oracle_full, small_inputs, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _shard_step(H, W, y, count_global, grad_loss, ws):
    n, d = H.shape
    v = W.shape[0]
    prob = flce.make_problem(n, d, v)
    lse = torch.empty(n, device="cuda")
    loss = torch.empty(1, device="cuda")
    dH = torch.empty(n, d, device="cuda")
    dW = torch.empty(v, d, device="cuda")
    buf = ws.get(prob)
    st = flce.flce_forward_backward_global(prob, H, W, y, count_global, grad_loss, lse, loss, dH, dW, buf)
    assert st == flce.Status.OK
    assert flce.flce_get_device_status(buf) == flce.Status.OK
    return loss, lse, dH, dW


@pytest.mark.parametrize("n,d,v,split", [(1000, 256, 5000, 600), (700, 128, 30000, 256), (300, 64, 4096, 0)])
def test_two_row_shards_with_a_global_count_match_the_whole_batch(n, d, v, split):
    inp = small_inputs(n, d, v, seed=40 + n, targets="zipf", ignore=0.08)
    H, W, y = to_device(inp)
    shards = [(H[:split], y[:split]), (H[split:], y[split:])]
    counts = []
    for Hs, ys in shards:
        c = torch.zeros(1, dtype=torch.int64, device="cuda")
        assert flce.flce_count_valid(flce.make_problem(Hs.shape[0], d, v), ys, c) == flce.Status.OK
        counts.append(c)
    total = counts[0] + counts[1]          # the all-reduce of two ranks
    assert int(total.item()) == int((y != -100).sum().item())
    ws = flce.Workspace()
    outs = [_shard_step(Hs.contiguous(), W, ys.contiguous(), total, 1.25, ws) for Hs, ys in shards]
    got = {"loss": float((outs[0][0] + outs[1][0]).item()),
           "lse": torch.cat([outs[0][1], outs[1][1]]).cpu().numpy(),
           "dH": torch.cat([outs[0][2], outs[1][2]]).cpu().numpy(),
           "dW": (outs[0][3] + outs[1][3]).cpu().numpy()}
    ref = oracle_full(inp, grad_loss=1.25)
    e = assert_parity(got, ref)
    print("two shards vs whole batch", e)


def test_single_process_data_parallel_step_is_the_plain_call():
    inp = small_inputs(900, 256, 8000, seed=44, targets="zipf", ignore=0.05)
    H, W, y = to_device(inp)
    step = flce.DataParallelStep(900, 256, 8000)
    loss, lse, dH, dW, count = step(H, W, y)
    assert step.device_status() == flce.Status.OK
    ref_loss, ref_lse, ref_dH, ref_dW = flce.forward_backward(H, W, y)
    assert int(count.item()) == int((y != -100).sum().item())
    # Same kernels in the same order: identical bits.
    assert torch.equal(loss.view(()), ref_loss) and torch.equal(lse, ref_lse)
    assert torch.equal(dH, ref_dH) and torch.equal(dW, ref_dW)
    assert_parity({"loss": float(loss.item()), "lse": lse.cpu().numpy(), "dH": dH.cpu().numpy(),
                   "dW": dW.cpu().numpy()}, oracle_full(inp))


# Two processes on the one GPU, each a rank of a gloo process group (NCCL takes
# one rank per GPU). Each rank runs DataParallelStep on its own rows; the
# all-reduces go through torch.distributed on the host, so no rank's kernels
# wait on the other's. The result must equal the oracle on the whole batch.
_DP_SHAPE = (900, 256, 6000, 350)   # rows, hidden, vocab, rows of rank 0


def _dp_rank(rank, world, port, q):
    import os
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        n, d, v, split = _DP_SHAPE
        inp = small_inputs(n, d, v, seed=77, targets="zipf", ignore=0.1)
        H, W, y = to_device(inp)
        rows = slice(0, split) if rank == 0 else slice(split, n)
        Hr, yr = H[rows].contiguous(), y[rows].contiguous()
        step = flce.DataParallelStep(Hr.shape[0], d, v, "cuda")
        loss, lse, dH, dW, count = step(Hr, W, yr, grad_loss=0.75)
        torch.cuda.synchronize()
        assert step.device_status() == flce.Status.OK
        q.put((rank, float(loss.item()), lse.cpu().numpy(), dH.cpu().numpy(), dW.cpu().numpy(), int(count.item())))
    finally:
        dist.destroy_process_group()


def test_two_process_data_parallel_step_matches_the_whole_batch():
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_dp_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(2):
        r = q.get(timeout=300)
        got[r[0]] = r
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    n, d, v, split = _DP_SHAPE
    inp = small_inputs(n, d, v, seed=77, targets="zipf", ignore=0.1)
    ref = oracle_full(inp, grad_loss=0.75)
    assert got[0][5] == got[1][5] == ref["count"]
    for rank in (0, 1):
        assert got[rank][1] == got[0][1]                        # every rank holds the global loss
        assert np.array_equal(got[rank][4], got[0][4])          # and the same summed dW
    whole = {"loss": got[0][1], "lse": np.concatenate([got[0][2], got[1][2]]),
             "dH": np.concatenate([got[0][3], got[1][3]]), "dW": got[0][4]}
    print("two processes vs whole batch", assert_parity(whole, ref))
