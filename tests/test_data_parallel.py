"""Data parallelism over rows, host logic on CPU: two gloo ranks each hold a
different number of rows (and of ignored rows) and the whole W. The
exchange sums their counts before the step, then the loss shares and the
dW contributions. With the oracle as each rank's local computation, the
result must equal the oracle on the whole batch: the mean is over the valid
rows of both ranks, not of either one.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from lm_head_loss_gb300.data_parallel import exchange_step

N, D, V = 37, 6, 23
SPLIT = 15            # rank 0 holds rows [0, 15), rank 1 rows [15, 37)


def _batch():
    rng = np.random.default_rng(3)
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * 0.7
    y = rng.integers(0, V, size=N).astype(np.int64)
    y[[1, 2, 20, 30, 31, 33]] = -100        # 2 ignored rows on rank 0, 4 on rank 1
    return H, W, y


def _oracle_rank(H, W, y, g):
    """This rank's local work, written with the oracle: the valid count, and
    the step with the mean over a given count (a sum, scaled by g / count)."""
    def local_count():
        return torch.tensor([oracle.valid_count(y)], dtype=torch.int64)

    def local_step(count):
        c = max(int(count.item()), 1)
        r = oracle.forward_backward_ex(H, W, y, reduction="sum", grad=g / c)
        return (torch.tensor([r["loss"] / c], dtype=torch.float64), torch.from_numpy(r["lse"]),
                torch.from_numpy(r["dH"]), torch.from_numpy(r["dW"]))
    return local_count, local_step


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        H, W, y = _batch()
        rows = slice(0, SPLIT) if rank == 0 else slice(SPLIT, N)
        local_count, local_step = _oracle_rank(H[rows], W, y[rows], g=1.5)
        loss, lse, dH, dW, count = exchange_step(local_count, local_step,
                                                 lambda t: dist.all_reduce(t, op=dist.ReduceOp.SUM))
        q.put((rank, float(loss.item()), lse.numpy(), dH.numpy(), dW.numpy(), int(count.item())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_equal_the_whole_batch():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(2):
        r = q.get(timeout=180)
        got[r[0]] = r
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    H, W, y = _batch()
    lse, loss, dH, dW, count = oracle.forward_backward(H, W, y, grad_loss=1.5)
    for rank, rows in ((0, slice(0, SPLIT)), (1, slice(SPLIT, N))):
        _, l, r_lse, r_dH, r_dW, c = got[rank]
        assert c == count == N - 6
        assert l == pytest.approx(loss, rel=1e-12)
        np.testing.assert_allclose(r_dW, dW, rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(r_dH, dH[rows], rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(r_lse, lse[rows], rtol=1e-12)


def test_single_rank_exchange_is_the_plain_step():
    H, W, y = _batch()
    local_count, local_step = _oracle_rank(H, W, y, g=1.0)
    loss, lse, dH, dW, count = exchange_step(local_count, local_step, lambda t: None)
    r_lse, r_loss, r_dH, r_dW, r_count = oracle.forward_backward(H, W, y)
    assert int(count.item()) == r_count
    assert float(loss.item()) == pytest.approx(r_loss, rel=1e-12)
    np.testing.assert_allclose(dW.numpy(), r_dW, rtol=1e-10, atol=1e-13)


def test_a_local_count_would_be_wrong():
    # The reason for the first exchange: with uneven valid counts, scaling
    # by each rank's own count and summing does not give the global mean.
    H, W, y = _batch()
    shares = []
    for rows in (slice(0, SPLIT), slice(SPLIT, N)):
        shares.append(oracle.forward(H[rows], W, y[rows])[1])
    whole = oracle.forward(H, W, y)[1]
    assert abs(sum(shares) / 2 - whole) > 1e-3
