"""GPU parity of the sorted-vocabulary backward (Cut Cross-Entropy, Sec. 4.3
"Vocabulary sorting") against the fp64 oracle: the average logits and their
order, unchanged results with the filter off, and with the filter on the
tile mask cut along the sorted order."""

import numpy as np
import pytest
import torch

import lm_head_loss_gb300 as flce
import oracle
import synth
from gpu_common import GRAD_REL, LOSS_REL, LSE_ABS, dh_filter_rows, errors, small_inputs, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _rel(a, b):
    s = float(np.max(np.abs(b)))
    return float(np.max(np.abs(a - b))) / s if s > 0 else float(np.max(np.abs(a)))


def _run_sorted(inp, filter_eps=0.0, bias=None, flags=0, ignore_index=-100):
    """forward_ex + backward_ex (reduction mean) with FLCE_FLAG_SORT_VOCAB."""
    H, W, y = to_device(inp)
    n, d, v = H.shape[0], H.shape[1], W.shape[0]
    prob = flce.make_problem(n, d, v, ignore_index, filter_eps, flce.FLAG_SORT_VOCAB | flags)
    ws = flce.Workspace().get(prob)
    b = torch.tensor(bias, dtype=torch.float32, device="cuda") if bias is not None else None
    lse = torch.empty(n, device="cuda")
    loss = torch.empty((), device="cuda")
    assert flce.flce_forward_ex(prob, 0, H, W, b, y, lse, loss, ws) == flce.Status.OK
    grad = torch.ones(1, device="cuda")
    dH = torch.empty(n, d, device="cuda")
    dW = torch.empty(v, d, device="cuda")
    db = torch.empty(v, device="cuda") if bias is not None else None
    assert flce.flce_backward_ex(prob, 0, H, W, b, y, lse, grad, dH, dW, db, ws) == flce.Status.OK
    order = torch.empty(v, dtype=torch.int32, device="cuda")
    avg = torch.empty(v, device="cuda")
    assert flce.flce_get_vocab_order(prob, ws, order, avg) == flce.Status.OK
    out = {"loss": loss.item(), "lse": lse.cpu().numpy(), "dH": dH.cpu().numpy(), "dW": dW.cpu().numpy(),
           "db": db.cpu().numpy() if db is not None else None, "order": order.cpu().numpy().astype(np.int64),
           "avg": avg.cpu().numpy(), "status": flce.flce_get_device_status(ws)}
    if filter_eps > 0:
        out["skipped"] = flce.flce_get_filter_stats(ws)
    return out


def _check_order(got, H64, W64, y, bias=None, ignore_index=-100):
    """The averages against the oracle's fp64 ones; the order is the stable
    descending sort of the GPU's own averages; both sorted sequences agree."""
    ref = oracle.average_logits(H64, W64, y, bias, ignore_index)
    valid = y != ignore_index
    count = max(int(valid.sum()), 1)
    scale = np.abs(W64) @ (np.abs(H64[valid]).sum(axis=0) / count)
    if bias is not None:
        scale = scale + np.abs(bias)
    tol = 1e-4 * scale + 1e-6
    avg = got["avg"].astype(np.float64)
    assert np.all(np.abs(avg - ref) <= tol), float(np.max(np.abs(avg - ref) / tol))
    assert np.array_equal(got["order"], np.argsort(-got["avg"], kind="stable"))
    ref_order = oracle.vocabulary_order(ref)
    assert np.all(np.abs(avg[got["order"]] - ref[ref_order]) <= tol.max())
    return ref_order


@pytest.mark.parametrize("n,d,v,with_bias", [(300, 64, 1000, False), (1000, 136, 5000, True),
                                             (8192 + 300, 64, 2 * 8192 + 100, False), (5, 8, 3, True),
                                             (8192 + 300, 64, 9000, True)])
def test_sorted_backward_matches_the_unsorted_oracle(n, d, v, with_bias):
    inp = small_inputs(n, d, v, seed=70 + n, targets="zipf", ignore=0.1)
    bias = np.random.default_rng(n).standard_normal(v) * 0.5 if with_bias else None
    got = _run_sorted(inp, bias=bias)
    assert got["status"] == flce.Status.OK
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    ref = oracle.forward_backward_ex(H64, W64, inp["y"], bias=bias)
    assert abs(got["loss"] - ref["loss"]) <= LOSS_REL * abs(ref["loss"])
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= LSE_ABS
    assert _rel(got["dH"], ref["dH"]) <= GRAD_REL
    assert _rel(got["dW"], ref["dW"]) <= GRAD_REL
    if with_bias:
        assert _rel(got["db"], ref["db"]) <= GRAD_REL
    _check_order(got, H64, W64, inp["y"], bias)


def test_sorted_backward_with_ignore_index_inside_the_vocabulary():
    n, d, v = 700, 64, 3000
    inp = small_inputs(n, d, v, seed=81, targets="zipf", ignore=0.0)
    y = inp["y"].copy()
    y[::5] = 7                       # 7 is the ignore index; other rows may still target a sorted position 7
    inp["y"] = y
    got = _run_sorted(inp, ignore_index=7)
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    lse, loss, dH, dW, count = oracle.forward_backward(H64, W64, y, ignore_index=7)
    assert abs(got["loss"] - loss) <= LOSS_REL * abs(loss)
    assert _rel(got["dH"], dH) <= GRAD_REL and _rel(got["dW"], dW) <= GRAD_REL
    assert np.all(got["dH"][::5] == 0.0)
    _check_order(got, H64, W64, y, ignore_index=7)


def test_sorted_backward_is_bitwise_deterministic():
    inp = small_inputs(3000, 128, 9000, seed=82, targets="zipf", ignore=0.05)
    a, b = _run_sorted(inp), _run_sorted(inp)
    for k in ("dH", "dW", "order", "avg"):
        assert np.array_equal(a[k], b[k]), k


def test_sorting_groups_the_filtered_tiles():
    # Rows share a component, so every token carries a common logit offset;
    # sorted by average logit, the tokens that never matter fill whole tiles.
    wl = synth.Workload("prior_filter", 1024, 128, 32768, 9.0, "top16", 0.0, h_shared=2.0)
    inp = synth.make_inputs(wl, seed=13)
    eps = 2.0 ** -12
    got = _run_sorted(inp, filter_eps=eps)
    assert got["status"] == flce.Status.OK
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    y = inp["y"]
    ref_order = _check_order(got, H64, W64, y)
    # The tiles are cut from the same sets of ids on both sides.
    v = W64.shape[0]
    for j in range(0, v, 256):
        assert set(got["order"][j:j + 256]) == set(ref_order[j:j + 256]), j
    rows = dh_filter_rows()
    lse, loss, dH, dW, _, frac = oracle.forward_backward_filtered(H64, W64, y, eps, 128, 256, dH_tile_rows=rows,
                                                                  vocab_order=ref_order)
    *_, frac_unsorted = oracle.forward_backward_filtered(H64, W64, y, eps, 128, 256, dH_tile_rows=rows)
    print("skipped: sorted", got["skipped"], frac, "unsorted", frac_unsorted)
    assert frac > 0.5 and frac_unsorted < 0.05
    assert abs(got["skipped"] - frac) <= 0.02
    e = errors(got, {"loss": loss, "lse": lse, "dH": dH, "dW": dW})
    assert e["dH_rel"] <= 1e-2 and e["dW_rel"] <= 1e-2
    full = oracle.forward_backward(H64, W64, y)
    assert abs(got["loss"] - full[1]) <= LOSS_REL * abs(full[1])


def test_sorting_with_compaction():
    n, d, v = 2500, 128, 7000
    inp = small_inputs(n, d, v, seed=83, targets="zipf", ignore=0.4)
    H, W, y = to_device(inp)
    flags = flce.FLAG_SORT_VOCAB | flce.FLAG_COMPACT_IGNORED
    loss, lse, dH, dW = flce.forward_backward(H, W, y, flags=flags)
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    ref = oracle.forward_backward_ex(H64, W64, inp["y"])
    assert abs(loss.item() - ref["loss"]) <= LOSS_REL * abs(ref["loss"])
    assert _rel(dH.cpu().numpy(), ref["dH"]) <= GRAD_REL
    assert _rel(dW.cpu().numpy(), ref["dW"]) <= GRAD_REL
    assert np.all(dH.cpu().numpy()[inp["y"] == -100] == 0.0)


def test_autograd_with_sorted_vocabulary():
    n, d, v = 600, 64, 2000
    inp = small_inputs(n, d, v, seed=84, targets="zipf", ignore=0.1)
    H, W, y = to_device(inp)
    H.requires_grad_(True)
    W.requires_grad_(True)
    bias = np.random.default_rng(3).standard_normal(v) * 0.5
    b = torch.tensor(bias, dtype=torch.float32, device="cuda", requires_grad=True)
    g = torch.tensor(np.random.default_rng(4).standard_normal(n), dtype=torch.float32, device="cuda")
    loss = flce.linear_cross_entropy(H, W, y, b, reduction="none", sort_vocab=True)
    loss.backward(g)
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    ref = oracle.forward_backward_ex(H64, W64, inp["y"], bias=bias, reduction="none", grad=g.cpu().numpy())
    assert np.max(np.abs(loss.detach().cpu().numpy() - ref["loss"])) <= LSE_ABS
    assert _rel(H.grad.float().cpu().numpy(), ref["dH"]) <= GRAD_REL
    assert _rel(W.grad.float().cpu().numpy(), ref["dW"]) <= GRAD_REL
    assert _rel(b.grad.cpu().numpy(), ref["db"]) <= GRAD_REL
