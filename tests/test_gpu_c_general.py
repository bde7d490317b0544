"""GPU parity of the general entry points (bias; reduction mean, sum, none;
per-row upstream gradients) and of the autograd wrapper, against the fp64
oracle's general form."""

import numpy as np
import pytest
import torch

import lm_head_loss_gb300 as flce
import oracle
from gpu_common import GRAD_REL, LOSS_REL, LSE_ABS, dh_filter_rows, small_inputs, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _bias(v, seed):
    return np.random.default_rng(seed).standard_normal(v) * 0.5


def _rel(a, b):
    s = float(np.max(np.abs(b)))
    return float(np.max(np.abs(a - b))) / s if s > 0 else float(np.max(np.abs(a)))


def _check(got, ref, reduction):
    if reduction == "none":
        assert np.max(np.abs(got["loss"] - ref["loss"])) <= LSE_ABS
    else:
        assert abs(got["loss"] - ref["loss"]) <= LOSS_REL * max(abs(ref["loss"]), 1e-6)
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= LSE_ABS
    assert _rel(got["dH"], ref["dH"]) <= GRAD_REL
    assert _rel(got["dW"], ref["dW"]) <= GRAD_REL
    if ref["db"] is not None:
        assert _rel(got["db"], ref["db"]) <= GRAD_REL


def _run_ex(inp, bias, reduction, grad):
    H, W, y = to_device(inp)
    n, d, v = H.shape[0], H.shape[1], W.shape[0]
    prob = flce.make_problem(n, d, v)
    ws = flce.Workspace().get(prob)
    red = flce.REDUCTIONS[reduction]
    b = None if bias is None else torch.tensor(bias, dtype=torch.float32, device="cuda")
    lse = torch.empty(n, device="cuda")
    loss = torch.empty((n,) if reduction == "none" else (), device="cuda")
    assert flce.flce_forward_ex(prob, red, H, W, b, y, lse, loss, ws) == flce.Status.OK
    g = torch.tensor(np.asarray(grad, dtype=np.float32).reshape(-1), device="cuda")
    dH = torch.empty(n, d, device="cuda")
    dW = torch.empty(v, d, device="cuda")
    db = torch.empty(v, device="cuda") if b is not None else None
    assert flce.flce_backward_ex(prob, red, H, W, b, y, lse, g, dH, dW, db, ws) == flce.Status.OK
    assert flce.flce_get_device_status(ws) == flce.Status.OK
    out = {"loss": loss.cpu().numpy() if reduction == "none" else loss.item(), "lse": lse.cpu().numpy(),
           "dH": dH.cpu().numpy(), "dW": dW.cpu().numpy()}
    out["db"] = db.cpu().numpy() if db is not None else None
    return out


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("n,d,v", [(300, 136, 1000), (8192 + 300, 64, 9000)])
def test_general_entry_points(reduction, with_bias, n, d, v):
    inp = small_inputs(n, d, v, seed=n + v + (7 if with_bias else 0), targets="zipf", ignore=0.05)
    bias = _bias(v, 3) if with_bias else None
    grad = np.random.default_rng(4).standard_normal(n) if reduction == "none" else 1.7
    got = _run_ex(inp, bias, reduction, grad)
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    b64 = None if bias is None else np.asarray(bias, dtype=np.float32).astype(np.float64)
    g64 = np.asarray(grad, dtype=np.float32).astype(np.float64) if reduction == "none" else float(np.float32(grad))
    ref = oracle.forward_backward_ex(H64, W64, inp["y"], bias=b64, reduction=reduction, grad=g64)
    _check(got, ref, reduction)


def test_forward_ex_mean_equals_forward():
    inp = small_inputs(500, 128, 3000, seed=41)
    H, W, y = to_device(inp)
    loss_a, lse_a = flce.forward(H, W, y)
    prob = flce.make_problem(500, 128, 3000)
    ws = flce.Workspace().get(prob)
    lse = torch.empty(500, device="cuda")
    loss = torch.empty((), device="cuda")
    assert flce.flce_forward_ex(prob, 0, H, W, None, y, lse, loss, ws) == flce.Status.OK
    assert loss.item() == loss_a.item() and torch.equal(lse, lse_a)


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_autograd_wrapper(reduction):
    inp = small_inputs(700, 128, 5000, seed=42, targets="zipf")
    H, W, y = to_device(inp)
    H.requires_grad_(True)
    W.requires_grad_(True)
    b = torch.tensor(_bias(5000, 5), dtype=torch.float32, device="cuda", requires_grad=True)
    loss = flce.linear_cross_entropy(H, W, y, bias=b, reduction=reduction)
    if reduction == "none":
        g = torch.randn(700, device="cuda", generator=torch.Generator("cuda").manual_seed(0))
        loss.backward(g, retain_graph=True)
        g_np = g.cpu().numpy().astype(np.float64)
    else:
        loss.backward(retain_graph=True)
        g_np = 1.0
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    ref = oracle.forward_backward_ex(H64, W64, inp["y"], bias=b.detach().cpu().numpy().astype(np.float64),
                                     reduction=reduction, grad=g_np)
    got_loss = loss.detach().cpu().numpy() if reduction == "none" else loss.item()
    if reduction == "none":
        assert np.max(np.abs(got_loss - ref["loss"])) <= LSE_ABS
    else:
        assert abs(got_loss - ref["loss"]) <= LOSS_REL * abs(ref["loss"])
    # Leaves are bf16, so the gradients arrive cast to bf16 (relative 2^-9).
    assert _rel(H.grad.float().cpu().numpy(), ref["dH"]) <= GRAD_REL
    assert _rel(W.grad.float().cpu().numpy(), ref["dW"]) <= GRAD_REL
    assert _rel(b.grad.cpu().numpy(), ref["db"]) <= GRAD_REL
    # The backward recomputes from the saved LSE, so it can run again.
    first = b.grad.clone()
    b.grad = None
    if reduction == "none":
        loss.backward(g)
    else:
        loss.backward()
    assert torch.equal(b.grad, first)


@pytest.mark.parametrize("flag,filter_dH,filter_dW", [(flce.FLAG_FILTER_FULL_DW, True, False),
                                                      (flce.FLAG_FILTER_FULL_DH, False, True)])
def test_filter_full_variants(flag, filter_dH, filter_dW):
    # Peaky logits (std ~ 30) so that many 128x256 tiles are filtered.
    import synth
    wl = synth.Workload("peaky_filter", 512, 64, 262144, 900.0, "top16", 0.0)
    inp = synth.make_inputs(wl, seed=12)
    eps = 2.0 ** -12
    H, W, y = to_device(inp)
    loss, lse, dH, dW = flce.forward_backward(H, W, y, filter_eps=eps, flags=flag)
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    r = oracle.forward_backward_filtered(H64, W64, inp["y"], eps, 128, 256, filter_dH=filter_dH,
                                         filter_dW=filter_dW, dH_tile_rows=dh_filter_rows())
    assert r[5] > 0.5
    assert _rel(dH.cpu().numpy(), r[2]) <= GRAD_REL
    assert _rel(dW.cpu().numpy(), r[3]) <= GRAD_REL


@pytest.mark.parametrize("n,d,v,ignore", [(8192 + 300, 64, 9000, 0.3), (1000, 136, 3000, 0.0), (500, 64, 2000, 1.0)])
def test_ignored_row_compaction(n, d, v, ignore):
    inp = small_inputs(n, d, v, seed=50 + n, targets="zipf", ignore=ignore)
    H, W, y = to_device(inp)
    loss, lse, dH, dW = flce.forward_backward(H, W, y, flags=flce.FLAG_COMPACT_IGNORED)
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    r = oracle.forward_backward_ex(H64, W64, inp["y"])
    got_dH = dH.cpu().numpy()
    ign = inp["y"] == -100
    assert np.all(got_dH[ign] == 0.0)
    if r["count"] > 0:
        assert abs(loss.item() - r["loss"]) <= LOSS_REL * abs(r["loss"])
        assert _rel(got_dH, r["dH"]) <= GRAD_REL
        assert _rel(dW.cpu().numpy(), r["dW"]) <= GRAD_REL
    else:
        assert loss.item() == 0.0 and torch.all(dW == 0).item()
    assert np.max(np.abs(lse.cpu().numpy() - r["lse"])) <= LSE_ABS


def test_compaction_with_bias_and_row_gradients():
    n, d, v = 3000, 128, 7000
    inp = small_inputs(n, d, v, seed=61, targets="zipf", ignore=0.4)
    bias = _bias(v, 9)
    grad = np.random.default_rng(10).standard_normal(n)
    H, W, y = to_device(inp)
    prob = flce.make_problem(n, d, v, flags=flce.FLAG_COMPACT_IGNORED)
    ws = flce.Workspace().get(prob)
    b = torch.tensor(bias, dtype=torch.float32, device="cuda")
    lse = torch.empty(n, device="cuda")
    loss = torch.empty(n, device="cuda")
    assert flce.flce_forward_ex(prob, 2, H, W, b, y, lse, loss, ws) == flce.Status.OK
    g = torch.tensor(grad, dtype=torch.float32, device="cuda")
    dH = torch.empty(n, d, device="cuda")
    dW = torch.empty(v, d, device="cuda")
    db = torch.empty(v, device="cuda")
    assert flce.flce_backward_ex(prob, 2, H, W, b, y, lse, g, dH, dW, db, ws) == flce.Status.OK
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    r = oracle.forward_backward_ex(H64, W64, inp["y"], bias=np.float32(bias).astype(np.float64), reduction="none",
                                   grad=np.float32(grad).astype(np.float64))
    assert _rel(dH.cpu().numpy(), r["dH"]) <= GRAD_REL
    assert _rel(dW.cpu().numpy(), r["dW"]) <= GRAD_REL
    assert _rel(db.cpu().numpy(), r["db"]) <= GRAD_REL
