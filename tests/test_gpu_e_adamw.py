"""GPU parity of flce_forward_backward_adamw (W's AdamW step fused into the dW
contraction, as the FORGE explainer describes) against the fp64 oracle's
two-phase step: gradient, then AdamW on the fp32 master weights."""

import numpy as np
import pytest
import torch

import lm_head_loss_gb300 as flce
import oracle
import synth
from gpu_common import GRAD_REL, LOSS_REL, LSE_ABS, small_inputs, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

HP = {"lr": 2e-3, "beta1": 0.9, "beta2": 0.95, "eps": 1e-8, "weight_decay": 0.1}


def _state(inp, seed):
    """fp32 master weights near the bf16 W, and moments of a run in progress."""
    rng = np.random.default_rng(seed)
    w = synth.bf16_bits_to_f32(inp["W"])
    master = (w + rng.standard_normal(w.shape).astype(np.float32) * np.float32(1e-3) * np.abs(w)).astype(np.float32)
    m = (rng.standard_normal(w.shape) * 1e-4).astype(np.float32)
    v = (rng.random(w.shape) * 1e-7 + 1e-8).astype(np.float32)
    return master, m, v


def _gpu_step(inp, master, m, v, step, flags=0):
    H, W, y = to_device(inp)
    dev = H.device
    tm, tmm, tv = (torch.from_numpy(a.copy()).to(dev) for a in (master, m, v))
    w_out = torch.empty(W.shape, dtype=torch.bfloat16, device=dev)
    hp = flce.adamw_hparams(HP["lr"], step, (HP["beta1"], HP["beta2"]), HP["eps"], HP["weight_decay"], dev)
    ws = flce.Workspace(dev)
    loss, lse, dH = flce.forward_backward_adamw(H, W, y, tm, tmm, tv, w_out, hp, flags=flags, workspace=ws)
    return {"loss": loss.item(), "lse": lse.cpu().numpy(), "dH": dH.cpu().numpy(), "master": tm.cpu().numpy(),
            "m": tmm.cpu().numpy(), "v": tv.cpu().numpy(),
            "w_out": w_out.view(torch.int16).cpu().numpy().view(np.uint16), "status": flce.device_status(ws)}


def _tolerances(H64, W64, y, ref, step):
    """Per-element bounds on the kernel's m, v and master after one step.

    G is rounded to bf16 (relative 2^-9) before the fp32 contraction, so the
    kernel's dW_vd is within 2^-7 * sum_n |dZ_nv| |H_nd| of the exact one;
    that bound is carried through one AdamW step to first order."""
    dZ = oracle.dlogits(H64, W64, y)
    dg = 2.0 ** -7 * (np.abs(dZ).T @ np.abs(H64))
    b1, b2, lr, eps = HP["beta1"], HP["beta2"], HP["lr"], HP["eps"]
    bc1, bc2 = 1 - b1 ** step, 1 - b2 ** step
    tol_m = (1 - b1) * dg + 1e-6 * np.abs(ref["m"]) + 1e-12
    tol_v = (1 - b2) * (2 * np.abs(ref["dW"]) + dg) * dg + 1e-5 * ref["v"] + 1e-20
    denom = np.sqrt(ref["v"] / bc2) + eps
    d_denom = tol_v / (2 * np.sqrt(bc2) * np.sqrt(np.maximum(ref["v"], 1e-30)))
    tol_p = lr / bc1 * (tol_m / denom + np.abs(ref["m"]) * d_denom / denom ** 2) * 1.5 + \
        4 * 2.0 ** -24 * np.abs(ref["master"]) + 1e-12
    return tol_m, tol_v, tol_p


def _check(got, inp, master, m, v, step):
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    ref = oracle.forward_backward_adamw(H64, W64, inp["y"], master.astype(np.float64), m.astype(np.float64),
                                        v.astype(np.float64), {**HP, "step": step})
    assert got["status"] == flce.Status.OK
    assert abs(got["loss"] - ref["loss"]) <= LOSS_REL * max(abs(ref["loss"]), 1e-6)
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= LSE_ABS
    s = float(np.max(np.abs(ref["dH"])))
    assert float(np.max(np.abs(got["dH"] - ref["dH"]))) <= GRAD_REL * s if s > 0 else np.all(got["dH"] == 0)
    tol_m, tol_v, tol_p = _tolerances(H64, W64, inp["y"], ref, step)
    assert np.all(np.abs(got["m"] - ref["m"]) <= tol_m)
    assert np.all(np.abs(got["v"] - ref["v"]) <= tol_v)
    err_p = np.abs(got["master"] - ref["master"])
    assert np.all(err_p <= tol_p), float(np.max(err_p / tol_p))
    # The bf16 copy is the round-to-nearest-even of the kernel's own fp32 result.
    assert np.array_equal(got["w_out"], synth.f64_to_bf16_bits(got["master"].astype(np.float64)))
    # The step moved the weights by about lr, far more than the tolerance.
    assert float(np.median(np.abs(ref["master"] - master))) > 20 * float(np.median(tol_p))
    return ref


@pytest.mark.parametrize("n,d,v,step", [(1000, 128, 5000, 3), (300, 72, 1000, 1), (4000, 64, 8192 + 100, 7)])
def test_fused_adamw_matches_two_phase_oracle(n, d, v, step):
    inp = small_inputs(n, d, v, seed=90 + n, targets="zipf", ignore=0.1)
    master, m, vv = _state(inp, n)
    got = _gpu_step(inp, master, m, vv, step)
    _check(got, inp, master, m, vv, step)


@pytest.mark.parametrize("flags", [flce.FLAG_SORT_VOCAB, flce.FLAG_COMPACT_IGNORED,
                                   flce.FLAG_SORT_VOCAB | flce.FLAG_COMPACT_IGNORED])
def test_fused_adamw_with_sorting_and_compaction(flags):
    inp = small_inputs(2000, 128, 6000, seed=95, targets="zipf", ignore=0.4)
    master, m, v = _state(inp, 5)
    got = _gpu_step(inp, master, m, v, 4, flags)
    _check(got, inp, master, m, v, 4)


def test_fused_adamw_with_every_row_ignored_takes_a_zero_gradient_step():
    inp = small_inputs(500, 64, 3000, seed=96, targets="zipf", ignore=1.0)
    master, m, v = _state(inp, 6)
    for flags in (0, flce.FLAG_COMPACT_IGNORED):
        got = _gpu_step(inp, master, m, v, 2, flags)
        assert got["loss"] == 0.0 and np.all(got["dH"] == 0.0)
        _, m_ref, v_ref = oracle.adamw_step(master, np.zeros_like(master), m, v, 2, **HP)
        assert np.max(np.abs(got["m"] - m_ref)) <= 1e-6 * np.max(np.abs(m_ref))
        assert np.max(np.abs(got["v"] - v_ref)) <= 1e-6 * np.max(v_ref)


def test_fused_adamw_rejects_bad_hyperparameters_on_the_device():
    inp = small_inputs(200, 64, 1000, seed=97)
    master, m, v = _state(inp, 7)
    got = _gpu_step(inp, master, m, v, 0)              # step 0 has no bias correction
    assert got["status"] == flce.Status.ERR_INVALID_ARGUMENT
    assert np.array_equal(got["master"], master) and np.array_equal(got["m"], m) and np.array_equal(got["v"], v)


def test_fused_adamw_head_three_steps():
    # The wrapper keeps the state and alternates the two bf16 copies. It is
    # started from a run in progress (moments set, ten steps taken) so that
    # every step is well conditioned and the per-step bounds add up.
    n, d, v = 1500, 128, 4000
    inp = small_inputs(n, d, v, seed=98, targets="zipf", ignore=0.05)
    H, W, y = to_device(inp)
    head = flce.FusedAdamWHead(W, lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                               weight_decay=HP["weight_decay"])
    _, m0, v0 = _state(inp, 8)
    head.m.copy_(torch.from_numpy(m0))
    head.v.copy_(torch.from_numpy(v0))
    head.steps = 10
    H64 = oracle.inputs_f64(inp["H"], inp["W"])[0]
    p = synth.bf16_bits_to_f64(inp["W"])
    p0 = p.copy()
    mo, vo = m0.astype(np.float64), v0.astype(np.float64)
    tol = np.zeros_like(p)
    for t in range(11, 14):
        w_cur = head.weight
        loss, lse, dH = head.step(H, y)
        assert head.weight.data_ptr() != w_cur.data_ptr()
        w_bf16 = synth.bf16_bits_to_f64(synth.f64_to_bf16_bits(p))
        r = oracle.forward_backward_adamw(H64, w_bf16, inp["y"], p, mo, vo, {**HP, "step": t})
        assert abs(loss.item() - r["loss"]) <= LOSS_REL * abs(r["loss"])
        tol += _tolerances(H64, w_bf16, inp["y"], r, t)[2]
        p, mo, vo = r["master"], r["m"], r["v"]
    got = head.master.cpu().numpy()
    assert np.all(np.abs(got - p) <= 2 * tol), float(np.max(np.abs(got - p) / tol))
    assert float(np.median(np.abs(p - p0))) > 20 * float(np.median(tol))
    assert flce.device_status(head.workspace) == flce.Status.OK


def test_standalone_adamw_step_matches_the_oracle():
    n = 1_000_003                      # a tail of 3 after the 4-wide part
    rng = np.random.default_rng(99)
    p0 = rng.standard_normal(n).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    m0 = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v0 = (rng.random(n) * 1e-6 + 1e-8).astype(np.float32)
    dev = torch.device("cuda")
    tp, tm, tv, tg = (torch.from_numpy(a.copy()).to(dev) for a in (p0, m0, v0, g))
    w = torch.empty(n, dtype=torch.bfloat16, device=dev)
    hp = flce.adamw_hparams(HP["lr"], 5, (HP["beta1"], HP["beta2"]), HP["eps"], HP["weight_decay"], dev)
    ws = torch.zeros(1024, dtype=torch.uint8, device=dev)     # status word clear
    assert flce.flce_adamw_step(hp, tg, tp, tm, tv, w, n, ws) == flce.Status.OK
    assert flce.flce_get_device_status(ws) == flce.Status.OK
    p, m, v = oracle.adamw_step(p0, g, m0, v0, 5, **HP)
    gp, gm, gv = tp.cpu().numpy(), tm.cpu().numpy(), tv.cpu().numpy()
    # fp32 arithmetic on fp32 inputs: a few roundings of each term.
    b1, b2 = HP["beta1"], HP["beta2"]
    assert np.all(np.abs(gm - m) <= 1e-6 * (b1 * np.abs(m0) + (1 - b1) * np.abs(g)) + 1e-15)
    assert np.all(np.abs(gv - v) <= 1e-6 * (b2 * v0 + (1 - b2) * g * g) + 1e-20)
    assert np.all(np.abs(gp - p) <= 1e-5 * HP["lr"] + 2.0 ** -22 * np.abs(p))
    assert np.array_equal(w.view(torch.int16).cpu().numpy().view(np.uint16),
                          synth.f64_to_bf16_bits(gp.astype(np.float64)))


def test_fused_step_equals_gradient_then_standalone_step_bit_for_bit():
    # The fused epilogue applies the same update to the same fp32 gradient
    # the two-phase path stores as dW, so both give identical bits.
    inp = small_inputs(2000, 128, 6000, seed=100, targets="zipf", ignore=0.1)
    master, m, v = _state(inp, 9)
    fused = _gpu_step(inp, master, m, v, 6)
    H, W, y = to_device(inp)
    dev = H.device
    tm, tmm, tv = (torch.from_numpy(a.copy()).to(dev) for a in (master, m, v))
    w_out = torch.empty(W.shape, dtype=torch.bfloat16, device=dev)
    hp = flce.adamw_hparams(HP["lr"], 6, (HP["beta1"], HP["beta2"]), HP["eps"], HP["weight_decay"], dev)
    ws = flce.Workspace(dev)
    loss, lse, dH, dW = flce.forward_backward(H, W, y, workspace=ws)
    assert flce.flce_adamw_step(hp, dW, tm, tmm, tv, w_out, W.numel(), ws.buf) == flce.Status.OK
    assert np.array_equal(tm.cpu().numpy(), fused["master"])
    assert np.array_equal(tmm.cpu().numpy(), fused["m"]) and np.array_equal(tv.cpu().numpy(), fused["v"])
    assert np.array_equal(w_out.view(torch.int16).cpu().numpy().view(np.uint16), fused["w_out"])
    assert np.array_equal(dH.cpu().numpy(), fused["dH"])


def test_fused_step_in_a_cuda_graph_reads_each_replays_hyperparameters():
    # The hyper-parameters live in device memory, so one captured graph serves
    # every step: replays with new values written into the same buffer match
    # eager calls with those values, bit for bit.
    inp = small_inputs(1200, 128, 5000, seed=101, targets="zipf", ignore=0.05)
    master, m, v = _state(inp, 10)
    H, W, y = to_device(inp)
    dev = H.device
    n, d, vv = H.shape[0], H.shape[1], W.shape[0]
    prob = flce.make_problem(n, d, vv)
    ws = torch.empty(flce.flce_workspace_bytes(prob), dtype=torch.uint8, device=dev)
    lse, loss = torch.empty(n, device=dev), torch.empty((), device=dev)
    dH = torch.empty(n, d, device=dev)
    w_out = torch.empty(W.shape, dtype=torch.bfloat16, device=dev)
    state = [torch.from_numpy(a.copy()).to(dev) for a in (master, m, v)]
    hp = flce.adamw_hparams(HP["lr"], 1, (HP["beta1"], HP["beta2"]), HP["eps"], HP["weight_decay"], dev)

    def call(stream=None):
        return flce.flce_forward_backward_adamw(prob, H, W, y, 1.0, lse, loss, dH, *state, w_out, hp, ws,
                                                stream=stream)

    def set_step(t, lr):
        hp.copy_(flce.adamw_hparams(lr, t, (HP["beta1"], HP["beta2"]), HP["eps"], HP["weight_decay"], dev))

    # Eager reference: two steps with different step counts and learning rates.
    assert call() == flce.Status.OK                      # also sets the device up before capture
    for t, a in zip(state, (master, m, v)):
        t.copy_(torch.from_numpy(a))
    eager = []
    for t, lr in ((3, 1e-3), (4, 5e-4)):
        set_step(t, lr)
        assert call() == flce.Status.OK
        eager.append([x.clone() for x in state] + [w_out.clone(), dH.clone(), loss.clone()])
    # The same two steps as replays of one graph.
    for t, a in zip(state, (master, m, v)):
        t.copy_(torch.from_numpy(a))
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    set_step(1, 0.0)
    torch.cuda.synchronize()
    saved = [x.clone() for x in state]
    with torch.cuda.graph(graph, stream=side):
        assert call(stream=side) == flce.Status.OK
    for x, s0 in zip(state, saved):                       # capture runs nothing; restore anyway
        x.copy_(s0)
    for (t, lr), ref in zip(((3, 1e-3), (4, 5e-4)), eager):
        set_step(t, lr)
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip(state + [w_out, dH, loss], ref):
            assert torch.equal(a, b)


def test_fused_step_with_filter_equals_filtered_gradient_then_step():
    # With the filter on, tiles whose gradient was left out reach the fused
    # update as exact zeros, as they reach a stored dW: the two paths agree
    # bit for bit (the filtered gradient itself is checked against the
    # oracle's tile mask in the parity tests).
    wl = synth.Workload("peaky_filter", 512, 64, 262144, 900.0, "top16", 0.0)
    inp = synth.make_inputs(wl, seed=12)
    master, m, v = _state(inp, 11)
    H, W, y = to_device(inp)
    dev = H.device
    eps = 2.0 ** -12
    hp = flce.adamw_hparams(HP["lr"], 2, (HP["beta1"], HP["beta2"]), HP["eps"], HP["weight_decay"], dev)
    fused = [torch.from_numpy(a.copy()).to(dev) for a in (master, m, v)]
    w_f = torch.empty(W.shape, dtype=torch.bfloat16, device=dev)
    ws = flce.Workspace(dev)
    loss_f, _, dH_f = flce.forward_backward_adamw(H, W, y, *fused, w_f, hp, filter_eps=eps, workspace=ws)
    skipped = flce.flce_get_filter_stats(ws.buf)
    assert skipped > 0.5
    two = [torch.from_numpy(a.copy()).to(dev) for a in (master, m, v)]
    w_t = torch.empty(W.shape, dtype=torch.bfloat16, device=dev)
    ws2 = flce.Workspace(dev)
    loss_t, _, dH_t, dW = flce.forward_backward(H, W, y, filter_eps=eps, workspace=ws2)
    assert flce.flce_adamw_step(hp, dW, *two, w_t, W.numel(), ws2.buf) == flce.Status.OK
    for a, b in zip(fused + [w_f, dH_f, loss_f], two + [w_t, dH_t, loss_t]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("flags", [0, flce.FLAG_SORT_VOCAB])
def test_fused_adamw_over_several_row_chunks(flags):
    # 8492 rows: two row chunks, so each vocabulary chunk's dW is summed over
    # both in the workspace before its AdamW step.
    inp = small_inputs(8192 + 300, 64, 9000, seed=102, targets="zipf", ignore=0.1)
    master, m, v = _state(inp, 12)
    got = _gpu_step(inp, master, m, v, 5, flags)
    _check(got, inp, master, m, v, 5)
    # The same bits as the stored gradient followed by the standalone step.
    H, W, y = to_device(inp)
    dev = H.device
    two = [torch.from_numpy(a.copy()).to(dev) for a in (master, m, v)]
    w_t = torch.empty(W.shape, dtype=torch.bfloat16, device=dev)
    hp = flce.adamw_hparams(HP["lr"], 5, (HP["beta1"], HP["beta2"]), HP["eps"], HP["weight_decay"], dev)
    ws = flce.Workspace(dev)
    loss, lse, dH, dW = flce.forward_backward(H, W, y, flags=flags, workspace=ws)
    assert flce.flce_adamw_step(hp, dW, *two, w_t, W.numel(), ws.buf) == flce.Status.OK
    assert np.array_equal(two[0].cpu().numpy(), got["master"])
    assert np.array_equal(two[1].cpu().numpy(), got["m"]) and np.array_equal(two[2].cpu().numpy(), got["v"])
    assert np.array_equal(w_t.view(torch.int16).cpu().numpy().view(np.uint16), got["w_out"])
    assert np.array_equal(dH.cpu().numpy(), got["dH"])
