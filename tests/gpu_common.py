"""Helpers shared by the GPU parity tests: device upload of the seeded inputs,
calls through the C-ABI, and the parity tolerances.

Tolerances (filter off): mean-loss relative error <= 1e-3, per-row LSE
absolute error <= 2e-3, dH and dW max absolute error <= 1e-2 * max|ref|.
"""

import os

import numpy as np
import torch

import lm_head_loss_gb300 as flce
import oracle
import synth

LOSS_REL = 1e-3
LSE_ABS = 2e-3
GRAD_REL = 1e-2


def to_device(inp, device="cuda"):
    H = torch.from_numpy(np.ascontiguousarray(inp["H"]).view(np.int16)).view(torch.bfloat16).to(device)
    W = torch.from_numpy(np.ascontiguousarray(inp["W"]).view(np.int16)).view(torch.bfloat16).to(device)
    y = torch.from_numpy(np.ascontiguousarray(inp["y"])).to(device)
    return H, W, y


def small_inputs(n, d, v, seed=0, ignore=0.05, targets="uniform", w_var=1.0):
    wl = synth.Workload(f"case_{n}_{d}_{v}", n, d, v, w_var, targets, ignore)
    return synth.make_inputs(wl, seed=seed)


def gpu_fwd_bwd(inp, grad_loss=1.0, filter_eps=0.0, ws=None, lse_out=True):
    H, W, y = to_device(inp)
    ws = ws or flce.Workspace(H.device)
    prob = flce.make_problem(H.shape[0], H.shape[1], W.shape[0], -100, filter_eps, 0)
    buf = ws.get(prob)
    lse = torch.empty(H.shape[0], dtype=torch.float32, device=H.device) if lse_out else None
    loss = torch.empty((), dtype=torch.float32, device=H.device)
    dH = torch.empty(H.shape, dtype=torch.float32, device=H.device)
    dW = torch.empty(W.shape, dtype=torch.float32, device=H.device)
    st = flce.flce_forward_backward(prob, H, W, y, grad_loss, lse, loss, dH, dW, buf)
    assert st == flce.Status.OK, st
    dev = flce.flce_get_device_status(buf)
    out = {"loss": loss.item(), "dH": dH.cpu().numpy(), "dW": dW.cpu().numpy(), "status": dev}
    if lse_out:
        out["lse"] = lse.cpu().numpy()
    if filter_eps > 0:
        out["skipped"] = flce.flce_get_filter_stats(buf)
    return out


def gpu_fwd(inp, ws=None):
    H, W, y = to_device(inp)
    ws = ws or flce.Workspace(H.device)
    loss, lse = flce.forward(H, W, y, workspace=ws)
    return {"loss": loss.item(), "lse": lse.cpu().numpy(), "status": flce.device_status(ws)}


def oracle_full(inp, grad_loss=1.0):
    H64, W64 = oracle.inputs_f64(inp["H"], inp["W"])
    lse, loss, dH, dW, count = oracle.forward_backward(H64, W64, inp["y"], grad_loss=grad_loss)
    return {"lse": lse, "loss": loss, "dH": dH, "dW": dW, "count": count}


def errors(got, ref):
    e = {}
    if "loss" in got:
        e["loss_rel"] = abs(got["loss"] - ref["loss"]) / max(abs(ref["loss"]), 1e-30)
    if "lse" in got and "lse" in ref:
        e["lse_abs"] = float(np.max(np.abs(got["lse"] - ref["lse"]))) if got["lse"].size else 0.0
    for k in ("dH", "dW"):
        if k in got and k in ref and ref[k].size:
            scale = float(np.max(np.abs(ref[k])))
            e[k + "_rel"] = float(np.max(np.abs(got[k] - ref[k]))) / scale if scale > 0 else float(
                np.max(np.abs(got[k])))
    return e


def assert_parity(got, ref, loss_rel=LOSS_REL, lse_abs=LSE_ABS, grad_rel=GRAD_REL):
    e = errors(got, ref)
    assert e.get("loss_rel", 0.0) <= loss_rel, e
    assert e.get("lse_abs", 0.0) <= lse_abs, e
    assert e.get("dH_rel", 0.0) <= grad_rel, e
    assert e.get("dW_rel", 0.0) <= grad_rel, e
    return e


def dh_filter_rows() -> int:
    """Height of the dH tile mask of the GEMM variant in use: the default pair
    kernel leaves a dH k-block out only when both of its 128-row halves are
    filtered; the 1-CTA variant filters 128-row tiles."""
    return 128 if os.environ.get("FLCE_GEMM_MODE") == "cta1" else 256
