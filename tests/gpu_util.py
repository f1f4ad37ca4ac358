"""Helpers for the GPU parity tests: run the library through its C ABI on
seeded inputs and compare against the fp64 oracle with the stated tolerances.

Tolerances (fixed for the whole project):
  gathered indices  bit-exact
  loss              relative error <= 1e-3
  lse, row_kl       absolute error <= 2e-3
  dh, dW            relative L2 error <= 1e-2
"""

from __future__ import annotations

import numpy as np
import torch

import chunked_top_kl_logit_b300 as kd

LOSS_RTOL = 1e-3
LSE_ATOL = 2e-3
GRAD_RL2 = 1e-2


def to_device(x: dict, dev="cuda") -> dict:
    out = dict(x)
    for k in ("h", "W"):
        out[k] = x[k].to(dev, dtype=torch.bfloat16).contiguous()
    out["teacher_idx"] = x["teacher_idx"].to(dev).contiguous()
    out["teacher_logits"] = x["teacher_logits"].to(dev).contiguous()
    out["valid"] = x["valid"].to(dev).contiguous()
    return out


def oracle_inputs(x: dict) -> dict:
    """The values the GPU sees, exactly, as fp64 numpy (bf16 -> fp64 is exact)."""
    return dict(h=x["h"].to(torch.bfloat16).double().cpu().numpy(),
                W=x["W"].to(torch.bfloat16).double().cpu().numpy(),
                teacher_idx=x["teacher_idx"].cpu().numpy(),
                teacher_logits=x["teacher_logits"].double().cpu().numpy(),
                valid=x["valid"].cpu().numpy(), tau=float(x["tau"]))


def run_sweep(x: dict, chunk: int, grad_loss: float = 1.0):
    """The one-call training step (kd_topk_kl_forward_backward, the single
    sweep) through the library; returns numpy outputs."""
    g = to_device(x)
    T, d = g["h"].shape
    V = g["W"].shape[0]
    K = g["teacher_idx"].shape[1]
    m = kd.TopKKL(T, V, d, K, chunk, fused=True)
    m.forward_backward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"],
                       g["tau"], grad_loss)
    torch.cuda.synchronize()
    out = dict(status=int(m.status.item()), loss=float(m.loss.item()),
               lse=m.lse.double().cpu().numpy(), row_kl=m.row_kl.double().cpu().numpy(),
               dh=m.dh.double().cpu().numpy(), dW=m.dW.double().cpu().numpy())
    del m
    return out


def run_gpu(x: dict, chunk: int, grad_loss: float = 1.0, backward: bool = True):
    """Forward (+ backward) through the library; returns numpy outputs."""
    g = to_device(x)
    T, d = g["h"].shape
    V = g["W"].shape[0]
    K = g["teacher_idx"].shape[1]
    m = kd.TopKKL(T, V, d, K, chunk)
    gidx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    m.forward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"],
              gathered_idx=gidx)
    torch.cuda.synchronize()
    fwd_status = int(m.status.item())
    out = dict(loss=float(m.loss.item()), lse=m.lse.double().cpu().numpy(),
               row_kl=m.row_kl.double().cpu().numpy(), gathered_idx=gidx.cpu().numpy(),
               fwd_status=fwd_status)
    if backward:
        m.backward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"],
                   grad_loss)
        torch.cuda.synchronize()
        out["bwd_status"] = int(m.status.item())
        out["dh"] = m.dh.double().cpu().numpy()
        out["dW"] = m.dW.double().cpu().numpy()
    del m
    return out


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    if nb == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def assert_forward_parity(gpu: dict, ref: dict, rows=None):
    sel = slice(None) if rows is None else rows
    assert gpu["fwd_status"] == 0, kd.status_string(gpu["fwd_status"])
    np.testing.assert_array_equal(gpu["gathered_idx"], ref["gathered_idx"])
    err_lse = np.abs(gpu["lse"][sel] - ref["lse"]).max()
    assert err_lse <= LSE_ATOL, f"lse abs err {err_lse}"
    err_kl = np.abs(gpu["row_kl"][sel] - ref["row_kl"]).max()
    assert err_kl <= LSE_ATOL, f"row_kl abs err {err_kl}"
    if rows is None:
        denom = max(abs(ref["loss"]), 1e-30)
        assert abs(gpu["loss"] - ref["loss"]) <= LOSS_RTOL * denom, (gpu["loss"], ref["loss"])
