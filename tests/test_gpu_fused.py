"""The single-call training step kd_topk_kl_forward_backward (the single
sweep), the dW accumulation flag and the loss-only forward, through the C ABI.

The sweep forms each row's logits once: its lse arithmetic is the forward's,
so loss, lse and row_kl must equal the separate forward and backward bit for
bit; its G is bf16 logits relative to a per-row offset times a per-row
scale, so dh and dW agree with the separate calls to within bf16 rounding
(relative L2 <= SWEEP_RL2) and with the fp64 oracle to the project's
tolerance, also where the stored values span a wide range or leave it (the
chunk's G is then recomputed).  With KD_ACCUMULATE_DW, dW must equal the
previous contents plus this batch's dW (fp32 rounding of the extra addition
only); the loss-only forward (lse = NULL) must give the same loss."""

import numpy as np
import pytest
import torch

import chunked_top_kl_logit_b300 as kd
from oracle import kd_oracle as O
from synth import make_inputs, workload
from tests.gpu_util import GRAD_RL2, LOSS_RTOL, LSE_ATOL, oracle_inputs, rel_l2, to_device

pytestmark = pytest.mark.gpu

# relative L2 between the sweep's and the separate calls' dh and dW.  Each route
# rounds G to bf16 once, at scales that differ by a non-power-of-two factor, so
# the two roundings are independent; the sweep's dW also rounds the scaled
# h_c^T.  One bf16 rounding of log-uniform values has an RMS relative error of
# 2^-7 sqrt(0.541 / 12) = 1.7e-3, so up to three independent ones give about
# 2.9e-3.
SWEEP_RL2 = 5e-3

CASES = [
    ("T600_V5000_d256_chunk200", dict(T=600, d=256, V=5000, K=50, tau=1.5), 200),
    ("packed_T520_V3000_d320", dict(T=520, d=320, V=3000, K=64, tau=2.0, mask_kind="packed",
                                    seq_len=130, pad=30), 1000),
]


def _separate(g, chunk, grad_loss):
    T, d = g["h"].shape
    V, K = g["W"].shape[0], g["teacher_idx"].shape[1]
    m = kd.TopKKL(T, V, d, K, chunk)
    args = (g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"])
    m.forward(*args)
    m.backward(*args, grad_loss)
    torch.cuda.synchronize()
    kd.check_device_status(m.status, "separate")
    return m


@pytest.mark.parametrize("name,over,chunk", CASES, ids=[c[0] for c in CASES])
def test_fused_matches_separate(name, over, chunk):
    x = make_inputs(workload("small_4k", **over))
    g = to_device(x)
    a = _separate(g, chunk, 0.75)
    T, d = g["h"].shape
    V, K = g["W"].shape[0], g["teacher_idx"].shape[1]
    b = kd.TopKKL(T, V, d, K, chunk)
    b.forward_backward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"],
                       0.75)
    torch.cuda.synchronize()
    kd.check_device_status(b.status, "fused")
    for k in ("loss", "lse", "row_kl"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
    for k in ("dh", "dW"):
        assert rel_l2(getattr(b, k).double().cpu().numpy(),
                      getattr(a, k).double().cpu().numpy()) <= SWEEP_RL2, k
    assert bool((b.dh[g["valid"] == 0] == 0).all())
    # and the oracle
    P = oracle_inputs(x)
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])
    f = O.forward(*args)
    dh, dW = O.backward(*args, 0.75, lse=f["lse"])
    assert rel_l2(b.dh.double().cpu().numpy(), dh) <= GRAD_RL2
    assert rel_l2(b.dW.double().cpu().numpy(), dW) <= GRAD_RL2


def test_fused_parity_with_oracle():
    x = make_inputs(workload("small_4k", T=700, d=192, V=6000, K=40, tau=1.0))
    g = to_device(x)
    T, d = g["h"].shape
    V, K = g["W"].shape[0], g["teacher_idx"].shape[1]
    m = kd.TopKKL(T, V, d, K, 256)
    m.forward_backward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"],
                       1.0)
    torch.cuda.synchronize()
    kd.check_device_status(m.status, "fused")
    P = oracle_inputs(x)
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])
    f = O.forward(*args)
    dh, dW = O.backward(*args, 1.0, lse=f["lse"])
    assert abs(float(m.loss.item()) - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert np.abs(m.lse.double().cpu().numpy() - f["lse"]).max() <= LSE_ATOL
    assert rel_l2(m.dh.double().cpu().numpy(), dh) <= GRAD_RL2
    assert rel_l2(m.dW.double().cpu().numpy(), dW) <= GRAD_RL2


@pytest.mark.parametrize("chunk", [96, 1000])
def test_accumulate_dW_adds_to_previous_contents(chunk):
    x = make_inputs(workload("small_4k", T=500, d=192, V=3000, K=32, tau=1.0, idx_kind="uniform"))
    g = to_device(x)
    T, d = g["h"].shape
    V, K = g["W"].shape[0], g["teacher_idx"].shape[1]
    ref = kd.TopKKL(T, V, d, K, chunk)
    ref.forward_backward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"],
                         g["tau"], 1.0)
    m = kd.TopKKL(T, V, d, K, chunk)
    prev = torch.randn(V, d, device="cuda", generator=torch.Generator("cuda").manual_seed(4))
    m.dW.copy_(prev)
    m.forward_backward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"],
                       1.0, accumulate_dW=True)
    torch.cuda.synchronize()
    kd.check_device_status(m.status, "accumulate")
    assert torch.equal(m.dh, ref.dh)
    expect = prev.double() + ref.dW.double()
    err = (m.dW.double() - expect).abs().max().item()
    assert err <= 1e-6 * expect.abs().max().item(), err
    # a second accumulation adds the same dW again
    m.forward_backward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"],
                       1.0, accumulate_dW=True)
    torch.cuda.synchronize()
    expect2 = expect + ref.dW.double()
    assert (m.dW.double() - expect2).abs().max().item() <= 2e-6 * expect2.abs().max().item()


def test_accumulate_with_no_valid_rows_leaves_dW():
    x = make_inputs(workload("small_4k", T=130, d=128, V=1024, K=20, idx_kind="uniform"))
    x["valid"] = torch.zeros_like(x["valid"])
    g = to_device(x)
    m = kd.TopKKL(130, 1024, 128, 20, 64)
    prev = torch.randn(1024, 128, device="cuda")
    m.dW.copy_(prev)
    m.forward_backward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"],
                       1.0, accumulate_dW=True)
    torch.cuda.synchronize()
    kd.check_device_status(m.status, "accumulate")
    assert float(m.loss.item()) == 0.0
    assert torch.equal(m.dW, prev) and bool((m.dh == 0).all())


def test_loss_only_forward():
    x = make_inputs(workload("small_4k", T=300, d=128, V=2000, K=30, tau=1.0))
    g = to_device(x)
    a = _separate(g, 128, 1.0)
    loss = torch.empty(1, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kd.kd_topk_kl_workspace_size(300, 2000, 128, 30, 128)[0], dtype=torch.uint8,
                     device="cuda")
    kd.kd_topk_kl_forward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"],
                          g["tau"], 128, loss, None, ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(loss, a.loss)


RANGE_CASES = [
    # (W scale, scale of the second chunk's rows of h): the student's logits
    # have standard deviation about W scale x h scale
    ("wide_range_unflagged", 5.0, 1.0),   # stored values up to about 2^40
    ("all_chunks_recomputed", 40.0, 1.0),
    ("second_chunk_recomputed", 1.0, 30.0),
]


@pytest.mark.parametrize("name,wscale,hscale", RANGE_CASES, ids=[c[0] for c in RANGE_CASES])
def test_sweep_stored_value_range(name, wscale, hscale):
    """Rows whose largest logit lies far above the logit at the teacher's top
    cached entry (uniform teacher indices, large logits): up to 64 ln 2 tau
    the stored values carry it; beyond, the chunk's G is recomputed.  Either
    way the sweep matches the separate calls (loss, lse, row_kl bit for bit)
    and the oracle."""
    T, chunk = 600, 300
    x = make_inputs(workload("small_4k", T=T, d=256, V=5000, K=50, tau=1.0, mask_kind="all",
                             idx_kind="uniform"))
    x["W"] = (x["W"].float() * wscale).to(torch.bfloat16)
    h = x["h"].float()
    h[chunk:] *= hscale
    x["h"] = h.to(torch.bfloat16)
    g = to_device(x)
    a = _separate(g, chunk, 1.0)
    b = kd.TopKKL(T, 5000, 256, 50, chunk, fused=True)
    b.forward_backward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"],
                       1.0)
    torch.cuda.synchronize()
    kd.check_device_status(b.status, name)
    for k in ("loss", "lse", "row_kl"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
    P = oracle_inputs(x)
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])
    f = O.forward(*args)
    dh, dW = O.backward(*args, 1.0, lse=f["lse"])
    assert abs(float(b.loss.item()) - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert np.abs(b.lse.double().cpu().numpy() - f["lse"]).max() <= LSE_ATOL
    for k, ref in (("dh", dh), ("dW", dW)):
        got = getattr(b, k).double().cpu().numpy()
        assert np.all(np.isfinite(got)), k
        assert rel_l2(got, ref) <= GRAD_RL2, k
        assert rel_l2(got, getattr(a, k).double().cpu().numpy()) <= SWEEP_RL2, k


@pytest.mark.parametrize("chunk", [128, 250])
def test_valid_rows_only(chunk):
    """KD_VALID_ROWS_ONLY forms no logits for masked rows: their lse is NaN and
    their row_kl 0; the loss, the valid rows' lse and row_kl, dh and dW are bit
    for bit those of the step without the flag (chunk 250 leaves the masked rows
    of the row order spread over the last two chunks, and one chunk of
    masked rows only)."""
    x = make_inputs(workload("small_4k", T=600, d=192, V=3000, K=30, tau=1.0,
                             mask_kind="packed", seq_len=150, pad=40))
    g = to_device(x)
    T, d = g["h"].shape
    V, K = g["W"].shape[0], g["teacher_idx"].shape[1]
    args = (g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"], 0.5)
    a = kd.TopKKL(T, V, d, K, chunk, fused=True)
    a.forward_backward(*args)
    b = kd.TopKKL(T, V, d, K, chunk, fused=True)
    b.forward_backward(*args, valid_rows_only=True)
    torch.cuda.synchronize()
    kd.check_device_status(a.status, "all rows")
    kd.check_device_status(b.status, "valid rows only")
    v = g["valid"] != 0
    assert int((~v).sum()) == 4 * 40
    assert torch.equal(a.loss, b.loss)
    assert torch.equal(a.lse[v], b.lse[v]) and bool(torch.isnan(b.lse[~v]).all())
    assert torch.equal(a.row_kl, b.row_kl) and bool((b.row_kl[~v] == 0).all())
    assert torch.equal(a.dh, b.dh) and torch.equal(a.dW, b.dW)
    P = oracle_inputs(x)
    f = O.forward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])
    assert abs(float(b.loss.item()) - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert np.abs(b.lse[v].double().cpu().numpy() - f["lse"][P["valid"] != 0]).max() <= LSE_ATOL


def test_sweep_duplicate_indices():
    """Repeated teacher indices in a row: the cached-column pass writes each
    repeated column once, from the probabilities of all its slots."""
    x = make_inputs(workload("small_4k", T=200, d=128, V=1024, K=32, tau=1.0, idx_kind="uniform"))
    idx = x["teacher_idx"].clone()
    idx[::3, 5] = idx[::3, 0]
    idx[1::3, 31] = idx[1::3, 30]
    idx[2::7, 10] = idx[2::7, 11]
    idx[2::7, 12] = idx[2::7, 11]
    x["teacher_idx"] = idx
    g = to_device(x)
    a = _separate(g, 64, 1.0)
    b = kd.TopKKL(200, 1024, 128, 32, 64, fused=True)
    b.forward_backward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"],
                       1.0)
    torch.cuda.synchronize()
    kd.check_device_status(b.status, "sweep")
    for k in ("loss", "lse", "row_kl"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
    P = oracle_inputs(x)
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])
    f = O.forward(*args)
    dh, dW = O.backward(*args, 1.0, lse=f["lse"])
    assert rel_l2(b.dh.double().cpu().numpy(), dh) <= GRAD_RL2
    assert rel_l2(b.dW.double().cpu().numpy(), dW) <= GRAD_RL2
