"""The residual-mass variant (kd_topk_kl_forward_residual / _backward_residual,
and the one-call kd_topk_kl_forward_backward_residual) through the C ABI
against its fp64 oracle, with the project's tolerances, on seeded inputs
spanning several tiles with ragged tails; plus the special case with no
residual mass, which must agree with the main loss."""

import numpy as np
import pytest
import torch

import chunked_top_kl_logit_b300 as kd
from oracle import kd_oracle as O
from oracle import kd_residual_oracle as RO
from synth import make_inputs, teacher_full_lse, workload
from tests.gpu_util import GRAD_RL2, LOSS_RTOL, LSE_ATOL, oracle_inputs, rel_l2, run_gpu, to_device

pytestmark = pytest.mark.gpu

MASS_ATOL = 1e-4


def run_gpu_resid(x, tlse, chunk, grad_loss=1.0, backward=True):
    g = to_device(x)
    T, d = g["h"].shape
    V, K = g["W"].shape[0], g["teacher_idx"].shape[1]
    dev = torch.device("cuda")
    fwd, bwd = kd.kd_topk_kl_workspace_size(T, V, d, K, chunk)
    ws = torch.empty(max(fwd, bwd), dtype=torch.uint8, device=dev)
    st = torch.full((1,), -1, dtype=torch.int32, device=dev)
    loss = torch.empty(1, device=dev)
    lse = torch.empty(T, device=dev)
    row_kl = torch.empty(T, device=dev)
    mass = torch.empty(T, device=dev)
    tl_d = tlse.to(dev).contiguous()
    kd.kd_topk_kl_forward_residual(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], tl_d,
                                   g["valid"], g["tau"], chunk, loss, lse, row_kl, mass, ws=ws,
                                   dev_status=st)
    torch.cuda.synchronize()
    out = dict(fwd_status=int(st.item()), loss=float(loss.item()), lse=lse.double().cpu().numpy(),
               row_kl=row_kl.double().cpu().numpy(), outside_mass=mass.double().cpu().numpy())
    if backward:
        dh = torch.empty(T, d, device=dev)
        dW = torch.empty(V, d, device=dev)
        kd.kd_topk_kl_backward_residual(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"],
                                        tl_d, g["valid"], g["tau"], chunk, lse, mass, grad_loss,
                                        dh, dW, ws=ws, dev_status=st)
        torch.cuda.synchronize()
        out.update(bwd_status=int(st.item()), dh=dh.double().cpu().numpy(),
                   dW=dW.double().cpu().numpy())
    return out


CASES = [
    ("teacher_T300_V5000_d256", dict(T=300, d=256, V=5000, tau=1.0), 128),
    ("packed_T520_V3000_d320_tau2", dict(T=520, d=320, V=3000, K=64, tau=2.0, mask_kind="packed",
                                         seq_len=130, pad=30), 200),
    ("uniform_T1000_V8192_d384", dict(T=1000, d=384, V=8192, K=100, tau=1.5, idx_kind="uniform"),
     512),
]


@pytest.mark.parametrize("name,over,chunk", CASES, ids=[c[0] for c in CASES])
def test_residual_parity(name, over, chunk):
    x = make_inputs(workload("small_4k", **over))
    tlse = teacher_full_lse(x["teacher_logits"], x["tau"])
    gpu = run_gpu_resid(x, tlse, chunk, grad_loss=0.8)
    assert gpu["fwd_status"] == 0 and gpu["bwd_status"] == 0
    P = oracle_inputs(x)
    tl64 = tlse.double().numpy()
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], tl64, P["valid"], P["tau"])
    f = RO.forward(*args)
    dh, dW = RO.backward(*args, 0.8, f["lse"], f["topk_mass"])
    assert abs(gpu["loss"] - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert np.abs(gpu["lse"] - f["lse"]).max() <= LSE_ATOL
    assert np.abs(gpu["row_kl"] - f["row_kl"]).max() <= LSE_ATOL
    assert np.abs(gpu["outside_mass"] - (1.0 - f["topk_mass"])).max() <= MASS_ATOL
    assert rel_l2(gpu["dh"], dh) <= GRAD_RL2
    assert rel_l2(gpu["dW"], dW) <= GRAD_RL2
    assert np.all(gpu["dh"][P["valid"] == 0] == 0.0)


def test_no_residual_mass_matches_main_loss():
    """teacher_lse = logsumexp of the cached logits: no mass outside the cache,
    so the variant is the renormalised main loss (up to fp32 rounding of the
    two normalisations; the variant assembles lse from the columns outside the
    cache and the cached ones, so it agrees with the main loss's to a few
    ulps, not bit for bit)."""
    x = make_inputs(workload("small_4k", T=400, d=192, V=4000, K=50, tau=1.0))
    a = x["teacher_logits"].double() / x["tau"]
    tlse = torch.logsumexp(a, dim=1).float()
    res = run_gpu_resid(x, tlse, 128)
    main = run_gpu(x, 128)
    assert abs(res["loss"] - main["loss"]) <= LOSS_RTOL * abs(main["loss"])
    assert np.abs(res["row_kl"] - main["row_kl"]).max() <= LSE_ATOL
    assert np.abs(res["lse"] - main["lse"]).max() <= 2e-5
    assert rel_l2(res["dh"], main["dh"]) <= 1e-3
    assert rel_l2(res["dW"], main["dW"]) <= 1e-3


def test_residual_full_vocab_small_4k_sampled():
    """T=4096, V=201088, d=2880: the oracle checks sampled rows (lse, row KL,
    student mass outside the cache, dh, all from the oracle's own forward of
    those rows) and dW column sums vanish."""
    w = workload("small_4k")
    x = make_inputs(w)
    tlse = teacher_full_lse(x["teacher_logits"], x["tau"])
    gpu = run_gpu_resid(x, tlse, w.chunk)
    assert gpu["fwd_status"] == 0 and gpu["bwd_status"] == 0
    P = oracle_inputs(x)
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(w.T, 12, replace=False))
    tl64 = tlse.double().numpy()
    sub = dict(h=P["h"][rows], idx=P["teacher_idx"][rows], tl=P["teacher_logits"][rows],
               tlse=tl64[rows], valid=np.ones(len(rows), dtype=np.uint8))
    f = RO.forward(sub["h"], P["W"], sub["idx"], sub["tl"], sub["tlse"], sub["valid"], P["tau"])
    assert np.abs(gpu["lse"][rows] - f["lse"]).max() <= LSE_ATOL
    assert np.abs(gpu["outside_mass"][rows] - (1.0 - f["topk_mass"])).max() <= MASS_ATOL
    kl = np.where(P["valid"][rows] > 0, f["row_kl"], 0.0)
    assert np.abs(gpu["row_kl"][rows] - kl).max() <= LSE_ATOL
    n_valid = int((P["valid"] > 0).sum())
    lse_r, mass_r = np.zeros(w.T), np.zeros(w.T)
    lse_r[rows], mass_r[rows] = f["lse"], f["topk_mass"]
    G = RO.grad_logits_rows(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], tl64,
                            P["valid"], P["tau"], 1.0, lse_r, mass_r, n_valid, rows)
    assert rel_l2(gpu["dh"][rows], G @ P["W"]) <= GRAD_RL2
    col = gpu["dW"].sum(axis=0)
    assert np.linalg.norm(col) <= 1e-2 * np.linalg.norm(gpu["dW"])


def test_residual_student_mass_concentrated_on_the_cache():
    """The well-distilled regime: the cache holds the student's own top-64
    and W is scaled so that the student puts at least 0.999 of its mass on
    them in nearly every row (the mass left outside, Q, reaches 1e-10), while
    the teacher leaves R ~ U(0.05, 0.5) outside its cache.  Q must come out
    without cancellation: 1 - sum_k q_k in fp32 would round it to 0 and make
    the loss infinite.  (The fp64 oracle forms Q as 1 - sum_k q_k too; down to
    Q ~ 1e-11 its own rounding stays below 1e-4 of Q.)"""
    rng = np.random.default_rng(29)
    T, d, V, K, tau = 384, 256, 8192, 64, 1.0
    h = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy((rng.standard_normal((V, d)) * 10.0 / np.sqrt(d)).astype(np.float32))
    W = W.to(torch.bfloat16)
    z = h.double().numpy() @ W.double().numpy().T
    idx = np.argsort(-z, axis=1, kind="stable")[:, :K].astype(np.int32)
    first = 8.0 + rng.gumbel(0.0, 1.0, size=(T, 1))
    tl = np.concatenate([first, first - np.cumsum(rng.exponential(0.3, (T, K - 1)), axis=1)],
                        axis=1).astype(np.float32)
    valid = np.ones(T, dtype=np.uint8)
    valid[rng.choice(T, T // 10, replace=False)] = 0
    x = dict(h=h, W=W, teacher_idx=torch.from_numpy(idx), teacher_logits=torch.from_numpy(tl),
             valid=torch.from_numpy(valid), tau=tau)
    tlse = teacher_full_lse(x["teacher_logits"], tau, seed=29)
    P = oracle_inputs(x)
    tl64 = tlse.double().numpy()
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], tl64, P["valid"], P["tau"])
    f = RO.forward(*args)
    Q = 1.0 - f["topk_mass"]
    assert (f["topk_mass"] >= 0.999).mean() >= 0.9 and (Q < 1e-9).any() and Q.min() > 1e-11
    gpu = run_gpu_resid(x, tlse, 128, grad_loss=1.0)
    assert gpu["fwd_status"] == 0 and gpu["bwd_status"] == 0
    assert abs(gpu["loss"] - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert np.abs(gpu["lse"] - f["lse"]).max() <= LSE_ATOL
    assert np.abs(gpu["row_kl"] - f["row_kl"]).max() <= LSE_ATOL
    # the mass outside the cache, to a relative error far below what the loss needs
    assert np.all(np.abs(gpu["outside_mass"] - Q) <= 1e-3 * Q)
    dh, dW = RO.backward(*args, 1.0, f["lse"], f["topk_mass"])
    assert rel_l2(gpu["dh"], dh) <= GRAD_RL2
    assert rel_l2(gpu["dW"], dW) <= GRAD_RL2


def run_sweep_resid(x, tlse, chunk, grad_loss=1.0, valid_rows_only=False):
    """The residual variant's one-call training step (the single sweep)."""
    g = to_device(x)
    T, d = g["h"].shape
    V, K = g["W"].shape[0], g["teacher_idx"].shape[1]
    m = kd.TopKKL(T, V, d, K, chunk, fused=True)
    m.forward_backward_residual(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"],
                                tlse.to("cuda").contiguous(), g["valid"], g["tau"], grad_loss,
                                valid_rows_only=valid_rows_only)
    torch.cuda.synchronize()
    out = dict(status=int(m.status.item()), loss=float(m.loss.item()),
               lse=m.lse.double().cpu().numpy(), row_kl=m.row_kl.double().cpu().numpy(),
               outside_mass=m.outside_mass.double().cpu().numpy(),
               dh=m.dh.double().cpu().numpy(), dW=m.dW.double().cpu().numpy())
    del m
    return out


# sweep against the separate calls: up to three independent bf16 roundings of G
# and h_c^T (see test_gpu_fused.py)
SWEEP_RL2 = 5e-3


@pytest.mark.parametrize("name,over,chunk", CASES, ids=[c[0] for c in CASES])
def test_residual_sweep_matches_split_and_oracle(name, over, chunk):
    """The residual variant's training step in one call: loss, lse, row_kl and
    the mass outside the cache bit for bit those of the separate calls, dh and
    dW within bf16 rounding of them, everything held to the oracle."""
    x = make_inputs(workload("small_4k", **over))
    tlse = teacher_full_lse(x["teacher_logits"], x["tau"])
    a = run_gpu_resid(x, tlse, chunk, grad_loss=0.8)
    b = run_sweep_resid(x, tlse, chunk, grad_loss=0.8)
    assert b["status"] == 0
    assert a["loss"] == b["loss"]
    for k in ("lse", "row_kl", "outside_mass"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    for k in ("dh", "dW"):
        assert rel_l2(b[k], a[k]) <= SWEEP_RL2, k
    P = oracle_inputs(x)
    tl64 = tlse.double().numpy()
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], tl64, P["valid"], P["tau"])
    f = RO.forward(*args)
    dh, dW = RO.backward(*args, 0.8, f["lse"], f["topk_mass"])
    assert abs(b["loss"] - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert rel_l2(b["dh"], dh) <= GRAD_RL2 and rel_l2(b["dW"], dW) <= GRAD_RL2
    assert np.all(b["dh"][P["valid"] == 0] == 0.0)


@pytest.mark.parametrize("case", ["concentrated", "recomputed"])
def test_residual_sweep_concentrated_and_recomputed(case):
    """The residual sweep where the student puts nearly all its mass on its
    cache (the cache holds the student's own top entries; the stored values
    carry it), and where the student's logits lie far above its logit at the
    teacher's top entry (random cache, logits of standard deviation about 400:
    the stored values would leave their range, so every chunk's G is recomputed
    from the lse), against the oracle."""
    rng = np.random.default_rng(31)
    T, d, V, K, tau = 320, 256, 6144, 48, 1.0
    wscale = 1.0 if case == "concentrated" else 40.0
    h = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    Ws = rng.standard_normal((V, d)) * (10.0 * wscale / np.sqrt(d))
    W = torch.from_numpy(Ws.astype(np.float32)).to(torch.bfloat16)
    z = h.double().numpy() @ W.double().numpy().T
    order = np.argsort(-z, axis=1, kind="stable")
    if case == "concentrated":
        idx = order[:, :K].astype(np.int32)
    else:  # random entries away from the student's top 64, so that Q stays near 1
        idx = np.stack([rng.choice(order[t, 64:], K, replace=False) for t in range(T)])
        idx = idx.astype(np.int32)
    first = 8.0 + rng.gumbel(0.0, 1.0, size=(T, 1))
    tl = np.concatenate([first, first - np.cumsum(rng.exponential(0.3, (T, K - 1)), axis=1)],
                        axis=1).astype(np.float32)
    valid = np.ones(T, dtype=np.uint8)
    valid[rng.choice(T, T // 8, replace=False)] = 0
    x = dict(h=h, W=W, teacher_idx=torch.from_numpy(idx), teacher_logits=torch.from_numpy(tl),
             valid=torch.from_numpy(valid), tau=tau)
    tlse = teacher_full_lse(x["teacher_logits"], tau, seed=31)
    b = run_sweep_resid(x, tlse, 128)
    assert b["status"] == 0
    P = oracle_inputs(x)
    tl64 = tlse.double().numpy()
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], tl64, P["valid"], P["tau"])
    f = RO.forward(*args)
    assert abs(b["loss"] - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert np.abs(b["lse"] - f["lse"]).max() <= LSE_ATOL
    Q = 1.0 - f["topk_mass"]
    if case == "concentrated":
        assert np.all(np.abs(b["outside_mass"] - Q) <= 1e-3 * Q)
    dh, dW = RO.backward(*args, 1.0, f["lse"], f["topk_mass"])
    for k, ref in (("dh", dh), ("dW", dW)):
        assert np.all(np.isfinite(b[k])), k
        assert rel_l2(b[k], ref) <= GRAD_RL2, k


def test_residual_sweep_duplicates_and_valid_rows_only():
    """The residual one-call step with repeated teacher indices (a column named
    by c slots carries c (R/Q) q) and packed masking, with and without
    KD_VALID_ROWS_ONLY: the flag leaves everything bit for bit the same except
    the masked rows' lse and outside mass (NaN); both against the oracle."""
    x = make_inputs(workload("small_4k", T=390, d=192, V=2048, K=24, tau=1.3, idx_kind="uniform",
                             mask_kind="packed", seq_len=130, pad=25))
    idx = x["teacher_idx"].clone()
    idx[::4, 3] = idx[::4, 2]
    idx[1::5, 23] = idx[1::5, 0]
    x["teacher_idx"] = idx
    tlse = teacher_full_lse(x["teacher_logits"], x["tau"])
    a = run_sweep_resid(x, tlse, 100)
    b = run_sweep_resid(x, tlse, 100, valid_rows_only=True)
    assert a["status"] == 0 and b["status"] == 0
    v = x["valid"].numpy() != 0
    assert a["loss"] == b["loss"]
    for k in ("lse", "outside_mass"):
        np.testing.assert_array_equal(a[k][v], b[k][v], err_msg=k)
        assert np.all(np.isnan(b[k][~v])), k
    for k in ("row_kl", "dh", "dW"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    s = run_gpu_resid(x, tlse, 100)
    assert s["loss"] == a["loss"]
    np.testing.assert_array_equal(s["outside_mass"], a["outside_mass"])
    P = oracle_inputs(x)
    tl64 = tlse.double().numpy()
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], tl64, P["valid"], P["tau"])
    f = RO.forward(*args)
    dh, dW = RO.backward(*args, 1.0, f["lse"], f["topk_mass"])
    assert abs(a["loss"] - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert rel_l2(a["dh"], dh) <= GRAD_RL2 and rel_l2(a["dW"], dW) <= GRAD_RL2


def test_residual_sweep_full_vocab_small_4k_sampled():
    """T=4096, V=201088, d=2880: the residual one-call step against the
    separate calls (loss, lse, row_kl and the outside mass bit for bit; dh and
    dW within bf16 rounding) and, on sampled rows, against the oracle."""
    w = workload("small_4k")
    x = make_inputs(w)
    tlse = teacher_full_lse(x["teacher_logits"], x["tau"])
    a = run_gpu_resid(x, tlse, w.chunk)
    b = run_sweep_resid(x, tlse, w.chunk)
    assert b["status"] == 0
    assert a["loss"] == b["loss"]
    for k in ("lse", "row_kl", "outside_mass"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    for k in ("dh", "dW"):
        assert rel_l2(b[k], a[k]) <= SWEEP_RL2, k
    P = oracle_inputs(x)
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(w.T, 12, replace=False))
    tl64 = tlse.double().numpy()
    f = RO.forward(P["h"][rows], P["W"], P["teacher_idx"][rows], P["teacher_logits"][rows],
                   tl64[rows], np.ones(len(rows), dtype=np.uint8), P["tau"])
    assert np.abs(b["lse"][rows] - f["lse"]).max() <= LSE_ATOL
    assert np.abs(b["outside_mass"][rows] - (1.0 - f["topk_mass"])).max() <= MASS_ATOL
    n_valid = int((P["valid"] > 0).sum())
    lse_r, mass_r = np.zeros(w.T), np.zeros(w.T)
    lse_r[rows], mass_r[rows] = f["lse"], f["topk_mass"]
    G = RO.grad_logits_rows(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], tl64,
                            P["valid"], P["tau"], 1.0, lse_r, mass_r, n_valid, rows)
    assert rel_l2(b["dh"][rows], G @ P["W"]) <= GRAD_RL2


def test_residual_sweep_ctx_32k_sampled():
    """The headline shapes (T=32768, V=201088, d=2880, chunk 8192) for the
    residual variant: the one-call step against the separate calls (forward
    outputs bit for bit, gradients within bf16 rounding) and sampled rows of
    both against the oracle."""
    w = workload("ctx_32k")
    x = make_inputs(w)
    tlse = teacher_full_lse(x["teacher_logits"], x["tau"])
    b = run_sweep_resid(x, tlse, w.chunk)
    assert b["status"] == 0
    a = run_gpu_resid(x, tlse, w.chunk)
    assert a["fwd_status"] == 0 and a["bwd_status"] == 0
    assert a["loss"] == b["loss"]
    for k in ("lse", "row_kl", "outside_mass"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    for k in ("dh", "dW"):
        assert rel_l2(b[k], a[k]) <= SWEEP_RL2, k
    P = oracle_inputs(x)
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(w.T, 16, replace=False))
    tl64 = tlse.double().numpy()
    f = RO.forward(P["h"][rows], P["W"], P["teacher_idx"][rows], P["teacher_logits"][rows],
                   tl64[rows], np.ones(len(rows), dtype=np.uint8), P["tau"])
    assert np.abs(b["lse"][rows] - f["lse"]).max() <= LSE_ATOL
    assert np.abs(b["outside_mass"][rows] - (1.0 - f["topk_mass"])).max() <= MASS_ATOL
    kl = np.where(P["valid"][rows] > 0, f["row_kl"], 0.0)
    assert np.abs(b["row_kl"][rows] - kl).max() <= LSE_ATOL
    n_valid = int((P["valid"] > 0).sum())
    lse_r, mass_r = np.zeros(w.T), np.zeros(w.T)
    lse_r[rows], mass_r[rows] = f["lse"], f["topk_mass"]
    G = RO.grad_logits_rows(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], tl64,
                            P["valid"], P["tau"], 1.0, lse_r, mass_r, n_valid, rows)
    assert rel_l2(b["dh"][rows], G @ P["W"]) <= GRAD_RL2


def test_residual_sweep_teacher_and_student_mass_equal():
    """Rows where the teacher leaves out exactly the student's mass outside the
    cache (R = Q, so 1 - R/Q vanishes up to rounding and the row factor cannot
    carry the cached columns): the one-call step recomputes those chunks' G
    and still matches the separate calls and the oracle."""
    x = make_inputs(workload("small_4k", T=384, d=128, V=4096, K=32, tau=1.0, idx_kind="uniform"))
    P = oracle_inputs(x)
    a64 = P["teacher_logits"] / P["tau"]
    m = a64.max(axis=1, keepdims=True)
    lse_k = (m + np.log(np.exp(a64 - m).sum(axis=1, keepdims=True)))[:, 0]
    tlse = teacher_full_lse(x["teacher_logits"], x["tau"]).double().numpy()
    f0 = RO.forward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], tlse, P["valid"],
                    P["tau"])
    rows = np.arange(0, 384, 5)
    tlse[rows] = lse_k[rows] - np.log(f0["topk_mass"][rows])  # R = 1 - sum P = Q
    tl32 = torch.from_numpy(tlse.astype(np.float32))
    tl64 = tl32.double().numpy()
    a = run_gpu_resid(x, tl32, 128)
    b = run_sweep_resid(x, tl32, 128)
    assert b["status"] == 0
    assert a["loss"] == b["loss"]
    for k in ("lse", "row_kl", "outside_mass"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], tl64, P["valid"], P["tau"])
    f = RO.forward(*args)
    dh, dW = RO.backward(*args, 1.0, f["lse"], f["topk_mass"])
    assert abs(b["loss"] - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    for k, ref in (("dh", dh), ("dW", dW)):
        assert np.all(np.isfinite(b[k])), k
        assert rel_l2(b[k], ref) <= GRAD_RL2, k
        assert rel_l2(b[k], a[k]) <= SWEEP_RL2, k
