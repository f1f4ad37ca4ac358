"""Pins for the fp64 oracle, independent of the oracle's own code.

Each check ties the oracle to something other than itself: hand-derived worked
examples, closed forms (W = 0; teacher equal to student), a special case that
reduces to library routines (torch log_softmax / kl_div and autograd), central
finite differences, a pure-Python brute force, and invariants (KL >= 0,
gradient rows summing to zero, permutation invariance, exact power-of-two
scaling).  The planted-mistake tests at the end break the oracle on purpose
(on the CPU) and show that some pin fails for each plausible error.
"""

import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

from oracle import kd_oracle as O
from synth import make_inputs, workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def rand_problem(T, d, V, K, tau, seed, masked=(), dup_rows=(), grad_loss=1.0):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d)) / math.sqrt(d)
    idx = np.stack([rng.choice(V, size=K, replace=False) for _ in range(T)]).astype(np.int32)
    for r in dup_rows:
        idx[r, -1] = idx[r, 0]
    tl = rng.normal(0.0, 2.0, size=(T, K))
    valid = np.ones(T, dtype=np.uint8)
    valid[list(masked)] = 0
    return dict(h=h, W=W, teacher_idx=idx, teacher_logits=tl, valid=valid, tau=tau,
                grad_loss=grad_loss)


def run(P, mod=O):
    f = mod.forward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])
    dh, dW = mod.backward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"],
                          P["tau"], P["grad_loss"], lse=f["lse"])
    return f, dh, dW


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = max(np.linalg.norm(b), 1e-300)
    return np.linalg.norm(a - b) / den


# --------------------------------------------------------------------------
# worked examples (tests/golden), derived by hand
# --------------------------------------------------------------------------

with open(GOLDEN) as _f:
    _CASES = json.load(_f)["cases"]


@pytest.mark.parametrize("case", _CASES, ids=[c["name"] for c in _CASES])
def test_worked_examples(case):
    P = dict(h=np.array(case["h"]), W=np.array(case["W"]),
             teacher_idx=np.array(case["teacher_idx"], dtype=np.int32),
             teacher_logits=np.array(case["teacher_logits"]),
             valid=np.array(case["valid"], dtype=np.uint8), tau=case["tau"],
             grad_loss=case["grad_loss"])
    f, dh, dW = run(P)
    np.testing.assert_allclose(f["lse"], case["lse"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(f["row_kl"], case["row_kl"], rtol=0, atol=1e-12)
    assert abs(f["loss"] - case["loss"]) <= 1e-12
    np.testing.assert_allclose(dh, case["dh"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dW, case["dW"], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(f["gathered_idx"], P["teacher_idx"])


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def check_w_zero(mod, tau):
    """W = 0: q = 1/V, lse = log V, row_kl = sum p log p + log V, dh = 0,
    dW[v] = sum_t g valid_t / (N tau) (1/V - P_t[v]) h_t."""
    x = make_inputs(workload("tiny_fp32"))
    h = x["h"].double().numpy()
    idx = x["teacher_idx"].numpy()
    tl = x["teacher_logits"].double().numpy()
    T, V = h.shape[0], 4096
    W = np.zeros((V, h.shape[1]))
    valid = np.ones(T, dtype=np.uint8)
    valid[::5] = 0
    g = 0.75
    P = dict(h=h, W=W, teacher_idx=idx, teacher_logits=tl, valid=valid, tau=tau, grad_loss=g)
    f, dh, dW = run(P, mod)
    logp = scipy.special.log_softmax(tl / tau, axis=1)
    p = np.exp(logp)
    n = int(valid.sum())
    np.testing.assert_allclose(f["lse"], np.full(T, math.log(V)), rtol=0, atol=1e-12)
    expect_kl = np.where(valid > 0, (p * logp).sum(1) + math.log(V), 0.0)
    np.testing.assert_allclose(f["row_kl"], expect_kl, rtol=0, atol=1e-12)
    assert abs(f["loss"] - expect_kl.sum() / n) <= 1e-12
    assert np.all(dh == 0.0)
    Pd = np.zeros((T, V))
    for t in range(T):
        for k in range(idx.shape[1]):
            Pd[t, idx[t, k]] += p[t, k]
    s = g * valid / n / tau
    expect_dW = (s[:, None] * (1.0 / V - Pd)).T @ h
    assert rel(dW, expect_dW) < 1e-12


@pytest.mark.parametrize("tau", [1.0, 0.5, 3.0])
def test_w_zero_closed_form(tau):
    check_w_zero(O, tau)


def test_teacher_equals_student_gives_zero():
    """K = V = 64, tau = 1, teacher logits = student logits at a permutation of
    all 64 entries: p == q, so row_kl = 0 and every gradient vanishes."""
    rng = np.random.default_rng(3)
    T, d, V = 16, 32, 64
    h = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d)) / math.sqrt(d)
    z = h @ W.T
    idx = np.stack([rng.permutation(V) for _ in range(T)]).astype(np.int32)
    tl = np.take_along_axis(z, idx.astype(np.int64), axis=1)
    P = dict(h=h, W=W, teacher_idx=idx, teacher_logits=tl, valid=np.ones(T, np.uint8),
             tau=1.0, grad_loss=1.0)
    f, dh, dW = run(P)
    assert np.abs(f["row_kl"]).max() < 1e-12
    assert abs(f["loss"]) < 1e-12
    assert np.abs(dh).max() < 1e-12 and np.abs(dW).max() < 1e-12


# --------------------------------------------------------------------------
# special case that reduces to library routines: torch dense KL + autograd
# --------------------------------------------------------------------------

def torch_dense(P):
    """Dense formulation with torch library calls.  With distinct indices per
    row, the renormalised top-K teacher is a dense distribution that is zero
    off the cached entries, and the loss is torch's kl_div(log_softmax(z/tau),
    P_dense) summed over the vocabulary and averaged over valid rows."""
    h = torch.tensor(P["h"], dtype=torch.float64, requires_grad=True)
    W = torch.tensor(P["W"], dtype=torch.float64, requires_grad=True)
    tau = P["tau"]
    idx = torch.tensor(P["teacher_idx"], dtype=torch.int64)
    tl = torch.tensor(P["teacher_logits"], dtype=torch.float64)
    valid = torch.tensor(P["valid"], dtype=torch.float64)
    z = h @ W.T
    logq = torch.nn.functional.log_softmax(z / tau, dim=1)
    p = torch.softmax(tl / tau, dim=1)
    Pd = torch.zeros_like(z).scatter(1, idx, p)
    row = torch.nn.functional.kl_div(logq, Pd, reduction="none").sum(1) * valid
    n = valid.sum()
    loss = row.sum() / n * P["grad_loss"]
    loss.backward()
    return (torch.logsumexp(z / tau, 1).detach().numpy(), row.detach().numpy(),
            float(loss.detach()) / P["grad_loss"], h.grad.numpy(), W.grad.numpy())


def check_torch(mod, tau):
    P = rand_problem(37, 24, 300, 20, tau, seed=11, masked=(0, 5, 36), grad_loss=1.7)
    f, dh, dW = run(P, mod)
    lse_t, row_t, loss_t, dh_t, dW_t = torch_dense(P)
    assert rel(f["lse"], lse_t) < 1e-12
    assert rel(f["row_kl"], row_t) < 1e-10
    assert abs(f["loss"] - loss_t) <= 1e-10 * abs(loss_t)
    assert rel(dh, dh_t) < 1e-10
    assert rel(dW, dW_t) < 1e-10


@pytest.mark.parametrize("tau", [1.0, 2.5])
def test_torch_dense_kl_and_autograd(tau):
    check_torch(O, tau)


# --------------------------------------------------------------------------
# finite differences
# --------------------------------------------------------------------------

def check_fd(mod):
    """Central differences of the loss in fp64 against the explicit gradients
    (T=4, d=8, V=32, K=4, one masked row, tau=2, grad_loss=1.3)."""
    P = rand_problem(4, 8, 32, 4, 2.0, seed=5, masked=(2,), grad_loss=1.3)
    _, dh, dW = run(P, mod)

    def loss(h, W):
        return P["grad_loss"] * mod.forward(h, W, P["teacher_idx"], P["teacher_logits"],
                                            P["valid"], P["tau"])["loss"]

    eps = 1e-6
    num_h = np.zeros_like(P["h"])
    for i in np.ndindex(*P["h"].shape):
        hp = P["h"].copy(); hp[i] += eps
        hm = P["h"].copy(); hm[i] -= eps
        num_h[i] = (loss(hp, P["W"]) - loss(hm, P["W"])) / (2 * eps)
    num_W = np.zeros_like(P["W"])
    for i in np.ndindex(*P["W"].shape):
        Wp = P["W"].copy(); Wp[i] += eps
        Wm = P["W"].copy(); Wm[i] -= eps
        num_W[i] = (loss(P["h"], Wp) - loss(P["h"], Wm)) / (2 * eps)
    assert rel(dh, num_h) < 1e-7
    assert rel(dW, num_W) < 1e-7
    assert np.all(dh[2] == 0.0)


def test_finite_differences():
    check_fd(O)


# --------------------------------------------------------------------------
# pure-Python brute force (no numpy matmul), duplicates included
# --------------------------------------------------------------------------

def brute(P):
    h, W, idx, tl = P["h"].tolist(), P["W"].tolist(), P["teacher_idx"].tolist(), P["teacher_logits"].tolist()
    valid, tau, g = P["valid"].tolist(), P["tau"], P["grad_loss"]
    T, d, V, K = len(h), len(h[0]), len(W), len(idx[0])
    lse, rows, G = [], [], []
    n = sum(1 for v in valid if v)
    for t in range(T):
        zs = [sum(h[t][j] * W[v][j] for j in range(d)) / tau for v in range(V)]
        m = max(zs)
        l = m + math.log(sum(math.exp(x - m) for x in zs))
        a = [x / tau for x in tl[t]]
        ma = max(a)
        la = ma + math.log(sum(math.exp(x - ma) for x in a))
        logp = [x - la for x in a]
        kl = sum(math.exp(lp) * (lp - (zs[idx[t][k]] - l)) for k, lp in enumerate(logp))
        rows.append(kl if valid[t] else 0.0)
        lse.append(l)
        s = g * valid[t] / n / tau
        gr = [s * math.exp(x - l) for x in zs]
        for k in range(K):
            gr[idx[t][k]] -= s * math.exp(logp[k])
        G.append(gr)
    dh = [[sum(G[t][v] * W[v][j] for v in range(V)) for j in range(d)] for t in range(T)]
    dW = [[sum(G[t][v] * h[t][j] for t in range(T)) for j in range(d)] for v in range(V)]
    return lse, rows, sum(rows) / n, dh, dW


def test_bruteforce_python():
    P = rand_problem(8, 16, 64, 8, 1.3, seed=7, masked=(6,), dup_rows=(1, 4), grad_loss=0.9)
    f, dh, dW = run(P)
    lse, rows, loss, dh_b, dW_b = brute(P)
    assert rel(f["lse"], lse) < 1e-12
    assert rel(f["row_kl"], rows) < 1e-12
    assert abs(f["loss"] - loss) < 1e-12 * abs(loss)
    assert rel(dh, dh_b) < 1e-12
    assert rel(dW, dW_b) < 1e-12


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def test_kl_nonnegative_and_gradient_rows_sum_to_zero():
    for seed, tau in [(1, 1.0), (2, 0.7), (3, 4.0)]:
        P = rand_problem(50, 16, 500, 30, tau, seed=seed, masked=(3, 4))
        f, dh, dW = run(P)
        assert f["row_kl"].min() >= -1e-12           # Gibbs: sum_k q_idx <= 1
        # sum_v G_tv = 0 for every row, hence the column sums of dW vanish
        assert np.abs(dW.sum(axis=0)).max() <= 1e-12 * np.abs(dW).max() * dW.shape[0]
        n = int(P["valid"].sum())
        G = O.grad_logits_rows(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"],
                               P["valid"], tau, 1.0, f["lse"], n, np.arange(50))
        assert np.abs(G.sum(axis=1)).max() < 1e-15 * 500
        assert np.all(dh[[3, 4]] == 0.0)


def test_tiny_workload_properties():
    x = make_inputs(workload("tiny_fp32"))
    P = dict(h=x["h"].double().numpy(), W=x["W"].double().numpy(),
             teacher_idx=x["teacher_idx"].numpy(), teacher_logits=x["teacher_logits"].double().numpy(),
             valid=x["valid"].numpy(), tau=1.0, grad_loss=1.0)
    f, dh, dW = run(P)
    assert f["row_kl"].min() >= -1e-12 and f["n_valid"] == 256
    assert np.abs(dW.sum(axis=0)).max() < 1e-12 * np.abs(dW).sum()


def test_no_valid_rows():
    P = rand_problem(6, 8, 40, 5, 1.0, seed=9, masked=range(6))
    f, dh, dW = run(P)
    assert f["loss"] == 0.0 and f["n_valid"] == 0
    assert np.all(f["row_kl"] == 0) and np.all(dh == 0) and np.all(dW == 0)
    assert np.all(np.isfinite(f["lse"]))


def test_permutation_invariance():
    P = rand_problem(20, 12, 200, 16, 1.5, seed=13, masked=(7,), dup_rows=(2,))
    f, dh, dW = run(P)
    rng = np.random.default_rng(0)
    perm = np.stack([rng.permutation(16) for _ in range(20)])
    Q = dict(P, teacher_idx=np.take_along_axis(P["teacher_idx"], perm, 1),
             teacher_logits=np.take_along_axis(P["teacher_logits"], perm, 1))
    g, dh2, dW2 = run(Q)
    assert rel(g["row_kl"], f["row_kl"]) < 1e-14
    assert abs(g["loss"] - f["loss"]) < 1e-14 * abs(f["loss"])
    assert rel(dh2, dh) < 1e-13 and rel(dW2, dW) < 1e-13


def test_power_of_two_scaling_is_exact():
    """(h, teacher_logits, tau) -> (2h, 2 teacher_logits, 2 tau) leaves z/tau and
    the teacher distribution bitwise unchanged; G halves exactly, so
    dh' = dh / 2 and dW' = G'^T (2h) = dW, bit for bit."""
    P = rand_problem(24, 16, 256, 10, 1.25, seed=17, masked=(1,), grad_loss=1.1)
    f, dh, dW = run(P)
    Q = dict(P, h=2 * P["h"], teacher_logits=2 * P["teacher_logits"], tau=2 * P["tau"])
    g, dh2, dW2 = run(Q)
    np.testing.assert_array_equal(g["lse"], f["lse"])
    np.testing.assert_array_equal(g["row_kl"], f["row_kl"])
    assert g["loss"] == f["loss"]
    np.testing.assert_array_equal(dh2, dh / 2)
    np.testing.assert_array_equal(dW2, dW)


def test_block_invariance():
    P = rand_problem(40, 8, 100, 6, 0.8, seed=19, masked=(0, 39))
    f = O.forward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], 0.8, block=256)
    dh, dW = O.backward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], 0.8, block=256)
    for b in (1, 7):
        g = O.forward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], 0.8, block=b)
        dh2, dW2 = O.backward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], 0.8, block=b)
        assert rel(g["lse"], f["lse"]) < 1e-14 and rel(g["row_kl"], f["row_kl"]) < 1e-14
        assert rel(dh2, dh) < 1e-13 and rel(dW2, dW) < 1e-13


def test_sampled_helpers_match_full():
    P = rand_problem(64, 16, 700, 12, 1.7, seed=23, masked=(5, 9), dup_rows=(3,), grad_loss=2.0)
    f, dh, dW = run(P)
    n = f["n_valid"]
    rows = np.array([0, 5, 17, 63])
    vrows = np.array([0, 3, 350, 699] + list(P["teacher_idx"][3, :3]))
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])
    assert rel(O.dh_rows(*args, 2.0, f["lse"], n, rows), dh[rows]) < 1e-13
    assert rel(O.dW_rows(*args, 2.0, f["lse"], n, vrows, block=10), dW[vrows]) < 1e-13
    assert rel(O.row_kl_rows(*args, rows), f["row_kl"][rows]) < 1e-14
    assert rel(O.student_lse(P["h"], P["W"], P["tau"], rows), f["lse"][rows]) < 1e-14


def test_index_out_of_range_raises():
    P = rand_problem(3, 4, 10, 2, 1.0, seed=1)
    P["teacher_idx"][1, 0] = 10
    with pytest.raises(ValueError):
        run(P)


# --------------------------------------------------------------------------
# planted mistakes: each plausible error in the oracle trips at least one pin
# --------------------------------------------------------------------------

def _mutant(monkeypatch, name, fn):
    monkeypatch.setattr(O, name, fn)
    return O


def test_planted_gradient_without_inverse_tau(monkeypatch):
    good = O.grad_logits_rows

    def bad(h, W, idx, tl, valid, tau, g, lse, n, rows):
        return good(h, W, idx, tl, valid, tau, g, lse, n, rows) * tau
    _mutant(monkeypatch, "grad_logits_rows", bad)
    with pytest.raises(AssertionError):
        check_fd(O)


def test_planted_gradient_sign_flip(monkeypatch):
    good = O.grad_logits_rows
    _mutant(monkeypatch, "grad_logits_rows", lambda *a: -good(*a))
    with pytest.raises(AssertionError):
        check_fd(O)


def test_planted_student_logits_without_tau(monkeypatch):
    good = O.student_scaled_logits
    _mutant(monkeypatch, "student_scaled_logits", lambda h, W, tau, rows=None: good(h, W, 1.0, rows))
    with pytest.raises(AssertionError):
        check_torch(O, 2.5)


def test_planted_teacher_not_renormalised(monkeypatch):
    # softmax over the cached entries replaced by exp(a) (no normaliser)
    def bad(tl, tau):
        a = np.asarray(tl, dtype=np.float64) / tau
        return a, np.exp(a)
    _mutant(monkeypatch, "teacher_topk_logprobs", bad)
    with pytest.raises(AssertionError):
        check_torch(O, 1.0)


def test_planted_teacher_without_tau(monkeypatch):
    good = O.teacher_topk_logprobs
    _mutant(monkeypatch, "teacher_topk_logprobs", lambda tl, tau: good(tl, 1.0))
    with pytest.raises(AssertionError):
        check_torch(O, 2.5)


def test_planted_mean_over_all_rows(monkeypatch):
    good = O.forward

    def bad(h, W, idx, tl, valid, tau, block=256):
        f = good(h, W, idx, tl, valid, tau, block)
        f["loss"] = float(f["row_kl"].sum() / len(valid))
        return f
    _mutant(monkeypatch, "forward", bad)
    with pytest.raises(AssertionError):
        check_w_zero(O, 1.0)


def test_planted_missing_teacher_scatter(monkeypatch):
    def bad(h, W, idx, tl, valid, tau, g, lse, n, rows):
        rows = np.asarray(rows)
        q = np.exp(O.student_scaled_logits(h, W, tau, rows) - np.asarray(lse)[rows][:, None])
        s = g * np.asarray(valid)[rows] / n / tau
        return s[:, None] * q
    _mutant(monkeypatch, "grad_logits_rows", bad)
    with pytest.raises(AssertionError):
        check_fd(O)


# --------------------------------------------------------------------------
# teacher-entropy token filter (asibiont.com, "Distillation Token Filtering")
# --------------------------------------------------------------------------

from oracle import entropy_filter as EF  # noqa: E402


def test_entropy_closed_forms():
    K = 7
    # equal logits: uniform over K entries, H = log K for any tau
    assert np.allclose(EF.teacher_entropy(np.full((3, K), 2.5), 0.7), math.log(K), atol=1e-14)
    # one dominant logit: H -> 0
    tl = np.zeros((1, K))
    tl[0, 3] = 800.0
    assert EF.teacher_entropy(tl, 1.0)[0] < 1e-300 or EF.teacher_entropy(tl, 1.0)[0] == 0.0
    # two entries: binary entropy of sigmoid(a - b)
    a, b, tau = 1.3, -0.4, 1.7
    s = 1.0 / (1.0 + math.exp(-(a - b) / tau))
    hb = -(s * math.log(s) + (1 - s) * math.log(1 - s))
    assert abs(EF.teacher_entropy(np.array([[a, b]]), tau)[0] - hb) < 1e-14
    # scipy's entropy of the softmax, as an independent routine
    rng = np.random.default_rng(3)
    tl = rng.normal(0, 2, size=(5, 11))
    ref = scipy.stats.entropy(scipy.special.softmax(tl / 1.3, axis=1), axis=1)
    assert np.allclose(EF.teacher_entropy(tl, 1.3), ref, atol=1e-13)


def test_entropy_temperature_scaling():
    rng = np.random.default_rng(4)
    tl = rng.normal(0, 3, size=(6, 9))
    assert np.allclose(EF.teacher_entropy(tl, 2.0), EF.teacher_entropy(tl / 2.0, 1.0), atol=1e-14)
    # higher temperature flattens the distribution: entropy does not decrease
    assert np.all(EF.teacher_entropy(tl, 3.0) >= EF.teacher_entropy(tl, 1.0) - 1e-12)


def test_keep_count_exact():
    assert EF.keep_count(10, 3, 10) == 3
    assert EF.keep_count(10, 31, 100) == 4
    assert EF.keep_count(0, 1, 2) == 0
    assert EF.keep_count(7, 0, 5) == 0
    assert EF.keep_count(7, 5, 5) == 7
    for n in range(50):
        for num, den in ((1, 3), (2, 7), (70, 100)):
            assert EF.keep_count(n, num, den) == math.ceil(n * num / den - 1e-12)


def test_entropy_filter_bruteforce():
    """Against an exhaustive check: every kept row has (H, -row) above every
    dropped candidate, the count is exact and non-candidates are never kept."""
    rng = np.random.default_rng(5)
    for trial in range(30):
        T = int(rng.integers(1, 40))
        H = rng.choice([0.0, 0.5, 1.0, 1.5], size=T) if trial % 2 else rng.random(T)
        valid = (rng.random(T) < 0.7).astype(np.uint8)
        num, den = int(rng.integers(0, 11)), 10
        out = EF.entropy_filter(H, valid, num, den)
        cand = np.nonzero(valid)[0]
        assert out.sum() == EF.keep_count(len(cand), num, den)
        assert np.all(out[valid == 0] == 0)
        kept = [t for t in cand if out[t]]
        dropped = [t for t in cand if not out[t]]
        for a in kept:
            for b in dropped:
                assert (H[a] > H[b]) or (H[a] == H[b] and a < b)


def test_entropy_filter_extremes():
    H = np.array([0.3, 0.1, 0.3, 0.9])
    valid = np.array([1, 1, 0, 1], dtype=np.uint8)
    assert np.array_equal(EF.entropy_filter(H, valid, 1, 1), valid)
    assert EF.entropy_filter(H, valid, 0, 1).sum() == 0
    # one of three: the highest entropy among candidates (row 3)
    assert np.array_equal(EF.entropy_filter(H, valid, 1, 3), [0, 0, 0, 1])
    # ties: rows 0 and 2 share H, row 2 is not a candidate; row 0 before row 1
    assert np.array_equal(EF.entropy_filter(H, valid, 2, 3), [1, 0, 0, 1])


# --------------------------------------------------------------------------
# residual-mass variant (teacher full-vocabulary normaliser cached with the
# top-K; one extra "everything else" outcome)
# --------------------------------------------------------------------------

from oracle import kd_residual_oracle as RO  # noqa: E402


def resid_problem(T, d, V, K, tau, seed, masked=(), r_lo=0.05, r_hi=0.5, grad_loss=1.0):
    P = rand_problem(T, d, V, K, tau, seed, masked=masked, grad_loss=grad_loss)
    a = P["teacher_logits"] / tau
    r = np.random.default_rng(seed + 1).uniform(r_lo, r_hi, size=T)
    P["teacher_lse"] = scipy.special.logsumexp(a, axis=1) - np.log1p(-r)
    P["r"] = r
    return P


def run_resid(P, mod=RO):
    f = mod.forward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["teacher_lse"],
                    P["valid"], P["tau"])
    dh, dW = mod.backward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"],
                          P["teacher_lse"], P["valid"], P["tau"], P["grad_loss"], f["lse"],
                          f["topk_mass"])
    return f, dh, dW


def test_residual_zero_reduces_to_main_loss():
    """teacher_lse = logsumexp of the cached logits leaves no residual mass:
    the variant is the renormalised loss exactly."""
    P = rand_problem(12, 8, 40, 6, 1.5, seed=21, masked=(3,))
    P["teacher_lse"] = scipy.special.logsumexp(P["teacher_logits"] / P["tau"], axis=1)
    f, dh, dW = run_resid(P)
    g, dh0, dW0 = run(P)
    assert abs(f["loss"] - g["loss"]) < 1e-12
    assert np.allclose(f["row_kl"], g["row_kl"], atol=1e-12)
    assert rel(dh, dh0) < 1e-10 and rel(dW, dW0) < 1e-10


def test_residual_bucket_kl_with_scipy():
    """Row KL against scipy's rel_entr on the explicit K+1-outcome
    distributions built from a full-vocabulary softmax."""
    P = resid_problem(9, 6, 30, 5, 0.8, seed=22)
    f, _, _ = run_resid(P)
    z = P["h"] @ P["W"].T / P["tau"]
    q = scipy.special.softmax(z, axis=1)
    for t in range(9):
        pt = np.exp(P["teacher_logits"][t] / P["tau"] - P["teacher_lse"][t])
        qt = q[t, P["teacher_idx"][t]]
        p_full = np.append(pt, 1.0 - pt.sum())
        q_full = np.append(qt, 1.0 - qt.sum())
        assert abs(p_full[-1] - P["r"][t]) < 1e-12
        assert abs(scipy.special.rel_entr(p_full, q_full).sum() - f["row_kl"][t]) < 1e-12
    assert np.all(f["row_kl"] >= 0)


@pytest.mark.parametrize("tau", [1.0, 2.0])
def test_residual_gradient_with_autograd(tau):
    """dh and dW against torch autograd of the bucketed loss (fp64)."""
    P = resid_problem(10, 7, 25, 4, tau, seed=23, masked=(0, 6), grad_loss=0.7)
    f, dh, dW = run_resid(P)
    h = torch.tensor(P["h"], requires_grad=True)
    W = torch.tensor(P["W"], requires_grad=True)
    idx = torch.tensor(P["teacher_idx"], dtype=torch.long)
    logq = torch.log_softmax(h @ W.T / tau, dim=1)
    lqk = torch.gather(logq, 1, idx)
    pk = torch.exp(torch.tensor(P["teacher_logits"]) / tau - torch.tensor(P["teacher_lse"])[:, None])
    R = 1.0 - pk.sum(1)
    Q = 1.0 - torch.exp(lqk).sum(1)
    kl = (pk * (torch.log(pk) - lqk)).sum(1) + R * (torch.log(R) - torch.log(Q))
    valid = torch.tensor(P["valid"], dtype=torch.float64)
    loss = (kl * valid).sum() / valid.sum()
    (loss * P["grad_loss"]).backward()
    assert abs(loss.item() - f["loss"]) < 1e-12
    assert rel(dh, h.grad.numpy()) < 1e-10
    assert rel(dW, W.grad.numpy()) < 1e-10


def test_residual_finite_differences():
    P = resid_problem(4, 5, 16, 3, 1.3, seed=24, masked=(2,))
    f, dh, dW = run_resid(P)
    eps = 1e-6
    for (M, G) in ((P["h"], dh), (P["W"], dW)):
        for i in range(M.shape[0]):
            for j in range(M.shape[1]):
                old = M[i, j]
                M[i, j] = old + eps
                lp = RO.forward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"],
                                P["teacher_lse"], P["valid"], P["tau"])["loss"]
                M[i, j] = old - eps
                lm = RO.forward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"],
                                P["teacher_lse"], P["valid"], P["tau"])["loss"]
                M[i, j] = old
                assert abs((lp - lm) / (2 * eps) - G[i, j]) < 1e-7


def test_residual_gradient_rows_sum_to_zero():
    P = resid_problem(8, 6, 50, 7, 1.0, seed=25)
    f = RO.forward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["teacher_lse"],
                   P["valid"], P["tau"])
    G = RO.grad_logits_rows(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"],
                            P["teacher_lse"], P["valid"], P["tau"], 1.0, f["lse"],
                            f["topk_mass"], f["n_valid"], np.arange(8))
    assert np.abs(G.sum(axis=1)).max() < 1e-15


def test_planted_residual_gradient_without_bucket_term(monkeypatch):
    """Dropping the R/Q terms of the gradient is caught by the autograd pin."""
    orig = RO.grad_logits_rows

    def broken(h, W, idx, tl, tlse, valid, tau, g, lse, tm, nv, rows):
        z = np.zeros_like(np.asarray(tm))
        return orig(h, W, idx, tl, tlse, valid, tau, g, lse, np.full_like(z, -np.inf), nv, rows)
    monkeypatch.setattr(RO, "grad_logits_rows", broken)
    with pytest.raises(AssertionError):
        test_residual_gradient_with_autograd(1.0)


# --------------------------------------------------------------------------
# teacher-side top-K cache producer
# --------------------------------------------------------------------------

from oracle import teacher_topk_oracle as TK  # noqa: E402


def test_teacher_topk_bruteforce_python():
    """Pure-Python selection (no numpy sort) on small random problems with ties."""
    rng = np.random.default_rng(31)
    for trial in range(6):
        T, d, V, K = 5, 4, 40, 7
        h = rng.integers(-2, 3, size=(T, d)).astype(np.float64)
        W = rng.integers(-2, 3, size=(V, d)).astype(np.float64)  # many exact ties
        idx, val, lse = TK.teacher_topk(h, W, K, 1.3)
        for t in range(T):
            z = [sum(h[t, j] * W[v, j] for j in range(d)) for v in range(V)]
            ref = sorted(range(V), key=lambda v: (-z[v], v))[:K]
            assert list(idx[t]) == ref
            assert list(val[t]) == [z[v] for v in ref]
            m = max(z)
            assert abs(lse[t] - (m / 1.3 + math.log(sum(math.exp((x - m) / 1.3) for x in z)))) < 1e-12


def test_teacher_topk_with_torch_topk_and_closed_forms():
    rng = np.random.default_rng(32)
    h = rng.standard_normal((9, 16))
    W = rng.standard_normal((300, 16)) / 4
    idx, val, lse = TK.teacher_topk(h, W, 25, 2.0)
    vals, ids = torch.topk(torch.tensor(h @ W.T), 25, dim=1)  # continuous: no ties
    assert np.array_equal(idx, ids.numpy()) and np.allclose(val, vals.numpy(), atol=0)
    assert np.allclose(lse, scipy.special.logsumexp(h @ W.T / 2.0, axis=1), atol=1e-12)
    # W = 0: every logit is 0, the first K indices in order, lse = log V
    idx0, val0, lse0 = TK.teacher_topk(h, np.zeros_like(W), 10, 0.5)
    assert np.array_equal(idx0, np.tile(np.arange(10), (9, 1))) and np.all(val0 == 0)
    assert np.allclose(lse0, math.log(300), atol=1e-12)
    # K = V: the whole row sorted
    idx_all, val_all, _ = TK.teacher_topk(h[:2], W[:30], 30, 1.0)
    assert np.all(np.diff(val_all, axis=1) <= 0) and sorted(idx_all[0]) == list(range(30))
