"""Plain fp64 CPU oracle of the residual-mass variant of the top-K KL loss.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import it; the library never calls it.

The pages cache only the teacher's top-100 logits per position (aipuls.nl
summary, section "Summary") and say nothing about the probability mass the
cache leaves out.  The main loss renormalises the teacher over its K cached
entries.  This variant is the other plain reading: the cache also keeps the
teacher's full-vocabulary log-normaliser at temperature tau,

    L_t = log sum_v exp(teacher_logit_tv / tau),

so the teacher's probabilities of the cached entries are P_tk = exp(a_tk - L_t)
(a = teacher_logits / tau) and the rest of its mass, R_t = 1 - sum_k P_tk, goes
to one extra "everything else" outcome.  The student is grouped the same way:
q_tk = exp(z_t,idx_tk / tau - lse_t) for the cached entries and
Q_t = 1 - sum_k q_tk for the rest.  The row loss is the KL divergence between
these two distributions over K + 1 outcomes:

    row_kl_t = sum_k P_tk (log P_tk - log q_tk) + R_t (log R_t - log Q_t),

with 0 log 0 = 0 (R_t = 0 drops the last term).  Every cached slot is its own
outcome (the teacher's top-K are distinct vocabulary entries; a row with a
repeated index counts it once per slot, as in the main loss).  Reduction,
masking and temperature follow the main loss: mean over valid rows, no tau^2.

Gradient (explicit, derived from the definition; s_t = g valid_t / N_valid,
c_tv = number of slots of row t holding v, P~_tv = sum of P_tk over those
slots, q_tv = exp(z_tv / tau - lse_t)):

    G_tv = (s_t / tau) (q_tv (1 - R_t / Q_t) + (R_t / Q_t) c_tv q_tv - P~_tv)

and dh = G W, dW = G^T h.
"""

from __future__ import annotations

import numpy as np

from oracle.kd_oracle import _f64, _logsumexp_rows, student_scaled_logits

__all__ = ["teacher_probs", "forward", "grad_logits_rows", "backward"]


def teacher_probs(teacher_logits, teacher_lse, tau: float):
    """(log P, P, R) of the cached entries under the teacher's full-vocabulary
    normaliser; R = 1 - sum_k P (the mass the cache leaves out)."""
    a = _f64(teacher_logits) / float(tau)
    logP = a - _f64(teacher_lse)[:, None]
    P = np.exp(logP)
    R = 1.0 - P.sum(axis=1)
    return logP, P, R


def _xlogy_ratio(R, Q):
    """R (log R - log Q) with the convention 0 log 0 = 0."""
    out = np.zeros_like(R)
    nz = R > 0
    out[nz] = R[nz] * (np.log(R[nz]) - np.log(Q[nz]))
    return out


def forward(h, W, teacher_idx, teacher_logits, teacher_lse, valid, tau: float, block: int = 256):
    """Loss, lse, row_kl and the student's cached-entry mass sum_k q_tk."""
    h = _f64(h)
    W = _f64(W)
    idx = np.asarray(teacher_idx).astype(np.int64)
    T, K = idx.shape
    logP, P, R = teacher_probs(teacher_logits, teacher_lse, tau)
    lse = np.empty(T)
    zg = np.empty((T, K))
    for r0 in range(0, T, block):
        r1 = min(T, r0 + block)
        zs = student_scaled_logits(h, W, tau, np.arange(r0, r1))
        lse[r0:r1] = _logsumexp_rows(zs)
        zg[r0:r1] = np.take_along_axis(zs, idx[r0:r1], axis=1)
    logq = zg - lse[:, None]
    s = np.exp(logq).sum(axis=1)
    Q = 1.0 - s
    kl = (P * (logP - logq)).sum(axis=1) + _xlogy_ratio(R, Q)
    valid_b = np.asarray(valid).astype(bool)
    row_kl = np.where(valid_b, kl, 0.0)
    n_valid = int(valid_b.sum())
    loss = float(row_kl.sum() / n_valid) if n_valid else 0.0
    return {"loss": loss, "lse": lse, "row_kl": row_kl, "topk_mass": s, "n_valid": n_valid}


def grad_logits_rows(h, W, teacher_idx, teacher_logits, teacher_lse, valid, tau: float,
                     grad_loss: float, lse, topk_mass, n_valid: int, rows) -> np.ndarray:
    """G rows by the explicit formula in the module docstring."""
    rows = np.asarray(rows)
    V = W.shape[0]
    if n_valid == 0:
        return np.zeros((len(rows), V))
    _, P, R = teacher_probs(np.asarray(teacher_logits)[rows], _f64(teacher_lse)[rows], tau)
    idx = np.asarray(teacher_idx)[rows].astype(np.int64)
    q = np.exp(student_scaled_logits(h, W, tau, rows) - _f64(lse)[rows][:, None])
    Q = 1.0 - _f64(topk_mass)[rows]
    ratio = np.where(R > 0, R / Q, 0.0)
    rr = np.repeat(np.arange(len(rows)), idx.shape[1])
    count = np.zeros_like(q)
    np.add.at(count, (rr, idx.ravel()), 1.0)
    Psc = np.zeros_like(q)
    np.add.at(Psc, (rr, idx.ravel()), P.ravel())
    s = float(grad_loss) * np.asarray(valid)[rows].astype(np.float64) / float(n_valid)
    inner = q * (1.0 - ratio[:, None]) + ratio[:, None] * count * q - Psc
    return (s / float(tau))[:, None] * inner


def backward(h, W, teacher_idx, teacher_logits, teacher_lse, valid, tau: float,
             grad_loss: float, lse, topk_mass, block: int = 256):
    """dh = G W, dW = G^T h."""
    h = _f64(h)
    W = _f64(W)
    T = h.shape[0]
    n_valid = int(np.asarray(valid).astype(bool).sum())
    dh = np.zeros_like(h)
    dW = np.zeros_like(W)
    for r0 in range(0, T, block):
        rows = np.arange(r0, min(T, r0 + block))
        G = grad_logits_rows(h, W, teacher_idx, teacher_logits, teacher_lse, valid, tau,
                             grad_loss, lse, topk_mass, n_valid, rows)
        dh[rows] = G @ W
        dW += G.T @ h[rows]
    return dh, dW
