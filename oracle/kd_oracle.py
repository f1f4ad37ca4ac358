"""Plain, slow fp64 CPU oracle for the top-K KL distillation loss.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this module.  The
library path (the CUDA kernels behind the C ABI) never imports, links or calls
it, and this module imports nothing from the library.

Sources (cited by page and section):

* [aipuls]  "Making Knowledge Distillation Cheap Enough to Run at Scale",
  aipuls.nl summary, section "Summary", second paragraph: the teacher's top-100
  logits per token position are cached offline, and the student is trained with
  a KL-divergence loss computed as a fused, chunked kernel that never forms the
  full sequence-by-vocabulary matrix.
* [gateway] "Hugging Face and Multiverse Computing cut KD memory costs",
  agent-gateway.com news, paragraphs on the second bottleneck: the loss is
  computed chunk by chunk instead of over a dense sequence x vocabulary tensor.
* [asibiont] asibiont.com blog rewrite, section "A Concrete Implementation
  Sketch": a dense loss of the form kl_div(log_softmax(student), softmax(teacher))
  summed over the vocabulary and averaged over the selected tokens.  Used only
  for the direction of the KL and for the mean over valid tokens.

The pages print no equation for the method.  The definitions below are the
plainest reading that the pages support; every reading is listed here:

1. Student distribution: q_t = softmax(z_t / tau) over the FULL vocabulary,
   z = h W^T, so lse_t = log sum_v exp(z_tv / tau) (natural log, of z/tau).
2. Teacher distribution: p_t = softmax(a_t) with a = teacher_logits / tau over
   the K cached entries only, i.e. renormalised over the top-K (no residual
   mass bucket).
3. Direction: KL(p_t || q_t) = sum_k p_tk (log p_tk - log q_t[idx_tk]).
   Each cached entry k counts separately, so duplicate indices in a row are
   well defined (their gradient contributions add).
4. Temperature divides both sides; no tau^2 factor.
5. Reduction: loss = sum over valid rows of row_kl / N_valid (0 if N_valid = 0);
   invalid rows still get lse, have row_kl = 0 and get zero gradient.
6. Gradient (explicit, no autograd):
   G_tv = g * (valid_t / N_valid) * (q_tv - sum_{k: idx_tk = v} p_tk) / tau,
   dh = G W, dW = G^T h.

Every floating-point step is fp64 on whatever values are passed in (the GPU
path receives bf16-rounded h and W; converting those to fp64 is exact).  The
student logits are formed in row blocks only to bound host memory; a block is
the plain definition applied to a subset of rows, with no reordering inside a
row.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "teacher_topk_logprobs",
    "student_scaled_logits",
    "student_lse",
    "forward",
    "grad_logits_rows",
    "backward",
    "dh_rows",
    "dW_rows",
    "row_kl_rows",
]


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _logsumexp_rows(x: np.ndarray) -> np.ndarray:
    """Natural-log sum of exponentials along axis 1, shifted by the row max."""
    m = x.max(axis=1)
    return m + np.log(np.exp(x - m[:, None]).sum(axis=1))


def teacher_topk_logprobs(teacher_logits, tau: float):
    """Teacher distribution over the K cached entries of each row.

    [aipuls] Summary: only the top-K logits per position are kept.  Reading 2:
    softmax of teacher_logits / tau over those K entries (renormalised).
    Returns (log p, p), both [T, K] fp64.
    """
    a = _f64(teacher_logits) / float(tau)
    logp = a - _logsumexp_rows(a)[:, None]
    return logp, np.exp(logp)


def student_scaled_logits(h, W, tau: float, rows=None) -> np.ndarray:
    """z / tau for the given rows (all rows if None): [len(rows), V] fp64.

    z = h W^T is the student's LM-head output ([aipuls] Summary).
    """
    h = _f64(h)
    if rows is not None:
        h = h[np.asarray(rows)]
    return (h @ _f64(W).T) / float(tau)


def student_lse(h, W, tau: float, rows=None, block: int = 256) -> np.ndarray:
    """lse_t = log sum_v exp(z_tv / tau) over the full vocabulary (reading 1)."""
    T = h.shape[0]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    out = np.empty(len(rows), dtype=np.float64)
    for b0 in range(0, len(rows), block):
        r = rows[b0:b0 + block]
        out[b0:b0 + len(r)] = _logsumexp_rows(student_scaled_logits(h, W, tau, r))
    return out


def row_kl_rows(h, W, teacher_idx, teacher_logits, valid, tau: float, rows,
                lse=None) -> np.ndarray:
    """row_kl_t for the given rows only (reading 3, 5).  lse may be supplied."""
    rows = np.asarray(rows)
    idx = np.asarray(teacher_idx)[rows].astype(np.int64)
    logp, p = teacher_topk_logprobs(np.asarray(teacher_logits)[rows], tau)
    zs = student_scaled_logits(h, W, tau, rows)
    lse_r = _logsumexp_rows(zs) if lse is None else _f64(lse)[rows]
    zg = np.take_along_axis(zs, idx, axis=1)
    kl = (p * (logp - (zg - lse_r[:, None]))).sum(axis=1)
    return np.where(np.asarray(valid)[rows].astype(bool), kl, 0.0)


def forward(h, W, teacher_idx, teacher_logits, valid, tau: float, block: int = 256):
    """Loss, per-row lse, per-row KL and the gathered indices.

    [aipuls] Summary + [gateway]: KL between the cached teacher top-K and the
    student's full-vocabulary softmax.  Readings 1-5.  Returns a dict with
    loss (float), lse [T], row_kl [T], gathered_idx [T, K] (the vocabulary
    column read for each cached slot, i.e. teacher_idx itself), n_valid (int).
    """
    h = _f64(h)
    W = _f64(W)
    idx = np.asarray(teacher_idx).astype(np.int64)
    T, K = idx.shape
    V = W.shape[0]
    if idx.size and (idx.min() < 0 or idx.max() >= V):
        raise ValueError("teacher index out of range")
    valid_b = np.asarray(valid).astype(bool)
    logp, p = teacher_topk_logprobs(teacher_logits, tau)
    lse = np.empty(T, dtype=np.float64)
    zg = np.empty((T, K), dtype=np.float64)
    for r0 in range(0, T, block):
        r1 = min(T, r0 + block)
        zs = student_scaled_logits(h, W, tau, np.arange(r0, r1))
        lse[r0:r1] = _logsumexp_rows(zs)
        zg[r0:r1] = np.take_along_axis(zs, idx[r0:r1], axis=1)
    kl = (p * (logp - (zg - lse[:, None]))).sum(axis=1)
    row_kl = np.where(valid_b, kl, 0.0)
    n_valid = int(valid_b.sum())
    loss = float(row_kl.sum() / n_valid) if n_valid > 0 else 0.0
    return {
        "loss": loss,
        "lse": lse,
        "row_kl": row_kl,
        "gathered_idx": idx.astype(np.int32).copy(),
        "n_valid": n_valid,
    }


def grad_logits_rows(h, W, teacher_idx, teacher_logits, valid, tau: float,
                     grad_loss: float, lse, n_valid: int, rows) -> np.ndarray:
    """G rows: dLoss/dz for the given rows, [len(rows), V] fp64 (reading 6).

    G_tv = g * valid_t / N_valid * (exp(z_tv/tau - lse_t) - sum_{k: idx_tk=v} p_tk) / tau.
    The teacher mass is scatter-added, so duplicate indices add up.
    """
    rows = np.asarray(rows)
    V = W.shape[0]
    if n_valid == 0:
        return np.zeros((len(rows), V), dtype=np.float64)
    _, p = teacher_topk_logprobs(np.asarray(teacher_logits)[rows], tau)
    idx = np.asarray(teacher_idx)[rows].astype(np.int64)
    q = np.exp(student_scaled_logits(h, W, tau, rows) - _f64(lse)[rows][:, None])
    scatter = np.zeros_like(q)
    np.add.at(scatter, (np.repeat(np.arange(len(rows)), idx.shape[1]), idx.ravel()), p.ravel())
    s = float(grad_loss) * np.asarray(valid)[rows].astype(np.float64) / float(n_valid)
    return (s / float(tau))[:, None] * (q - scatter)


def backward(h, W, teacher_idx, teacher_logits, valid, tau: float, grad_loss: float = 1.0,
             lse=None, block: int = 256):
    """dh = G W and dW = G^T h by explicit formula (reading 6); returns (dh, dW)."""
    h = _f64(h)
    W = _f64(W)
    T = h.shape[0]
    n_valid = int(np.asarray(valid).astype(bool).sum())
    if lse is None:
        lse = student_lse(h, W, tau)
    dh = np.zeros_like(h)
    dW = np.zeros_like(W)
    for r0 in range(0, T, block):
        rows = np.arange(r0, min(T, r0 + block))
        G = grad_logits_rows(h, W, teacher_idx, teacher_logits, valid, tau, grad_loss,
                             lse, n_valid, rows)
        dh[rows] = G @ W
        dW += G.T @ h[rows]
    return dh, dW


def dh_rows(h, W, teacher_idx, teacher_logits, valid, tau: float, grad_loss: float,
            lse, n_valid: int, rows) -> np.ndarray:
    """dh for a sample of rows only: G[rows] W."""
    G = grad_logits_rows(h, W, teacher_idx, teacher_logits, valid, tau, grad_loss,
                         lse, n_valid, rows)
    return G @ _f64(W)


def dW_rows(h, W, teacher_idx, teacher_logits, valid, tau: float, grad_loss: float,
            lse, n_valid: int, vrows, block: int = 1024) -> np.ndarray:
    """dW for a sample of vocabulary rows only: dW[v] = sum_t G_tv h_t.

    Needs the full-row lse (from ``forward``) but only the logits of the sampled
    vocabulary columns, so its cost is T * len(vrows) * d.
    """
    h = _f64(h)
    W = _f64(W)
    vrows = np.asarray(vrows).astype(np.int64)
    T = h.shape[0]
    out = np.zeros((len(vrows), h.shape[1]), dtype=np.float64)
    if n_valid == 0:
        return out
    idx = np.asarray(teacher_idx).astype(np.int64)
    valid_f = np.asarray(valid).astype(np.float64)
    lse = _f64(lse)
    Ws = W[vrows]
    # column of the sample that each vocabulary entry maps to (-1: not sampled);
    # a vocabulary row sampled twice keeps its last position, so callers pass
    # distinct vrows.
    vpos = np.full(W.shape[0], -1, dtype=np.int64)
    vpos[vrows] = np.arange(len(vrows))
    for r0 in range(0, T, block):
        r1 = min(T, r0 + block)
        _, p = teacher_topk_logprobs(np.asarray(teacher_logits)[r0:r1], tau)
        q = np.exp((h[r0:r1] @ Ws.T) / float(tau) - lse[r0:r1, None])
        # teacher mass landing on each sampled column: sum over k of p where idx == v
        scatter = np.zeros_like(q)
        col = vpos[idx[r0:r1]]
        rr, kk = np.nonzero(col >= 0)
        np.add.at(scatter, (rr, col[rr, kk]), p[rr, kk])
        s = float(grad_loss) * valid_f[r0:r1] / float(n_valid) / float(tau)
        G = s[:, None] * (q - scatter)
        out += G.T @ h[r0:r1]
    return out
