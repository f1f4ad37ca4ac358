"""Seeded synthetic inputs for the top-K KL distillation loss.

Shared by the tests, the oracle checks and the benchmark.  It draws random
numbers and lays them out; it holds none of the loss's arithmetic.  The one
non-random step, choosing each row's 20 largest student logits for the
"teacher" index recipe, is an input recipe (the teacher's cache agrees with the
student on its top entries) and uses a plain library matmul + top-k.

Workloads (the pages' setting is a 120B teacher with a ~201k vocabulary at 8k
and 32k context; a synthetic cache of the same shape stands in for it):

  tiny_fp32    T=256   d=128  V=4096   K=16  tau=1  chunk=64   fp32, all valid
  small_4k     T=4096  d=2880 V=201088 K=100 tau=1  bf16, 10% rows masked
  ctx_8k       T=8192  d=2880 V=201088 K=100 tau=2  bf16, 10% rows masked
  ctx_32k      T=32768 d=2880 V=201088 K=100 tau=1  bf16, 10% rows masked
  vocab_152k   T=16384 d=4096 V=151936 K=100 tau=1  bf16, 4x4096 packed,
               last 1024 rows of each sequence masked

Draw order from numpy.random.default_rng(seed): h, W, mask, indices, logits.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "workload", "teacher_full_lse"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    V: int
    K: int
    tau: float
    chunk: int
    dtype: str = "bf16"          # storage type of h and W handed to the library
    idx_kind: str = "teacher"    # "uniform" | "teacher"
    mask_kind: str = "random10"  # "all" | "random10" | "packed"
    seq_len: int = 0             # packed mask: sequence length
    pad: int = 0                 # packed mask: padded rows at each sequence end

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 256, 128, 4096, 16, 1.0, 64, dtype="fp32",
                          idx_kind="uniform", mask_kind="all"),
    "small_4k": Workload("small_4k", 4096, 2880, 201088, 100, 1.0, 4096),
    "ctx_8k": Workload("ctx_8k", 8192, 2880, 201088, 100, 2.0, 4096),
    "ctx_32k": Workload("ctx_32k", 32768, 2880, 201088, 100, 1.0, 8192),
    "vocab_152k": Workload("vocab_152k", 16384, 4096, 151936, 100, 1.0, 8192,
                           mask_kind="packed", seq_len=4096, pad=1024),
}


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return w.replace(**overrides) if overrides else w


def _distinct_draws(rng: np.random.Generator, T: int, n: int, V: int,
                    exclude: np.ndarray | None) -> np.ndarray:
    """Per row, n distinct uniform draws from [0, V) avoiding `exclude[row]`.

    Rejection sampling: draw a batch of candidates per row, drop excluded
    values and repeats, keep the first n in draw order.  Rows that come up
    short (vanishingly rare for n << V) draw again from the same generator.
    """
    out = np.empty((T, n), dtype=np.int64)
    m = max(2 * n, n + 32)
    cand = rng.integers(0, V, size=(T, m), dtype=np.int64)
    keep = np.ones((T, m), dtype=bool)
    if exclude is not None and exclude.shape[1] > 0:
        for b0 in range(0, T, 4096):
            b1 = min(T, b0 + 4096)
            keep[b0:b1] &= ~(cand[b0:b1, :, None] == exclude[b0:b1, None, :]).any(axis=2)
    # drop repeats: keep the first occurrence in draw order
    order = np.argsort(cand, axis=1, kind="stable")
    sc = np.take_along_axis(cand, order, axis=1)
    rep = np.zeros_like(keep)
    rep_sorted = np.zeros((T, m), dtype=bool)
    rep_sorted[:, 1:] = sc[:, 1:] == sc[:, :-1]
    np.put_along_axis(rep, order, rep_sorted, axis=1)
    keep &= ~rep
    counts = keep.sum(axis=1)
    for t in range(T):
        if counts[t] >= n:
            out[t] = cand[t][keep[t]][:n]
            continue
        chosen = list(cand[t][keep[t]])
        seen = set(chosen) | (set(exclude[t].tolist()) if exclude is not None else set())
        while len(chosen) < n:
            c = int(rng.integers(0, V))
            if c not in seen:
                seen.add(c)
                chosen.append(c)
        out[t] = np.asarray(chosen, dtype=np.int64)
    return out


def _student_top(h: torch.Tensor, W: torch.Tensor, k: int, device) -> np.ndarray:
    """Indices of each row's k largest entries of h W^T (fp32 product of the
    stored values), in descending order; ties go to the lower index."""
    dev = torch.device(device)
    Wd = W.to(dev, dtype=torch.float32)
    T = h.shape[0]
    out = np.empty((T, k), dtype=np.int64)
    blk = 1024 if dev.type == "cuda" else 256
    prev_tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        for r0 in range(0, T, blk):
            r1 = min(T, r0 + blk)
            z = h[r0:r1].to(dev, dtype=torch.float32) @ Wd.T
            # stable descending sort on (value desc, index asc): topk then re-sort
            vals, ids = torch.topk(z, k, dim=1, largest=True, sorted=True)
            key = torch.stack([-vals.double(), ids.double()], dim=2)
            # resolve exact ties by index
            order = np.lexsort((key[..., 1].cpu().numpy(), key[..., 0].cpu().numpy()), axis=1)
            out[r0:r1] = np.take_along_axis(ids.cpu().numpy(), order, axis=1)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev_tf32
    return out


def make_inputs(w: Workload, seed: int = 0, device=None) -> dict:
    """Build (h, W, teacher_idx, teacher_logits, valid) on the CPU.

    h, W are torch bfloat16 (round-to-nearest-even from fp32 draws) unless
    w.dtype == "fp32"; teacher_idx int32 [T, K]; teacher_logits fp32 [T, K];
    valid uint8 [T].  `device` is only used for the student top-20 product of
    the "teacher" recipe (default: CUDA when present).
    """
    rng = np.random.default_rng(seed)
    T, d, V, K = w.T, w.d, w.V, w.K
    h32 = rng.standard_normal((T, d), dtype=np.float32)
    W32 = rng.standard_normal((V, d), dtype=np.float32)
    W32 *= np.float32(1.0 / np.sqrt(d))
    if w.dtype == "fp32":
        h = torch.from_numpy(h32)
        W = torch.from_numpy(W32)
    else:
        h = torch.from_numpy(h32).to(torch.bfloat16)
        W = torch.from_numpy(W32).to(torch.bfloat16)
    del h32, W32

    valid = np.ones(T, dtype=np.uint8)
    if w.mask_kind == "random10":
        n_bad = int(round(0.1 * T))
        valid[rng.choice(T, size=n_bad, replace=False)] = 0
    elif w.mask_kind == "packed":
        L, P = w.seq_len, w.pad
        for s0 in range(0, T, L):
            valid[max(s0, min(T, s0 + L) - P):min(T, s0 + L)] = 0
    elif w.mask_kind != "all":
        raise ValueError(w.mask_kind)

    if w.idx_kind == "uniform":
        idx = _distinct_draws(rng, T, K, V, None)
        tl = np.sort(rng.normal(0.0, 2.0, size=(T, K)).astype(np.float32), axis=1)[:, ::-1].copy()
    elif w.idx_kind == "teacher":
        n_top = min(20, K)
        if device is None:
            device = "cuda" if torch.cuda.is_available() else "cpu"
        top = _student_top(h, W, n_top, device)
        rest = _distinct_draws(rng, T, K - n_top, V, top)
        idx = np.concatenate([top, rest], axis=1)
        first = 8.0 + rng.gumbel(0.0, 1.0, size=(T, 1))
        gaps = rng.exponential(0.3, size=(T, K - 1))
        tl = np.concatenate([first, first - np.cumsum(gaps, axis=1)], axis=1).astype(np.float32)
    else:
        raise ValueError(w.idx_kind)

    return {
        "h": h.contiguous(),
        "W": W.contiguous(),
        "teacher_idx": torch.from_numpy(np.ascontiguousarray(idx.astype(np.int32))),
        "teacher_logits": torch.from_numpy(np.ascontiguousarray(tl)),
        "valid": torch.from_numpy(valid),
        "tau": float(w.tau),
        "workload": w,
    }


def teacher_full_lse(teacher_logits: torch.Tensor, tau: float, seed: int = 0,
                     lo: float = 0.05, hi: float = 0.5) -> torch.Tensor:
    """Full-vocabulary log-normaliser of a synthetic teacher, for the
    residual-mass variant of the loss: per row a share r ~ U(lo, hi) of the
    teacher's probability mass (at temperature tau) lies outside its cached
    entries, so L = logsumexp(teacher_logits / tau) - log(1 - r).  fp32 [T].
    Draws from its own generator (seed), after the other inputs."""
    rng = np.random.default_rng(seed + 7919)
    a = teacher_logits.double().numpy() / float(tau)
    m = a.max(axis=1)
    lse_k = m + np.log(np.exp(a - m[:, None]).sum(axis=1))
    r = rng.uniform(lo, hi, size=a.shape[0])
    return torch.from_numpy((lse_k - np.log1p(-r)).astype(np.float32))
