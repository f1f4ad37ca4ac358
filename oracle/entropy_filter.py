"""Plain fp64 CPU oracle of the teacher-entropy token filter.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import it; the library never calls it.

Source: asibiont.com rewrite of "Making Knowledge Distillation Cheap Enough to
Run at Scale", section "Distillation Token Filtering": score every token by the
entropy of the teacher's distribution, skip the near-deterministic (low
entropy) tokens, and, for a batch, keep a fixed percentage of the tokens with
the highest entropy.

Readings (the section gives no formula):

1. The teacher distribution is the one the loss uses: softmax of
   teacher_logits / tau over the K cached entries (renormalised top-K), and
   H_t = -sum_k p_tk log p_tk (natural log).
2. Only rows already valid (valid_in != 0) are candidates; the kept count is
   n_keep = ceil(N_in * keep_num / keep_den) in exact integer arithmetic, the
   fixed percentage being given as the fraction keep_num / keep_den.
3. The kept rows are the n_keep candidates of largest H; equal entropies are
   ordered by row index, the lower row first.
"""

from __future__ import annotations

import numpy as np

from oracle.kd_oracle import teacher_topk_logprobs

__all__ = ["teacher_entropy", "keep_count", "entropy_filter"]


def teacher_entropy(teacher_logits, tau: float) -> np.ndarray:
    """H_t of the renormalised top-K teacher distribution (reading 1), fp64 [T]."""
    logp, p = teacher_topk_logprobs(teacher_logits, tau)
    return -(p * logp).sum(axis=1)


def keep_count(n_in: int, keep_num: int, keep_den: int) -> int:
    """ceil(n_in * keep_num / keep_den) with integers only (reading 2)."""
    return -((-n_in * keep_num) // keep_den)


def entropy_filter(entropy, valid_in, keep_num: int, keep_den: int) -> np.ndarray:
    """uint8 [T] mask of the kept rows for the given per-row entropies
    (readings 2 and 3): sort the candidate rows by (-H, row) and keep the first
    n_keep."""
    H = np.asarray(entropy, dtype=np.float64)
    cand = [int(t) for t in np.nonzero(np.asarray(valid_in))[0]]
    n_keep = keep_count(len(cand), keep_num, keep_den)
    order = sorted(cand, key=lambda t: (-H[t], t))
    out = np.zeros(H.shape[0], dtype=np.uint8)
    out[order[:n_keep]] = 1
    return out
