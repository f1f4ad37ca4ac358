"""Plain fp64 CPU oracle of the teacher-side top-K cache producer.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import it; the library never calls it.

Source: aipuls.nl summary of "Making Knowledge Distillation Cheap Enough to
Run at Scale", section "Summary": the teacher runs once and its top-100
logits per token position are cached offline.  The pages do not say how ties
are broken or what else goes into the cache.  Readings:

1. The cached logits are the raw teacher logits z = h W^T (no temperature);
   per row the K largest, in descending order, with their vocabulary indices.
2. Equal logits are ordered by vocabulary index, the lower index first (so the
   result is unique: the first K of the row sorted by (-z, index)).
3. With the cache the producer also returns the teacher's full-vocabulary
   log-normaliser at temperature tau, L_t = log sum_v exp(z_tv / tau), which the
   residual-mass variant of the loss consumes.
"""

from __future__ import annotations

import numpy as np

from oracle.kd_oracle import _f64, _logsumexp_rows

__all__ = ["teacher_topk"]


def teacher_topk(h, W, K: int, tau: float, block: int = 256):
    """(idx int64 [T, K], logits fp64 [T, K], full_lse fp64 [T]) by the plain
    definition: form each row's logits, sort by (-z, index), keep the first K."""
    h = _f64(h)
    W = _f64(W)
    T = h.shape[0]
    V = W.shape[0]
    idx = np.empty((T, K), dtype=np.int64)
    val = np.empty((T, K))
    lse = np.empty(T)
    cols = np.arange(V)
    for r0 in range(0, T, block):
        r1 = min(T, r0 + block)
        z = h[r0:r1] @ W.T
        lse[r0:r1] = _logsumexp_rows(z / float(tau))
        for i in range(r1 - r0):
            order = np.lexsort((cols, -z[i]))[:K]
            idx[r0 + i] = order
            val[r0 + i] = z[i, order]
    return idx, val, lse
