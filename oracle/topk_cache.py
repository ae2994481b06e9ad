"""Float64 CPU oracle of the offline teacher cache: top-K logits per position.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (same rules as ``oracle/dense_kl.py``).

"Efficient Knowledge Distillation for LLMs: Offline Top-K Logits and a Fused Chunked KL
Loss", section "Two systems changes", paragraph "Offline distillation": the teacher is run
once, and for every position the 100 most likely tokens and their logits are stored and
reused.  With the teacher's final hidden states Ht [T, d] and LM head Wt [V, d]:

    s = Ht Wt^T                      teacher logits, [T, V]
    row t of the cache: the K ids with the largest s[t, id], ordered by logit descending,
                        ties broken by the lower id; and those logits.

The softmax is monotone, so "most likely" and "largest logit" select the same ids.  The
pages do not say how ties are broken; the lower id first is the plainest deterministic rule.
"""
from __future__ import annotations

import numpy as np


def teacher_topk(Ht, Wt, K: int, chunk: int = 64):
    """(ids int64 [T, K], logits float64 [T, K]) of the K largest teacher logits per row."""
    Ht = np.asarray(Ht, dtype=np.float64)
    Wt = np.asarray(Wt, dtype=np.float64)
    T, V = Ht.shape[0], Wt.shape[0]
    if not 1 <= K <= V:
        raise ValueError("need 1 <= K <= V")
    ids = np.zeros((T, K), dtype=np.int64)
    vals = np.zeros((T, K))
    cols = np.arange(V)
    for b0 in range(0, T, chunk):
        s = Ht[b0:b0 + chunk] @ Wt.T
        for r in range(s.shape[0]):
            order = np.lexsort((cols, -s[r]))[:K]  # by -logit, then by id
            ids[b0 + r] = order
            vals[b0 + r] = s[r, order]
    return ids, vals


def logits_at(Ht, Wt, ids):
    """s[t, ids[t, k]] in float64 (the teacher logit of given ids, one dot product each)."""
    Ht = np.asarray(Ht, dtype=np.float64)
    Wt = np.asarray(Wt, dtype=np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    return np.einsum("td,tkd->tk", Ht, Wt[ids])
