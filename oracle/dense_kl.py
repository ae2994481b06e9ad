"""Float64 CPU oracle of the KL distillation loss against a cached teacher top-K.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference leg may import or call this module.  The CUDA
library never calls it and shares no code with it.

What it computes follows "Efficient Knowledge Distillation for LLMs: Offline Top-K Logits
and a Fused Chunked KL Loss" (Hugging Face blog post, section "Two systems changes"):

* the teacher is represented only by its cached top-K (id, logit) pairs per position
  (paragraph "Offline distillation");
* the loss is computed the way the post's "Dense KL" paragraph describes the
  correctness baseline: the student's full row of logits over the vocabulary is
  materialised (here one block of rows at a time) and compared with the teacher's
  distribution rebuilt from the cached top-K;
* the post says the three formulations (dense, forward-chunked, fused chunked) are
  mathematically equivalent, so this plain dense computation is the value the fused
  GPU path must reproduce.

The pages print no formula.  The one used here (and its readings of what the pages
leave open) is:

    s   = H W^T                      student logits, [T, V]
    a   = s / tau                    tempered student logits
    lse_t = log sum_v exp(a_tv)      natural log, over the full vocabulary
    p_t = softmax(z_t / tau)         over the K cached teacher slots only
    KL_t = sum_k p_tk (log p_tk - (a_{t, id_tk} - lse_t)),   0 * log 0 = 0
    L   = tau^2 / N * sum_{t valid} KL_t,   N = number of valid tokens (L = 0 if N = 0)

and its exact gradient, with g the upstream gradient of L:

    dS_tv = g * tau / N * (q_tv - ptilde_tv)   for valid t, 0 for masked t
    q_tv  = exp(a_tv - lse_t),  ptilde_t = p_t scattered (added) to the ids of row t
    dH = dS W,   dW = dS^T H

The post names this the "closed-form gradient behind the fused chunked loss" without
printing it; the expression above is the derivative of L and is checked against finite
differences and torch.autograd in the tests.

Normalisation (the pages mention sequence packing without fixing the loss's normaliser).
``norm="tokens"`` is the formula above.  ``norm="sequences"`` averages per packed sequence
first: with seq_ids[t] the sequence of token t, N_s the valid tokens of sequence s and S the
number of sequences with N_s > 0,

    L = tau^2 / S * sum_{s : N_s > 0} (1 / N_s) * sum_{t valid, seq t = s} KL_t,

i.e. every token carries the weight w_t = 1 / (S N_{s(t)}) instead of 1 / N, and the gradient
is the same expression with tau / N replaced by tau * w_t.

A batch split over several calls (token shards on data-parallel GPUs, or micro-batches).  The
pages' GPT-OSS 20B run trains on one node of several GPUs ("Scaling to long context lengths")
without saying how the loss is normalised across them; the plainest reading is the loss of the
whole batch.  ``count`` is then the whole batch's N (or S, each sequence within one shard),
given to every shard in place of its own: shard r computes tau^2 / count * sum over its valid
tokens of KL_t, and the shards' losses and gradients add up to the whole batch's.  ``count``
must not be below the shard's own count.

Everything is float64.  H and W arrive as bfloat16 on the GPU path; ``to_f64`` widens
them exactly.  Rows are processed in blocks of ``chunk`` rows (a dense [chunk, V] block
of logits at a time); the result does not depend on ``chunk`` beyond float64 rounding.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np


def to_f64(x) -> np.ndarray:
    """Exact widening of a torch tensor (bf16/fp32/int) or array to a float64 ndarray."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover - torch is always present in this repo
        pass
    return np.asarray(x, dtype=np.float64)


def _np(x, dtype=None) -> np.ndarray:
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu").numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=dtype)


def teacher_probs(topk_logits, tau: float):
    """p = softmax(z / tau) over the K cached slots of each row, and log p.

    Slots whose logit is -inf get p = 0 and log p = -inf.  A row whose logits are all
    -inf has no distribution and is rejected.
    """
    z = _np(topk_logits, np.float64) / float(tau)
    zmax = np.max(z, axis=1, keepdims=True)
    if not np.all(np.isfinite(zmax)):
        raise ValueError("a teacher row has no finite logit")
    e = np.exp(z - zmax)
    Z = np.sum(e, axis=1, keepdims=True)
    p = e / Z
    with np.errstate(divide="ignore"):
        logp = (z - zmax) - np.log(Z)
    return p, logp


def _own_count(n: int, count) -> int:
    """The mean's count: the batch's ``count`` when given (not below this shard's own n)."""
    if count is None:
        return n
    if int(count) < n:
        raise ValueError("count is below the shard's own count")
    return int(count)


def token_weights(mask, T: int, norm: str = "tokens", seq_ids=None, count=None) -> np.ndarray:
    """w_t, the weight of token t's KL in the loss (before tau^2): 1/N for valid tokens under
    the token mean; 1/(S N_s) under the sequence mean; 0 for masked tokens.  ``count``
    replaces N (or S) by the whole batch's when the batch is split over several calls."""
    msk = np.ones(T, dtype=bool) if mask is None else _np(mask).astype(bool)
    w = np.zeros(T)
    if norm == "tokens":
        n = _own_count(int(msk.sum()), count)
        if n:
            w[msk] = 1.0 / n
        return w
    if norm != "sequences":
        raise ValueError(norm)
    if seq_ids is None:
        raise ValueError("seq_ids are needed for the sequence mean")
    sid = _np(seq_ids, np.int64)
    if sid.shape != (T,) or (T and sid.min() < 0):
        raise ValueError("seq_ids must be [T] non-negative")
    counts = {}
    for t in np.flatnonzero(msk):
        counts[int(sid[t])] = counts.get(int(sid[t]), 0) + 1
    S = _own_count(len(counts), count)
    for t in np.flatnonzero(msk):
        w[t] = 1.0 / (S * counts[int(sid[t])])
    return w


def _check(H, W, idx, V):
    if H.ndim != 2 or W.ndim != 2 or H.shape[1] != W.shape[1]:
        raise ValueError("H must be [T, d] and W [V, d]")
    if idx.size and (idx.min() < 0 or idx.max() >= V):
        raise ValueError("teacher id out of range [0, V)")


def _row_terms(s_blk: np.ndarray, idx_blk: np.ndarray, p_blk: np.ndarray, logp_blk: np.ndarray,
               tau: float):
    """lse and KL for one block of rows, from its dense logits s_blk [rows, V]."""
    a = s_blk / tau
    m = np.max(a, axis=1, keepdims=True)
    lse = (m + np.log(np.sum(np.exp(a - m), axis=1, keepdims=True)))[:, 0]
    log_q_at_ids = np.take_along_axis(a, idx_blk, axis=1) - lse[:, None]
    safe_logp = np.where(p_blk > 0, logp_blk, 0.0)  # 0 * log 0 = 0
    return lse, np.sum(p_blk * (safe_logp - log_q_at_ids), axis=1)


def forward(H, W, topk_idx, topk_logits, mask, tau: float, chunk: int = 64,
            rows: Optional[Sequence[int]] = None, norm: str = "tokens", seq_ids=None, count=None):
    """Loss, per-token lse and per-token KL.

    H [T, d] and W [V, d] are float64 arrays (see ``to_f64``); topk_idx [T, K] ints;
    topk_logits [T, K]; mask [T] (1 = valid, None = all valid).

    With ``rows`` given, lse and KL are computed only for those rows (returned in that
    order) and the loss is computed only if every valid row is among them; otherwise
    ``loss`` is None.  This keeps exact checks affordable at full vocabulary size.
    ``norm`` / ``seq_ids`` select the normaliser and ``count`` the whole batch's count of a
    split batch (module docstring).
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = _np(topk_idx, np.int64)
    T, V = H.shape[0], W.shape[0]
    _check(H, W, idx, V)
    msk = np.ones(T, dtype=bool) if mask is None else _np(mask).astype(bool)
    n_valid = int(msk.sum())
    sel = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    p, logp = teacher_probs(_np(topk_logits)[sel] if len(sel) else np.zeros((0, idx.shape[1])), tau)
    lse = np.zeros(len(sel))
    kl = np.zeros(len(sel))
    for b0 in range(0, len(sel), chunk):
        r = sel[b0:b0 + chunk]
        s_blk = H[r] @ W.T
        lse[b0:b0 + chunk], kl[b0:b0 + chunk] = _row_terms(
            s_blk, idx[r], p[b0:b0 + chunk], logp[b0:b0 + chunk], tau)
    loss = None
    covered = set(sel.tolist())
    if all(t in covered for t in np.flatnonzero(msk).tolist()):
        if n_valid == 0:
            loss = 0.0
        elif norm == "tokens":
            valid_sel = msk[sel]
            loss = float(tau) ** 2 / _own_count(n_valid, count) * float(np.sum(kl[valid_sel]))
        else:
            wts = token_weights(mask, T, norm, seq_ids, count)[sel]
            loss = float(tau) ** 2 * float(np.sum(wts * kl))
    return {"loss": loss, "lse": lse, "kl": kl, "n_valid": n_valid, "rows": sel}


def _ds_block(s_blk, idx_blk, p_blk, valid_blk, tau, scale):
    """dS for one block of rows: scale * (q - ptilde), zero on masked rows.  ``scale`` is a
    number or one value per row."""
    a = s_blk / tau
    m = np.max(a, axis=1, keepdims=True)
    e = np.exp(a - m)
    q = e / np.sum(e, axis=1, keepdims=True)
    ptilde = np.zeros_like(q)
    rr = np.repeat(np.arange(q.shape[0]), idx_blk.shape[1])
    np.add.at(ptilde, (rr, idx_blk.reshape(-1)), p_blk.reshape(-1))
    scale = np.asarray(scale, dtype=np.float64)
    ds = (scale[:, None] if scale.ndim else scale) * (q - ptilde)
    ds[~valid_blk] = 0.0
    return ds


def backward(H, W, topk_idx, topk_logits, mask, tau: float, grad: float = 1.0, chunk: int = 64,
             norm: str = "tokens", seq_ids=None, count=None):
    """dH [T, d] and dW [V, d] in float64, the exact gradient of ``forward``'s loss."""
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = _np(topk_idx, np.int64)
    T, V = H.shape[0], W.shape[0]
    _check(H, W, idx, V)
    msk = np.ones(T, dtype=bool) if mask is None else _np(mask).astype(bool)
    n_valid = int(msk.sum())
    dH = np.zeros_like(H)
    dW = np.zeros_like(W)
    if n_valid == 0:
        return dH, dW
    row_scale = float(grad) * float(tau) * token_weights(mask, T, norm, seq_ids, count)
    p, _ = teacher_probs(topk_logits, tau)
    for b0 in range(0, T, chunk):
        r = slice(b0, min(T, b0 + chunk))
        s_blk = H[r] @ W.T
        ds = _ds_block(s_blk, idx[r], p[r], msk[r], tau, row_scale[r])
        dH[r] = ds @ W
        dW += ds.T @ H[r]
    return dH, dW


def dH_rows(H, W, topk_idx, topk_logits, mask, tau: float, rows: Sequence[int], grad: float = 1.0,
            chunk: int = 64, count=None):
    """Selected rows of dH.  Row t of dH needs only row t of the logits, so this is exact
    at any size."""
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = _np(topk_idx, np.int64)
    T = H.shape[0]
    msk = np.ones(T, dtype=bool) if mask is None else _np(mask).astype(bool)
    n_valid = int(msk.sum())
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), H.shape[1]))
    if n_valid == 0:
        return out
    scale = float(grad) * float(tau) / _own_count(n_valid, count)
    p, _ = teacher_probs(_np(topk_logits)[rows], tau)
    for b0 in range(0, len(rows), chunk):
        r = rows[b0:b0 + chunk]
        ds = _ds_block(H[r] @ W.T, idx[r], p[b0:b0 + chunk], msk[r], tau, scale)
        out[b0:b0 + chunk] = ds @ W
    return out


def dW_rows(H, W, topk_idx, topk_logits, mask, tau: float, vocab_rows: Sequence[int],
            grad: float = 1.0, chunk: int = 64, count=None):
    """Selected rows of dW.  Row v of dW sums dS[t, v] H[t] over the valid tokens, so it
    needs lse of every valid token: affordable when few tokens are valid."""
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = _np(topk_idx, np.int64)
    T = H.shape[0]
    msk = np.ones(T, dtype=bool) if mask is None else _np(mask).astype(bool)
    n_valid = int(msk.sum())
    vrows = np.asarray(vocab_rows, dtype=np.int64)
    out = np.zeros((len(vrows), H.shape[1]))
    if n_valid == 0:
        return out
    scale = float(grad) * float(tau) / _own_count(n_valid, count)
    valid = np.flatnonzero(msk)
    p, _ = teacher_probs(_np(topk_logits)[valid], tau)
    for b0 in range(0, len(valid), chunk):
        r = valid[b0:b0 + chunk]
        ds = _ds_block(H[r] @ W.T, idx[r], p[b0:b0 + chunk], np.ones(len(r), bool), tau, scale)
        out += ds[:, vrows].T @ H[r]
    return out
