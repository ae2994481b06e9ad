"""Float64 CPU oracle of the distillation loss under other divergences than KL(p || q).

TEST INFRASTRUCTURE, NOT PRODUCT CODE (same rules as ``oracle/dense_kl.py``): only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU leg may import it; the CUDA
library never calls it and shares no code with it.

Source.  "Efficient Knowledge Distillation for LLMs: Offline Top-K Logits and a Fused
Chunked KL Loss" (Hugging Face blog post, closing section) says that the paper also
ablates the choice of loss function, without naming the alternatives.  The reading taken
here: divergences D(ptilde_t || q_t) between the teacher's distribution ptilde_t (the
softmax of the K cached logits over the K slots, scattered onto the vocabulary and added
where an id repeats; zero at every other id) and the student's full softmax q_t, restricted
to those that stay finite where ptilde has zeros, so that a top-K teacher can be used
without a tail bucket:

    "kl"        KL(p || q)            = sum_v p log(p / q)
    "jsd"       JSD_b(p, q)           = b KL(p || m) + (1 - b) KL(q || m),  m = b p + (1 - b) q,
                                        0 < b < 1 (b = 1/2: the Jensen-Shannon divergence)
    "skew_kl"   SKL_a(p, q)           = KL(p || a p + (1 - a) q),   0 <= a < 1  (a = 0: KL)
    "skew_rkl"  SRKL_a(p, q)          = KL(q || a q + (1 - a) p),   0 < a <= 1
    "tv"        TV(p, q)              = 1/2 sum_v |p - q|

with p = ptilde_t, q = q_t = softmax(s_t / tau) over all V ids, 0 log 0 = 0, and the loss

    L = tau^2 sum_t w_t D(ptilde_t || q_t)

with the token weights of ``dense_kl.token_weights`` (1/N, or 1/(S N_s) for the sequence
mean; 0 for masked tokens).  The tau^2 factor is kept for every divergence, as for KL.

Gradient.  D is a function of the vector q.  With gamma_v = dD/dq_v taken with the entries of
q as independent variables, and dq_u/ds_v = q_u (delta_uv - q_v) / tau,

    dD/ds_v  = q_v (gamma_v - sum_u q_u gamma_u) / tau,
    dS_tv    = g tau w_t q_tv (gamma_tv - sum_u q_tu gamma_tu),    dH = dS W,  dW = dS^T H,

where, elementwise in (p, q) = (ptilde_tv, q_tv):

    kl        gamma = -p / q
    jsd       gamma = (1 - b) log(q / m)
    skew_kl   gamma = -(1 - a) p / (a p + (1 - a) q)
    skew_rkl  gamma = log(q / m') + 1 - a q / m',    m' = a q + (1 - a) p
    tv        gamma = -sign(p - q) / 2               (sign(0) = 0: a subgradient)

Everything below evaluates these over the dense [rows, V] block of logits, one block of
rows at a time, as written; the tests pin the divergences to SciPy's routines and brute
force and the gradients to finite differences of ``forward``.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .dense_kl import _check, _np, teacher_probs, token_weights

KINDS = ("kl", "jsd", "skew_kl", "skew_rkl", "tv")


def check_param(kind: str, param: float) -> float:
    """The divergence's parameter (b for "jsd", a for the skew forms; ignored otherwise)."""
    if kind not in KINDS:
        raise ValueError(f"unknown divergence {kind!r}")
    param = float(param)
    if kind == "jsd" and not 0.0 < param < 1.0:
        raise ValueError("jsd needs 0 < b < 1")
    if kind == "skew_kl" and not 0.0 <= param < 1.0:
        raise ValueError("skew_kl needs 0 <= a < 1")
    if kind == "skew_rkl" and not 0.0 < param <= 1.0:
        raise ValueError("skew_rkl needs 0 < a <= 1")
    return param


def _xlogy_ratio(x, y):
    """x log(x / y) elementwise with 0 log(0 / y) = 0."""
    out = np.zeros_like(x)
    nz = x > 0
    out[nz] = x[nz] * np.log(x[nz] / y[nz])
    return out


def divergence_rows(p, q, kind: str, param: float) -> np.ndarray:
    """D(p_r || q_r) for each row r of dense distributions p, q [rows, V]."""
    b = a = param
    if kind == "kl":
        return np.sum(_xlogy_ratio(p, q), axis=1)
    if kind == "jsd":
        m = b * p + (1.0 - b) * q
        return b * np.sum(_xlogy_ratio(p, m), axis=1) + (1.0 - b) * np.sum(_xlogy_ratio(q, m), axis=1)
    if kind == "skew_kl":
        return np.sum(_xlogy_ratio(p, a * p + (1.0 - a) * q), axis=1)
    if kind == "skew_rkl":
        return np.sum(_xlogy_ratio(q, a * q + (1.0 - a) * p), axis=1)
    if kind == "tv":
        return 0.5 * np.sum(np.abs(p - q), axis=1)
    raise ValueError(kind)


def gamma(p, q, kind: str, param: float) -> np.ndarray:
    """dD/dq elementwise (module docstring), for q > 0."""
    b = a = param
    if kind == "kl":
        return -p / q
    if kind == "jsd":
        return (1.0 - b) * np.log(q / (b * p + (1.0 - b) * q))
    if kind == "skew_kl":
        return -(1.0 - a) * p / (a * p + (1.0 - a) * q)
    if kind == "skew_rkl":
        m = a * q + (1.0 - a) * p
        return np.log(q / m) + 1.0 - a * q / m
    if kind == "tv":
        return -0.5 * np.sign(p - q)
    raise ValueError(kind)


def _dense_block(s_blk, idx_blk, p_blk, tau):
    """(q, ptilde, lse) of one block of rows from its dense logits [rows, V]."""
    a = s_blk / tau
    mx = np.max(a, axis=1, keepdims=True)
    lse = mx + np.log(np.sum(np.exp(a - mx), axis=1, keepdims=True))
    q = np.exp(a - lse)
    pt = np.zeros_like(q)
    rr = np.repeat(np.arange(q.shape[0]), idx_blk.shape[1])
    np.add.at(pt, (rr, idx_blk.reshape(-1)), p_blk.reshape(-1))
    return q, pt, lse[:, 0]


def forward(H, W, topk_idx, topk_logits, mask, tau: float, kind: str, param: float = 0.5,
            chunk: int = 64, rows: Optional[Sequence[int]] = None, norm: str = "tokens",
            seq_ids=None):
    """Loss, lse, per-token divergence and the student logits at the cached ids.

    Arguments as ``dense_kl.forward``.  Returns dict(loss, lse [rows], div [rows],
    s_at_ids [rows, K], rows); ``loss`` is None unless every valid row is among ``rows``.
    """
    param = check_param(kind, param)
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = _np(topk_idx, np.int64)
    T, V = H.shape[0], W.shape[0]
    _check(H, W, idx, V)
    msk = np.ones(T, dtype=bool) if mask is None else _np(mask).astype(bool)
    sel = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    K = idx.shape[1]
    p, _ = teacher_probs(_np(topk_logits)[sel] if len(sel) else np.zeros((0, K)), tau)
    lse = np.zeros(len(sel))
    div = np.zeros(len(sel))
    s_ids = np.zeros((len(sel), K))
    for b0 in range(0, len(sel), chunk):
        r = sel[b0:b0 + chunk]
        s_blk = H[r] @ W.T
        q, pt, lse[b0:b0 + chunk] = _dense_block(s_blk, idx[r], p[b0:b0 + chunk], tau)
        div[b0:b0 + chunk] = divergence_rows(pt, q, kind, param)
        s_ids[b0:b0 + chunk] = np.take_along_axis(s_blk, idx[r], axis=1)
    loss = None
    covered = set(sel.tolist())
    if all(t in covered for t in np.flatnonzero(msk).tolist()):
        wts = token_weights(mask, T, norm, seq_ids)[sel]
        loss = float(tau) ** 2 * float(np.sum(wts * div))
    return {"loss": loss, "lse": lse, "div": div, "s_at_ids": s_ids, "rows": sel}


def ds_block(s_blk, idx_blk, p_blk, tau, row_scale, kind: str, param: float):
    """dS of one block of rows: row_scale_t * q (gamma - sum_u q gamma) with row_scale_t =
    g tau w_t (zero rows stay zero)."""
    q, pt, _ = _dense_block(s_blk, idx_blk, p_blk, tau)
    gm = gamma(pt, q, kind, param)
    gbar = np.sum(q * gm, axis=1, keepdims=True)
    ds = np.asarray(row_scale, dtype=np.float64)[:, None] * q * (gm - gbar)
    ds[np.asarray(row_scale) == 0] = 0.0
    return ds


def backward(H, W, topk_idx, topk_logits, mask, tau: float, kind: str, param: float = 0.5,
             grad: float = 1.0, chunk: int = 64, norm: str = "tokens", seq_ids=None):
    """dH [T, d] and dW [V, d] in float64, the gradient of ``forward``'s loss."""
    param = check_param(kind, param)
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = _np(topk_idx, np.int64)
    T, V = H.shape[0], W.shape[0]
    _check(H, W, idx, V)
    dH = np.zeros_like(H)
    dW = np.zeros_like(W)
    row_scale = float(grad) * float(tau) * token_weights(mask, T, norm, seq_ids)
    if not np.any(row_scale):
        return dH, dW
    p, _ = teacher_probs(topk_logits, tau)
    for b0 in range(0, T, chunk):
        r = slice(b0, min(T, b0 + chunk))
        ds = ds_block(H[r] @ W.T, idx[r], p[r], tau, row_scale[r], kind, param)
        dH[r] = ds @ W
        dW += ds.T @ H[r]
    return dH, dW


def dH_rows(H, W, topk_idx, topk_logits, mask, tau: float, kind: str, param: float, rows: Sequence[int],
            grad: float = 1.0, chunk: int = 64, norm: str = "tokens", seq_ids=None):
    """Selected rows of dH: row t needs only row t of the logits (exact at any size)."""
    param = check_param(kind, param)
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = _np(topk_idx, np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    row_scale = float(grad) * float(tau) * token_weights(mask, H.shape[0], norm, seq_ids)[rows]
    p, _ = teacher_probs(_np(topk_logits)[rows], tau)
    out = np.zeros((len(rows), H.shape[1]))
    for b0 in range(0, len(rows), chunk):
        r = rows[b0:b0 + chunk]
        ds = ds_block(H[r] @ W.T, idx[r], p[b0:b0 + chunk], tau, row_scale[b0:b0 + chunk], kind, param)
        out[b0:b0 + chunk] = ds @ W
    return out


def dW_rows(H, W, topk_idx, topk_logits, mask, tau: float, kind: str, param: float,
            vocab_rows: Sequence[int], grad: float = 1.0, chunk: int = 64, norm: str = "tokens",
            seq_ids=None):
    """Selected rows of dW: row v sums dS[t, v] H[t] over the tokens with a nonzero weight, so it
    needs those tokens' logits (affordable when few tokens are valid)."""
    param = check_param(kind, param)
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = _np(topk_idx, np.int64)
    vr = np.asarray(vocab_rows, dtype=np.int64)
    scale = float(grad) * float(tau) * token_weights(mask, H.shape[0], norm, seq_ids)
    live = np.flatnonzero(scale)
    p, _ = teacher_probs(_np(topk_logits)[live], tau)
    out = np.zeros((len(vr), H.shape[1]))
    for b0 in range(0, len(live), chunk):
        r = live[b0:b0 + chunk]
        ds = ds_block(H[r] @ W.T, idx[r], p[b0:b0 + chunk], tau, scale[r], kind, param)
        out += ds[:, vr].T @ H[r]
    return out
