"""Seeded synthetic workloads for the fused chunked KL distillation loss.

This module only draws random inputs.  It holds none of the loss arithmetic, so both
the CUDA path (through the tests and the benchmark) and the float64 oracle can be
fed from it without sharing any code with each other.

The five workloads mirror the shapes the pages' experiments use:

* a tiny case the oracle finishes in milliseconds;
* a Llama-3.2-3B-like student at 8K tokens (vocabulary 128,256, d = 3072), the
  8K distillation setting of "Efficient Knowledge Distillation for LLMs"
  ("What this changes in practice");
* a gpt-oss-20b-like student at 32K tokens (vocabulary 201,088, d = 2880), the
  32,768-token GPT-OSS 20B setting ("Scaling to long context lengths");
* the same student at 256K tokens, the long-context projection-only setting;
* a packed batch of four 16K sequences with temperature 2 and trailing padding.

Every input is synthetic: there is no teacher model and no corpus.  The teacher cache
(top-K ids and logits per position, "Two systems changes", offline distillation) is
drawn directly: K distinct ids per row and K logits sorted in descending order.

Every workload draws from ``numpy.random.SeedSequence(1000 + number)``, split into five
child streams in a fixed order: W, H, ids (with the vocabulary permutation), logits, mask.
W and H are drawn in blocks of 4096 rows, block b from child b of their stream, so blocks
can be drawn on several threads and the first rows of H do not depend on how many rows are
drawn.  Floats are drawn in float32 and H, W are rounded to bfloat16 with
round-to-nearest-even (``torch.Tensor.to``).
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and value distributions of one synthetic workload."""

    number: int
    name: str
    T: int
    d: int
    V: int
    K: int
    tau: float
    chunk: int
    w_std: float
    logit_mean: float
    logit_std: float
    ids: str  # "uniform" or "zipf80"
    mask: str  # "none", "random2pct" or "trailing10pct4seq"
    n_seq: int = 1

    @property
    def seed(self) -> int:
        return 1000 + self.number

    @property
    def flops_fwd_bwd(self) -> float:
        """8*T*V*d: forward projection, recompute, dH and dW products (2*T*V*d each)."""
        return 8.0 * self.T * self.V * self.d


WORKLOADS = {
    "tiny": Workload(1, "tiny", T=256, d=256, V=4096, K=16, tau=1.0, chunk=64,
                     w_std=0.02, logit_mean=5.0, logit_std=3.0, ids="uniform", mask="none"),
    "llama3b_8k": Workload(2, "llama3b_8k", T=8192, d=3072, V=128256, K=100, tau=1.0, chunk=1024,
                           w_std=0.02, logit_mean=8.0, logit_std=3.0, ids="uniform",
                           mask="random2pct"),
    "gptoss20b_32k": Workload(3, "gptoss20b_32k", T=32768, d=2880, V=201088, K=100, tau=1.0,
                              chunk=2048, w_std=0.02, logit_mean=8.0, logit_std=3.0,
                              ids="zipf80", mask="none"),
    "gptoss20b_256k": Workload(4, "gptoss20b_256k", T=262144, d=2880, V=201088, K=100, tau=1.0,
                               chunk=4096, w_std=0.02, logit_mean=8.0, logit_std=3.0,
                               ids="zipf80", mask="none"),
    "packed4x16k_tau2": Workload(5, "packed4x16k_tau2", T=65536, d=4096, V=151936, K=100, tau=2.0,
                                 chunk=4096, w_std=0.015, logit_mean=6.0, logit_std=4.0,
                                 ids="uniform", mask="trailing10pct4seq", n_seq=4),
}


@dataclasses.dataclass
class Inputs:
    """One batch of host-side inputs (CPU tensors)."""

    H: torch.Tensor            # bf16 [T, d]
    W: torch.Tensor            # bf16 [V, d]
    topk_idx: torch.Tensor     # int32 [T, K]
    topk_logits: torch.Tensor  # float32 [T, K], descending per row
    mask: torch.Tensor         # uint8 [T], 1 = valid token
    tau: float
    chunk: int


def _normal_f32(rng: np.random.Generator, shape, std: float, mean: float = 0.0) -> np.ndarray:
    out = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    if mean != 0.0:
        out += np.float32(mean)
    return out


ROW_BLOCK = 4096


def _normal_bf16_rows(seq: np.random.SeedSequence, rows: int, cols: int, std: float,
                      keep: int) -> torch.Tensor:
    """N(0, std^2) bf16 matrix [keep, cols]: the first `keep` of `rows` rows, block b of
    ROW_BLOCK rows drawn from child b of `seq` (on several threads)."""
    nblocks = (rows + ROW_BLOCK - 1) // ROW_BLOCK
    children = seq.spawn(nblocks)
    out = torch.empty((keep, cols), dtype=torch.bfloat16)
    need = (keep + ROW_BLOCK - 1) // ROW_BLOCK

    def block(b):
        r0 = b * ROW_BLOCK
        r1 = min(keep, r0 + ROW_BLOCK)
        full = min(rows, r0 + ROW_BLOCK) - r0
        x = _normal_f32(np.random.default_rng(children[b]), (full, cols), std)
        out[r0:r1] = torch.from_numpy(x[: r1 - r0])

    workers = max(1, min(16, len(os.sched_getaffinity(0))))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(block, range(need)))
    return out


def _first_distinct_in_draw_order(draws: np.ndarray, want: int, skip: int = 0) -> Optional[np.ndarray]:
    """Per row, the first ``want`` values that do not repeat an earlier value of the row.

    Values at positions < ``skip`` count as already taken but are not returned.  This is
    rejection sampling of distinct values, done for many rows at once.  Returns None when
    some row has too few distinct values (the caller redraws).
    """
    R, B = draws.shape
    order = np.argsort(draws, axis=1, kind="stable")
    srt = np.take_along_axis(draws, order, axis=1)
    first_sorted = np.ones_like(srt, dtype=bool)
    first_sorted[:, 1:] = srt[:, 1:] != srt[:, :-1]
    is_first = np.empty_like(first_sorted)
    np.put_along_axis(is_first, order, first_sorted, axis=1)
    is_first[:, :skip] = False
    if (is_first.sum(axis=1) < want).any():
        return None
    pos = np.argsort(~is_first, axis=1, kind="stable")[:, :want]
    return np.take_along_axis(draws, pos, axis=1)


def _distinct_uniform(rng: np.random.Generator, T: int, K: int, V: int) -> np.ndarray:
    out = np.empty((T, K), dtype=np.int64)
    margin = max(8, 2 * K * K // max(V, 1) + 8)
    for r0 in range(0, T, 8192):
        r1 = min(T, r0 + 8192)
        while True:
            draws = rng.integers(0, V, size=(r1 - r0, K + margin), dtype=np.int64)
            got = _first_distinct_in_draw_order(draws, K)
            if got is not None:
                break
            margin *= 2
        out[r0:r1] = got
    return out


def _zipf80_uniform20(rng: np.random.Generator, T: int, K: int, V: int, s: float = 1.1) -> np.ndarray:
    """80% of each row: distinct draws of finite Zipf(s) over ranks 1..V, mapped through one
    seeded vocabulary permutation; the rest: distinct uniform ids not already in the row."""
    n_zipf = int(round(0.8 * K))
    n_unif = K - n_zipf
    perm = rng.permutation(V).astype(np.int64)
    ranks = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    out = np.empty((T, K), dtype=np.int64)
    for r0 in range(0, T, 4096):
        r1 = min(T, r0 + 4096)
        batch = 6 * n_zipf + 64
        while True:
            u = rng.random((r1 - r0, batch))
            draws = np.minimum(np.searchsorted(cdf, u, side="right"), V - 1)  # rank - 1
            got = _first_distinct_in_draw_order(draws, n_zipf)
            if got is not None:
                break
            batch *= 2
        zipf_ids = perm[got]
        extra = 2 * n_unif + 16
        while True:
            unif = rng.integers(0, V, size=(r1 - r0, extra), dtype=np.int64)
            both = np.concatenate([zipf_ids, unif], axis=1)
            got_u = _first_distinct_in_draw_order(both, n_unif, skip=n_zipf)
            if got_u is not None:
                break
            extra *= 2
        out[r0:r1, :n_zipf] = zipf_ids
        out[r0:r1, n_zipf:] = got_u
    return out


def _mask(w: Workload, rng: np.random.Generator) -> np.ndarray:
    mask = np.ones(w.T, dtype=np.uint8)
    if w.mask == "random2pct":
        n = int(round(0.02 * w.T))
        mask[rng.choice(w.T, size=n, replace=False)] = 0
    elif w.mask == "trailing10pct4seq":
        L = w.T // w.n_seq
        pad = int(math.floor(0.1 * L))
        for s in range(w.n_seq):
            mask[(s + 1) * L - pad:(s + 1) * L] = 0
    elif w.mask != "none":
        raise ValueError(w.mask)
    return mask


def make_inputs(w: Workload | str, rows: Optional[int] = None) -> Inputs:
    """Draw the seeded inputs of workload ``w``.

    ``rows`` keeps only the first ``rows`` tokens (the draws are the same, truncated), which
    gives a bounded sample of the workload for CPU timing.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    n = w.T if rows is None else rows
    sW, sH, sI, sL, sM = np.random.SeedSequence(w.seed).spawn(5)
    W = _normal_bf16_rows(sW, w.V, w.d, w.w_std, w.V)
    H = _normal_bf16_rows(sH, w.T, w.d, 1.0, n)
    rng = np.random.default_rng(sI)
    if w.ids == "uniform":
        idx = _distinct_uniform(rng, w.T, w.K, w.V)
    elif w.ids == "zipf80":
        idx = _zipf80_uniform20(rng, w.T, w.K, w.V)
    else:
        raise ValueError(w.ids)
    logits = _normal_f32(np.random.default_rng(sL), (w.T, w.K), w.logit_std, w.logit_mean)
    logits = -np.sort(-logits, axis=1)
    mask = _mask(w, np.random.default_rng(sM))
    return Inputs(H=H, W=W,
                  topk_idx=torch.from_numpy(idx[:n].astype(np.int32)),
                  topk_logits=torch.from_numpy(np.ascontiguousarray(logits[:n])),
                  mask=torch.from_numpy(mask[:n].copy()), tau=w.tau, chunk=w.chunk)


def make_random(T: int, d: int, V: int, K: int, tau: float = 1.0, chunk: int = 64, seed: int = 0,
                w_std: float = 0.02, logit_mean: float = 5.0, logit_std: float = 3.0,
                mask_frac: float = 0.0) -> Inputs:
    """Small ad-hoc case with the same distributions (ragged shapes for parity tests)."""
    rng = np.random.default_rng(seed)
    W = torch.from_numpy(_normal_f32(rng, (V, d), w_std)).to(torch.bfloat16)
    H = torch.from_numpy(_normal_f32(rng, (T, d), 1.0)).to(torch.bfloat16)
    idx = _distinct_uniform(rng, T, K, V)
    logits = -np.sort(-_normal_f32(rng, (T, K), logit_std, logit_mean), axis=1)
    mask = np.ones(T, dtype=np.uint8)
    if mask_frac > 0 and T > 0:
        n = int(round(mask_frac * T))
        mask[rng.choice(T, size=n, replace=False)] = 0
    return Inputs(H=H, W=W, topk_idx=torch.from_numpy(idx.astype(np.int32)),
                  topk_logits=torch.from_numpy(np.ascontiguousarray(logits)),
                  mask=torch.from_numpy(mask), tau=tau, chunk=chunk)
