"""Token-sharded data parallelism for the fused chunked KL loss.

Every rank holds a replica of the LM head W and its own shard of the batch's tokens (hidden
states, teacher cache, mask).  The loss of the whole batch is

    L = tau^2 / N * sum over the batch's valid tokens of KL_t,   N = the batch's valid tokens,

so a rank's share is tau^2 / N * sum over its own valid tokens: it needs the batch's N, not
its own.  One step on one rank is

  1. n_r = fkl_local_count(mask_r)                  its own count (a device int64)
  2. N = all-reduce-sum(n_r)                         8 bytes over the process group
  3. loss_r, lse_r = fkl_forward(..., global_count=N)
  4. dH_r, dW_r = fkl_backward(..., global_count=N)  dH_r is the batch's dH on its rows
  5. dW = all-reduce-sum(dW_r)                       the usual data-parallel gradient all-reduce
     loss = all-reduce-sum(loss_r)                   (a scalar, for logging)

The pages' GPT-OSS 20B run trains on one node of several GPUs and reports per-GPU throughput
(the post's "Scaling to long context lengths"); how it splits the batch and normalises the
loss across GPUs is not stated.  Token sharding with the batch's own count is the plainest
reading: the result is the single-GPU loss and gradient of the whole batch.  With
FKL_NORM_SEQUENCES the count is the batch's sequences with a valid token, and each packed
sequence must lie within one rank's shard.

The collectives are torch.distributed calls on the current stream (NCCL for CUDA tensors);
every step of the loss itself runs in the library's kernels.  No TMA multicast or peer memory
is involved: the ranks exchange only through the collectives.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch


def _dist():
    import torch.distributed as dist

    return dist if dist.is_available() and dist.is_initialized() else None


def _all_reduce_sum(t: torch.Tensor, group) -> torch.Tensor:
    dist = _dist()
    if dist is not None and dist.get_world_size(group) > 1:
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return t


class _LibraryOps:
    """The library's calls (the default engine of ShardedStep)."""

    def local_count(self, mask, T, device, seq_ids, num_seqs, workspace):
        from . import local_count

        return local_count(mask, T, device=device, seq_ids=seq_ids, num_seqs=num_seqs, workspace=workspace)

    def forward(self, H, W, idx, z, mask, tau, chunk, **kw):
        from . import forward

        return forward(H, W, idx, z, mask, tau, chunk, **kw)

    def backward(self, H, W, idx, z, mask, lse, tau, chunk, **kw):
        from . import backward

        return backward(H, W, idx, z, mask, lse, None, tau, chunk, **kw)


class ShardedStep:
    """One rank's forward + backward of the loss on its token shard of a global batch.

    ``group`` is the data-parallel process group (None: the default group; a single process
    without torch.distributed runs the plain single-GPU step).  ``reduce_dw`` all-reduces dW
    over the ranks after the backward (turn it off when an optimizer or a gradient bucketing
    scheme does that reduction itself).  ``ops`` replaces the library's calls (tests drive the
    same control flow with a CPU reference)."""

    def __init__(self, group=None, reduce_dw: bool = True, ops=None):
        self.group = group
        self.reduce_dw = reduce_dw
        self.ops = ops if ops is not None else _LibraryOps()

    def global_count(self, mask: Optional[torch.Tensor], T: int, device, seq_ids=None, num_seqs=None,
                     workspace=None) -> torch.Tensor:
        """The batch's count: this rank's count summed over the group (steps 1 and 2)."""
        from . import all_reduce_count

        n = self.ops.local_count(mask, T, device, seq_ids, num_seqs, workspace)
        return all_reduce_count(n, self.group)

    def __call__(self, H, W, topk_idx, topk_logits, mask=None, tau: float = 1.0, chunk: int = 2048,
                 workspace=None, out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None,
                 seq_ids=None, num_seqs=None, grad_dtype: torch.dtype = torch.float32,
                 **div) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
        """(loss of the whole batch, dH of this rank's rows, dW of the whole batch).

        The loss is summed over the ranks; dW too when ``reduce_dw`` (else it is this rank's
        term).  ``out`` receives dH and dW as in ``backward``; ``div`` (divergence, div_param,
        student_topk_logits) goes to both passes as in ``forward`` and ``backward``."""
        T = H.shape[0]
        N = self.global_count(mask, T, H.device, seq_ids, num_seqs, workspace)
        kw = dict(workspace=workspace, seq_ids=seq_ids, num_seqs=num_seqs, global_count=N, **div)
        loss, lse = self.ops.forward(H, W, topk_idx, topk_logits, mask, tau, chunk, **kw)
        dH, dW = self.ops.backward(H, W, topk_idx, topk_logits, mask, lse, tau, chunk, out=out,
                                   grad_dtype=grad_dtype, **kw)
        loss = _all_reduce_sum(loss, self.group)
        if self.reduce_dw:
            dW = _all_reduce_sum(dW, self.group)
        return loss, dH, dW
