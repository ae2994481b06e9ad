"""Fused chunked KL distillation loss for GB300 (sm_103a): Python binding.

The loss is the one of "Efficient Knowledge Distillation for LLMs: Offline Top-K Logits and a
Fused Chunked KL Loss" (section "Two systems changes"): the LM-head projection s = H W^T is
fused into a KL divergence against the teacher's cached top-K logits, chunk by chunk, and
the backward recomputes each chunk.  Every step runs in the CUDA kernels of ``libfkl.so``
(C ABI in include/fkl.h); this module only checks and marshals PyTorch tensors (device
memory and streams) into that ABI.

    loss = fused_kl(H, W, topk_idx, topk_logits, mask=None, tau=1.0, chunk=2048)
    loss.backward()          # gradients for H and W

or the explicit calls ``forward`` / ``backward`` with a reusable ``Workspace``.  Other
divergences than KL(teacher || student) over the same top-K support: ``divergence="jsd"``
(``div_param`` = b, default 0.5), ``"skew_kl"`` / ``"skew_rkl"`` (``div_param`` = a, default
0.1) and ``"tv"``; their backward needs the student logits at the cached ids that the
forward returns in ``student_topk_logits`` (``fused_kl`` keeps them itself).

A batch split over several calls (token shards on data-parallel ranks, or the micro-batches
of one accumulated step) is normalised by the whole batch's count: sum ``local_count`` over
the shards (``all_reduce_count`` across ranks) and pass it as ``global_count`` to every
shard's forward and backward; the shards' losses then add up to the batch's loss, their dH
rows are the batch's, and their dW summed (the usual data-parallel gradient all-reduce, or
``accumulate=True``) is the batch's dW.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from ._lib import (DIVERGENCES, FKL_ACCUMULATE_DH, FKL_ACCUMULATE_DW, FKL_NORM_SEQUENCES,  # noqa: F401
                   FKL_NORM_TOKENS, FKL_OK, STATUS, FklError, FklOptions, check, lib)

_DEFAULT_PARAM = {"kl": 0.0, "jsd": 0.5, "skew_kl": 0.1, "skew_rkl": 0.1, "tv": 0.0}

__all__ = ["workspace_size", "Workspace", "forward", "backward", "read_status", "fused_kl",
           "FusedKL", "FklError", "STATUS", "teacher_topk", "local_count", "all_reduce_count"]


def workspace_size(T: int, d: int, V: int, K: int, chunk: int, bf16_grads: bool = False) -> int:
    """Workspace bytes for forward and backward; ``bf16_grads`` sizes it for bf16 gradients."""
    fn = lib().fkl_backward_bf16_workspace_size if bf16_grads else lib().fkl_workspace_size
    n = fn(T, d, V, K, chunk)
    if n == 0:
        raise FklError(1, "fkl_workspace_size", f"unsupported shape T={T} d={d} V={V} K={K} chunk={chunk}")
    return int(n)


class Workspace:
    """Device scratch buffer for fkl_forward / fkl_backward, grown on demand and reused."""

    def __init__(self, device=None):
        self.device = torch.device(device) if device is not None else None
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int, device) -> torch.Tensor:
        device = torch.device(device)
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != device:
            # release the old buffer first: both alive at once would raise the peak by its size
            # (the caching allocator hands it back to this stream only after its queued work)
            self.buf = None
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        return self.buf


_default_ws = {}


def _norm(device) -> torch.device:
    device = torch.device(device)
    if device.type == "cuda" and device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    return device


def _ws_for(workspace: Optional[Workspace], nbytes: int, device) -> torch.Tensor:
    device = _norm(device)
    if workspace is None:
        workspace = _default_ws.setdefault(device, Workspace(device))
    return workspace.get(nbytes, device)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_inputs(H, W, topk_idx, topk_logits, mask):
    if not (H.is_cuda and W.is_cuda and topk_idx.is_cuda and topk_logits.is_cuda):
        raise ValueError("H, W, topk_idx and topk_logits must be CUDA tensors")
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("H and W must be bfloat16")
    if topk_idx.dtype != torch.int32 or topk_logits.dtype != torch.float32:
        raise TypeError("topk_idx must be int32 and topk_logits float32")
    if H.dim() != 2 or W.dim() != 2 or H.shape[1] != W.shape[1]:
        raise ValueError("H must be [T, d] and W [V, d]")
    T, K = topk_idx.shape
    if T != H.shape[0] or tuple(topk_logits.shape) != (T, K):
        raise ValueError("topk_idx and topk_logits must be [T, K]")
    for name, t in (("H", H), ("W", W), ("topk_idx", topk_idx), ("topk_logits", topk_logits)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if mask is not None:
        if mask.dtype not in (torch.uint8, torch.bool) or tuple(mask.shape) != (T,) or not mask.is_cuda:
            raise ValueError("mask must be a CUDA uint8/bool tensor of shape [T]")
        mask = mask.contiguous().view(torch.uint8)
    return mask


def _divergence(divergence: str, div_param: Optional[float]):
    if divergence not in DIVERGENCES:
        raise ValueError(f"divergence must be one of {sorted(DIVERGENCES)}")
    return DIVERGENCES[divergence], float(_DEFAULT_PARAM[divergence] if div_param is None else div_param)


def _student_buf(t: Optional[torch.Tensor], T: int, K: int, device) -> Optional[torch.Tensor]:
    if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != (T, K) or not t.is_contiguous()
                          or t.device != device):
        raise ValueError(f"student_topk_logits must be a contiguous float32 [{T}, {K}] tensor on {device}")
    return t


def _count_tensor(t: Optional[torch.Tensor], device) -> Optional[torch.Tensor]:
    if t is None:
        return None
    if t.dtype != torch.int64 or t.numel() != 1 or t.device != device:
        raise ValueError(f"global_count must be a one-element int64 tensor on {device}")
    return t.reshape(()).contiguous()


def _options(T: int, seq_ids: Optional[torch.Tensor], num_seqs: Optional[int], accumulate: int = 0,
             divergence: str = "kl", div_param: Optional[float] = None,
             student_topk_logits: Optional[torch.Tensor] = None, global_count: Optional[torch.Tensor] = None):
    """fkl_options: sequence-mean normaliser (seq_ids given), accumulation flags, divergence,
    the whole batch's count (global_count given)."""
    o = FklOptions()
    o.accumulate = accumulate
    o.divergence, o.div_param = _divergence(divergence, div_param)
    if student_topk_logits is not None:
        o.student_topk_logits = student_topk_logits.data_ptr()
    if global_count is not None:
        o.global_count = global_count.data_ptr()
    if seq_ids is not None:
        if seq_ids.dtype != torch.int32 or tuple(seq_ids.shape) != (T,) or not seq_ids.is_cuda:
            raise ValueError("seq_ids must be a CUDA int32 tensor of shape [T]")
        seq_ids = seq_ids.contiguous()
        o.normalization = FKL_NORM_SEQUENCES
        o.num_seqs = int(num_seqs) if num_seqs is not None else max(1, int(seq_ids.max().item()) + 1 if T else 1)
        o.seq_ids = seq_ids.data_ptr()
    return o, seq_ids


def forward(H: torch.Tensor, W: torch.Tensor, topk_idx: torch.Tensor, topk_logits: torch.Tensor,
            mask: Optional[torch.Tensor] = None, tau: float = 1.0, chunk: int = 2048,
            workspace: Optional[Workspace] = None, seq_ids: Optional[torch.Tensor] = None,
            num_seqs: Optional[int] = None, divergence: str = "kl", div_param: Optional[float] = None,
            student_topk_logits: Optional[torch.Tensor] = None,
            global_count: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Loss (0-dim float32) and lse [T] (float32) on H's device and current stream.

    With ``seq_ids`` (int32 [T], the packed sequence of each token) the loss is the mean
    over sequences of each sequence's token mean; otherwise the mean over valid tokens.
    ``student_topk_logits`` (float32 [T, K], optional) receives the student's logit at each
    cached slot; the backward of every divergence but "kl" needs it.  ``global_count``
    (int64 scalar on the device) divides by the whole batch's count instead of this call's
    own (module docstring)."""
    mask = _check_inputs(H, W, topk_idx, topk_logits, mask)
    T, d = H.shape
    V, K = W.shape[0], topk_idx.shape[1]
    student_topk_logits = _student_buf(student_topk_logits, T, K, H.device)
    global_count = _count_tensor(global_count, H.device)
    ws = _ws_for(workspace, workspace_size(T, d, V, K, chunk), H.device)
    loss = torch.empty((), dtype=torch.float32, device=H.device)
    lse = torch.empty(T, dtype=torch.float32, device=H.device)
    opts, seq_ids = _options(T, seq_ids, num_seqs, 0, divergence, div_param, student_topk_logits, global_count)
    st = lib().fkl_forward_ex(_ptr(H), _ptr(W), _ptr(topk_idx), _ptr(topk_logits), _ptr(mask), T, d, V, K,
                              float(tau), chunk, ctypes.byref(opts), _ptr(loss), _ptr(lse), _ptr(ws), ws.numel(),
                              _stream(H.device))
    check(st, "fkl_forward_ex")
    return loss, lse


def backward(H: torch.Tensor, W: torch.Tensor, topk_idx: torch.Tensor, topk_logits: torch.Tensor,
             mask: Optional[torch.Tensor], lse: torch.Tensor, grad_loss: Optional[torch.Tensor] = None,
             tau: float = 1.0, chunk: int = 2048, workspace: Optional[Workspace] = None,
             out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None, seq_ids: Optional[torch.Tensor] = None,
             num_seqs: Optional[int] = None, accumulate: bool = False, divergence: str = "kl",
             div_param: Optional[float] = None,
             student_topk_logits: Optional[torch.Tensor] = None,
             grad_dtype: torch.dtype = torch.float32,
             global_count: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """dH [T, d] and dW [V, d], the gradient of g * loss (g = grad_loss or 1), in float32 or,
    with ``grad_dtype=torch.bfloat16``, in bfloat16 (fp32 sums rounded once by the library).

    ``accumulate=True`` adds into the float32 tensors given in ``out`` (gradient
    accumulation).  For every divergence but "kl", ``student_topk_logits`` is the forward's
    output of that name.  ``global_count`` as in ``forward`` (the same value)."""
    if grad_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("grad_dtype must be torch.float32 or torch.bfloat16")
    bf16 = grad_dtype == torch.bfloat16
    if bf16 and accumulate:
        raise ValueError("bf16 gradients do not accumulate; use float32 gradients with accumulate=True")
    mask = _check_inputs(H, W, topk_idx, topk_logits, mask)
    T, d = H.shape
    V, K = W.shape[0], topk_idx.shape[1]
    student_topk_logits = _student_buf(student_topk_logits, T, K, H.device)
    global_count = _count_tensor(global_count, H.device)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (T,) or not lse.is_cuda:
        raise ValueError("lse must be a CUDA float32 tensor of shape [T]")
    if grad_loss is not None:
        grad_loss = grad_loss.detach().to(device=H.device, dtype=torch.float32).reshape(()).contiguous()
    ws = _ws_for(workspace, workspace_size(T, d, V, K, chunk, bf16), H.device)
    if out is None:
        if accumulate:
            raise ValueError("accumulate=True needs the gradients to add into, in `out`")
        dH = torch.empty((T, d), dtype=grad_dtype, device=H.device)
        dW = torch.empty((V, d), dtype=grad_dtype, device=H.device)
    else:
        dH, dW = out
        for g, shape in ((dH, (T, d)), (dW, (V, d))):
            if g.dtype != grad_dtype or tuple(g.shape) != shape or not g.is_contiguous() or g.device != H.device:
                raise ValueError(f"out gradients must be contiguous {grad_dtype} {shape} on {H.device}")
    flags = (FKL_ACCUMULATE_DH | FKL_ACCUMULATE_DW) if accumulate else 0
    opts, seq_ids = _options(T, seq_ids, num_seqs, flags, divergence, div_param, student_topk_logits,
                             global_count)
    fn, name = (lib().fkl_backward_bf16, "fkl_backward_bf16") if bf16 else (lib().fkl_backward_ex, "fkl_backward_ex")
    st = fn(_ptr(H), _ptr(W), _ptr(topk_idx), _ptr(topk_logits), _ptr(mask), _ptr(lse.contiguous()),
            _ptr(grad_loss), T, d, V, K, float(tau), chunk, ctypes.byref(opts), _ptr(dH), _ptr(dW), _ptr(ws),
            ws.numel(), _stream(H.device))
    check(st, name)
    return dH, dW


def read_status(workspace: Optional[Workspace] = None, device=None) -> int:
    """Device-side status of the last call on ``workspace`` (syncs the current stream)."""
    if workspace is None:
        workspace = _default_ws[_norm(device or "cuda")]
    return int(lib().fkl_read_status(_ptr(workspace.buf), _stream(workspace.buf.device)))


def local_count(mask: Optional[torch.Tensor], T: int, device=None, seq_ids: Optional[torch.Tensor] = None,
                num_seqs: Optional[int] = None, workspace: Optional[Workspace] = None) -> torch.Tensor:
    """This shard's count (int64 scalar on the device, computed by the library): its valid
    tokens, or with ``seq_ids`` its sequences that have a valid token.  The sum over the
    shards of a batch is the ``global_count`` of each shard's forward and backward."""
    if mask is not None:
        if mask.dtype not in (torch.uint8, torch.bool) or tuple(mask.shape) != (T,) or not mask.is_cuda:
            raise ValueError("mask must be a CUDA uint8/bool tensor of shape [T]")
        mask = mask.contiguous().view(torch.uint8)
        device = mask.device
    device = _norm(device if device is not None else "cuda")
    ws = _ws_for(workspace, 256 + 4 * max(T, 1), device)
    count = torch.empty((), dtype=torch.int64, device=device)
    opts, seq_ids = _options(T, seq_ids, num_seqs)
    st = lib().fkl_local_count(_ptr(mask), T, ctypes.byref(opts), _ptr(count), _ptr(ws), ws.numel(), _stream(device))
    check(st, "fkl_local_count")
    return count


def all_reduce_count(count: torch.Tensor, group=None) -> torch.Tensor:
    """Sums a shard's count over the ranks of ``group`` (torch.distributed, in place, on the
    device with NCCL): the whole batch's ``global_count``.  Without an initialised process
    group, or with one rank, the count is returned as it is."""
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(count, op=dist.ReduceOp.SUM, group=group)
    return count


class FusedKL(torch.autograd.Function):
    """Autograd wrapper: forward saves lse (and, for divergences other than KL, the student
    logits at the cached ids); backward recomputes the projection chunk by chunk."""

    @staticmethod
    def forward(ctx, H, W, topk_idx, topk_logits, mask, tau, chunk, seq_ids=None, num_seqs=None,
                divergence="kl", div_param=None, global_count=None):
        s_ids = None
        if divergence != "kl":
            s_ids = torch.empty(topk_idx.shape, dtype=torch.float32, device=H.device)
        loss, lse = forward(H, W, topk_idx, topk_logits, mask, tau, chunk, seq_ids=seq_ids, num_seqs=num_seqs,
                            divergence=divergence, div_param=div_param, student_topk_logits=s_ids,
                            global_count=global_count)
        ctx.save_for_backward(H, W, topk_idx, topk_logits, lse)
        ctx.mask, ctx.seq_ids, ctx.num_seqs, ctx.global_count = mask, seq_ids, num_seqs, global_count
        ctx.tau, ctx.chunk, ctx.divergence, ctx.div_param, ctx.s_ids = tau, chunk, divergence, div_param, s_ids
        return loss

    @staticmethod
    def backward(ctx, grad):
        H, W, topk_idx, topk_logits, lse = ctx.saved_tensors
        # H and W are bf16: the library writes bf16 gradients (fp32 sums, rounded once)
        dH, dW = backward(H, W, topk_idx, topk_logits, ctx.mask, lse, grad, ctx.tau, ctx.chunk,
                          seq_ids=ctx.seq_ids, num_seqs=ctx.num_seqs, divergence=ctx.divergence,
                          div_param=ctx.div_param, student_topk_logits=ctx.s_ids, grad_dtype=torch.bfloat16,
                          global_count=ctx.global_count)
        return dH, dW, None, None, None, None, None, None, None, None, None, None


def fused_kl(H: torch.Tensor, W: torch.Tensor, topk_idx: torch.Tensor, topk_logits: torch.Tensor,
             mask: Optional[torch.Tensor] = None, tau: float = 1.0, chunk: int = 2048,
             seq_ids: Optional[torch.Tensor] = None, num_seqs: Optional[int] = None,
             divergence: str = "kl", div_param: Optional[float] = None,
             global_count: Optional[torch.Tensor] = None) -> torch.Tensor:
    """tau^2 * KL(teacher top-K || student) averaged over valid tokens (or, with seq_ids, over
    packed sequences of their token means); differentiable in H and W.  ``divergence`` picks
    another divergence over the same support ("jsd", "skew_kl", "skew_rkl", "tv").  With
    ``global_count`` this is one shard's term of a batch split over several calls."""
    return FusedKL.apply(H, W, topk_idx, topk_logits, mask, tau, chunk, seq_ids, num_seqs, divergence, div_param,
                         global_count)


def teacher_topk(Ht: torch.Tensor, Wt: torch.Tensor, K: int = 100,
                 workspace: Optional[Workspace] = None, max_bound_stride: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """Offline teacher cache: (topk_idx int32 [T, K], topk_logits float32 [T, K]) of the K
    largest teacher logits Ht Wt^T per row, by logit descending (ties: lower id first).

    ``max_bound_stride`` caps the first pass's vocabulary sampling (0: default 8; 1: every
    row, for a teacher whose sampled run reported FKL_ERR_TOPK_OVERFLOW)."""
    if not (Ht.is_cuda and Wt.is_cuda) or Ht.dtype != torch.bfloat16 or Wt.dtype != torch.bfloat16:
        raise TypeError("Ht and Wt must be bfloat16 CUDA tensors")
    if Ht.dim() != 2 or Wt.dim() != 2 or Ht.shape[1] != Wt.shape[1] or not (Ht.is_contiguous() and Wt.is_contiguous()):
        raise ValueError("Ht must be [T, d] and Wt [V, d], contiguous")
    T, d = Ht.shape
    V = Wt.shape[0]
    n = lib().fkl_teacher_topk_workspace_size(T, d, V, K)
    if n == 0:
        raise FklError(1, "fkl_teacher_topk_workspace_size", f"unsupported shape T={T} d={d} V={V} K={K}")
    ws = _ws_for(workspace, int(n), Ht.device)
    idx = torch.empty((T, K), dtype=torch.int32, device=Ht.device)
    val = torch.empty((T, K), dtype=torch.float32, device=Ht.device)
    st = lib().fkl_teacher_topk_ex(_ptr(Ht), _ptr(Wt), T, d, V, K, int(max_bound_stride), _ptr(idx), _ptr(val),
                                   _ptr(ws), ws.numel(), _stream(Ht.device))
    check(st, "fkl_teacher_topk_ex")
    return idx, val
