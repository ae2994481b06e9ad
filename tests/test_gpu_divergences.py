"""The other divergences over the top-K support (JSD, skew KL, skew reverse KL, total
variation) on the CUDA path against the float64 oracle (oracle/divergences.py), with the
loss's tolerances: loss relative error <= 1e-3, lse absolute error <= 1e-3, dH and dW
relative Frobenius error <= 2e-2 and max-abs error <= 5e-2 * max|ref|.  The student logits
at the cached ids, which the forward hands to the backward, are checked against float64
dot products."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import divergences as dv
from tests.test_gpu_parity import assert_grad_close, assert_parity, fkl, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu

S_RTOL = 1e-4  # fp32-accumulated logits against float64, relative to the row's largest |s|

KINDS = [("jsd", 0.5), ("jsd", 0.2), ("skew_kl", 0.1), ("skew_kl", 0.0), ("skew_rkl", 0.1),
         ("skew_rkl", 0.7), ("skew_rkl", 1.0), ("tv", None)]


def run_gpu(fkl, x, kind, param, grad=None, chunk=None, seq=None, num_seqs=None):
    H, W, idx, z, m = to_dev(x)
    chunk = x.chunk if chunk is None else chunk
    T, K = idx.shape
    s_ids = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
    sid = None if seq is None else torch.from_numpy(seq).cuda()
    loss, lse = fkl.forward(H, W, idx, z, m, x.tau, chunk, divergence=kind, div_param=param,
                            student_topk_logits=s_ids, seq_ids=sid, num_seqs=num_seqs)
    g = None if grad is None else torch.tensor(grad, dtype=torch.float32, device="cuda")
    dH, dW = fkl.backward(H, W, idx, z, m, lse, g, x.tau, chunk, divergence=kind, div_param=param,
                          student_topk_logits=s_ids, seq_ids=sid, num_seqs=num_seqs)
    torch.cuda.synchronize()
    return dict(loss=loss.item(), lse=lse.cpu().numpy().astype(np.float64), dH=dH.cpu().numpy().astype(np.float64),
                dW=dW.cpu().numpy().astype(np.float64), s_ids=s_ids.cpu().numpy().astype(np.float64),
                status=fkl.read_status(device="cuda"))


def run_oracle(x, kind, param, grad=1.0, seq=None):
    param = {"jsd": 0.5, "skew_kl": 0.1, "skew_rkl": 0.1}.get(kind, 0.0) if param is None else param
    H64, W64 = oracle.to_f64(x.H), oracle.to_f64(x.W)
    norm = "tokens" if seq is None else "sequences"
    f = dv.forward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau, kind, param, norm=norm, seq_ids=seq)
    dH, dW = dv.backward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau, kind, param, grad=grad,
                         norm=norm, seq_ids=seq)
    return dict(loss=f["loss"], lse=f["lse"], dH=dH, dW=dW, s_ids=f["s_at_ids"])


def assert_s_close(gpu, ref):
    scale = np.max(np.abs(ref), axis=1, keepdims=True)
    err = np.max(np.abs(gpu - ref) / scale)
    assert err <= S_RTOL, f"student logits at the ids: error {err:.3e} of the row's max|s|"


@pytest.mark.parametrize("kind,param", KINDS)
def test_divergence_parity(fkl, kind, param):
    x = workloads.make_random(300, 200, 5000, 16, tau=1.5, chunk=128, seed=50, mask_frac=0.1)
    gpu = run_gpu(fkl, x, kind, param, grad=-0.8)
    ref = run_oracle(x, kind, param, grad=-0.8)
    assert_parity(gpu, ref)
    assert_s_close(gpu["s_ids"], ref["s_ids"])


def test_divergence_token_blocks(fkl):
    # 4 token blocks x 3 vocabulary slabs in the backward (a long sequence, small vocabulary)
    x = workloads.make_random(4000, 64, 2999, 16, tau=1.2, chunk=512, seed=59, mask_frac=0.1)
    assert_parity(run_gpu(fkl, x, "skew_rkl", 0.2), run_oracle(x, "skew_rkl", 0.2))


@pytest.mark.parametrize("kind,param", [("jsd", 0.5), ("tv", None)])
def test_divergence_parity_wide_shape(fkl, kind, param):
    # several 256-row blocks and vocabulary slabs, ragged on every axis
    x = workloads.make_random(1100, 320, 20000, 64, tau=1.0, chunk=96, seed=51, mask_frac=0.05)
    assert_parity(run_gpu(fkl, x, kind, param), run_oracle(x, kind, param))


def test_repeated_ids_merge(fkl):
    x = workloads.make_random(200, 128, 3000, 12, tau=1.2, chunk=64, seed=52)
    x.topk_idx[::7, 3] = x.topk_idx[::7, 0]  # one id held by two slots in every 7th row
    x.topk_idx[::11, 5] = x.topk_idx[::11, 9]
    for kind, param in (("jsd", 0.3), ("skew_rkl", 0.2)):
        assert_parity(run_gpu(fkl, x, kind, param), run_oracle(x, kind, param))


def test_sequence_mean_with_divergence(fkl):
    x = workloads.make_random(300, 200, 5000, 16, tau=2.0, chunk=128, seed=53, mask_frac=0.1)
    seq = np.concatenate([np.full(n, i) for i, n in enumerate([40, 130, 37, 93])]).astype(np.int32)
    assert_parity(run_gpu(fkl, x, "skew_kl", 0.2, seq=seq, num_seqs=4), run_oracle(x, "skew_kl", 0.2, seq=seq))


def test_kl_can_return_student_logits_unchanged(fkl):
    # divergence="kl" with the buffer: same loss and gradients as without it, logits filled
    x = workloads.make_random(300, 200, 5000, 16, tau=1.5, chunk=128, seed=54, mask_frac=0.1)
    H, W, idx, z, m = to_dev(x)
    s_ids = torch.empty(idx.shape, dtype=torch.float32, device="cuda")
    l1, lse1 = fkl.forward(H, W, idx, z, m, x.tau, x.chunk, student_topk_logits=s_ids)
    l2, lse2 = fkl.forward(H, W, idx, z, m, x.tau, x.chunk)
    torch.cuda.synchronize()
    assert l1.item() == l2.item() and torch.equal(lse1, lse2)
    H64, W64 = oracle.to_f64(x.H), oracle.to_f64(x.W)
    assert_s_close(s_ids.cpu().numpy().astype(np.float64), oracle.logits_at(H64, W64, x.topk_idx))


def test_divergence_deterministic(fkl):
    x = workloads.make_random(300, 200, 5000, 16, tau=1.0, chunk=128, seed=55)
    a = run_gpu(fkl, x, "jsd", 0.5)
    b = run_gpu(fkl, x, "jsd", 0.5)
    assert a["loss"] == b["loss"]
    assert np.array_equal(a["dH"], b["dH"]) and np.array_equal(a["dW"], b["dW"])


def test_divergence_chunk_invariance(fkl):
    x = workloads.make_random(300, 200, 5000, 16, tau=1.0, chunk=128, seed=56)
    a = run_gpu(fkl, x, "skew_rkl", 0.1, chunk=1)
    b = run_gpu(fkl, x, "skew_rkl", 0.1, chunk=4096)
    assert a["loss"] == b["loss"]
    assert_grad_close(a["dW"], b["dW"], "dW across chunk sizes")


def test_divergence_autograd(fkl):
    x = workloads.make_random(300, 200, 5000, 16, tau=1.3, chunk=128, seed=57, mask_frac=0.2)
    H, W, idx, z, m = to_dev(x)
    H.requires_grad_(True)
    W.requires_grad_(True)
    loss = fkl.fused_kl(H, W, idx, z, m, tau=x.tau, chunk=64, divergence="jsd", div_param=0.4)
    (2.0 * loss).backward()
    ref = run_oracle(x, "jsd", 0.4, grad=2.0)
    assert abs(loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    assert_grad_close(H.grad.double().cpu().numpy(), ref["dH"], "H.grad")
    assert_grad_close(W.grad.double().cpu().numpy(), ref["dW"], "W.grad")


def test_divergence_zero_when_teacher_is_student(fkl):
    # the cache holds every id with the student's own logits: each divergence is ~0
    T, d, V = 64, 64, 512
    x = workloads.make_random(T, d, V, V, seed=58)
    s = (x.H.double() @ x.W.double().T).float()
    x.topk_idx = torch.arange(V, dtype=torch.int32).repeat(T, 1)
    x.topk_logits = s.contiguous()
    for kind, param in (("jsd", 0.5), ("skew_kl", 0.1), ("skew_rkl", 0.1), ("tv", None)):
        gpu = run_gpu(fkl, x, kind, param)
        assert gpu["status"] == 0 and abs(gpu["loss"]) < 1e-5, (kind, gpu["loss"])


@pytest.mark.parametrize("kind,param", [("jsd", 0.5), ("tv", None)])
def test_full_size_sparse_mask_exact(fkl, kind, param):
    # The 32K workload's shapes, chunk and slabs (the benchmark's launches) with one valid token
    # per 128-row block: the oracle then computes the exact loss and sampled rows of dH and dW.
    import dataclasses

    w = workloads.WORKLOADS["gptoss20b_32k"]
    x = workloads.make_inputs(w)
    rng = np.random.default_rng(8)
    valid = np.arange(0, w.T, 128) + rng.integers(0, 128, size=w.T // 128)
    mask = torch.zeros(w.T, dtype=torch.uint8)
    mask[valid] = 1
    x = dataclasses.replace(x, mask=mask)
    gpu = run_gpu(fkl, x, kind, param)
    assert gpu["status"] == 0
    prm = 0.5 if param is None and kind == "jsd" else (0.0 if param is None else param)
    H64, W64 = oracle.to_f64(x.H), oracle.to_f64(x.W)
    rows = np.unique(np.concatenate([valid, rng.choice(w.T, 16, replace=False)]))
    ref = dv.forward(H64, W64, x.topk_idx, x.topk_logits, mask, w.tau, kind, prm, rows=rows)
    assert ref["loss"] is not None
    assert abs(gpu["loss"] - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    assert np.max(np.abs(gpu["lse"][rows] - ref["lse"])) <= 1e-3
    assert_s_close(gpu["s_ids"][rows], ref["s_at_ids"])
    some = valid[:: max(1, len(valid) // 24)]
    dH_ref = dv.dH_rows(H64, W64, x.topk_idx, x.topk_logits, mask, w.tau, kind, prm, some)
    assert_grad_close(gpu["dH"][some], dH_ref, "dH rows")
    hot = np.unique(x.topk_idx.numpy()[valid[:4]].ravel())[:24]
    vr = np.unique(np.concatenate([hot, rng.choice(w.V, 24, replace=False), [0, w.V - 1]]))
    dW_ref = dv.dW_rows(H64, W64, x.topk_idx, x.topk_logits, mask, w.tau, kind, prm, vr)
    assert_grad_close(gpu["dW"][vr], dW_ref, "dW rows")
