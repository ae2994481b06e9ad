"""CUDA path against the oracle at the workloads' full sizes, in the launch configuration the
benchmark times (same shapes, chunk, tiles and backward blocks).

Exact checks (test_full_size_sparse_mask_exact, all four full-size workloads).  The inputs
are the workload's own; the mask keeps one valid token per 128-row block.  The backward's
block plan depends on the shape, not on the mask, so every tile, slab and token block of the
benchmark's run still executes (256K: 11 token blocks x 6 slabs).  With few valid rows the
oracle computes, in float64, everything that matters: the exact loss, lse of every valid row
and of random and edge rows, dH of valid rows (masked rows must be exactly 0), and rows of dW
at the valid rows' teacher ids (where p is scattered), at random ids and at both ends of the
vocabulary.

Consistency checks (test_full_size and test_long_context_256k, the workloads' own masks).
Here the oracle cannot compute every output, so the run is checked on what it computes one
row at a time and on properties that hold at any size:

* lse and dH of sampled rows (row t needs only row t of the logits);
* the loss against tau^2/N * sum over valid rows of (sum_k p log p - sum_k p s_id / tau + lse_t),
  with the teacher terms and the gathered student logits computed in float64 from the inputs
  and lse from the run (itself checked on samples): a consistency check of the reduction, not
  an independent value;
* dW through the identity sum_t dH_t . H_t = sum_v dW_v . W_v (both equal sum dS * S) and
  through sum_v dW_v = 0 (every valid row of dS sums to zero).

Tolerances as in test_gpu_parity: loss relative 1e-3, lse absolute 1e-3, gradient rows
relative Frobenius 2e-2 and max-abs 5e-2 of max |ref|."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

LOSS_RTOL, LSE_ATOL, FRO_RTOL, MAX_FRAC = 1e-3, 1e-3, 2e-2, 5e-2


@pytest.fixture(scope="module")
def fkl(cuda_device):
    from lm_head_top_tcgen05_gb300 import build

    build.build()
    import lm_head_top_tcgen05_gb300 as m

    return m


def run_gpu(fkl, x, mask=None):
    dev = "cuda"
    H, W = x.H.to(dev), x.W.to(dev)
    idx, z = x.topk_idx.to(dev), x.topk_logits.to(dev)
    m = (x.mask if mask is None else mask).to(dev)
    loss, lse = fkl.forward(H, W, idx, z, m, x.tau, x.chunk)
    dH, dW = fkl.backward(H, W, idx, z, m, lse, None, x.tau, x.chunk)
    torch.cuda.synchronize()
    status = fkl.read_status(device=dev)
    out = dict(loss=loss.item(), lse=lse.cpu().numpy().astype(np.float64), dH=dH.cpu(), dW=dW.cpu(),
               status=status)
    del H, W, idx, z, m, dH, dW
    torch.cuda.empty_cache()
    return out


def sample_rows(T, n, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, T - 1, T // 2], rng.choice(T, n, replace=False)]))


def close_rows(G, R, name):
    fro = np.linalg.norm(G - R) / np.linalg.norm(R)
    mx = np.max(np.abs(G - R)) / np.max(np.abs(R))
    assert fro <= FRO_RTOL and mx <= MAX_FRAC, f"{name}: fro {fro:.3e}, max {mx:.3e}"


def gathered_terms(x, W64, H):
    """Per row: c_t = sum_k p log p and g_t = sum_k p_k s_{t, id_k}, in float64 (rows in blocks)."""
    p, logp = oracle.teacher_probs(x.topk_logits, x.tau)
    c = np.sum(np.where(p > 0, p * np.where(p > 0, logp, 0.0), 0.0), axis=1)
    Wt = torch.from_numpy(W64)
    T = p.shape[0]
    g = np.zeros(T)
    for r0 in range(0, T, 16384):
        r1 = min(T, r0 + 16384)
        E = torch.nn.functional.embedding_bag(x.topk_idx[r0:r1].long(), Wt,
                                              per_sample_weights=torch.from_numpy(p[r0:r1]),
                                              mode="sum").numpy()  # sum_k p_k W[id_k]
        g[r0:r1] = np.einsum("td,td->t", oracle.to_f64(H[r0:r1]), E)
    return c, g


def loss_property(x, W64, gpu, tau):
    c, g = gathered_terms(x, W64, x.H)
    valid = x.mask.numpy() != 0
    kl = c - g / tau + gpu["lse"]
    return tau ** 2 * kl[valid].sum() / valid.sum()


def dw_identities(x, gpu):
    """sum_t dH_t . H_t = sum_v dW_v . W_v and sum_v dW_v = 0, accumulated in row blocks."""
    dH, dW = gpu["dH"], gpu["dW"]
    lhs = rhs = scale = 0.0
    for i in range(0, dH.shape[0], 16384):
        a, h = dH[i:i + 16384].double(), x.H[i:i + 16384].double()
        lhs += float((a * h).sum())
        scale += float((a.abs() * h.abs()).sum())
    d = dW.shape[1]
    colsum = torch.zeros(d, dtype=torch.float64)
    colabs = torch.zeros(d, dtype=torch.float64)
    for i in range(0, dW.shape[0], 16384):
        g = dW[i:i + 16384].double()
        rhs += float((g * x.W[i:i + 16384].double()).sum())
        colsum += g.sum(0)
        colabs += g.abs().sum(0)
    assert abs(lhs - rhs) <= 1e-3 * scale, (lhs, rhs, scale)
    assert colsum.abs().max().item() <= 1e-3 * colabs.max().item()


@pytest.mark.parametrize("name", ["llama3b_8k", "gptoss20b_32k", "packed4x16k_tau2"])
def test_full_size(fkl, name):
    # consistency checks with the workload's own mask (module docstring)
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w)
    gpu = run_gpu(fkl, x)
    assert gpu["status"] == 0 and np.isfinite(gpu["loss"])
    W64, H64 = oracle.to_f64(x.W), oracle.to_f64(x.H)

    rows = sample_rows(w.T, 40, 1)
    ref = oracle.forward(H64, W64, x.topk_idx, x.topk_logits, x.mask, w.tau, rows=rows)
    assert np.max(np.abs(gpu["lse"][rows] - ref["lse"])) <= LSE_ATOL
    dH_ref = oracle.dH_rows(H64, W64, x.topk_idx, x.topk_logits, x.mask, w.tau, rows)
    valid_rows = rows[x.mask.numpy()[rows] != 0]
    sel = np.isin(rows, valid_rows)
    close_rows(gpu["dH"].numpy()[rows][sel].astype(np.float64), dH_ref[sel], "dH rows")
    assert np.all(gpu["dH"].numpy()[rows][~sel] == 0)
    del H64

    loss_prop = loss_property(x, W64, gpu, w.tau)
    assert abs(gpu["loss"] - loss_prop) <= LOSS_RTOL * abs(loss_prop)
    dw_identities(x, gpu)


def sub_batch(x, rows, mask):
    """The rows `rows` of the batch, with the given mask restricted to them."""
    return dataclasses.replace(x, H=x.H[rows], topk_idx=x.topk_idx[rows], topk_logits=x.topk_logits[rows],
                               mask=mask[rows])


@pytest.mark.parametrize("name", ["llama3b_8k", "gptoss20b_32k", "gptoss20b_256k", "packed4x16k_tau2"])
def test_full_size_sparse_mask_exact(fkl, name):
    # exact checks: one valid token per 128-row block (module docstring)
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w)
    rng = np.random.default_rng(7)
    mask = torch.zeros(w.T, dtype=torch.uint8)
    valid = np.arange(0, w.T, 128) + rng.integers(0, 128, size=w.T // 128)
    mask[valid] = 1
    gpu = run_gpu(fkl, x, mask=mask)
    assert gpu["status"] == 0
    # every valid row plus random and edge rows: the loss, N and dW need only the valid rows,
    # so the oracle on this sub-batch is exact for the whole batch
    rows = np.unique(np.concatenate([valid, sample_rows(w.T, 16, 2)]))
    sub = sub_batch(x, rows, mask)
    W64, H64 = oracle.to_f64(x.W), oracle.to_f64(sub.H)
    ref = oracle.forward(H64, W64, sub.topk_idx, sub.topk_logits, sub.mask, w.tau)
    assert ref["n_valid"] == len(valid) and ref["loss"] is not None
    assert abs(gpu["loss"] - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"])
    assert np.max(np.abs(gpu["lse"][rows] - ref["lse"])) <= LSE_ATOL
    # dH: valid rows spread over the batch (every token block), and the masked rows are 0
    pos = np.flatnonzero(sub.mask.numpy())
    some = pos[:: max(1, len(pos) // 24)]
    dH_ref = oracle.dH_rows(H64, W64, sub.topk_idx, sub.topk_logits, sub.mask, w.tau, some)
    close_rows(gpu["dH"].numpy()[rows[some]].astype(np.float64), dH_ref, "dH rows")
    masked = rows[sub.mask.numpy() == 0]
    assert np.all(gpu["dH"].numpy()[masked] == 0)
    # dW rows: the teacher's ids of valid rows (where p is scattered), random rows, both ends
    hot = np.unique(x.topk_idx.numpy()[valid[:: max(1, len(valid) // 6)]][:, :8].ravel())[:32]
    vr = np.unique(np.concatenate([hot, rng.choice(w.V, 32, replace=False), [0, 1, w.V - 2, w.V - 1]]))
    dW_ref = oracle.dW_rows(H64, W64, sub.topk_idx, sub.topk_logits, sub.mask, w.tau, vr)
    close_rows(gpu["dW"].numpy()[vr].astype(np.float64), dW_ref, "dW rows")


def test_long_context_256k(fkl):
    # consistency checks at 256K with the workload's own (all-valid) mask: the backward runs in
    # token blocks x vocabulary slabs, dW accumulating over the token blocks
    w = workloads.WORKLOADS["gptoss20b_256k"]
    x = workloads.make_inputs(w)
    gpu = run_gpu(fkl, x)
    assert gpu["status"] == 0 and np.isfinite(gpu["loss"])
    W64 = oracle.to_f64(x.W)
    rows = sample_rows(w.T, 24, 3)
    sub = sub_batch(x, rows, x.mask)
    H64 = oracle.to_f64(sub.H)
    ref = oracle.forward(H64, W64, sub.topk_idx, sub.topk_logits, None, w.tau)
    assert np.max(np.abs(gpu["lse"][rows] - ref["lse"])) <= LSE_ATOL
    # dH rows scale with 1/N: the oracle's per-row formula with N = T
    dH_ref = oracle.dH_rows(H64, W64, sub.topk_idx, sub.topk_logits, None, w.tau, np.arange(len(rows)),
                            grad=len(rows) / w.T)
    close_rows(gpu["dH"].numpy()[rows].astype(np.float64), dH_ref, "dH rows")
    loss_prop = loss_property(x, W64, gpu, w.tau)
    assert abs(gpu["loss"] - loss_prop) <= LOSS_RTOL * abs(loss_prop)
    dw_identities(x, gpu)


@pytest.mark.parametrize("name", ["gptoss20b_32k", "gptoss20b_256k"])
def test_full_size_bf16_gradients(fkl, name):
    # the bf16 gradient outputs are the fp32 ones rounded to nearest even, bit for bit, with one
    # token block (32K: dW written once, dH summed over 18 slabs) and with 11 (256K: dW summed
    # over the token blocks in the workspace)
    x = workloads.make_inputs(workloads.WORKLOADS[name])
    dev = "cuda"
    H, W = x.H.to(dev), x.W.to(dev)
    idx, z, m = x.topk_idx.to(dev), x.topk_logits.to(dev), x.mask.to(dev)
    loss, lse = fkl.forward(H, W, idx, z, m, x.tau, x.chunk)
    dH, dW = fkl.backward(H, W, idx, z, m, lse, None, x.tau, x.chunk)
    ref_h, ref_w = dH.to(torch.bfloat16), dW.to(torch.bfloat16)
    del dH, dW
    dH16, dW16 = fkl.backward(H, W, idx, z, m, lse, None, x.tau, x.chunk, grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fkl.read_status(device=dev) == 0
    assert torch.equal(dH16.view(torch.int16), ref_h.view(torch.int16))
    assert torch.equal(dW16.view(torch.int16), ref_w.view(torch.int16))
    del H, W, idx, z, m, dH16, dW16, ref_h, ref_w
    torch.cuda.empty_cache()


def test_full_size_memory_has_no_txv_tensor(fkl):
    # the 32K step in the benchmark's configuration: beyond the inputs, outputs and the
    # caller's workspace nothing is allocated (the library allocates no device memory, and
    # no T x V tensor exists anywhere); the whole peak stays far below one bf16 T x V grid
    w = workloads.WORKLOADS["gptoss20b_32k"]
    x = workloads.make_inputs(w)
    dev = "cuda"
    H, W = x.H.to(dev), x.W.to(dev)
    idx, z, m = x.topk_idx.to(dev), x.topk_logits.to(dev), x.mask.to(dev)
    dH = torch.empty(w.T, w.d, device=dev)
    dW = torch.empty(w.V, w.d, device=dev)
    ws = fkl.Workspace(dev)
    ws.get(fkl.workspace_size(w.T, w.d, w.V, w.K, w.chunk), dev)

    def step():
        loss, lse = fkl.forward(H, W, idx, z, m, w.tau, w.chunk, workspace=ws)
        fkl.backward(H, W, idx, z, m, lse, None, w.tau, w.chunk, workspace=ws, out=(dH, dW))
        return loss

    # first call of the shape: kernels and tensor maps set up, and every module this test
    # launches from loaded (module loading takes device memory outside any allocator)
    loss = step()
    torch.cuda.synchronize()
    assert fkl.read_status(ws) == 0 and bool(torch.isfinite(loss))
    del loss
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated(dev)
    free0 = torch.cuda.mem_get_info(dev)[0]
    torch.cuda.reset_peak_memory_stats(dev)
    loss = step()
    torch.cuda.synchronize()
    assert fkl.read_status(ws) == 0 and bool(torch.isfinite(loss))
    peak = torch.cuda.max_memory_allocated(dev)
    assert peak - base < 1 << 20                       # loss and lse only
    assert abs(torch.cuda.mem_get_info(dev)[0] - free0) < 4 << 20   # nothing allocated outside torch
    assert peak < w.T * w.V * 2                        # far below one bf16 logits grid
    del H, W, idx, z, m, dH, dW, ws
    torch.cuda.empty_cache()
