"""A batch split over several calls with the batch's count (fkl_options.global_count).

On one GPU, the shards stand for data-parallel ranks or for the micro-batches of one
accumulated step: each shard's forward and backward divide by the whole batch's count (the
sum of fkl_local_count over the shards, added on the device as an all-reduce would), the
shards' losses are added and their dW accumulated into one buffer.  The result must equal the
float64 oracle on the whole batch within the parity tolerances (loss relative 1e-3, lse
absolute 1e-3, dH and dW relative Frobenius 2e-2 and max-abs 5e-2 of max |ref|)."""
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


def close(G, R, name):
    G, R = np.asarray(G, np.float64), np.asarray(R, np.float64)
    fro = np.linalg.norm(G - R) / np.linalg.norm(R)
    mx = np.max(np.abs(G - R)) / np.max(np.abs(R))
    assert fro <= FRO_RTOL and mx <= MAX_FRAC, f"{name}: fro {fro:.3e}, max {mx:.3e}"


def run_shards(fkl, x, cuts, seq_ids=None, num_seqs=None):
    dev = "cuda"
    H, W = x.H.to(dev), x.W.to(dev)
    idx, z, m = x.topk_idx.to(dev), x.topk_logits.to(dev), x.mask.to(dev)
    seq = None if seq_ids is None else seq_ids.to(dev)
    T, d = H.shape
    shard = lambda t, a, b: None if t is None else t[a:b]  # noqa: E731
    # each shard's own count, then their sum on the device (the all-reduce of a data-parallel run)
    counts = [fkl.local_count(m[a:b], b - a, seq_ids=shard(seq, a, b), num_seqs=num_seqs) for a, b in cuts]
    N = torch.stack(counts).sum()
    dH = torch.zeros(T, d, device=dev)
    dW = torch.zeros(W.shape[0], d, device=dev)
    loss = torch.zeros((), device=dev)
    lse = torch.empty(T, device=dev)
    for a, b in cuts:
        kw = dict(seq_ids=shard(seq, a, b), num_seqs=num_seqs, global_count=N)
        l_r, lse_r = fkl.forward(H[a:b], W, idx[a:b], z[a:b], m[a:b], x.tau, x.chunk, **kw)
        fkl.backward(H[a:b], W, idx[a:b], z[a:b], m[a:b], lse_r, None, x.tau, x.chunk, out=(dH[a:b], dW),
                     accumulate=True, **kw)
        loss += l_r
        lse[a:b] = lse_r
    torch.cuda.synchronize()
    assert fkl.read_status(device=dev) == 0
    return [int(c) for c in counts], int(N), loss.item(), lse.cpu().numpy(), dH.cpu().numpy(), dW.cpu().numpy()


def test_local_count(fkl):
    x = workloads.make_random(1000, 64, 1000, 8, seed=61, mask_frac=0.3)
    m = x.mask.cuda()
    assert int(fkl.local_count(m, 1000)) == int(x.mask.sum())
    assert int(fkl.local_count(None, 1000)) == 1000
    assert int(fkl.local_count(None, 0)) == 0
    seq = torch.arange(1000, dtype=torch.int32) // 100  # 10 sequences of 100 tokens
    m2 = x.mask.clone()
    m2[300:400] = 0                                    # sequence 3 has no valid token
    assert int(fkl.local_count(m2.cuda(), 1000, seq_ids=seq.cuda(), num_seqs=10)) == 9


@pytest.mark.parametrize("cuts", [[(0, 137), (137, 600), (600, 1000)], [(0, 1000)],
                                  [(0, 256), (256, 512), (512, 768), (768, 1000)]])
def test_token_shards_equal_the_whole_batch(fkl, cuts):
    x = workloads.make_random(1000, 200, 5000, 16, tau=1.5, chunk=64, seed=62, mask_frac=0.25)
    # make the shards' valid counts clearly uneven
    x.mask[:100] = 0
    counts, N, loss, lse, dH, dW = run_shards(fkl, x, cuts)
    assert N == int(x.mask.sum()) and sum(counts) == N
    H64, W64 = oracle.to_f64(x.H), oracle.to_f64(x.W)
    ref = oracle.forward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau)
    rdH, rdW = oracle.backward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau)
    assert abs(loss - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"])
    assert np.max(np.abs(lse - ref["lse"])) <= LSE_ATOL
    close(dH, rdH, "dH")
    close(dW, rdW, "dW")


def test_sequence_shards_equal_the_whole_batch(fkl):
    # packed sequences of unequal lengths, none crossing a shard boundary; each shard divides by
    # the batch's number of sequences with a valid token
    x = workloads.make_random(900, 128, 3000, 12, tau=2.0, chunk=128, seed=63, mask_frac=0.2)
    bounds = [0, 100, 350, 400, 700, 900]
    seq = torch.zeros(900, dtype=torch.int32)
    for s in range(len(bounds) - 1):
        seq[bounds[s]:bounds[s + 1]] = s
    x.mask[350:400] = 0  # sequence 2 has no valid token
    counts, N, loss, lse, dH, dW = run_shards(fkl, x, [(0, 350), (350, 700), (700, 900)], seq_ids=seq, num_seqs=5)
    assert N == 4
    H64, W64 = oracle.to_f64(x.H), oracle.to_f64(x.W)
    kw = dict(norm="sequences", seq_ids=seq.numpy())
    ref = oracle.forward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau, **kw)
    rdH, rdW = oracle.backward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau, **kw)
    assert abs(loss - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"])
    close(dH, rdH, "dH")
    close(dW, rdW, "dW")


def test_count_below_the_shards_own_is_reported(fkl):
    x = workloads.make_random(300, 64, 2000, 8, seed=64)
    dev = "cuda"
    H, W, idx, z = x.H.to(dev), x.W.to(dev), x.topk_idx.to(dev), x.topk_logits.to(dev)
    N = torch.tensor(299, dtype=torch.int64, device=dev)  # 300 valid tokens in this shard alone
    loss, lse = fkl.forward(H, W, idx, z, None, 1.0, 64, global_count=N)
    torch.cuda.synchronize()
    assert fkl.read_status(device=dev) == 11  # FKL_ERR_BAD_COUNT
    assert torch.isnan(loss)
    dH, dW = fkl.backward(H, W, idx, z, None, lse, None, 1.0, 64, global_count=N)
    torch.cuda.synchronize()
    assert fkl.read_status(device=dev) == 11
    assert torch.isnan(dH).all() and torch.isnan(dW).all()


def test_sharded_step_single_process(fkl):
    # ShardedStep without torch.distributed: the plain step of the batch it is given
    from lm_head_top_tcgen05_gb300.data_parallel import ShardedStep

    x = workloads.make_random(500, 128, 4000, 16, seed=65, mask_frac=0.1)
    dev = "cuda"
    args = (x.H.to(dev), x.W.to(dev), x.topk_idx.to(dev), x.topk_logits.to(dev), x.mask.to(dev), 1.0, 64)
    loss, dH, dW = ShardedStep()(*args)
    ref_loss, lse = fkl.forward(*args)
    ref_dH, ref_dW = fkl.backward(*args[:5], lse, None, 1.0, 64)
    torch.cuda.synchronize()
    assert loss.item() == ref_loss.item()
    assert torch.equal(dH, ref_dH) and torch.equal(dW, ref_dW)


def test_jsd_shards_equal_the_whole_batch(fkl):
    # the batch's count reaches the other divergences' token weights too (forward rows and
    # the backward's per-row factor): JSD over three shards against the whole batch
    x = workloads.make_random(700, 160, 4000, 12, tau=1.3, chunk=64, seed=66, mask_frac=0.2)
    x.mask[:80] = 0
    dev = "cuda"
    H, W = x.H.to(dev), x.W.to(dev)
    idx, z, m = x.topk_idx.to(dev), x.topk_logits.to(dev), x.mask.to(dev)
    cuts = [(0, 150), (150, 480), (480, 700)]
    N = torch.stack([fkl.local_count(m[a:b], b - a) for a, b in cuts]).sum()
    dH = torch.zeros(700, 160, device=dev)
    dW = torch.zeros(4000, 160, device=dev)
    loss = 0.0
    for a, b in cuts:
        s_ids = torch.empty(b - a, 12, device=dev)
        kw = dict(divergence="jsd", div_param=0.4, student_topk_logits=s_ids, global_count=N)
        l_r, lse_r = fkl.forward(H[a:b], W, idx[a:b], z[a:b], m[a:b], x.tau, x.chunk, **kw)
        fkl.backward(H[a:b], W, idx[a:b], z[a:b], m[a:b], lse_r, None, x.tau, x.chunk, out=(dH[a:b], dW),
                     accumulate=True, **kw)
        loss += l_r.item()
    torch.cuda.synchronize()
    assert fkl.read_status(device=dev) == 0
    H64, W64 = oracle.to_f64(x.H), oracle.to_f64(x.W)
    ref = oracle.divergences.forward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau, "jsd", 0.4)
    rdH, rdW = oracle.divergences.backward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau, "jsd", 0.4)
    assert abs(loss - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"])
    close(dH.cpu().numpy(), rdH, "dH")
    close(dW.cpu().numpy(), rdW, "dW")


def test_bf16_gradients_of_a_shard_with_the_batch_count(fkl):
    # a shard's bf16 gradients with the batch's count equal its fp32 ones rounded, bit for bit
    x = workloads.make_random(600, 128, 3000, 16, seed=67, mask_frac=0.15)
    dev = "cuda"
    H, W = x.H.to(dev), x.W.to(dev)
    idx, z, m = x.topk_idx.to(dev), x.topk_logits.to(dev), x.mask.to(dev)
    N = fkl.local_count(m, 600) * 3  # as if two more shards of the same count followed
    loss, lse = fkl.forward(H, W, idx, z, m, 1.0, 64, global_count=N)
    dH, dW = fkl.backward(H, W, idx, z, m, lse, None, 1.0, 64, global_count=N)
    dH16, dW16 = fkl.backward(H, W, idx, z, m, lse, None, 1.0, 64, global_count=N, grad_dtype=torch.bfloat16)
    ref_loss, ref_lse = fkl.forward(H, W, idx, z, m, 1.0, 64)
    torch.cuda.synchronize()
    assert fkl.read_status(device=dev) == 0
    assert torch.equal(dH16.view(torch.int16), dH.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(dW16.view(torch.int16), dW.to(torch.bfloat16).view(torch.int16))
    assert loss.item() == pytest.approx(ref_loss.item() / 3, rel=1e-6)  # a third of the shard's own mean
