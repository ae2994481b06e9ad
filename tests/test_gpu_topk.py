"""The offline teacher cache producer (fkl_teacher_topk) against the float64 oracle.

Floating point decides which ids make the top K: the GPU ranks fp32 logits accumulated by
the tensor cores, the oracle float64 ones.  So the set of ids is compared exactly except
where the oracle's logits lie within a rounding margin of the K-th largest (near-ties may
legitimately swap across the boundary); the logits the GPU returns are compared with the
oracle's float64 logits at the GPU's own ids; and the order is checked on the GPU's values
(descending, ties by lower id)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fkl(cuda_device):
    from lm_head_top_tcgen05_gb300 import build

    build.build()
    import lm_head_top_tcgen05_gb300 as m

    return m


def teacher(T, d, V, seed, w_std=0.02):
    g = torch.Generator().manual_seed(seed)
    Ht = torch.randn(T, d, generator=g).to(torch.bfloat16)
    Wt = (torch.randn(V, d, generator=g) * w_std).to(torch.bfloat16)
    return Ht, Wt


def check_cache(Ht, Wt, K, idx, val):
    H64, W64 = oracle.to_f64(Ht), oracle.to_f64(Wt)
    ref_ids, ref_vals = oracle.teacher_topk(H64, W64, K)
    idx, val = idx.cpu().numpy(), val.cpu().numpy().astype(np.float64)
    s = H64 @ W64.T
    margin = 1e-4 * np.abs(s).max() + 1e-6
    # values at the GPU's ids
    np.testing.assert_allclose(val, oracle.logits_at(H64, W64, idx), rtol=0, atol=margin)
    for t in range(idx.shape[0]):
        assert len(set(idx[t].tolist())) == K
        # order: descending values, ties by lower id
        for k in range(K - 1):
            assert val[t, k] > val[t, k + 1] or (val[t, k] == val[t, k + 1] and idx[t, k] < idx[t, k + 1])
        kth = ref_vals[t, K - 1]
        sure = set(ref_ids[t][ref_vals[t] > kth + margin].tolist())   # must be present
        allowed = set(np.flatnonzero(s[t] >= kth - margin).tolist())    # may be present
        got = set(idx[t].tolist())
        assert sure <= got, (t, sorted(sure - got)[:5])
        assert got <= allowed, (t, sorted(got - allowed)[:5])


@pytest.mark.parametrize("T,d,V,K", [(300, 200, 3000, 16),      # all-candidates path (V <= 4096)
                                     (257, 256, 20000, 100),     # bound pass
                                     (130, 136, 9000, 64),       # bound pass, ragged d and V
                                     (1, 64, 8192, 256)])        # one row, K at the limit
def test_teacher_topk_matches_oracle(fkl, T, d, V, K):
    Ht, Wt = teacher(T, d, V, seed=T + V)
    idx, val = fkl.teacher_topk(Ht.cuda(), Wt.cuda(), K)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 0
    check_cache(Ht, Wt, K, idx, val)


def test_teacher_topk_is_deterministic(fkl):
    Ht, Wt = teacher(200, 128, 12000, seed=3)
    a = fkl.teacher_topk(Ht.cuda(), Wt.cuda(), 100)
    b = fkl.teacher_topk(Ht.cuda(), Wt.cuda(), 100)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_ties_beyond_capacity_are_reported(fkl):
    Ht = torch.randn(64, 64).to(torch.bfloat16)
    Wt = torch.zeros(6000, 64, dtype=torch.bfloat16)  # every logit is 0: 6000 tied candidates
    idx, val = fkl.teacher_topk(Ht.cuda(), Wt.cuda(), 10)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 10  # FKL_ERR_TOPK_OVERFLOW
    assert (idx == -1).all() and torch.isnan(val).all()


def test_cache_feeds_the_loss(fkl):
    # the producer's cache is exactly what fkl_forward reads: distil a student from it
    Ht, Wt = teacher(256, 128, 10000, seed=5)
    idx, val = fkl.teacher_topk(Ht.cuda(), Wt.cuda(), 100)
    g = torch.Generator().manual_seed(6)
    H = torch.randn(256, 128, generator=g).to(torch.bfloat16)
    W = (torch.randn(10000, 128, generator=g) * 0.02).to(torch.bfloat16)
    loss, lse = fkl.forward(H.cuda(), W.cuda(), idx, val, None, 1.0, 64)
    ref = oracle.forward(oracle.to_f64(H), oracle.to_f64(W), idx.cpu(), val.cpu(), None, 1.0)
    assert abs(loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])


def test_teacher_whose_top_logits_avoid_the_sampled_rows(fkl):
    # Every 4th vocabulary row (every row the default first pass samples is among them) is
    # scaled down: its
    # bound is loose, far more logits reach it than the buffer holds, and the overflow is
    # reported; the exact first pass (max_bound_stride=1) gives the right cache.
    Ht, Wt = teacher(96, 128, 20000, seed=9)
    Wt[::4] = (Wt[::4].float() * 0.05).to(torch.bfloat16)
    idx, val = fkl.teacher_topk(Ht.cuda(), Wt.cuda(), 100)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 10  # FKL_ERR_TOPK_OVERFLOW
    idx, val = fkl.teacher_topk(Ht.cuda(), Wt.cuda(), 100, max_bound_stride=1)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 0
    check_cache(Ht, Wt, 100, idx, val)


def test_teacher_topk_production_vocabulary(fkl):
    # the gpt-oss-like teacher head at its full size (V = 201088, d = 2880, K = 100): the bound
    # pass samples every 8th vocabulary row (25136 rows, 32 splits of several 256-wide tiles),
    # so the multi-tile top-8 insertion of the bound pass and the candidate pass at full V are
    # checked against the float64 oracle on every row
    Ht, Wt = teacher(320, 2880, 201088, seed=11)
    idx, val = fkl.teacher_topk(Ht.cuda(), Wt.cuda(), 100)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 0
    check_cache(Ht, Wt, 100, idx, val)


def test_forced_stride_8_matches_oracle(fkl):
    # stride 8 forced on a smaller vocabulary (15 one-tile splits), against the oracle itself
    Ht, Wt = teacher(200, 192, 30000, seed=10)
    idx, val = fkl.teacher_topk(Ht.cuda(), Wt.cuda(), 100, max_bound_stride=8)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 0
    check_cache(Ht, Wt, 100, idx, val)


@pytest.mark.parametrize("stride", [1, 2, 4, 8])
def test_every_bound_stride_gives_the_same_cache(fkl, stride):
    Ht, Wt = teacher(200, 192, 30000, seed=10)
    a = fkl.teacher_topk(Ht.cuda(), Wt.cuda(), 100, max_bound_stride=stride)
    b = fkl.teacher_topk(Ht.cuda(), Wt.cuda(), 100, max_bound_stride=1)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
