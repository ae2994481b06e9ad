"""The seeded synthetic inputs have the structure the workloads promise."""
import dataclasses

import numpy as np
import torch

import workloads


def _distinct_rows(idx):
    s = np.sort(idx, axis=1)
    return bool((s[:, 1:] != s[:, :-1]).all())


def test_tiny_workload_structure():
    x = workloads.make_inputs("tiny")
    assert x.H.dtype == torch.bfloat16 and tuple(x.H.shape) == (256, 256)
    assert x.W.dtype == torch.bfloat16 and tuple(x.W.shape) == (4096, 256)
    assert x.topk_idx.dtype == torch.int32 and tuple(x.topk_idx.shape) == (256, 16)
    assert x.topk_logits.dtype == torch.float32
    assert x.mask.dtype == torch.uint8 and int(x.mask.sum()) == 256
    idx = x.topk_idx.numpy()
    assert idx.min() >= 0 and idx.max() < 4096 and _distinct_rows(idx)
    assert (np.diff(x.topk_logits.numpy(), axis=1) <= 0).all()
    assert x.H.is_contiguous() and x.W.is_contiguous()


def test_seeded_and_reproducible():
    a, b = workloads.make_inputs("tiny"), workloads.make_inputs("tiny")
    assert torch.equal(a.H, b.H) and torch.equal(a.W, b.W) and torch.equal(a.topk_idx, b.topk_idx)
    c = workloads.make_inputs("tiny", rows=40)
    assert torch.equal(c.H, a.H[:40]) and torch.equal(c.topk_idx, a.topk_idx[:40])


def test_zipf_rows_distinct_and_skewed():
    rng = np.random.default_rng(0)
    V = 201088
    idx = workloads._zipf80_uniform20(rng, 512, 100, V)
    assert idx.shape == (512, 100) and _distinct_rows(idx)
    assert idx.min() >= 0 and idx.max() < V
    # the Zipf part concentrates on few ids; the uniform part does not
    head_counts = np.bincount(idx[:, :80].ravel(), minlength=V)
    tail_counts = np.bincount(idx[:, 80:].ravel(), minlength=V)
    assert head_counts.max() >= 400  # the top-ranked id appears in nearly every row
    assert tail_counts.max() <= 5


def test_packed_trailing_mask():
    w = dataclasses.replace(workloads.WORKLOADS["packed4x16k_tau2"], T=4 * 40, d=16, V=64, K=8)
    rng = np.random.default_rng(0)
    m = workloads._mask(w, rng)
    assert m.sum() == 4 * (40 - 4)
    for s in range(4):
        assert (m[s * 40:s * 40 + 36] == 1).all() and (m[s * 40 + 36:(s + 1) * 40] == 0).all()


def test_random_mask_count():
    w = dataclasses.replace(workloads.WORKLOADS["llama3b_8k"], T=1000)
    m = workloads._mask(w, np.random.default_rng(0))
    assert int((m == 0).sum()) == 20


def test_published_shapes():
    w = workloads.WORKLOADS
    assert (w["gptoss20b_32k"].T, w["gptoss20b_32k"].V, w["gptoss20b_32k"].d) == (32768, 201088, 2880)
    assert w["gptoss20b_32k"].flops_fwd_bwd == 8.0 * 32768 * 201088 * 2880
    assert w["packed4x16k_tau2"].tau == 2.0 and w["packed4x16k_tau2"].T == 65536
    assert [x.seed for x in w.values()] == [1001, 1002, 1003, 1004, 1005]
