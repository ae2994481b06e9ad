"""Pins of the teacher-cache oracle (top-K logits per position) to library routines and
to cases whose answer is fixed by hand."""
import numpy as np
import pytest
import torch

import oracle


def rand(T=7, d=9, V=50, seed=0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((T, d)), rng.standard_normal((V, d))


@pytest.mark.parametrize("K", [1, 5, 50])
def test_matches_torch_topk_on_distinct_logits(K):
    Ht, Wt = rand(seed=K)
    ids, vals = oracle.teacher_topk(Ht, Wt, K)
    tv, ti = torch.topk(torch.tensor(Ht @ Wt.T), K, dim=1, largest=True, sorted=True)
    np.testing.assert_array_equal(ids, ti.numpy())
    np.testing.assert_allclose(vals, tv.numpy(), rtol=0, atol=0)


def test_k1_is_argmax_and_ties_take_lower_id():
    Ht = np.array([[1.0, 0.0], [0.0, 1.0]])
    Wt = np.array([[1.0, 2.0], [3.0, 2.0], [3.0, -1.0], [0.0, 2.0]])  # row 0: 1,3,3,0  row 1: 2,2,-1,2
    ids, vals = oracle.teacher_topk(Ht, Wt, 1)
    assert ids.tolist() == [[1], [0]] and vals.tolist() == [[3.0], [2.0]]
    ids, vals = oracle.teacher_topk(Ht, Wt, 3)
    assert ids.tolist() == [[1, 2, 0], [0, 1, 3]]
    assert vals.tolist() == [[3.0, 3.0, 1.0], [2.0, 2.0, 2.0]]


def test_k_equals_v_is_a_full_sort():
    Ht, Wt = rand(T=3, V=20, seed=4)
    ids, vals = oracle.teacher_topk(Ht, Wt, 20)
    s = Ht @ Wt.T
    for t in range(3):
        assert sorted(ids[t].tolist()) == list(range(20))
        assert np.all(np.diff(vals[t]) <= 0)
        np.testing.assert_array_equal(vals[t], np.sort(s[t])[::-1])


def test_logits_at_and_chunking():
    Ht, Wt = rand(T=11, d=6, V=40, seed=5)
    a = oracle.teacher_topk(Ht, Wt, 7, chunk=3)
    b = oracle.teacher_topk(Ht, Wt, 7, chunk=64)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_allclose(oracle.logits_at(Ht, Wt, a[0]), a[1], rtol=1e-15)


def test_cache_is_what_the_loss_reads():
    # a teacher identical to the student gives KL = 0 when the cache holds every id
    Ht, Wt = rand(T=4, d=5, V=12, seed=6)
    ids, vals = oracle.teacher_topk(Ht, Wt, 12)
    f = oracle.forward(Ht, Wt, ids, vals, None, 1.0)
    assert abs(f["loss"]) < 1e-13
