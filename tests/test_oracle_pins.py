"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped term, tau in the
wrong place, a wrong sign, a transposed operand, a wrong index, a wrong normaliser)
breaks at least one of them:

* closed-form special cases derived by hand (tests/golden/closed_form_cases.json);
* KL = 0 when the teacher cache holds the whole vocabulary with the student's logits;
* KL >= 0 (Gibbs' inequality; the top-K support carries at most all of q's mass);
* K = 1 reduces to cross-entropy, checked against torch.nn.functional.cross_entropy;
* the rebuilt dense teacher grid checked against torch.nn.functional.kl_div, and lse
  against torch.logsumexp (the pages' "Dense KL" baseline, via library routines);
* the tau identity L(tau; s, z) = tau^2 L(1; s/tau, z/tau);
* gradients against central finite differences and against torch.autograd;
* invariance to the row-block size, to slot order, and to the contents of masked rows.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


def rand_case(T=6, d=8, V=32, K=5, seed=0, tau=1.0, mask=None, distinct=True, w_scale=0.5):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d)) * w_scale
    if distinct:
        idx = np.stack([rng.permutation(V)[:K] for _ in range(T)])
    else:
        idx = rng.integers(0, V, size=(T, K))
    z = -np.sort(-(rng.standard_normal((T, K)) * 2.0 + 1.0), axis=1)
    m = np.ones(T, np.uint8) if mask is None else np.asarray(mask, np.uint8)
    return H, W, idx, z, m, tau


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_closed_form_cases(case):
    H, W = np.array(case["H"], float), np.array(case["W"], float)
    ids, z, mask, tau = np.array(case["ids"]), np.array(case["z"], float), np.array(case["mask"]), case["tau"]
    norm, seq, count = case.get("norm", "tokens"), case.get("seq_ids"), case.get("count")
    f = oracle.forward(H, W, ids, z, mask, tau, norm=norm, seq_ids=seq, count=count)
    assert f["loss"] == pytest.approx(case["loss"], rel=1e-13, abs=1e-14)
    np.testing.assert_allclose(f["lse"], case["lse"], rtol=1e-13)
    dH, dW = oracle.backward(H, W, ids, z, mask, tau, norm=norm, seq_ids=seq, count=count)
    np.testing.assert_allclose(dH, case["dH"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dW, case["dW"], rtol=1e-12, atol=1e-14)


def test_golden_file_is_its_derivations():
    # the stored values are what the committed derivation script computes from the formulas
    import importlib.util

    spec = importlib.util.spec_from_file_location("make_closed_form_cases",
                                                  os.path.join(os.path.dirname(GOLDEN), "make_closed_form_cases.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    assert mod.differences() == []


@pytest.mark.parametrize("tau", [1.0, 2.0, 0.7])
def test_kl_zero_when_teacher_is_student(tau):
    T, d, V = 5, 7, 24
    rng = np.random.default_rng(3)
    H, W = rng.standard_normal((T, d)), rng.standard_normal((V, d))
    s = H @ W.T
    idx = np.stack([rng.permutation(V) for _ in range(T)])  # K = V, every id once
    z = np.take_along_axis(s, idx, axis=1)                  # teacher logits = student logits
    f = oracle.forward(H, W, idx, z, None, tau)
    assert np.max(np.abs(f["kl"])) < 1e-13
    assert abs(f["loss"]) < 1e-13
    dH, dW = oracle.backward(H, W, idx, z, None, tau)
    assert np.max(np.abs(dH)) < 1e-12 and np.max(np.abs(dW)) < 1e-12


@pytest.mark.parametrize("seed", range(5))
def test_kl_nonnegative(seed):
    H, W, idx, z, m, tau = rand_case(T=16, V=40, K=7, seed=seed, tau=1.0 + seed * 0.3)
    f = oracle.forward(H, W, idx, z, m, tau)
    assert np.all(f["kl"] >= -1e-13)
    assert f["loss"] > 0


@pytest.mark.parametrize("tau", [1.0, 1.5])
def test_single_slot_is_cross_entropy(tau):
    T, d, V = 9, 6, 30
    rng = np.random.default_rng(11)
    H, W = rng.standard_normal((T, d)), rng.standard_normal((V, d))
    idx = rng.integers(0, V, size=(T, 1))
    z = rng.standard_normal((T, 1))
    mask = np.array([1, 1, 0, 1, 1, 1, 0, 1, 1], np.uint8)
    f = oracle.forward(H, W, idx, z, mask, tau)
    logits = torch.tensor(H @ W.T / tau)
    ce = torch.nn.functional.cross_entropy(logits, torch.tensor(idx[:, 0]), reduction="none").numpy()
    valid = mask.astype(bool)
    assert f["loss"] == pytest.approx(tau ** 2 * ce[valid].mean(), rel=1e-13)
    np.testing.assert_allclose(f["kl"], ce, rtol=1e-12)


def test_dense_grid_matches_torch_kl_div_and_logsumexp():
    H, W, idx, z, m, tau = rand_case(T=12, d=9, V=50, K=8, seed=5, tau=1.3,
                                     mask=[1] * 10 + [0, 1])
    f = oracle.forward(H, W, idx, z, m, tau)
    logits = torch.tensor(H @ W.T / tau)
    logq = torch.log_softmax(logits, dim=1)
    P = torch.zeros_like(logq)
    p = torch.softmax(torch.tensor(z / tau), dim=1)
    P.scatter_(1, torch.tensor(idx), p)       # the dense teacher grid rebuilt from the cache
    kl_rows = torch.nn.functional.kl_div(logq, P, reduction="none").sum(1).numpy()
    np.testing.assert_allclose(f["kl"], kl_rows, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(f["lse"], torch.logsumexp(logits, 1).numpy(), rtol=1e-14)
    valid = m.astype(bool)
    assert f["loss"] == pytest.approx(tau ** 2 * kl_rows[valid].sum() / valid.sum(), rel=1e-13)


def test_tau_identity():
    H, W, idx, z, m, _ = rand_case(T=10, d=5, V=33, K=6, seed=8)
    tau = 2.5
    a = oracle.forward(H, W, idx, z, m, tau)["loss"]
    b = oracle.forward(H / tau, W, idx, z / tau, m, 1.0)["loss"]
    assert a == pytest.approx(tau ** 2 * b, rel=1e-12)


def _loss(H, W, idx, z, m, tau):
    return oracle.forward(H, W, idx, z, m, tau)["loss"]


@pytest.mark.parametrize("tau,distinct", [(1.0, True), (1.7, True), (1.0, False)])
def test_gradient_finite_differences(tau, distinct):
    H, W, idx, z, m, _ = rand_case(T=8, d=16, V=64, K=8, seed=2, distinct=distinct,
                                   mask=[1, 1, 1, 0, 1, 1, 1, 1])
    if not distinct:
        idx[0, 1] = idx[0, 0]  # a repeated id in one row: the per-slot sum scatters with add
    dH, dW = oracle.backward(H, W, idx, z, m, tau, grad=1.0)
    h = 1e-6
    for X, G in ((H, dH), (W, dW)):
        num = np.zeros_like(X)
        for i in np.ndindex(X.shape):
            old = X[i]
            X[i] = old + h
            lp = _loss(H, W, idx, z, m, tau)
            X[i] = old - h
            lm = _loss(H, W, idx, z, m, tau)
            X[i] = old
            num[i] = (lp - lm) / (2 * h)
        err = np.linalg.norm(num - G) / np.linalg.norm(G)
        assert err < 1e-6, err


def test_gradient_matches_autograd_on_dense_formula():
    H, W, idx, z, m, tau = rand_case(T=10, d=12, V=40, K=6, seed=4, tau=1.4,
                                     mask=[1, 0, 1, 1, 1, 1, 1, 1, 0, 1])
    g = 0.37
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    logq = torch.log_softmax(Ht @ Wt.T / tau, dim=1)
    P = torch.zeros(10, 40, dtype=torch.float64).scatter_(1, torch.tensor(idx),
                                                          torch.softmax(torch.tensor(z / tau), 1))
    valid = torch.tensor(m.astype(bool))
    L = tau ** 2 * torch.nn.functional.kl_div(logq[valid], P[valid], reduction="sum") / valid.sum()
    (L * g).backward()
    dH, dW = oracle.backward(H, W, idx, z, m, tau, grad=g)
    np.testing.assert_allclose(dH, Ht.grad.numpy(), rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-11, atol=1e-15)
    assert oracle.forward(H, W, idx, z, m, tau)["loss"] == pytest.approx(L.item(), rel=1e-13)


def test_chunk_invariance():
    H, W, idx, z, m, tau = rand_case(T=29, d=10, V=70, K=9, seed=6, tau=1.2,
                                     mask=[1] * 20 + [0] * 3 + [1] * 6)
    ref = oracle.forward(H, W, idx, z, m, tau, chunk=29)
    refg = oracle.backward(H, W, idx, z, m, tau, chunk=29)
    for c in (1, 7, 64):
        f = oracle.forward(H, W, idx, z, m, tau, chunk=c)
        assert f["loss"] == pytest.approx(ref["loss"], rel=1e-14)
        np.testing.assert_allclose(f["lse"], ref["lse"], rtol=1e-14)
        g = oracle.backward(H, W, idx, z, m, tau, chunk=c)
        np.testing.assert_allclose(g[0], refg[0], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(g[1], refg[1], rtol=1e-12, atol=1e-15)


def test_slot_permutation_invariance():
    H, W, idx, z, m, tau = rand_case(T=7, d=6, V=30, K=5, seed=9, tau=1.1)
    rng = np.random.default_rng(0)
    perm = np.stack([rng.permutation(5) for _ in range(7)])
    a = oracle.forward(H, W, idx, z, m, tau)
    b = oracle.forward(H, W, np.take_along_axis(idx, perm, 1), np.take_along_axis(z, perm, 1), m, tau)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-14)
    ga = oracle.backward(H, W, idx, z, m, tau)
    gb = oracle.backward(H, W, np.take_along_axis(idx, perm, 1), np.take_along_axis(z, perm, 1), m, tau)
    np.testing.assert_allclose(ga[1], gb[1], rtol=1e-12, atol=1e-15)


def test_masked_rows_change_nothing():
    mask = np.array([1, 0, 1, 1, 0, 1], np.uint8)
    H, W, idx, z, m, tau = rand_case(T=6, d=5, V=20, K=4, seed=12, mask=mask)
    a = oracle.forward(H, W, idx, z, m, tau)
    ga = oracle.backward(H, W, idx, z, m, tau)
    H2, idx2, z2 = H.copy(), idx.copy(), z.copy()
    H2[[1, 4]] += 3.0
    idx2[[1, 4]] = idx2[[1, 4]][:, ::-1] + 0  # different teacher content on masked rows
    z2[[1, 4]] = 0.0
    b = oracle.forward(H2, W, idx2, z2, m, tau)
    gb = oracle.backward(H2, W, idx2, z2, m, tau)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-14)
    assert np.all(ga[0][[1, 4]] == 0) and np.all(gb[0][[1, 4]] == 0)
    np.testing.assert_allclose(ga[1], gb[1], rtol=1e-12, atol=1e-15)
    assert a["n_valid"] == 4
    # lse stays defined on masked rows and is a property of the projection alone
    np.testing.assert_allclose(a["lse"][[0, 2, 3, 5]], b["lse"][[0, 2, 3, 5]], rtol=1e-14)


def test_no_valid_token():
    H, W, idx, z, _, tau = rand_case(T=4, seed=1)
    m = np.zeros(4, np.uint8)
    f = oracle.forward(H, W, idx, z, m, tau)
    assert f["loss"] == 0.0 and f["n_valid"] == 0
    dH, dW = oracle.backward(H, W, idx, z, m, tau)
    assert not dH.any() and not dW.any()


def test_minus_inf_slots_get_zero_mass():
    H, W, idx, z, m, tau = rand_case(T=3, d=4, V=16, K=4, seed=7)
    z[:, -1] = -np.inf
    f = oracle.forward(H, W, idx, z, m, tau)
    g = oracle.forward(H, W, idx[:, :3], z[:, :3], m, tau)
    assert f["loss"] == pytest.approx(g["loss"], rel=1e-14)
    z[1, :] = -np.inf
    with pytest.raises(ValueError):
        oracle.forward(H, W, idx, z, m, tau)


def test_rejects_out_of_range_ids():
    H, W, idx, z, m, tau = rand_case(T=3, d=4, V=16, K=4, seed=7)
    idx[2, 1] = 16
    with pytest.raises(ValueError):
        oracle.forward(H, W, idx, z, m, tau)


def test_sampled_rows_agree_with_full():
    H, W, idx, z, _, tau = rand_case(T=20, d=7, V=45, K=6, seed=13, tau=1.6)
    m = np.zeros(20, np.uint8)
    m[[2, 5, 11, 17]] = 1
    full = oracle.forward(H, W, idx, z, m, tau)
    part = oracle.forward(H, W, idx, z, m, tau, rows=[17, 2, 5, 11, 0])
    assert part["loss"] == pytest.approx(full["loss"], rel=1e-14)
    np.testing.assert_allclose(part["lse"], full["lse"][[17, 2, 5, 11, 0]], rtol=1e-14)
    assert oracle.forward(H, W, idx, z, m, tau, rows=[2, 5])["loss"] is None
    dH, dW = oracle.backward(H, W, idx, z, m, tau, grad=0.5)
    np.testing.assert_allclose(oracle.dH_rows(H, W, idx, z, m, tau, [11, 3], grad=0.5), dH[[11, 3]],
                               rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(oracle.dW_rows(H, W, idx, z, m, tau, [44, 0, 9], grad=0.5), dW[[44, 0, 9]],
                               rtol=1e-12, atol=1e-15)


def test_to_f64_is_exact_for_bf16():
    x = torch.randn(1000).to(torch.bfloat16)
    y = oracle.to_f64(x)
    assert y.dtype == np.float64
    assert np.array_equal(y, x.float().numpy().astype(np.float64))
    assert math.isclose(float(oracle.to_f64(torch.tensor([1.5], dtype=torch.bfloat16))[0]), 1.5)


# ---------------------------------------------------------------- sequence-mean normaliser

def test_sequence_mean_of_one_sequence_is_token_mean():
    H, W, idx, z, m, tau = rand_case(T=9, d=6, V=30, K=5, seed=21, tau=1.3, mask=[1, 1, 0, 1, 1, 1, 1, 0, 1])
    seq = np.zeros(9, np.int64)
    a = oracle.forward(H, W, idx, z, m, tau)["loss"]
    b = oracle.forward(H, W, idx, z, m, tau, norm="sequences", seq_ids=seq)["loss"]
    assert a == pytest.approx(b, rel=1e-14)
    ga = oracle.backward(H, W, idx, z, m, tau)
    gb = oracle.backward(H, W, idx, z, m, tau, norm="sequences", seq_ids=seq)
    np.testing.assert_allclose(ga[1], gb[1], rtol=1e-13, atol=1e-16)


def test_sequence_mean_with_equal_counts_is_token_mean():
    H, W, idx, z, _, tau = rand_case(T=12, d=6, V=30, K=5, seed=22)
    seq = np.repeat(np.arange(3), 4)
    m = np.array([1, 1, 1, 0] * 3, np.uint8)  # three valid tokens in every sequence
    a = oracle.forward(H, W, idx, z, m, tau)["loss"]
    b = oracle.forward(H, W, idx, z, m, tau, norm="sequences", seq_ids=seq)["loss"]
    assert a == pytest.approx(b, rel=1e-14)


def test_sequence_mean_weights_unequal_sequences():
    seq = np.array([0, 0, 0, 1, 2, 2, 3, 3])
    m = np.array([1, 1, 0, 1, 1, 1, 0, 0], np.uint8)  # sequence 3 has no valid token
    w = oracle.token_weights(m, 8, "sequences", seq)
    np.testing.assert_allclose(w, [1 / 6, 1 / 6, 0, 1 / 3, 1 / 6, 1 / 6, 0, 0])
    assert w.sum() == pytest.approx(1.0)


def test_sequence_mean_gradient_finite_differences():
    seq = np.array([0, 0, 0, 1, 1, 2, 2, 2])
    H, W, idx, z, m, tau = rand_case(T=8, d=10, V=40, K=6, seed=23, tau=1.4, mask=[1, 1, 0, 1, 1, 1, 1, 0])
    dH, dW = oracle.backward(H, W, idx, z, m, tau, grad=0.8, norm="sequences", seq_ids=seq)
    h = 1e-6
    for X, G in ((H, dH), (W, dW)):
        num = np.zeros_like(X)
        for i in np.ndindex(X.shape):
            old = X[i]
            X[i] = old + h
            lp = oracle.forward(H, W, idx, z, m, tau, norm="sequences", seq_ids=seq)["loss"]
            X[i] = old - h
            lm = oracle.forward(H, W, idx, z, m, tau, norm="sequences", seq_ids=seq)["loss"]
            X[i] = old
            num[i] = 0.8 * (lp - lm) / (2 * h)
        assert np.linalg.norm(num - G) / np.linalg.norm(G) < 1e-6


def test_sequence_mean_matches_autograd():
    seq = np.array([0, 0, 1, 1, 1, 1, 2, 3, 3, 3])
    H, W, idx, z, m, tau = rand_case(T=10, d=12, V=40, K=6, seed=24, tau=1.1,
                                     mask=[1, 1, 0, 1, 1, 1, 1, 1, 0, 1])
    Ht, Wt = torch.tensor(H, requires_grad=True), torch.tensor(W, requires_grad=True)
    logq = torch.log_softmax(Ht @ Wt.T / tau, dim=1)
    P = torch.zeros(10, 40, dtype=torch.float64).scatter_(1, torch.tensor(idx),
                                                          torch.softmax(torch.tensor(z / tau), 1))
    kl = torch.nn.functional.kl_div(logq, P, reduction="none").sum(1)
    valid = torch.tensor(m.astype(bool))
    per_seq = [kl[(torch.tensor(seq) == s) & valid].mean() for s in range(4)
               if ((torch.tensor(seq) == s) & valid).any()]
    L = tau ** 2 * torch.stack(per_seq).mean()
    L.backward()
    assert oracle.forward(H, W, idx, z, m, tau, norm="sequences", seq_ids=seq)["loss"] == pytest.approx(L.item(), rel=1e-13)
    dH, dW = oracle.backward(H, W, idx, z, m, tau, norm="sequences", seq_ids=seq)
    np.testing.assert_allclose(dH, Ht.grad.numpy(), rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-11, atol=1e-15)


def test_shards_with_the_batch_count_add_up_to_the_batch():
    # A batch split into three uneven shards with unequal valid counts (as over data-parallel
    # ranks or micro-batches); every shard divides by the whole batch's N.  The shards' losses
    # add up to the batch's, their dH rows are the batch's rows, and their dW add up to its dW.
    H, W, idx, z, m, tau = rand_case(T=11, d=8, V=30, K=5, seed=31, tau=1.3,
                                     mask=[1, 0, 1, 1, 1, 0, 0, 1, 1, 1, 1])
    whole = oracle.forward(H, W, idx, z, m, tau)["loss"]
    dH, dW = oracle.backward(H, W, idx, z, m, tau, grad=0.7)
    N = int(m.sum())
    loss, dW_sum = 0.0, np.zeros_like(W)
    for a, b in [(0, 2), (2, 7), (7, 11)]:
        sh = (H[a:b], W, idx[a:b], z[a:b], m[a:b], tau)
        loss += oracle.forward(*sh, count=N)["loss"]
        h, w = oracle.backward(*sh, grad=0.7, count=N)
        np.testing.assert_allclose(h, dH[a:b], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(oracle.dH_rows(*sh, rows=np.arange(b - a), grad=0.7, count=N), h,
                                   rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(oracle.dW_rows(*sh, vocab_rows=np.arange(30), grad=0.7, count=N), w,
                                   rtol=1e-12, atol=1e-15)
        dW_sum += w
    assert loss == pytest.approx(whole, rel=1e-13)
    np.testing.assert_allclose(dW_sum, dW, rtol=1e-12, atol=1e-15)


def test_sequence_shards_with_the_batch_count_add_up_to_the_batch():
    # packed sequences, each inside one shard; every shard divides by the batch's S
    seq = np.array([0, 0, 0, 1, 1, 2, 2, 2, 2, 3])
    H, W, idx, z, m, tau = rand_case(T=10, d=6, V=24, K=4, seed=32, tau=0.9,
                                     mask=[1, 1, 0, 1, 0, 1, 1, 1, 0, 1])
    kw = dict(norm="sequences")
    whole = oracle.forward(H, W, idx, z, m, tau, seq_ids=seq, **kw)["loss"]
    dH, dW = oracle.backward(H, W, idx, z, m, tau, seq_ids=seq, **kw)
    loss, dW_sum = 0.0, np.zeros_like(W)
    for a, b in [(0, 3), (3, 9), (9, 10)]:
        sh = (H[a:b], W, idx[a:b], z[a:b], m[a:b], tau)
        loss += oracle.forward(*sh, seq_ids=seq[a:b], count=4, **kw)["loss"]
        h, w = oracle.backward(*sh, seq_ids=seq[a:b], count=4, **kw)
        np.testing.assert_allclose(h, dH[a:b], rtol=1e-12, atol=1e-15)
        dW_sum += w
    assert loss == pytest.approx(whole, rel=1e-13)
    np.testing.assert_allclose(dW_sum, dW, rtol=1e-12, atol=1e-15)


def test_batch_count_defaults_and_limits():
    H, W, idx, z, m, tau = rand_case(T=6, seed=33, mask=[1, 1, 0, 1, 1, 1])
    own = oracle.forward(H, W, idx, z, m, tau)["loss"]
    assert oracle.forward(H, W, idx, z, m, tau, count=5)["loss"] == own
    assert oracle.forward(H, W, idx, z, m, tau, count=10)["loss"] == pytest.approx(own / 2, rel=1e-14)
    with pytest.raises(ValueError):
        oracle.forward(H, W, idx, z, m, tau, count=4)  # below the shard's own 5 valid tokens
