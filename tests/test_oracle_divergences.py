"""Pins of the float64 oracle of the other divergences (oracle/divergences.py) to facts that
do not come from the oracle itself:

* each divergence against SciPy's routines on the dense rows (Jensen-Shannon distance,
  relative entropy) or, for total variation, against brute force over all events of a
  small vocabulary and the identity TV = 1 - sum min(p, q);
* special cases: every divergence is 0 when the cache holds the whole vocabulary with the
  student's own logits; skew KL with a = 0 is the default KL loss; skew reverse KL with
  a = 1 is 0; bounds 0 <= JSD_1/2 <= log 2 and 0 <= TV <= 1;
* gradients against central finite differences of the oracle's own loss;
* repeated ids add their probabilities (same value as one slot carrying the sum), the tau
  identity, and invariance to the contents of masked rows.
"""
import itertools
import math

import numpy as np
import pytest
from scipy.spatial.distance import jensenshannon
from scipy.special import softmax
from scipy.stats import entropy

import oracle
from oracle import divergences as dv

PARAMS = [("kl", 0.0), ("jsd", 0.5), ("jsd", 0.2), ("skew_kl", 0.1), ("skew_kl", 0.0),
          ("skew_rkl", 0.1), ("skew_rkl", 0.7), ("tv", 0.0)]


def rand_case(T=6, d=8, V=32, K=5, seed=0, w_scale=0.5, distinct=True):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d)) * w_scale
    if distinct:
        idx = np.stack([rng.permutation(V)[:K] for _ in range(T)])
    else:
        idx = rng.integers(0, V, size=(T, K))
    z = -np.sort(-(rng.standard_normal((T, K)) * 2.0 + 1.0), axis=1)
    return H, W, idx, z


def dense_rows(H, W, idx, z, tau):
    """Dense teacher and student rows built with SciPy's softmax (test side)."""
    q = softmax(H @ W.T / tau, axis=1)
    pk = softmax(z / tau, axis=1)
    p = np.zeros_like(q)
    for t in range(q.shape[0]):
        for k in range(idx.shape[1]):
            p[t, idx[t, k]] += pk[t, k]
    return p, q


@pytest.mark.parametrize("tau", [1.0, 1.7])
def test_jsd_half_is_scipy_jensen_shannon(tau):
    H, W, idx, z = rand_case(seed=1)
    f = dv.forward(H, W, idx, z, None, tau, "jsd", 0.5)
    p, q = dense_rows(H, W, idx, z, tau)
    ref = np.array([jensenshannon(p[t], q[t]) ** 2 for t in range(len(p))])  # natural log
    np.testing.assert_allclose(f["div"], ref, rtol=1e-10)
    assert np.all(f["div"] <= math.log(2) + 1e-12)


@pytest.mark.parametrize("b", [0.1, 0.35, 0.9])
def test_generalised_jsd_against_relative_entropy(b):
    H, W, idx, z = rand_case(seed=2)
    f = dv.forward(H, W, idx, z, None, 1.3, "jsd", b)
    p, q = dense_rows(H, W, idx, z, 1.3)
    m = b * p + (1 - b) * q
    ref = np.array([b * entropy(p[t], m[t]) + (1 - b) * entropy(q[t], m[t]) for t in range(len(p))])
    np.testing.assert_allclose(f["div"], ref, rtol=1e-10)


@pytest.mark.parametrize("a", [0.0, 0.1, 0.6])
def test_skew_kl_against_relative_entropy(a):
    H, W, idx, z = rand_case(seed=3)
    f = dv.forward(H, W, idx, z, None, 1.0, "skew_kl", a)
    p, q = dense_rows(H, W, idx, z, 1.0)
    ref = np.array([entropy(p[t], a * p[t] + (1 - a) * q[t]) for t in range(len(p))])
    np.testing.assert_allclose(f["div"], ref, rtol=1e-10)


@pytest.mark.parametrize("a", [0.05, 0.1, 0.6, 1.0])
def test_skew_reverse_kl_against_relative_entropy(a):
    H, W, idx, z = rand_case(seed=4)
    f = dv.forward(H, W, idx, z, None, 0.8, "skew_rkl", a)
    p, q = dense_rows(H, W, idx, z, 0.8)
    ref = np.array([entropy(q[t], a * q[t] + (1 - a) * p[t]) for t in range(len(p))])
    np.testing.assert_allclose(f["div"], ref, rtol=1e-10, atol=1e-15)
    if a == 1.0:
        np.testing.assert_allclose(f["div"], 0.0, atol=1e-15)


def test_total_variation_brute_force_over_events():
    # TV(p, q) = max over sets A of the vocabulary of p(A) - q(A)
    H, W, idx, z = rand_case(T=4, V=10, K=4, seed=5)
    f = dv.forward(H, W, idx, z, None, 1.0, "tv")
    p, q = dense_rows(H, W, idx, z, 1.0)
    for t in range(len(p)):
        best = 0.0
        for r in range(11):
            for A in itertools.combinations(range(10), r):
                A = list(A)
                best = max(best, p[t, A].sum() - q[t, A].sum())
        assert f["div"][t] == pytest.approx(best, rel=1e-12)
        assert f["div"][t] == pytest.approx(1.0 - np.minimum(p[t], q[t]).sum(), rel=1e-12)
        assert 0.0 <= f["div"][t] <= 1.0


def test_skew_kl_zero_is_the_default_kl_loss():
    H, W, idx, z = rand_case(seed=6)
    mask = np.array([1, 0, 1, 1, 1, 1], np.uint8)
    a = dv.forward(H, W, idx, z, mask, 1.4, "skew_kl", 0.0)
    b = oracle.forward(H, W, idx, z, mask, 1.4)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-12)
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=1e-13)
    dH1, dW1 = dv.backward(H, W, idx, z, mask, 1.4, "skew_kl", 0.0, grad=0.7)
    dH2, dW2 = oracle.backward(H, W, idx, z, mask, 1.4, grad=0.7)
    np.testing.assert_allclose(dH1, dH2, rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(dW1, dW2, rtol=1e-10, atol=1e-15)


@pytest.mark.parametrize("kind,param", PARAMS)
def test_zero_when_teacher_is_student(kind, param):
    T, d, V = 4, 6, 16
    rng = np.random.default_rng(7)
    H, W = rng.standard_normal((T, d)), rng.standard_normal((V, d)) * 0.7
    idx = np.stack([rng.permutation(V) for _ in range(T)])
    z = np.take_along_axis(H @ W.T, idx, axis=1)
    f = dv.forward(H, W, idx, z, None, 1.3, kind, param)
    np.testing.assert_allclose(f["div"], 0.0, atol=1e-14)
    if kind == "tv":
        return  # |p - q| has no derivative at p = q; rounding picks the subgradient's sign
    dH, dW = dv.backward(H, W, idx, z, None, 1.3, kind, param)
    np.testing.assert_allclose(dH, 0.0, atol=1e-13)
    np.testing.assert_allclose(dW, 0.0, atol=1e-13)


@pytest.mark.parametrize("kind,param", PARAMS)
def test_nonnegative(kind, param):
    H, W, idx, z = rand_case(seed=8, T=10)
    f = dv.forward(H, W, idx, z, None, 1.0, kind, param)
    assert np.all(f["div"] >= -1e-15)


@pytest.mark.parametrize("kind,param", PARAMS)
def test_gradients_finite_differences(kind, param):
    T, d, V, K, tau = 4, 5, 12, 4, 1.3
    H, W, idx, z = rand_case(T=T, d=d, V=V, K=K, seed=9)
    mask = np.array([1, 1, 0, 1], np.uint8)
    g = -0.6
    dH, dW = dv.backward(H, W, idx, z, mask, tau, kind, param, grad=g)

    def loss(H_, W_):
        return g * dv.forward(H_, W_, idx, z, mask, tau, kind, param)["loss"]

    h = 1e-6
    for X, dX, is_h in ((H, dH, True), (W, dW, False)):
        num = np.zeros_like(X)
        for i in range(X.shape[0]):
            for j in range(X.shape[1]):
                Xp, Xm = X.copy(), X.copy()
                Xp[i, j] += h
                Xm[i, j] -= h
                lp = loss(Xp, W) if is_h else loss(H, Xp)
                lm = loss(Xm, W) if is_h else loss(H, Xm)
                num[i, j] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - dX)) / np.max(np.abs(num))
        assert err < 1e-6, f"{kind} {'dH' if is_h else 'dW'} relative error {err:.2e}"


@pytest.mark.parametrize("kind,param", PARAMS)
def test_repeated_ids_add_their_probabilities(kind, param):
    # Row 0 holds id 3 twice.  The same row with one slot carrying the summed probability
    # (logit tau * log(e^{z1/tau} + e^{z2/tau})) and the other slot at -inf gives the same value.
    H, W, idx, z = rand_case(T=2, d=6, V=20, K=4, seed=10)
    tau = 1.2
    idx = idx.copy()
    idx[0] = [3, 7, 3, 11]
    z = z.copy()
    z[0] = [2.0, 1.0, 0.5, -0.3]
    idx2, z2 = idx.copy(), z.copy()
    idx2[0, 2] = 15
    z2[0, 0] = tau * np.logaddexp(z[0, 0] / tau, z[0, 2] / tau)
    z2[0, 2] = -np.inf
    a = dv.forward(H, W, idx, z, None, tau, kind, param)
    b = dv.forward(H, W, idx2, z2, None, tau, kind, param)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-12)
    dHa, dWa = dv.backward(H, W, idx, z, None, tau, kind, param)
    dHb, dWb = dv.backward(H, W, idx2, z2, None, tau, kind, param)
    np.testing.assert_allclose(dHa, dHb, rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(dWa, dWb, rtol=1e-10, atol=1e-15)


@pytest.mark.parametrize("kind,param", [("jsd", 0.3), ("skew_rkl", 0.2), ("tv", 0.0)])
def test_tau_identity(kind, param):
    H, W, idx, z = rand_case(seed=11)
    tau = 2.5
    a = dv.forward(H, W, idx, z, None, tau, kind, param)["loss"]
    b = dv.forward(H / tau, W, idx, z / tau, None, 1.0, kind, param)["loss"]
    assert a == pytest.approx(tau ** 2 * b, rel=1e-12)


@pytest.mark.parametrize("kind,param", [("jsd", 0.5), ("skew_kl", 0.1), ("tv", 0.0)])
def test_masked_rows_do_not_matter(kind, param):
    H, W, idx, z = rand_case(seed=12)
    mask = np.array([1, 0, 1, 0, 1, 1], np.uint8)
    H2, z2, idx2 = H.copy(), z.copy(), idx.copy()
    H2[[1, 3]] = 5.0
    z2[[1, 3]] = -z2[[1, 3]]
    idx2[[1, 3]] = idx2[[1, 3]][:, ::-1]
    a = dv.forward(H, W, idx, z, mask, 1.0, kind, param)["loss"]
    b = dv.forward(H2, W, idx2, z2, mask, 1.0, kind, param)["loss"]
    assert a == pytest.approx(b, rel=1e-13)
    dH, _ = dv.backward(H2, W, idx2, z2, mask, 1.0, kind, param)
    assert np.all(dH[[1, 3]] == 0.0)


def test_parameter_ranges():
    with pytest.raises(ValueError):
        dv.check_param("jsd", 0.0)
    with pytest.raises(ValueError):
        dv.check_param("skew_kl", 1.0)
    with pytest.raises(ValueError):
        dv.check_param("skew_rkl", 0.0)
    with pytest.raises(ValueError):
        dv.check_param("reverse_kl", 0.5)


@pytest.mark.parametrize("kind,param", [("jsd", 0.3), ("skew_rkl", 0.2), ("tv", 0.0)])
def test_row_samplers_match_the_full_backward(kind, param):
    # dH_rows / dW_rows (used at full vocabulary size) are rows of the finite-difference-pinned
    # backward
    H, W, idx, z = rand_case(T=9, d=7, V=40, K=6, seed=13)
    mask = np.array([1, 0, 1, 1, 0, 1, 1, 1, 0], np.uint8)
    dH, dW = dv.backward(H, W, idx, z, mask, 1.4, kind, param, grad=0.6)
    rows = [0, 3, 4, 8]
    np.testing.assert_allclose(dv.dH_rows(H, W, idx, z, mask, 1.4, kind, param, rows, grad=0.6, chunk=3),
                               dH[rows], rtol=1e-12, atol=1e-15)
    vr = [0, 5, 17, 39]
    np.testing.assert_allclose(dv.dW_rows(H, W, idx, z, mask, 1.4, kind, param, vr, grad=0.6, chunk=2),
                               dW[vr], rtol=1e-12, atol=1e-15)
