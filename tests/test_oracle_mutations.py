"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch each.

This is what makes the pins worth trusting: a mistake that no pin notices would let a
wrong oracle certify a wrong kernel.  Each mutation replaces one internal step of
``oracle.dense_kl`` for the duration of one test.
"""
import numpy as np
import pytest

import oracle.dense_kl as dk
from tests import test_oracle_pins as pins

PIN_CALLS = [
    lambda: [pins.test_closed_form_cases(c) for c in pins.json.load(open(pins.GOLDEN))["cases"]],
    lambda: pins.test_kl_zero_when_teacher_is_student(2.0),
    lambda: pins.test_kl_nonnegative(1),
    lambda: pins.test_single_slot_is_cross_entropy(1.5),
    pins.test_dense_grid_matches_torch_kl_div_and_logsumexp,
    pins.test_tau_identity,
    lambda: pins.test_gradient_finite_differences(1.7, True),
    lambda: pins.test_gradient_finite_differences(1.0, False),
    pins.test_gradient_matches_autograd_on_dense_formula,
    pins.test_chunk_invariance,
    pins.test_masked_rows_change_nothing,
    pins.test_no_valid_token,
    pins.test_sequence_mean_of_one_sequence_is_token_mean,
    pins.test_sequence_mean_weights_unequal_sequences,
    pins.test_sequence_mean_matches_autograd,
    pins.test_shards_with_the_batch_count_add_up_to_the_batch,
    pins.test_sequence_shards_with_the_batch_count_add_up_to_the_batch,
]


def failing_pins():
    failed = 0
    for call in PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                call()
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed += 1
    return failed


def test_unmutated_oracle_passes_every_pin():
    assert failing_pins() == 0


orig_row_terms = dk._row_terms
orig_ds_block = dk._ds_block
orig_teacher_probs = dk.teacher_probs


def row_terms_no_student_tau(s, idx, p, logp, tau):
    return orig_row_terms(s * tau, idx, p, logp, tau)


def row_terms_drop_entropy(s, idx, p, logp, tau):
    return orig_row_terms(s, idx, p, np.zeros_like(logp), tau)


def row_terms_wrong_index(s, idx, p, logp, tau):
    return orig_row_terms(s, (idx + 1) % s.shape[1], p, logp, tau)


def ds_sign_flip(s, idx, p, valid, tau, scale):
    return -orig_ds_block(s, idx, p, valid, tau, scale)


def ds_scatter_assign(s, idx, p, valid, tau, scale):
    a = s / tau
    q = np.exp(a - a.max(1, keepdims=True))
    q /= q.sum(1, keepdims=True)
    pt = np.zeros_like(q)
    np.put_along_axis(pt, idx, p, axis=1)  # assignment: repeated ids lose mass
    ds = scale * (q - pt)
    ds[~valid] = 0
    return ds


def ds_missing_tau(s, idx, p, valid, tau, scale):
    return orig_ds_block(s, idx, p, valid, tau, scale / tau)


orig_token_weights = dk.token_weights


def weights_ignore_mask(mask, T, norm="tokens", seq_ids=None, count=None):
    return orig_token_weights(None, T, norm, seq_ids, count)


def weights_sequence_by_total_count(mask, T, norm="tokens", seq_ids=None, count=None):
    w = orig_token_weights(mask, T, norm, seq_ids, count)
    if norm == "sequences":  # divides by the total valid count instead of each sequence's
        w = orig_token_weights(mask, T, "tokens", count=count)
    return w


def own_count_ignores_batch_count(n, count):
    return n  # a split batch normalised by each shard's own count


def own_count_in_forward_only(n, count):
    # the batch's count reaches the loss but not the gradient's scale: dH_rows / dW_rows / the
    # backward's token weights keep the shard's own count
    import inspect

    caller = inspect.stack()[1].function
    return n if caller in ("dH_rows", "dW_rows", "token_weights") else (n if count is None else int(count))


def probs_no_teacher_tau(z, tau):
    return orig_teacher_probs(z, 1.0)


def lse_log2(s, idx, p, logp, tau):
    lse, kl = orig_row_terms(s, idx, p, logp, tau)
    return lse / np.log(2.0), kl


MUTATIONS = {
    "_row_terms": [row_terms_no_student_tau, row_terms_drop_entropy, row_terms_wrong_index, lse_log2],
    "_ds_block": [ds_sign_flip, ds_scatter_assign, ds_missing_tau],
    "token_weights": [weights_ignore_mask, weights_sequence_by_total_count],
    "_own_count": [own_count_ignores_batch_count, own_count_in_forward_only],
    "teacher_probs": [probs_no_teacher_tau],
}


@pytest.mark.parametrize("target,mutant", [(t, m) for t, ms in MUTATIONS.items() for m in ms],
                         ids=lambda x: getattr(x, "__name__", x))
def test_planted_mistake_is_caught(monkeypatch, target, mutant):
    monkeypatch.setattr(dk, target, mutant)
    assert failing_pins() >= 1


def test_loss_normaliser_mistake_is_caught(monkeypatch):
    orig_forward = dk.forward

    def forward_over_all_tokens(H, W, idx, z, mask, tau, chunk=64, rows=None, **kw):
        out = orig_forward(H, W, idx, z, mask, tau, chunk, rows, **kw)
        if out["loss"] is not None and out["n_valid"]:
            out["loss"] *= out["n_valid"] / len(out["lse"])  # divides by T, not N_valid
        return out

    monkeypatch.setattr(dk, "forward", forward_over_all_tokens)
    import oracle
    monkeypatch.setattr(oracle, "forward", forward_over_all_tokens)
    assert failing_pins() >= 1


# ---- the other divergences (oracle/divergences.py) against their own pins

import oracle.divergences as dvm  # noqa: E402
from tests import test_oracle_divergences as dpins  # noqa: E402

DIV_PIN_CALLS = [
    lambda: dpins.test_jsd_half_is_scipy_jensen_shannon(1.0),
    lambda: dpins.test_generalised_jsd_against_relative_entropy(0.35),
    lambda: dpins.test_skew_kl_against_relative_entropy(0.1),
    lambda: dpins.test_skew_reverse_kl_against_relative_entropy(0.1),
    dpins.test_total_variation_brute_force_over_events,
    dpins.test_skew_kl_zero_is_the_default_kl_loss,
] + [(lambda k=k, a=a: dpins.test_gradients_finite_differences(k, a)) for k, a in dpins.PARAMS] + [
    (lambda k=k, a=a: dpins.test_repeated_ids_add_their_probabilities(k, a)) for k, a in dpins.PARAMS]


def failing_div_pins():
    failed = 0
    for call in DIV_PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                call()
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed += 1
    return failed


orig_div_rows = dvm.divergence_rows
orig_gamma = dvm.gamma
orig_dense_block = dvm._dense_block


def div_jsd_mixture_swapped(p, q, kind, param):
    return orig_div_rows(p, q, kind, 1.0 - param if kind == "jsd" else param)


def div_tv_no_half(p, q, kind, param):
    return orig_div_rows(p, q, kind, param) * (2.0 if kind == "tv" else 1.0)


def div_skew_rkl_as_skew_kl(p, q, kind, param):
    return orig_div_rows(p, q, "skew_kl" if kind == "skew_rkl" else kind, min(param, 0.99))


def gamma_skew_rkl_drops_terms(p, q, kind, param):
    g = orig_gamma(p, q, kind, param)
    if kind == "skew_rkl":
        m = param * q + (1 - param) * p
        g = g - 1.0 + param * q / m
    return g


def gamma_jsd_drops_weight(p, q, kind, param):
    g = orig_gamma(p, q, kind, param)
    return g / (1.0 - param) if kind == "jsd" else g


def dense_block_assigns_repeats(s_blk, idx_blk, p_blk, tau):
    q, pt, lse = orig_dense_block(s_blk, idx_blk, p_blk, tau)
    pt = np.zeros_like(q)
    pt[np.arange(q.shape[0])[:, None], idx_blk] = p_blk
    return q, pt, lse


DIV_MUTATIONS = {
    "divergence_rows": [div_jsd_mixture_swapped, div_tv_no_half, div_skew_rkl_as_skew_kl],
    "gamma": [gamma_skew_rkl_drops_terms, gamma_jsd_drops_weight],
    "_dense_block": [dense_block_assigns_repeats],
}


def test_unmutated_divergence_oracle_passes_every_pin():
    assert failing_div_pins() == 0


@pytest.mark.parametrize("target,mutant", [(t, m) for t, ms in DIV_MUTATIONS.items() for m in ms],
                         ids=lambda x: getattr(x, "__name__", x))
def test_planted_divergence_mistake_is_caught(monkeypatch, target, mutant):
    monkeypatch.setattr(dvm, target, mutant)
    assert failing_div_pins() > 0
