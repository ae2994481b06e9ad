"""Seeded random shapes through the whole path against the float64 oracle.

Each case draws T, d, V, K, tau, chunk, a mask fraction and a divergence, so that the
planning on the host (vocabulary splits, grouped unit order, backward blocks of tokens x
vocabulary slabs, tile widths along d) meets shapes that the hand-picked cases do not:
ragged everywhere, long sequences against small vocabularies (several token blocks),
chunk from 1 to larger than T.  Tolerances as in test_gpu_parity."""
import numpy as np
import pytest

import workloads
from tests.test_gpu_divergences import run_gpu as run_gpu_div
from tests.test_gpu_divergences import run_oracle as run_oracle_div
from tests.test_gpu_parity import assert_parity, fkl, run_gpu, run_oracle  # noqa: F401

pytestmark = pytest.mark.gpu

N_CASES = 32


def draw(i):
    # odd cases: long sequences against small vocabularies, where the backward takes several
    # token blocks; even cases: anything
    rng = np.random.default_rng(9000 + i)
    if i % 2:
        T = int(rng.integers(2000, 6001))
        V = int(rng.integers(100, 1501))
        chunk = int(rng.choice([128, 256, 512]))
    else:
        T = int(rng.integers(1, 3001))
        V = int(rng.integers(100, 6001))
        chunk = int(rng.choice([1, 7, 64, 256, 1024, 100000]))
    d = 8 * int(rng.integers(1, 41))
    K = int(rng.integers(1, min(64, V) + 1))
    tau = float(np.round(rng.uniform(0.3, 3.0), 2))
    mask_frac = float(rng.choice([0.0, 0.1, 0.5]))
    kind = str(rng.choice(["kl", "kl", "jsd", "skew_kl", "skew_rkl", "tv"]))
    return T, d, V, K, tau, chunk, mask_frac, kind


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(fkl, i):
    T, d, V, K, tau, chunk, mf, kind = draw(i)
    x = workloads.make_random(T, d, V, K, tau=tau, chunk=chunk, seed=700 + i, mask_frac=mf)
    if kind == "kl":
        assert_parity(run_gpu(fkl, x), run_oracle(x))
    else:
        assert_parity(run_gpu_div(fkl, x, kind, None), run_oracle_div(x, kind, None))
