"""Token-sharded data parallelism (lm_head_top_tcgen05_gb300.data_parallel) on CPU ranks.

Two gloo ranks each hold an uneven shard of one batch (different numbers of tokens and of
valid tokens).  ShardedStep's control flow - the count all-reduce before the loss, the loss
and dW all-reduces after the backward - runs with the float64 oracle standing in for the
library's kernels.  The ranks' results must equal the oracle on the whole batch: the loss and
dW of the whole batch on every rank, and each rank's dH rows."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

T, D, V, K, TAU = 16, 8, 40, 5, 1.3
CUT = 6  # rank 0 holds rows [0, 6), rank 1 rows [6, 16)
MASK = np.array([1, 0, 1, 1, 1, 1, 0, 0, 1, 1, 1, 0, 1, 1, 1, 1], np.uint8)
SEQ = np.array([0, 0, 0, 1, 1, 1, 2, 2, 2, 2, 3, 3, 4, 4, 4, 4])  # no sequence crosses the cut


def batch():
    rng = np.random.default_rng(41)
    H = rng.standard_normal((T, D))
    W = rng.standard_normal((V, D)) * 0.5
    idx = np.stack([rng.permutation(V)[:K] for _ in range(T)])
    z = -np.sort(-(rng.standard_normal((T, K)) * 2.0 + 1.0), axis=1)
    return H, W, idx, z


class OracleOps:
    """The library's three calls, computed by the float64 oracle on CPU tensors."""

    def __init__(self, norm="tokens"):
        self.norm = norm

    def local_count(self, mask, T, device, seq_ids, num_seqs, workspace):
        m = mask.numpy().astype(bool)
        if self.norm == "tokens":
            return torch.tensor(int(m.sum()), dtype=torch.int64)
        return torch.tensor(len(set(seq_ids.numpy()[m].tolist())), dtype=torch.int64)

    def forward(self, H, W, idx, z, mask, tau, chunk, workspace=None, seq_ids=None, num_seqs=None,
                global_count=None):
        import oracle

        f = oracle.forward(H.numpy(), W.numpy(), idx.numpy(), z.numpy(), mask.numpy(), tau, norm=self.norm,
                           seq_ids=None if seq_ids is None else seq_ids.numpy(), count=int(global_count))
        return torch.tensor(f["loss"], dtype=torch.float64), torch.from_numpy(f["lse"])

    def backward(self, H, W, idx, z, mask, lse, tau, chunk, out=None, grad_dtype=None, workspace=None,
                 seq_ids=None, num_seqs=None, global_count=None):
        import oracle

        dH, dW = oracle.backward(H.numpy(), W.numpy(), idx.numpy(), z.numpy(), mask.numpy(), tau, norm=self.norm,
                                 seq_ids=None if seq_ids is None else seq_ids.numpy(), count=int(global_count))
        return torch.from_numpy(dH), torch.from_numpy(dW)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, norm, out):
    import torch.distributed as dist

    from lm_head_top_tcgen05_gb300.data_parallel import ShardedStep

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        H, W, idx, z = batch()
        rows = slice(0, CUT) if rank == 0 else slice(CUT, T)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))  # noqa: E731
        step = ShardedStep(ops=OracleOps(norm))
        seq = t(SEQ[rows]) if norm == "sequences" else None
        n = step.global_count(t(MASK[rows]), rows.stop - rows.start, "cpu", seq_ids=seq)
        loss, dH, dW = step(t(H[rows]), t(W), t(idx[rows]), t(z[rows]), t(MASK[rows]), TAU, 64, seq_ids=seq)
        out[rank] = (int(n), float(loss), dH.numpy().copy(), dW.numpy().copy())
    finally:
        dist.destroy_process_group()


def _run(norm):
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, norm, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    return out[0], out[1]


@pytest.mark.parametrize("norm", ["tokens", "sequences"])
def test_two_gloo_ranks_reproduce_the_whole_batch(norm):
    import oracle

    H, W, idx, z = batch()
    seq = SEQ if norm == "sequences" else None
    whole = oracle.forward(H, W, idx, z, MASK, TAU, norm=norm, seq_ids=seq)
    dH, dW = oracle.backward(H, W, idx, z, MASK, TAU, norm=norm, seq_ids=seq)
    r0, r1 = _run(norm)
    want_n = int(MASK.sum()) if norm == "tokens" else len(set(SEQ[MASK.astype(bool)].tolist()))
    assert r0[0] == r1[0] == want_n                    # the batch's count on both ranks
    assert int(MASK[:CUT].sum()) != int(MASK[CUT:].sum())  # the shards are uneven
    for r in (r0, r1):
        assert r[1] == pytest.approx(whole["loss"], rel=1e-12)
        np.testing.assert_allclose(r[3], dW, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(r0[2], dH[:CUT], rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(r1[2], dH[CUT:], rtol=1e-11, atol=1e-14)


def test_single_process_step_is_the_plain_step():
    # without torch.distributed the step is the single-device loss of the batch it is given
    import oracle
    from lm_head_top_tcgen05_gb300.data_parallel import ShardedStep

    H, W, idx, z = batch()
    t = torch.from_numpy
    loss, dH, dW = ShardedStep(ops=OracleOps())(t(H), t(W), t(idx), t(z), t(MASK), TAU, 64)
    whole = oracle.forward(H, W, idx, z, MASK, TAU)
    rdH, rdW = oracle.backward(H, W, idx, z, MASK, TAU)
    assert float(loss) == pytest.approx(whole["loss"], rel=1e-13)
    np.testing.assert_allclose(dH.numpy(), rdH, rtol=1e-12)
    np.testing.assert_allclose(dW.numpy(), rdW, rtol=1e-12)
