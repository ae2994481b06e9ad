"""fkl_forward_noalloc: the forward for callers that cannot allocate device memory.

Such callers (an operator inside a runtime that owns the whole device memory pool, or a
latency-critical loop that must never call cudaMalloc) get the forward with its scratch in
a fixed device array inside the library.  This checks, through the C ABI, that two calls in
a row give the same loss and lse as fkl_forward with a caller-provided workspace, within the
parity tolerances, with and without a mask; that an empty batch gives a zero loss; and that
a shape too large for the fixed array is refused on the host.  The file is named so that
pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

LOSS_RTOL, LSE_ATOL = 1e-3, 1e-3


@pytest.fixture(scope="module")
def L(cuda_device):
    from lm_head_top_tcgen05_gb300 import build
    from lm_head_top_tcgen05_gb300._lib import lib

    build.build()
    return lib()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_noalloc_forward_matches_workspace_forward(L):
    import lm_head_top_tcgen05_gb300 as fkl

    cases = [(workloads.make_random(300, 200, 5000, 16, tau=2.0, seed=31, mask_frac=0.1), True),
             (workloads.make_random(1000, 256, 7000, 32, tau=1.0, seed=32), True),
             (workloads.make_random(700, 128, 3000, 8, tau=1.0, seed=33), False)]   # mask = NULL
    for x, with_mask in cases:
        H, W = x.H.cuda(), x.W.cuda()
        idx, z = x.topk_idx.cuda(), x.topk_logits.cuda()
        m = x.mask.cuda() if with_mask else None
        T, d = H.shape
        V, K = W.shape[0], idx.shape[1]
        ref_loss, ref_lse = fkl.forward(H, W, idx, z, m, x.tau, x.chunk)
        ref_loss, ref_lse = ref_loss.item(), ref_lse.cpu().numpy()
        for _ in range(2):  # two calls in a row share (and reuse) the fixed scratch
            loss = torch.full((), float("nan"), device="cuda")
            lse = torch.full((T,), float("nan"), device="cuda")
            st = L.fkl_forward_noalloc(_p(H), _p(W), _p(idx), _p(z), _p(m) if m is not None else None,
                                       T, d, V, K, x.tau,
                                       _p(loss), _p(lse), _stream())
            assert st == 0, L.fkl_last_error()
            torch.cuda.synchronize()
            assert abs(loss.item() - ref_loss) <= LOSS_RTOL * abs(ref_loss)
            assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_ATOL


def test_noalloc_empty_batch(L):
    # T = 0: no token, so the loss is 0 and nothing else is written
    W = torch.zeros(1000, 64, dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        loss = torch.full((), float("nan"), device="cuda")
        st = L.fkl_forward_noalloc(None, _p(W), None, None, None, 0, 64, 1000, 16, 1.0, _p(loss), None, _stream())
        assert st == 0, L.fkl_last_error()
        torch.cuda.synchronize()
        assert loss.item() == 0.0


def test_noalloc_rejects_shapes_beyond_its_scratch(L):
    # 100000 tokens at K = 100 need about 119 MB of forward scratch, more than the 64 MiB held.
    dummy = torch.zeros(64, dtype=torch.float32, device="cuda")
    st = L.fkl_forward_noalloc(_p(dummy), _p(dummy), _p(dummy), _p(dummy), None, 100000, 64, 1000, 100,
                               1.0, _p(dummy), _p(dummy), _stream())
    assert st == 4  # FKL_ERR_WORKSPACE, refused before any launch
    assert b"static scratch" in L.fkl_last_error()
