"""Arguments that are not device memory of the current device are refused on the host.

A host buffer passed by mistake (here pinned host memory, which a kernel could even reach
through unified addressing) must come back as FKL_ERR_INVALID_ARG naming the argument,
with nothing enqueued, from every entry point."""
import ctypes

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

INVALID = 1


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


@pytest.fixture(scope="module")
def case(cuda_device):
    x = workloads.make_random(300, 128, 2000, 8, seed=71)
    dev = "cuda"
    return dict(H=x.H.to(dev), W=x.W.to(dev), idx=x.topk_idx.to(dev), z=x.topk_logits.to(dev),
                z_host=x.topk_logits.pin_memory(), T=300, d=128, V=2000, K=8)


def test_forward_refuses_host_memory(L, case):
    c = case
    ws = torch.empty(L.fkl_workspace_size(c["T"], c["d"], c["V"], c["K"], 64), dtype=torch.uint8, device="cuda")
    loss = torch.zeros((), device="cuda")
    lse = torch.zeros(c["T"], device="cuda")
    loss_host = torch.zeros((), pin_memory=True)
    args = dict(z=c["z"], loss=loss)
    for name, over in (("topk_logits", dict(z=c["z_host"])), ("loss", dict(loss=loss_host))):
        a = dict(args, **over)
        st = L.fkl_forward(_p(c["H"]), _p(c["W"]), _p(c["idx"]), _p(a["z"]), None, c["T"], c["d"], c["V"], c["K"],
                           1.0, 64, _p(a["loss"]), _p(lse), _p(ws), ws.numel(), _stream())
        assert st == INVALID, name
        assert name.encode() in L.fkl_last_error()
    # the same call with device memory runs
    st = L.fkl_forward(_p(c["H"]), _p(c["W"]), _p(c["idx"]), _p(c["z"]), None, c["T"], c["d"], c["V"], c["K"],
                       1.0, 64, _p(loss), _p(lse), _p(ws), ws.numel(), _stream())
    assert st == 0
    torch.cuda.synchronize()
    assert torch.isfinite(loss)


def test_backward_and_count_refuse_host_memory(L, case):
    c = case
    ws = torch.empty(L.fkl_workspace_size(c["T"], c["d"], c["V"], c["K"], 64), dtype=torch.uint8, device="cuda")
    lse = torch.zeros(c["T"], device="cuda")
    dH = torch.empty(c["T"], c["d"], device="cuda")
    dW_host = torch.empty(c["V"], c["d"], pin_memory=True)
    st = L.fkl_backward(_p(c["H"]), _p(c["W"]), _p(c["idx"]), _p(c["z"]), None, _p(lse), None, c["T"], c["d"],
                        c["V"], c["K"], 1.0, 64, _p(dH), _p(dW_host), _p(ws), ws.numel(), _stream())
    assert st == INVALID and b"dW" in L.fkl_last_error()
    count_host = torch.zeros((), dtype=torch.int64, pin_memory=True)
    st = L.fkl_local_count(None, c["T"], None, _p(count_host), _p(ws), ws.numel(), _stream())
    assert st == INVALID and b"count" in L.fkl_last_error()


def test_teacher_topk_refuses_host_memory(L, case):
    c = case
    n = L.fkl_teacher_topk_workspace_size(c["T"], c["d"], c["V"], 8)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    idx = torch.empty(c["T"], 8, dtype=torch.int32, device="cuda")
    val_host = torch.empty(c["T"], 8, pin_memory=True)
    st = L.fkl_teacher_topk(_p(c["H"]), _p(c["W"]), c["T"], c["d"], c["V"], 8, _p(idx), _p(val_host), _p(ws), n,
                            _stream())
    assert st == INVALID and b"topk_logits" in L.fkl_last_error()
