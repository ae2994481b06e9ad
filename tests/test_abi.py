"""The C ABI library builds, loads without a GPU, exports every declared symbol, sizes its
workspace as documented and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
FKL_OK, INVALID, ALIGN, UNSUP, WS, CUDA = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def L():
    from lm_head_top_tcgen05_gb300 import build
    from lm_head_top_tcgen05_gb300._lib import lib

    build.build()
    return lib()


def declared_symbols():
    names = set()
    for h in (ROOT / "include").glob("*.h"):
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names |= set(re.findall(r"\b(fkl_[a-z_0-9]+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(L):
    from lm_head_top_tcgen05_gb300._lib import _SIGNATURES

    names = declared_symbols()
    assert {"fkl_forward", "fkl_backward", "fkl_workspace_size", "fkl_read_status"} <= names
    for n in names:
        assert hasattr(L, n), n
    assert names == set(_SIGNATURES), "binding signatures and headers disagree"


def test_status_strings(L):
    assert L.fkl_status_string(0) == b"ok"
    assert b"teacher id" in L.fkl_status_string(6)
    assert b"global count" in L.fkl_status_string(11)
    assert L.fkl_status_string(99) == b"unknown status"


def test_workspace_size_plan(L):
    ws = L.fkl_workspace_size
    assert ws(256, 256, 4096, 16, 64) > 0
    assert ws(256, 7, 4096, 16, 64) == 0       # d not a multiple of 8
    assert ws(256, 256, 0, 16, 64) == 0        # no vocabulary
    assert ws(256, 256, 4096, 0, 64) == 0      # K = 0
    assert ws(256, 256, 4096, 1025, 64) == 0   # K too large
    assert ws(256, 256, 4096, 16, 0) == 0      # chunk = 0
    assert ws(0, 256, 4096, 16, 64) > 0        # empty batch is fine
    # the dS slab obeys the chunk bound: at most chunk * V bf16 values (whole 256-wide tiles)
    T, d, V, K = 32768, 2880, 201088, 100
    fixed = ws(T, d, V, K, 1) - T * 256 * 2    # chunk=1 gives the one-tile minimum slab
    for chunk in (512, 2048, 4096):
        ds_bytes = ws(T, d, V, K, chunk) - fixed
        assert ds_bytes <= chunk * V * 2 + 256
        assert ds_bytes >= 0.75 * chunk * V * 2  # slabs are evened out, so a little below
    assert ws(T, d, V, K, 2048) < 2 * 2**30    # far below T * V * 2 = 13 GB
    assert ws(T, d, V, K, 2048) < T * V * 2 / 8


def _args(L, **over):
    a = dict(H=16, W=16, idx=16, z=16, mask=None, T=256, d=256, V=4096, K=16, tau=1.0, chunk=64,
             loss=16, lse=16, ws=256, ws_bytes=L.fkl_workspace_size(256, 256, 4096, 16, 64), stream=None)
    a.update(over)
    return a


def _fwd(L, **over):
    a = _args(L, **over)
    return L.fkl_forward(a["H"], a["W"], a["idx"], a["z"], a["mask"], a["T"], a["d"], a["V"], a["K"],
                         a["tau"], a["chunk"], a["loss"], a["lse"], a["ws"], a["ws_bytes"], a["stream"])


def test_forward_rejects_bad_arguments_on_host(L):
    # Pointers are fake (never dereferenced): every case fails before any CUDA call.
    assert _fwd(L, W=None) == INVALID
    assert _fwd(L, H=None) == INVALID
    assert _fwd(L, d=12) == INVALID
    assert _fwd(L, K=0) == INVALID
    assert _fwd(L, tau=0.0) == INVALID
    assert _fwd(L, tau=float("inf")) == INVALID
    assert _fwd(L, chunk=0) == INVALID
    assert _fwd(L, ws=None) == WS
    assert _fwd(L, ws_bytes=1024) == WS
    assert _fwd(L, ws=512 + 16) == ALIGN
    assert _fwd(L, H=16 + 2) == ALIGN
    assert _fwd(L, idx=16 + 2) == ALIGN
    assert b"workspace" in L.fkl_last_error() or True


def test_valid_call_without_gpu_fails_loudly(L):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd(L) in (CUDA, UNSUP)
    assert len(L.fkl_last_error()) > 0


def test_backward_rejects_bad_arguments_on_host(L):
    ws_bytes = L.fkl_workspace_size(256, 256, 4096, 16, 64)
    st = L.fkl_backward(16, 16, 16, 16, None, 16, None, 256, 256, 4096, 16, 1.0, 64, None, 16, 256,
                        ws_bytes, None)
    assert st == INVALID  # dH missing
    st = L.fkl_backward(16, 16, 16, 16, None, 16, None, 256, 256, 4096, 16, 1.0, 64, 16 + 4, 16, 256,
                        ws_bytes, None)
    assert st == ALIGN    # dH not 16-byte aligned


def test_bf16_backward_checks_and_workspace(L):
    from lm_head_top_tcgen05_gb300._lib import FklOptions

    T, d, V, K, chunk = 4000, 64, 2999, 16, 512
    n32 = L.fkl_workspace_size(T, d, V, K, chunk)
    n16 = L.fkl_backward_bf16_workspace_size(T, d, V, K, chunk)
    Ct, nt = _plan(L, T, d, V, K, chunk)[:2]
    assert nt > 1 and n16 >= n32 + Ct * d * 4 + V * d * 4    # dH of a block and dW over blocks
    T1 = 700
    Ct1, nt1 = _plan(L, T1, d, V, K, chunk)[:2]
    assert nt1 == 1 and L.fkl_backward_bf16_workspace_size(T1, d, V, K, chunk) >= \
        L.fkl_workspace_size(T1, d, V, K, chunk) + Ct1 * d * 4
    assert L.fkl_backward_bf16_workspace_size(T, 12, V, K, chunk) == 0
    # long sequences against a larger vocabulary: the slabs go outer, and the fp32 sums (all
    # of dH, one slab of dW) are smaller than one token block of dH plus all of dW
    T2, V2 = 2000, 3000
    Ct2, nt2, Vc2, ns2, Vmax2 = _plan(L, T2, d, V2, K, 256)
    assert nt2 > 1 and ns2 > 1
    extra = L.fkl_backward_bf16_workspace_size(T2, d, V2, K, 256) - L.fkl_workspace_size(T2, d, V2, K, 256)
    assert T2 * d * 4 + Vmax2 * d * 4 <= extra < Ct2 * d * 4 + V2 * d * 4
    o = FklOptions()
    o.accumulate = 3
    # bf16 gradients do not accumulate; the fp32 workspace is too small for bf16 gradients
    assert L.fkl_backward_bf16(16, 16, 16, 16, None, 16, None, T, d, V, K, 1.0, chunk, ctypes.byref(o), 256, 256,
                               256, n16, None) == INVALID
    assert L.fkl_backward_bf16(16, 16, 16, 16, None, 16, None, T, d, V, K, 1.0, chunk, None, 256, 256, 256, n32,
                               None) == WS
    assert L.fkl_backward_bf16(16, 16, 16, 16, None, 16, None, T, d, V, K, 1.0, chunk, None, 256 + 8, 256, 256, n16,
                               None) == ALIGN


def test_test_hooks_reject_bad_arguments(L):
    assert L.fkl_test_gemm(16, 16, 16, 0, 8, 8, 0, 0, 256, 0, 256, 256, None) == INVALID
    assert L.fkl_test_gemm(16, 16, 16, 8, 8, 8, 0, 0, 100, 0, 256, 256, None) == INVALID
    assert L.fkl_test_gemm(16, 16, 16, 8, 8, 12, 0, 0, 256, 0, 256, 256, None) == ALIGN
    assert L.fkl_test_wait_timeout(0, 256, 256, None) == INVALID
    assert L.fkl_test_wait_timeout(2_000_000_000, 256, 256, None) == INVALID


def test_python_binding_needs_cuda_tensors():
    import torch

    import lm_head_top_tcgen05_gb300 as fkl

    H = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fkl.forward(H, H, torch.zeros(4, 1, dtype=torch.int32), torch.zeros(4, 1))


def test_options_are_checked_on_host(L):
    from lm_head_top_tcgen05_gb300._lib import FklOptions

    ws_bytes = L.fkl_workspace_size(256, 256, 4096, 16, 64)

    def fwd(o):
        return L.fkl_forward_ex(16, 16, 16, 16, None, 256, 256, 4096, 16, 1.0, 64, ctypes.byref(o), 16, 16, 256,
                                ws_bytes, None)

    o = FklOptions()
    o.reserved = 1
    assert fwd(o) == INVALID
    o = FklOptions()
    o.normalization = 5
    assert fwd(o) == INVALID
    o = FklOptions()
    o.normalization = 1
    o.num_seqs = 3
    assert fwd(o) == INVALID          # seq_ids missing
    o.seq_ids = 16
    o.num_seqs = 0
    assert fwd(o) == INVALID          # no sequence
    o.num_seqs = 257
    assert fwd(o) == INVALID          # more sequences than tokens
    o.num_seqs = 3
    o.seq_ids = 18
    assert fwd(o) == ALIGN
    o = FklOptions()
    o.accumulate = 4
    assert fwd(o) == INVALID
    o = FklOptions()
    o.global_count = 20                # an int64 scalar must be 8-byte aligned
    assert fwd(o) == ALIGN


def test_local_count_is_checked_on_host(L):
    from lm_head_top_tcgen05_gb300._lib import FklOptions

    def cnt(T, opts, count, ws, nbytes):
        return L.fkl_local_count(None, T, ctypes.byref(opts) if opts is not None else None, count, ws, nbytes, None)

    assert cnt(-1, None, 16, 256, 4096) == INVALID
    assert cnt(100, None, None, 256, 4096) == INVALID       # no output
    assert cnt(100, None, 12, 256, 4096) == ALIGN           # int64 output 8-byte aligned
    assert cnt(100, None, 16, None, 4096) == WS
    assert cnt(100, None, 16, 128, 4096) == ALIGN           # workspace 256-byte aligned
    assert cnt(1000, None, 16, 256, 256 + 4 * 1000 - 1) == WS
    o = FklOptions()
    o.normalization, o.num_seqs = 1, 3
    assert cnt(100, o, 16, 256, 4096) == INVALID            # seq_ids missing
    # a valid call without a GPU fails on the device query, not before
    assert cnt(100, None, 16, 256, 4096) in (UNSUP, CUDA)


def test_divergence_options_are_checked_on_host(L):
    from lm_head_top_tcgen05_gb300._lib import FklOptions

    ws_bytes = L.fkl_workspace_size(256, 256, 4096, 16, 64)

    def fwd(o):
        return L.fkl_forward_ex(16, 16, 16, 16, None, 256, 256, 4096, 16, 1.0, 64, ctypes.byref(o), 16, 16, 256,
                                ws_bytes, None)

    def bwd(o):
        return L.fkl_backward_ex(16, 16, 16, 16, None, 16, None, 256, 256, 4096, 16, 1.0, 64, ctypes.byref(o),
                                 16, 16, 256, ws_bytes, None)

    for kind, param in ((5, 0.0), (-1, 0.0), (1, 0.0), (1, 1.0), (2, 1.0), (2, -0.1), (3, 0.0), (3, 1.5),
                        (1, float("nan"))):
        o = FklOptions()
        o.divergence, o.div_param = kind, param
        assert fwd(o) == INVALID, (kind, param)
    o = FklOptions()
    o.divergence, o.div_param = 1, 0.5
    o.student_topk_logits = 18
    assert fwd(o) == ALIGN
    o.student_topk_logits = None
    assert bwd(o) == INVALID  # the backward of a divergence other than KL needs the student logits


def test_options_struct_layout_matches_header(tmp_path):
    # Compile a probe against include/fkl.h and compare fkl_options' layout with the binding's.
    import subprocess

    from lm_head_top_tcgen05_gb300._lib import FklOptions

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "layout.c"
    fields = [f for f, _ in FklOptions._fields_]
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "fkl.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(fkl_options));\n'
                   + "".join(f'  printf("%zu\\n", offsetof(fkl_options, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(root, "include"), str(src), "-o", str(exe)], check=True)
    out = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(FklOptions)
    assert out[1:] == [getattr(FklOptions, f).offset for f in fields]


def test_teacher_topk_stride_is_checked_on_host(L):
    n = L.fkl_teacher_topk_workspace_size(64, 64, 8192, 16)
    for bad in (3, 16, -1):
        assert L.fkl_teacher_topk_ex(16, 16, 64, 64, 8192, 16, bad, 16, 16, 256, n, None) == INVALID


def _plan(L, T, d, V, K, chunk, sms=152):
    out = (ctypes.c_int64 * 5)()
    assert L.fkl_test_backward_plan(T, d, V, K, chunk, sms, out) == 0
    return tuple(out)


@pytest.mark.parametrize("T,d,V,K,chunk", [(32768, 2880, 201088, 100, 2048), (262144, 2880, 201088, 100, 4096),
                                           (65536, 4096, 151936, 100, 4096), (8192, 3072, 128256, 100, 1024),
                                           (4000, 64, 2999, 16, 512), (300, 200, 5000, 16, 128), (1, 64, 777, 8, 1)])
def test_backward_blocks_respect_the_chunk_bound(L, T, d, V, K, chunk):
    for sms in (152, 148, 132, 2):
        Ct, nt, Vc, ns, Vmax = _plan(L, T, d, V, K, chunk, sms)
        assert Vc % 256 == 0 and Vc >= 256 and ns * Vc >= V and (ns - 1) * Vc < V
        assert nt * Ct >= T and (nt - 1) * Ct < T
        assert Ct == T or Ct % 256 == 0
        # the dS buffer of one block: at most chunk * V values, or one 256-wide tile of Ct rows
        assert Vc <= Vmax and 2 * Vc >= Vmax - 256
        assert Ct * Vmax <= max(min(chunk, T) * V, Ct * 256)
    # no device here: the slab count is planned for a GB300's 152 SMs
    assert L.fkl_backward_slabs(T, d, V, K, chunk) == _plan(L, T, d, V, K, chunk)[1] * _plan(L, T, d, V, K, chunk)[3]


def test_backward_block_choice(L):
    # 32K: full-height slabs (dW written once); 256K and long sequences: lower blocks cut the
    # read-modify-write of dH, which otherwise grows with the number of narrow slabs
    assert _plan(L, 32768, 2880, 201088, 100, 2048)[1] == 1
    Ct, nt, Vc, ns, _ = _plan(L, 262144, 2880, 201088, 100, 4096)
    assert nt > 1 and Ct < 262144

    def rmw(T, d, V, nt, ns):
        return (2 * ns - 1) * T * d * 4 + (2 * nt - 1) * V * d * 4

    assert rmw(262144, 2880, 201088, nt, ns) < 0.3 * rmw(262144, 2880, 201088, 1, 66)
    assert _plan(L, 4000, 64, 2999, 16, 512)[1] > 1


def test_slab_width_fills_the_dw_waves(L):
    # 32K tokens, d = 2880 (12 tiles of 256): the widest slab the chunk allows is 49 tiles and
    # evening it over the slabs gives 47, whose dW GEMM has 47 x 12 = 564 one-tile units, 7.4
    # waves of 76 CTA pairs run as 8.  44-tile slabs give 528 units, 6.95 waves.
    Ct, nt, Vc, ns, Vmax = _plan(L, 32768, 2880, 201088, 100, 2048, 152)
    assert (Ct, nt, Vmax) == (32768, 1, 49 * 256)
    assert (Vc, ns) == (44 * 256, 18)
    units = Vc // 256 * 12
    assert units / 76 > 0.9 * -(-units // 76)
    # the slab width follows the device: half the pairs, other waves
    assert _plan(L, 32768, 2880, 201088, 100, 2048, 76)[2] != Vc
