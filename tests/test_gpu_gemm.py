"""The tcgen05 GEMM building block (TMA -> shared memory -> tcgen05.mma -> TMEM -> fp32)
against a float64 host product of the same bf16 operands, for every operand major-ness
and tile width the loss uses, on ragged shapes that leave partial tiles on every axis."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L(cuda_device):
    from lm_head_top_tcgen05_gb300 import build
    from lm_head_top_tcgen05_gb300._lib import lib

    build.build()
    return lib()


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def run_gemm(L, M, N, Kd, a_mn, b_mn, bn, accumulate=False, seed=0, force2d=False, pair=False, ksplit=False):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, Kd, generator=g).to(torch.bfloat16)
    B = torch.randn(N, Kd, generator=g).to(torch.bfloat16)
    D0 = torch.randn(M, N, generator=g) if accumulate else torch.zeros(M, N)
    Ad = (A.t().contiguous() if a_mn else A).cuda()
    Bd = (B.t().contiguous() if b_mn else B).cuda()
    D = D0.clone().cuda()
    # room for 80 partial tiles of 256 x 256 fp32 when the last wave is split along K
    nws = 256 + (80 * 256 * 256 * 4 if ksplit else 0)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    flags = int(accumulate) | (2 if force2d else 0) | (4 if pair else 0) | (8 if ksplit else 0)
    st = L.fkl_test_gemm(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, Kd, int(a_mn), int(b_mn), bn,
                         flags, ws.data_ptr(), nws, _stream())
    assert st == 0, L.fkl_last_error()
    assert L.fkl_read_status(ws.data_ptr(), _stream()) == 0
    ref = A.double() @ B.double().T + D0.double()
    err = ((D.cpu().double() - ref).abs().max() / ref.abs().max()).item()
    return err


def test_single_tile_k_major(L):
    assert run_gemm(L, 128, 256, 64, False, False, 256) < 1e-5


@pytest.mark.parametrize("bn", [256, 192, 128])
@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, False), (True, True)])
def test_ragged_all_majors(L, a_mn, b_mn, bn):
    assert run_gemm(L, 304, 520, 200, a_mn, b_mn, bn) < 1e-5


@pytest.mark.parametrize("a_mn,b_mn,bn", [(False, False, 256), (True, True, 192), (False, True, 192)])
def test_many_waves(L, a_mn, b_mn, bn):
    # more tiles than SMs: wraps the shared-memory ring and both TMEM accumulators many times
    assert run_gemm(L, 2048, 3072, 1024, a_mn, b_mn, bn, seed=3) < 2e-5


@pytest.mark.parametrize("force2d", [False, True])
@pytest.mark.parametrize("bn", [256, 192, 128])
def test_mn_major_box_paths(L, bn, force2d):
    # extents that are multiples of 64 take one 3-D box per tile (M = 320: the last 128-row
    # tile has one 64-wide block past the end, read as zeros); force2d takes 64-wide boxes
    assert run_gemm(L, 320, 1344, 200, True, True, bn, force2d=force2d) < 1e-5


@pytest.mark.parametrize("a_mn,b_mn", [(False, True), (True, True)])
def test_accumulate(L, a_mn, b_mn):
    assert run_gemm(L, 256, 384, 136, a_mn, b_mn, 192, accumulate=True, seed=5) < 1e-5


def test_long_k(L):
    # the dW product has K = T, thousands of k-blocks per tile
    assert run_gemm(L, 256, 192, 16384, True, True, 192, seed=7) < 5e-5


def test_timeout_probe_reports_status(L):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert L.fkl_test_wait_timeout(2_000_000, ws.data_ptr(), 256, _stream()) == 0
    assert L.fkl_read_status(ws.data_ptr(), _stream()) == 8  # FKL_ERR_TIMEOUT
    # the context is still usable afterwards
    assert run_gemm(L, 128, 256, 64, False, False, 256) < 1e-5


# ---- the two-SM (CTA pair, cta_group::2) kernel that the loss uses: 256-row tiles, each CTA
# ---- of a pair holding 128 rows of A and half of the B tile

def test_pair_single_tile(L):
    assert run_gemm(L, 256, 256, 64, False, False, 256, pair=True) < 1e-5


@pytest.mark.parametrize("bn", [256, 192, 128])
@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, False), (True, True)])
def test_pair_ragged_all_majors(L, a_mn, b_mn, bn):
    # M = 304: the second 256-row tile has 48 rows, so the odd CTA's half is all padding
    assert run_gemm(L, 304, 520, 200, a_mn, b_mn, bn, pair=True) < 1e-5


@pytest.mark.parametrize("bn", [256, 192])
@pytest.mark.parametrize("force2d", [False, True])
def test_pair_mn_major_box_paths(L, force2d, bn):
    # bn = 192: the 96-wide B halves use the 64-byte swizzle (three 32-wide atoms)
    assert run_gemm(L, 320, 1344, 200, True, True, bn, force2d=force2d, pair=True) < 1e-5


@pytest.mark.parametrize("a_mn,b_mn,bn", [(False, False, 256), (True, True, 256), (False, True, 128),
                                           (True, True, 192), (False, True, 192)])
def test_pair_many_waves(L, a_mn, b_mn, bn):
    assert run_gemm(L, 2048, 3072, 1024, a_mn, b_mn, bn, seed=3, pair=True) < 2e-5


def test_pair_accumulate_long_k(L):
    assert run_gemm(L, 512, 384, 8192, True, True, 128, accumulate=True, seed=9, pair=True) < 5e-5


# ---- a ragged last tile of 256-wide two-SM tiles at the d = 2880 shapes (8, 64 or 72 columns)

@pytest.mark.parametrize("N", [2880, 2824, 2888, 320])
@pytest.mark.parametrize("a_mn,b_mn", [(True, True), (False, True), (False, False)])
def test_pair_ragged_last_tile(L, N, a_mn, b_mn):
    # N = 2880 and 320: 64 columns in the last tile; 2824: 8; 2888: 72
    assert run_gemm(L, 512, N, 192, a_mn, b_mn, 256, seed=N, pair=True) < 1e-5


def test_pair_ragged_last_tile_accumulate(L):
    assert run_gemm(L, 264, 2880, 520, True, True, 256, accumulate=True, seed=13, pair=True) < 2e-5


def test_two_copies_of_the_library_in_one_process(L, tmp_path):
    # Each copy keeps its own per-kernel launch state (shared-memory limit, occupancy): the
    # second copy must raise the limit for its own kernels, not inherit the first's flag.
    import shutil

    from lm_head_top_tcgen05_gb300 import _lib

    assert run_gemm(L, 512, 512, 128, False, False, 256, pair=True) < 1e-5  # first copy, state set
    dup = tmp_path / "libfkl_copy.so"
    shutil.copy(_lib.LIB_PATH, dup)
    L2 = ctypes.CDLL(str(dup))
    for name, (res, args) in _lib._SIGNATURES.items():
        fn = getattr(L2, name)
        fn.restype, fn.argtypes = res, args
    assert run_gemm(L2, 512, 512, 128, False, False, 256, pair=True) < 1e-5


@pytest.mark.parametrize("M,N,Kd,a_mn,b_mn,bn,acc", [
    (1792, 768, 1000, False, True, 256, False),  # 21 units on 76 pairs: all split, 3 pieces each
    (2816, 2880, 1024, False, True, 256, True),  # 11 x 12 = 132 units: 56 left over, no split
    (2304, 2880, 2048, True, True, 256, True),   # 9 x 12 = 108: 32 left over, 2 pieces each
    (512, 2880, 1536, False, True, 256, False),  # 2 x 12 = 24: 3 pieces, ragged last column tile
    (304, 520, 4000, True, True, 192, True),     # 2 x 3 = 6 units: 12 pieces of 5-6 k-blocks
    (256, 256, 296, False, False, 256, False),   # 1 unit of 5 k-blocks: too short to split
    (1792, 300, 1000, False, False, 256, True),  # rows of 300 floats: element-wise output, 4 pieces
])
def test_last_wave_split_along_k(L, M, N, Kd, a_mn, b_mn, bn, acc):
    # the units of the last, partial wave are split along K into pieces that store partial
    # tiles, and a fixup kernel adds them in piece order into the output (or onto it)
    assert run_gemm(L, M, N, Kd, a_mn, b_mn, bn, accumulate=acc, seed=11, pair=True, ksplit=True) < 3e-5


def _random_split_case(i):
    # seeded shapes for the two-SM kernel with the last wave split along K: every operand
    # major-ness, tile widths 256 / 192 / 128, ragged tiles, plain and accumulating output
    import numpy as np

    rng = np.random.default_rng(5000 + i)
    a_mn, b_mn = bool(rng.integers(2)), bool(rng.integers(2))
    bn = int(rng.choice([256, 192, 128]))
    M = 8 * int(rng.integers(1, 200))
    N = 8 * int(rng.integers(1, 200))
    Kd = 8 * int(rng.integers(32, 400))
    return M, N, Kd, a_mn, b_mn, bn, bool(rng.integers(2))


@pytest.mark.parametrize("i", range(16))
def test_last_wave_split_random_shapes(L, i):
    M, N, Kd, a_mn, b_mn, bn, acc = _random_split_case(i)
    assert run_gemm(L, M, N, Kd, a_mn, b_mn, bn, accumulate=acc, seed=100 + i, pair=True, ksplit=True) < 5e-5
