"""CUDA path against the float64 oracle, element by element, on seeded inputs.

Tolerances (fixed for the loss): loss relative error <= 1e-3, lse absolute error <= 1e-3 on
every row, dH and dW relative Frobenius error <= 2e-2 and max-abs error <= 5e-2 * max|ref|.
Shapes span several tiles on every axis and leave ragged tails (T not a multiple of 128,
V not a multiple of 256, d not a multiple of 64), plus the degenerate cases."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

LOSS_RTOL, LSE_ATOL, FRO_RTOL, MAX_FRAC = 1e-3, 1e-3, 2e-2, 5e-2


@pytest.fixture(scope="module")
def fkl(cuda_device):
    from lm_head_top_tcgen05_gb300 import build

    build.build()
    import lm_head_top_tcgen05_gb300 as m

    return m


def to_dev(x, dev="cuda"):
    return (x.H.to(dev), x.W.to(dev), x.topk_idx.to(dev), x.topk_logits.to(dev), x.mask.to(dev))


def run_gpu(fkl, x, chunk=None, grad=None):
    H, W, idx, z, m = to_dev(x)
    chunk = x.chunk if chunk is None else chunk
    loss, lse = fkl.forward(H, W, idx, z, m, x.tau, chunk)
    g = None if grad is None else torch.tensor(grad, dtype=torch.float32, device="cuda")
    dH, dW = fkl.backward(H, W, idx, z, m, lse, g, x.tau, chunk)
    torch.cuda.synchronize()
    status = fkl.read_status(device="cuda")
    return dict(loss=loss.item(), lse=lse.cpu().numpy().astype(np.float64), dH=dH.cpu().numpy().astype(np.float64),
                dW=dW.cpu().numpy().astype(np.float64), status=status)


def run_oracle(x, grad=1.0):
    H64, W64 = oracle.to_f64(x.H), oracle.to_f64(x.W)
    f = oracle.forward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau)
    dH, dW = oracle.backward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau, grad=grad)
    return dict(loss=f["loss"], lse=f["lse"], dH=dH, dW=dW)


def assert_grad_close(G, R, name):
    nr = np.linalg.norm(R)
    if nr == 0:
        assert np.max(np.abs(G)) == 0, name
        return
    fro = np.linalg.norm(G - R) / nr
    mx = np.max(np.abs(G - R)) / np.max(np.abs(R))
    assert fro <= FRO_RTOL, f"{name}: relative Frobenius error {fro:.3e}"
    assert mx <= MAX_FRAC, f"{name}: max-abs error {mx:.3e} of max|ref|"


def assert_parity(gpu, ref):
    assert gpu["status"] == 0
    if ref["loss"] == 0:
        assert gpu["loss"] == 0
    else:
        rel = abs(gpu["loss"] - ref["loss"]) / abs(ref["loss"])
        assert rel <= LOSS_RTOL, f"loss {gpu['loss']} vs {ref['loss']} (rel {rel:.3e})"
    if len(ref["lse"]):
        err = np.max(np.abs(gpu["lse"] - ref["lse"]))
        assert err <= LSE_ATOL, f"lse max abs error {err:.3e}"
    assert_grad_close(gpu["dH"], ref["dH"], "dH")
    assert_grad_close(gpu["dW"], ref["dW"], "dW")


CASES = {
    # name: (T, d, V, K, tau, chunk, mask_frac, seed)
    "one_tile": (128, 64, 256, 4, 1.0, 128, 0.0, 1),
    "ragged_all_axes": (300, 200, 5000, 16, 2.0, 128, 0.1, 2),
    "small_vocab_many_slots": (130, 320, 1000, 50, 0.7, 4096, 0.0, 3),
    "single_slot": (257, 136, 300, 1, 1.0, 64, 0.05, 4),
    "one_token": (1, 64, 777, 8, 1.0, 1, 0.0, 5),
    "wide_d": (200, 1152, 3000, 32, 1.3, 512, 0.0, 6),
    # the ABI's limits and extremes
    "max_k": (136, 64, 3000, 1024, 1.0, 256, 0.0, 7),
    "min_d": (300, 8, 2000, 16, 1.0, 128, 0.1, 8),
    "d4096": (264, 4096, 2600, 24, 2.0, 512, 0.0, 9),
    "d8200": (130, 8200, 700, 8, 1.0, 256, 0.0, 14),  # 33 d-tiles, the last 8 columns wide
    "cold_tau": (200, 128, 3000, 16, 0.05, 256, 0.0, 10),
    "hot_tau": (200, 128, 3000, 16, 20.0, 256, 0.0, 11),
    "vocab_below_one_tile": (300, 96, 100, 20, 1.0, 64, 0.0, 12),
    # long sequence against a small vocabulary: the backward walks 4 token blocks x 3 slabs
    # (dW accumulates over the token blocks), the last block and slab ragged
    "token_blocks": (4000, 64, 2999, 16, 1.0, 512, 0.1, 13),
}


@pytest.mark.parametrize("name", list(CASES))
def test_parity_small(fkl, name):
    T, d, V, K, tau, chunk, mf, seed = CASES[name]
    x = workloads.make_random(T, d, V, K, tau=tau, chunk=chunk, seed=seed, mask_frac=mf)
    assert_parity(run_gpu(fkl, x), run_oracle(x))


def test_parity_tiny_workload(fkl):
    x = workloads.make_inputs("tiny")
    assert_parity(run_gpu(fkl, x), run_oracle(x))


def test_upstream_gradient_scales(fkl):
    x = workloads.make_random(160, 128, 2000, 10, seed=8)
    assert_parity(run_gpu(fkl, x, grad=-0.37), run_oracle(x, grad=-0.37))


def test_zero_upstream_gradient(fkl):
    # g = 0: every row's factor g tau w_t is 0, so dS and both gradients are exactly zero
    x = workloads.make_random(300, 128, 3000, 12, seed=9, mask_frac=0.1)
    out = run_gpu(fkl, x, grad=0.0)
    assert out["status"] == 0
    assert not np.any(out["dH"]) and not np.any(out["dW"])


def test_deterministic(fkl):
    x = workloads.make_random(300, 200, 5000, 16, tau=2.0, chunk=128, seed=2, mask_frac=0.1)
    a, b = run_gpu(fkl, x), run_gpu(fkl, x)
    assert a["loss"] == b["loss"]
    for k in ("lse", "dH", "dW"):
        assert np.array_equal(a[k], b[k]), k


def test_chunk_invariance(fkl):
    x = workloads.make_random(300, 200, 5000, 16, tau=1.0, seed=9)
    ref = run_oracle(x)
    outs = [run_gpu(fkl, x, chunk=c) for c in (1, 64, 300, 100000)]
    for o in outs:
        assert_parity(o, ref)
    for o in outs[1:]:
        assert o["loss"] == outs[0]["loss"]  # the forward does not depend on chunk at all
        assert_grad_close(o["dW"], outs[0]["dW"], "dW across chunks")


def test_masked_rows_have_zero_gradient(fkl):
    x = workloads.make_random(256, 128, 3000, 12, seed=10, mask_frac=0.3)
    g = run_gpu(fkl, x)
    masked = x.mask.numpy() == 0
    assert masked.sum() > 0
    assert np.all(g["dH"][masked] == 0)
    assert np.all(np.isfinite(g["lse"]))


def test_no_valid_token(fkl):
    x = workloads.make_random(100, 64, 1000, 8, seed=11)
    x.mask[:] = 0
    g = run_gpu(fkl, x)
    assert g["loss"] == 0 and g["status"] == 0
    assert not g["dH"].any() and not g["dW"].any()


def test_empty_batch(fkl):
    x = workloads.make_random(0, 64, 1000, 8, seed=12)
    g = run_gpu(fkl, x)
    assert g["loss"] == 0 and g["lse"].shape == (0,) and not g["dW"].any()


def test_duplicate_ids_follow_per_slot_definition(fkl):
    x = workloads.make_random(64, 64, 512, 6, seed=13)
    x.topk_idx[5, 1] = x.topk_idx[5, 0]
    x.topk_idx[9, 2:] = x.topk_idx[9, 1]
    assert_parity(run_gpu(fkl, x), run_oracle(x))


def test_minus_inf_teacher_slots(fkl):
    x = workloads.make_random(64, 64, 512, 6, seed=14)
    x.topk_logits[:, -2:] = -float("inf")
    assert_parity(run_gpu(fkl, x), run_oracle(x))


def test_bad_teacher_id_is_reported(fkl):
    x = workloads.make_random(64, 64, 512, 6, seed=15)
    x.topk_idx[3, 2] = 512
    g = run_gpu(fkl, x)
    assert g["status"] == 6 and np.isnan(g["loss"]) and np.isnan(g["dH"]).all()


def test_teacher_row_without_finite_logit_is_reported(fkl):
    x = workloads.make_random(64, 64, 512, 6, seed=16)
    x.topk_logits[7, :] = -float("inf")
    g = run_gpu(fkl, x)
    assert g["status"] == 7 and np.isnan(g["loss"])


def test_status_clears_on_next_good_call(fkl):
    x = workloads.make_random(64, 64, 512, 6, seed=17)
    assert run_gpu(fkl, x)["status"] == 0


def test_autograd_wrapper(fkl):
    x = workloads.make_random(200, 128, 2500, 10, tau=1.5, seed=18, mask_frac=0.1)
    H, W, idx, z, m = to_dev(x)
    H.requires_grad_(True)
    W.requires_grad_(True)
    loss = fkl.fused_kl(H, W, idx, z, m, tau=x.tau, chunk=64)
    (2.0 * loss).backward()
    ref = run_oracle(x, grad=2.0)
    assert abs(loss.item() - ref["loss"]) / ref["loss"] <= LOSS_RTOL
    assert H.grad.dtype == torch.bfloat16 and W.grad.dtype == torch.bfloat16
    assert_grad_close(H.grad.double().cpu().numpy(), ref["dH"], "H.grad")
    assert_grad_close(W.grad.double().cpu().numpy(), ref["dW"], "W.grad")


# ---------------------------------------------------------------- variants: packed sequences, accumulation

def run_oracle_seq(x, seq, grad=1.0):
    H64, W64 = oracle.to_f64(x.H), oracle.to_f64(x.W)
    f = oracle.forward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau, norm="sequences", seq_ids=seq)
    dH, dW = oracle.backward(H64, W64, x.topk_idx, x.topk_logits, x.mask, x.tau, grad=grad,
                             norm="sequences", seq_ids=seq)
    return dict(loss=f["loss"], lse=f["lse"], dH=dH, dW=dW)


def packed_case(seed=40):
    x = workloads.make_random(300, 200, 5000, 16, tau=2.0, chunk=128, seed=seed, mask_frac=0.1)
    lengths = [40, 130, 7, 90, 33]  # the third sequence is entirely masked below
    seq = np.concatenate([np.full(n, i) for i, n in enumerate(lengths)]).astype(np.int32)
    x.mask[170:177] = 0
    return x, seq


def test_sequence_mean_parity(fkl):
    x, seq = packed_case()
    H, W, idx, z, m = to_dev(x)
    sid = torch.from_numpy(seq).cuda()
    loss, lse = fkl.forward(H, W, idx, z, m, x.tau, x.chunk, seq_ids=sid, num_seqs=5)
    dH, dW = fkl.backward(H, W, idx, z, m, lse, None, x.tau, x.chunk, seq_ids=sid, num_seqs=5)
    torch.cuda.synchronize()
    gpu = dict(loss=loss.item(), lse=lse.cpu().numpy().astype(np.float64), dH=dH.cpu().numpy().astype(np.float64),
               dW=dW.cpu().numpy().astype(np.float64), status=fkl.read_status(device="cuda"))
    ref = run_oracle_seq(x, seq)
    tok = run_oracle(x)
    assert abs(ref["loss"] - tok["loss"]) > 1e-3 * abs(tok["loss"])  # the two normalisers differ here
    assert_parity(gpu, ref)


def test_sequence_mean_autograd(fkl):
    x, seq = packed_case(41)
    H, W, idx, z, m = to_dev(x)
    H.requires_grad_(True)
    W.requires_grad_(True)
    loss = fkl.fused_kl(H, W, idx, z, m, tau=x.tau, chunk=64, seq_ids=torch.from_numpy(seq).cuda(), num_seqs=5)
    loss.backward()
    ref = run_oracle_seq(x, seq)
    assert abs(loss.item() - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"])
    assert_grad_close(H.grad.double().cpu().numpy(), ref["dH"], "H.grad")


def test_bad_sequence_id_is_reported(fkl):
    x, seq = packed_case(42)
    seq[5] = 7  # outside [0, 5) on a valid token
    H, W, idx, z, m = to_dev(x)
    loss, _ = fkl.forward(H, W, idx, z, m, x.tau, x.chunk, seq_ids=torch.from_numpy(seq).cuda(), num_seqs=5)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 9 and np.isnan(loss.item())


def test_gradient_accumulation(fkl):
    x = workloads.make_random(300, 200, 5000, 16, tau=1.5, chunk=128, seed=43, mask_frac=0.1)
    H, W, idx, z, m = to_dev(x)
    loss, lse = fkl.forward(H, W, idx, z, m, x.tau, x.chunk)
    g = torch.Generator(device="cuda").manual_seed(0)
    dH0 = torch.randn(H.shape, device="cuda", generator=g)
    dW0 = torch.randn(W.shape, device="cuda", generator=g)
    dH, dW = dH0.clone(), dW0.clone()
    fkl.backward(H, W, idx, z, m, lse, None, x.tau, x.chunk, out=(dH, dW), accumulate=True)
    fkl.backward(H, W, idx, z, m, lse, None, x.tau, x.chunk, out=(dH, dW), accumulate=True)
    torch.cuda.synchronize()
    ref = run_oracle(x, grad=2.0)  # two micro-batches of the same gradient
    assert_grad_close((dH - dH0).double().cpu().numpy(), ref["dH"], "accumulated dH")
    assert_grad_close((dW - dW0).double().cpu().numpy(), ref["dW"], "accumulated dW")


def test_token_blocks_with_variants(fkl):
    # the blocked backward with the sequence mean and with accumulation into given gradients
    x = workloads.make_random(4000, 64, 2999, 16, tau=1.5, chunk=512, seed=44, mask_frac=0.1)
    seq = np.repeat(np.arange(5), 800).astype(np.int32)
    H, W, idx, z, m = to_dev(x)
    sid = torch.from_numpy(seq).cuda()
    loss, lse = fkl.forward(H, W, idx, z, m, x.tau, x.chunk, seq_ids=sid, num_seqs=5)
    g = torch.Generator(device="cuda").manual_seed(1)
    dH0 = torch.randn(H.shape, device="cuda", generator=g)
    dW0 = torch.randn(W.shape, device="cuda", generator=g)
    dH, dW = dH0.clone(), dW0.clone()
    fkl.backward(H, W, idx, z, m, lse, None, x.tau, x.chunk, out=(dH, dW), accumulate=True, seq_ids=sid, num_seqs=5)
    torch.cuda.synchronize()
    ref = run_oracle_seq(x, seq)
    assert abs(loss.item() - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"])
    assert_grad_close((dH - dH0).double().cpu().numpy(), ref["dH"], "accumulated dH")
    assert_grad_close((dW - dW0).double().cpu().numpy(), ref["dW"], "accumulated dW")


@pytest.mark.parametrize("accumulate", [False, True])
def test_gradients_16_but_not_32_byte_aligned(fkl, accumulate):
    # dH and dW 16 bytes past a 32-byte boundary: the products' epilogues and the K-split
    # fixup write them element by element instead of in 32-byte vectors
    x = workloads.make_random(700, 136, 3000, 16, tau=1.2, chunk=256, seed=61, mask_frac=0.1)
    H, W, idx, z, m = to_dev(x)
    loss, lse = fkl.forward(H, W, idx, z, m, x.tau, x.chunk)
    g = torch.Generator(device="cuda").manual_seed(3)
    bh = torch.zeros(H.numel() + 4, device="cuda")
    bw = torch.zeros(W.numel() + 4, device="cuda")
    dH, dW = bh[4:].view(H.shape), bw[4:].view(W.shape)
    assert dH.data_ptr() % 32 == 16 and dW.data_ptr() % 32 == 16
    dH0 = torch.randn(H.shape, device="cuda", generator=g) if accumulate else torch.zeros(H.shape, device="cuda")
    dW0 = torch.randn(W.shape, device="cuda", generator=g) if accumulate else torch.zeros(W.shape, device="cuda")
    dH.copy_(dH0)
    dW.copy_(dW0)
    fkl.backward(H, W, idx, z, m, lse, None, x.tau, x.chunk, out=(dH, dW), accumulate=accumulate)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 0
    ref = run_oracle(x)
    assert_grad_close(dH.cpu().numpy().astype(np.float64) - dH0.cpu().numpy(), ref["dH"], "dH")
    assert_grad_close(dW.cpu().numpy().astype(np.float64) - dW0.cpu().numpy(), ref["dW"], "dW")
    assert bh[:4].abs().max().item() == 0 and bw[:4].abs().max().item() == 0


# ---------------------------------------------------------------- bf16 gradient outputs

def _bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("T,d,V,K,chunk,div", [
    (300, 136, 3000, 16, 256, "kl"),      # K-split dW and dH, one token block, ragged everywhere
    (4000, 64, 2999, 16, 512, "kl"),      # several token blocks: dW summed over blocks in fp32
    (700, 200, 5000, 16, 100000, "kl"),   # one vocabulary slab: dH written once
    (513, 96, 4100, 12, 64, "jsd"),       # another divergence
    (2000, 64, 3000, 16, 256, "kl"),      # 3 token blocks x 4 slabs walked slabs outer (less fp32 scratch)
    (3000, 96, 5000, 12, 256, "jsd"),     # slabs outer, another divergence
])
def test_bf16_gradients_are_the_rounded_fp32_ones(fkl, T, d, V, K, chunk, div):
    # fkl_backward_bf16 keeps fp32 sums and rounds once: bit for bit the fp32 result rounded
    x = workloads.make_random(T, d, V, K, tau=1.3, chunk=chunk, seed=70 + T % 97, mask_frac=0.1)
    H, W, idx, z, m = to_dev(x)
    s = None if div == "kl" else torch.empty((T, K), dtype=torch.float32, device="cuda")
    loss, lse = fkl.forward(H, W, idx, z, m, x.tau, chunk, divergence=div, student_topk_logits=s)
    g = torch.tensor(0.75, device="cuda")
    dH, dW = fkl.backward(H, W, idx, z, m, lse, g, x.tau, chunk, divergence=div, student_topk_logits=s)
    dH16, dW16 = fkl.backward(H, W, idx, z, m, lse, g, x.tau, chunk, divergence=div, student_topk_logits=s,
                              grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 0
    assert dH16.dtype == torch.bfloat16 and dW16.dtype == torch.bfloat16
    assert (_bf16_bits(dH16) == _bf16_bits(dH.to(torch.bfloat16))).all()
    assert (_bf16_bits(dW16) == _bf16_bits(dW.to(torch.bfloat16))).all()


def test_bf16_gradients_edge_cases(fkl):
    x = workloads.make_random(64, 64, 512, 6, seed=19)
    H, W, idx, z, m = to_dev(x)
    loss, lse = fkl.forward(H, W, idx, z, m, x.tau, x.chunk)
    # accumulation is fp32 only
    with pytest.raises(ValueError):
        fkl.backward(H, W, idx, z, m, lse, None, x.tau, x.chunk, grad_dtype=torch.bfloat16, accumulate=True,
                     out=(torch.zeros(H.shape, dtype=torch.bfloat16, device="cuda"),
                          torch.zeros(W.shape, dtype=torch.bfloat16, device="cuda")))
    # T = 0: dW is zero
    dH, dW = fkl.backward(H[:0], W, idx[:0], z[:0], m[:0], lse[:0], None, x.tau, x.chunk,
                          grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert dW.dtype == torch.bfloat16 and dW.abs().max().item() == 0 and dH.numel() == 0
    # a device-side error poisons the bf16 gradients with NaN
    bad = idx.clone()
    bad[3, 2] = 512
    dH, dW = fkl.backward(H, W, bad, z, m, lse, None, x.tau, x.chunk, grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 6
    assert torch.isnan(dH.float()).all() and torch.isnan(dW.float()).all()
    assert fkl.read_status(device="cuda") == 6
    fkl.forward(H, W, idx, z, m, x.tau, x.chunk)
    torch.cuda.synchronize()
    assert fkl.read_status(device="cuda") == 0


def test_vocabulary_of_one(fkl):
    # V = 1: student and teacher both put all mass on the one entry, so the loss and the
    # gradients are zero; the kernels get there through lse = s and q = exp(s - lse) = 1 in
    # fp32, so zero up to rounding
    x = workloads.make_random(70, 64, 1, 1, tau=1.0, chunk=64, seed=15)
    g = run_gpu(fkl, x)
    ref = run_oracle(x)
    assert g["status"] == 0 and ref["loss"] == 0
    assert abs(g["loss"]) <= 1e-5
    assert np.max(np.abs(g["lse"] - ref["lse"])) <= LSE_ATOL
    assert np.max(np.abs(g["dH"])) <= 1e-5 and np.max(np.abs(g["dW"])) <= 1e-5
