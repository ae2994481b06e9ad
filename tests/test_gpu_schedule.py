"""Dynamic scheduling of the long GEMM launches (forward, teacher-cache passes).

Each pair of a dynamically scheduled launch starts on a fixed unit and then draws units from
a counter in the workspace header (the int32 at byte 16), so that the launches of one call
can share the counter with running bases: that only works if a launch takes exactly as many
values from the counter as it has units (one per drawn unit and one closing value per
pair).  These tests read the counter after a call and check that accounting, for grids
larger and smaller than the number of units, and that drawing units leaves the results
bitwise deterministic."""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fkl(cuda_device):
    from lm_head_top_tcgen05_gb300 import build

    build.build()
    import lm_head_top_tcgen05_gb300 as m

    return m


def counter(ws):
    return int(ws.buf[16:20].view(torch.int32).item())


def drawn_splits(m_tiles, n_tiles, pairs):
    """Splits of a drawn launch: units of at least 4 tiles unless that leaves fewer than two
    units per pair, at most one per tile and at most 64."""
    s = max(-(-n_tiles // 4), -(-2 * pairs // m_tiles))
    return min(s, n_tiles, 64)


def pairs():
    return torch.cuda.get_device_properties(0).multi_processor_count // 2


@pytest.mark.parametrize("T,V", [(1000, 20000), (4096, 50000), (10, 300), (256, 256)])
def test_forward_takes_one_value_per_unit(fkl, T, V):
    x = workloads.make_random(T, 128, V, 8, seed=T + V)
    ws = fkl.Workspace("cuda")
    loss, lse = fkl.forward(x.H.cuda(), x.W.cuda(), x.topk_idx.cuda(), x.topk_logits.cuda(), None, 1.0, 64,
                            workspace=ws)
    torch.cuda.synchronize()
    assert fkl.read_status(ws) == 0
    m_tiles, n_tiles = (T + 255) // 256, (V + 255) // 256
    assert counter(ws) == m_tiles * drawn_splits(m_tiles, n_tiles, pairs())  # row blocks x splits


def test_teacher_passes_share_the_counter(fkl):
    # the bound pass over every 8th vocabulary row (3750 rows: 15 tiles, one split each),
    # then the candidate pass over all 30000 (118 tiles): the counter ends at the
    # sum of both launches' units
    T, V = 600, 30000
    g = torch.Generator().manual_seed(12)
    Ht = torch.randn(T, 192, generator=g).to(torch.bfloat16).cuda()
    Wt = (torch.randn(V, 192, generator=g) * 0.02).to(torch.bfloat16).cuda()
    ws = fkl.Workspace("cuda")
    fkl.teacher_topk(Ht, Wt, 100, workspace=ws)
    torch.cuda.synchronize()
    assert fkl.read_status(ws) == 0
    m_tiles = (T + 255) // 256
    vs = (V + 7) // 8                      # rows the bound pass samples at stride 8
    bound_units = m_tiles * min(32, (vs + 255) // 256)
    cand_units = m_tiles * drawn_splits(m_tiles, (V + 255) // 256, pairs())
    assert counter(ws) == bound_units + cand_units


def test_drawn_units_are_deterministic(fkl):
    x = workloads.make_random(5000, 256, 60000, 16, seed=13, mask_frac=0.1)
    args = (x.H.cuda(), x.W.cuda(), x.topk_idx.cuda(), x.topk_logits.cuda(), x.mask.cuda(), 1.0, 256)
    outs = [fkl.forward(*args) for _ in range(3)]
    torch.cuda.synchronize()
    for loss, lse in outs[1:]:
        assert loss.item() == outs[0][0].item()
        assert torch.equal(lse, outs[0][1])
    assert np.isfinite(outs[0][0].item())
