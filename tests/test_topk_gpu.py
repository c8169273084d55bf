"""Parity of dsa_topk with the oracle's full-sort selection on the same fp32
logits (exact: the selected sets must be identical, ties to the lower
column)."""
import numpy as np
import pytest
import torch

import oracle
from dsa_check import gpu_topk, np_

pytestmark = pytest.mark.gpu


def sets_equal(sel, logits, L, k):
    ref = oracle.topk(np_(logits).astype(np.float64), np_(L), k)
    s = np_(sel)
    for i in range(s.shape[0]):
        assert sorted(s[i].tolist()) == sorted(ref[i].tolist()), f"row {i}"


@pytest.mark.parametrize("force", [0, 1, 2])
def test_topk_random_rows(force):
    g = torch.Generator(device="cuda").manual_seed(1)
    L = torch.tensor([0, 1, 2047, 2048, 2049, 4099, 8192, 33333, 65536, 70001, 131072],
                     dtype=torch.int32, device="cuda")
    ld = 131072
    logits = torch.randn(len(L), ld, generator=g, device="cuda")
    sel = gpu_topk(logits, ld, L, 2048, force_path=force)
    sets_equal(sel, logits, L, 2048)


@pytest.mark.parametrize("force", [1, 2])
def test_topk_heavy_ties(force):
    g = torch.Generator(device="cuda").manual_seed(2)
    L = torch.tensor([5000, 70000, 100000], dtype=torch.int32, device="cuda")
    ld = 100000
    logits = torch.randint(-6, 6, (3, ld), generator=g, device="cuda").float()
    logits[0, ::3] = -0.0
    logits[0, 1::3] = 0.0
    sel = gpu_topk(logits, ld, L, 1000, force_path=force)
    sets_equal(sel, logits, L, 1000)


def test_topk_all_equal_takes_exact_fallback():
    from deepseek_sparse_attention_02_gb300 import dsa
    dsa.dsa_get_device_error(clear=True)
    L = torch.tensor([90000], dtype=torch.int32, device="cuda")
    logits = torch.full((1, 90000), 0.25, device="cuda")
    sel = gpu_topk(logits, 90000, L, 2048, force_path=2)
    assert sorted(np_(sel)[0].tolist()) == list(range(2048))
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error(clear=True) == dsa.DEVERR_CAPACITY


def _sample_positions(L):
    """The columns the long-row path samples for its cutoff: 256 runs of 8
    consecutive scores, run i starting at (i (L - 8) / 255) rounded down to a
    multiple of 4 (16-byte loads)."""
    pos = []
    for i in range(256):
        g0 = ((i * (L - 8)) // 255) & ~3
        pos.extend(range(g0, g0 + 8))
    return pos


@pytest.mark.parametrize("Lr", [131072, 65536])
def test_topk_sample_overestimate_takes_exact_redo(Lr):
    """A row whose sampled columns hold its 2048 largest scores, spread over
    ten octaves (80 bins of the 12-bit key prefix the cutoff is read from):
    the cutoff estimated from the sample keeps only about 2k * 2048 / L of
    them, fewer than k, so the row is redone by the exact full-row select; the
    result is still exact and the device error word reports the missed
    estimate.  131072 columns run on a CTA pair, 65536 on one CTA."""
    from deepseek_sparse_attention_02_gb300 import dsa
    dsa.dsa_get_device_error(clear=True)
    g = torch.Generator(device="cuda").manual_seed(7)
    logits = torch.randn(1, Lr, generator=g, device="cuda")  # all below 8
    pos = _sample_positions(Lr)
    assert len(set(pos)) == 2048
    big = torch.exp2(3.0 + 10.0 * torch.rand(2048, generator=g, device="cuda"))  # [8, 8192)
    logits[0, torch.tensor(pos, device="cuda")] = big
    L = torch.tensor([Lr], dtype=torch.int32, device="cuda")
    sel = gpu_topk(logits, Lr, L, 2048)
    sets_equal(sel, logits, L, 2048)
    assert sorted(np_(sel)[0].tolist()) == sorted(pos)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error(clear=True) == dsa.DEVERR_CAPACITY


def test_topk_small_k_and_odd_sizes():
    g = torch.Generator(device="cuda").manual_seed(3)
    L = torch.tensor([3, 10, 17, 1000], dtype=torch.int32, device="cuda")
    logits = torch.randn(4, 1000, generator=g, device="cuda")
    for k in (1, 7, 16):
        sel = gpu_topk(logits, 1000, L, k)
        sets_equal(sel, logits, L, k)


def test_topk_column_map():
    g = torch.Generator(device="cuda").manual_seed(4)
    R, nb, bs = 3, 40, 64
    cols = nb * bs
    logits = torch.randn(R, cols, generator=g, device="cuda")
    L = torch.tensor([cols, cols - 17, 100], dtype=torch.int32, device="cuda")
    blocks = torch.stack([torch.randperm(500, generator=torch.Generator().manual_seed(r))[:nb]
                          for r in range(R)]).to(torch.int32).cuda()
    sel = gpu_topk(logits, cols, L, 256, col_blocks=blocks, bs=bs)
    ref = oracle.topk(np_(logits).astype(np.float64), np_(L), 256, col_blocks=np_(blocks), bs=bs)
    for i in range(R):
        assert sorted(np_(sel)[i].tolist()) == sorted(ref[i].tolist())


def test_topk_cutoff_at_or_below_zero():
    """Rows whose k-th largest score is negative or a (signed) zero, so the
    sampled cutoff of the long-row path is at or below +0.0; with positive
    cutoffs the compaction compares raw float bits instead of ordered keys."""
    g = torch.Generator(device="cuda").manual_seed(5)
    ld = 131072
    L = torch.tensor([131072, 131072, 100003], dtype=torch.int32, device="cuda")
    logits = -torch.randn(3, ld, generator=g, device="cuda").abs()
    # row 1: 1000 positive scores, then 3000 zeros of both signs around the k-th
    logits[1, :1000] = torch.rand(1000, generator=g, device="cuda") + 0.5
    logits[1, 5000:6500] = 0.0
    logits[1, 6500:8000] = -0.0
    # row 2: negative scores only, with many exact ties
    logits[2] = -torch.randint(1, 50, (ld,), generator=g, device="cuda").float()
    for force in (0, 2):
        sel = gpu_topk(logits, ld, L, 2048, force_path=force)
        sets_equal(sel, logits, L, 2048)


def test_topk_many_rows_one_cta_per_row():
    """More rows than half the SM count: one CTA per row (the pair split of
    the streaming pass is used only for fewer rows), mixed lengths so both the
    staged and the cutoff path run."""
    g = torch.Generator(device="cuda").manual_seed(6)
    R, ld = 100, 70004
    L = torch.randint(1, ld + 1, (R,), generator=g, device="cuda").to(torch.int32)
    L[:4] = torch.tensor([ld, 2048, 16384, 40961], dtype=torch.int32, device="cuda")
    logits = torch.randn(R, ld, generator=g, device="cuda")
    sel = gpu_topk(logits, ld, L, 2048)
    sets_equal(sel, logits, L, 2048)


@pytest.mark.parametrize("force", [0, 1, 2])
def test_topk_bf16_rows(force):
    """bf16 scores (many exact ties after rounding): the set equals the
    oracle's full sort of the same values, ties to the lower column; long rows
    take the two-CTA kernel, short ones the one-CTA kernel."""
    from deepseek_sparse_attention_02_gb300 import dsa
    g = torch.Generator(device="cuda").manual_seed(7)
    L = torch.tensor([0, 5, 2048, 2049, 9000, 40961, 70001, 131072], dtype=torch.int32,
                     device="cuda")
    ld = 131072
    logits = torch.randn(len(L), ld, generator=g, device="cuda").to(torch.bfloat16)
    logits[3, 100:2000] = 0.0
    logits[3, 2000:2049:2] = -0.0
    out = torch.full((len(L), 2048), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_topk_bf16(logits, ld, L, len(L), 2048, out, force_path=force)
    torch.cuda.synchronize()
    ref = oracle.topk(np_(logits.float()).astype(np.float64), np_(L), 2048)
    for i in range(len(L)):
        assert sorted(np_(out)[i].tolist()) == sorted(ref[i].tolist()), f"row {i}"


def test_topk_bf16_matches_f32_of_same_values():
    """A bf16 row and the f32 row of the same (widened) values select the same set."""
    from deepseek_sparse_attention_02_gb300 import dsa
    g = torch.Generator(device="cuda").manual_seed(8)
    R, ld, k = 64, 32768, 2048
    L = torch.full((R,), ld, dtype=torch.int32, device="cuda")
    b = (torch.randn(R, ld, generator=g, device="cuda") * 3).to(torch.bfloat16)
    o16 = torch.empty((R, k), dtype=torch.int32, device="cuda")
    o32 = torch.empty((R, k), dtype=torch.int32, device="cuda")
    dsa.dsa_topk_bf16(b, ld, L, R, k, o16)
    dsa.dsa_topk(b.float().contiguous(), ld, L, R, k, o32)
    torch.cuda.synchronize()
    assert torch.equal(torch.sort(o16, dim=1).values, torch.sort(o32, dim=1).values)
