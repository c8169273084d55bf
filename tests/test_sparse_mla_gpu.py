"""Parity of dsa_sparse_mla_decode (Eq. (2)) with the fp64 oracle."""
import numpy as np
import pytest
import torch

from dsa_check import LSE_ATOL, MLA_ATOL, gpu_mla, mla_oracle, np_
from deepseek_sparse_attention_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_case(ctx, next_n, k, seed, holes=0.0):
    layout = W.make_layout(ctx, seed, device="cuda")
    R = len(ctx) * next_n
    mla = W.make_mla_case(R, layout.num_pages, seed=seed, device="cuda")
    L = W.row_lengths(layout.ctx_len, next_n).tolist()
    idx = W.random_indices(L, k, seed=seed, device="cuda")
    if holes:
        g = torch.Generator(device="cuda").manual_seed(seed)
        idx[torch.rand(idx.shape, generator=g, device="cuda") < holes] = -1
    out, lse = gpu_mla(mla, layout.block_table, len(ctx), next_n, idx, layout.num_pages)
    torch.cuda.synchronize()
    return mla, layout, idx, out, lse


def compare(mla, layout, next_n, idx, out, lse, rows=None, rel=0.0):
    """rel adds rel * |ref| to the absolute bound, element by element: the
    output is stored in bf16, whose rounding to nearest is up to half an ulp,
    2^-8 * |ref| at worst (bf16 keeps 8 significant bits)."""
    o_ref, l_ref = mla_oracle(mla, layout.block_table, next_n, idx, rows=rows)
    got = np_(out.float())
    gl = np_(lse)
    if rows is not None:
        got, gl = got[rows], gl[rows]
    excess = np.abs(got - o_ref) - (MLA_ATOL + rel * np.abs(o_ref))
    err = np.abs(got - o_ref).max()
    assert excess.max() <= 0, f"max |out - ref| = {err}, worst excess {excess.max()}"
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(gl), fin)
    if fin.any():
        assert np.abs(gl[fin] - l_ref[fin]).max() <= LSE_ATOL
    return err


@pytest.mark.parametrize("ctx,next_n,k,holes", [
    ([3000, 5000, 2500], 1, 2048, 0.0),     # full tiles
    ([700, 3000], 2, 2048, 0.1),            # rows shorter than k (-1 tails) + holes
    ([4000], 1, 100, 0.0),                  # ragged last tile, split-K path
    ([9000, 9000, 9000, 9000], 1, 2048, 0.02),
    # 40 rows and more: one split per row (no combine), the pair's full
    # message / rescale protocol over 16 tiles
    ([3000] * 40, 1, 2048, 0.0),
    ([700, 3000] * 20, 2, 2048, 0.1),       # -1 tails + holes, 80 rows
    ([2500] * 48, 1, 300, 0.05),            # ragged last tile, 3 tiles
])
def test_mla_parity(ctx, next_n, k, holes):
    mla, layout, idx, out, lse = run_case(ctx, next_n, k, seed=5, holes=holes)
    from deepseek_sparse_attention_02_gb300 import dsa
    assert dsa.dsa_get_device_error() == 0
    compare(mla, layout, next_n, idx, out, lse)


def test_mla_no_valid_index_row():
    layout = W.make_layout([500], 1, device="cuda")
    mla = W.make_mla_case(1, layout.num_pages, seed=1, device="cuda")
    idx = torch.full((1, 256), -1, dtype=torch.int32, device="cuda")
    out, lse = gpu_mla(mla, layout.block_table, 1, 1, idx, layout.num_pages)
    assert torch.all(out.float() == 0) and torch.all(torch.isneginf(lse))


def test_mla_index_order_does_not_matter_and_is_not_a_prefix():
    mla, layout, idx, out, lse = run_case([6000], 1, 512, seed=7)
    perm = idx[:, torch.randperm(512, generator=torch.Generator().manual_seed(0)).cuda()]
    out2, _ = gpu_mla(mla, layout.block_table, 1, 1, perm.contiguous(), layout.num_pages)
    assert (out.float() - out2.float()).abs().max() <= MLA_ATOL
    prefix = torch.arange(512, dtype=torch.int32, device="cuda")[None]
    out3, _ = gpu_mla(mla, layout.block_table, 1, 1, prefix, layout.num_pages)
    assert (out.float() - out3.float()).abs().max() > 0.05


@pytest.mark.parametrize("nreq", [2, 40])
def test_mla_scores_growing_within_and_across_tiles(nreq):
    """Scores that rise inside a 128-token tile (second half) and from tile to
    tile, so the running softmax reference moves mid-tile (P already written
    for the tile's first half is brought to the new reference) and between
    tiles (O and l are rescaled).  Only the 64 rotary dimensions of the keys
    are scaled: they enter the scores but not the values, so the outputs keep
    their unit scale; but each output is then close to a single value row
    (up to ~4.5), so the bound adds one bf16 ulp of the reference (2^-8 |ref|)
    for the rounding of the stored output."""
    ctx, k = ([6000, 7000] * nreq)[:nreq], 512
    layout = W.make_layout(ctx, 7, device="cuda")
    mla = W.make_mla_case(nreq, layout.num_pages, seed=7, device="cuda")
    L = W.row_lengths(layout.ctx_len, 1).tolist()
    idx = W.random_indices(L, k, seed=7, device="cuda")
    kv = mla.kv.float()
    bt = layout.block_table
    for r in range(nreq):
        toks = idx[r].long()
        j = torch.arange(k, device="cuda")
        factor = 1.0 + 19.0 * ((j % 128) >= 64).float() + 10.0 * (j // 128).float()
        pages, slots = bt[r, toks // 64].long(), toks % 64
        kv[pages, slots, 512:] *= factor[:, None]
    mla.kv.copy_(kv.to(torch.bfloat16))
    out, lse = gpu_mla(mla, layout.block_table, nreq, 1, idx, layout.num_pages)
    torch.cuda.synchronize()
    compare(mla, layout, 1, idx, out, lse, rel=2.0 ** -8)
