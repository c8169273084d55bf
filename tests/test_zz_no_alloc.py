"""The no-allocation sparse MLA entry point (dsa_sparse_mla_decode_static).

Callers that may not call cudaMalloc -- a plug-in inside a host program that
owns all device memory, or a latency-critical loop that cannot take the
synchronisation an allocation may cause -- have no way to provide the split-K
workspace of dsa_sparse_mla_decode.  This entry point keeps that scratch in
an array compiled into the library.  The test calls it through the C ABI
twice in a row (different inputs, so leftovers of the first call would show)
and checks each result against dsa_sparse_mla_decode with a caller workspace:
the two calls split the work the same way and run the same kernels, so out
and lse must be bit for bit the same (a looser check, the sparse-attention
tolerance of the other parity tests, is asserted first so a failure says how
far apart they are).  It runs last (file name) and needs no state from other
tests.
"""
import pytest
import torch

from dsa_check import LSE_ATOL, MLA_ATOL, gpu_mla
from deepseek_sparse_attention_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _static(mla, bt, num_req, next_n, idx, num_pages):
    from deepseek_sparse_attention_02_gb300 import dsa
    R, k = idx.shape
    out = torch.full((R, W.MLA_HEADS, W.MLA_DV), float("nan"), dtype=torch.bfloat16,
                     device=idx.device)
    lse = torch.full((R, W.MLA_HEADS), float("nan"), device=idx.device)
    dsa.dsa_sparse_mla_decode_static(mla.q, mla.kv, 64 * 576 * 2, num_pages, bt, num_req, next_n,
                                     idx, k, mla.scale, out, lse)
    return out, lse


def _case(ctx, next_n, k, seed):
    layout = W.make_layout(ctx, seed, device="cuda")
    R = len(ctx) * next_n
    mla = W.make_mla_case(R, layout.num_pages, seed=seed, device="cuda")
    idx = W.random_indices(W.row_lengths(layout.ctx_len, next_n).tolist(), k, seed=seed,
                           device="cuda")
    return layout, mla, idx


def test_static_scratch_matches_workspace_entry_point_twice():
    from deepseek_sparse_attention_02_gb300 import dsa
    # batches small enough that the work is split over the selections, so the
    # scratch is really used (one row -> 32 splits; 3 rows x 2 -> 16 splits)
    for ctx, next_n, seed in (([20000], 1, 11), ([9000, 7000, 12000], 2, 12)):
        layout, mla, idx = _case(ctx, next_n, 2048, seed)
        R, k = idx.shape
        assert dsa.dsa_sparse_mla_workspace_size(R, k) > 0
        assert dsa.dsa_sparse_mla_workspace_size(R, k) <= dsa.dsa_sparse_mla_static_scratch_bytes()
        ref_out, ref_lse = gpu_mla(mla, layout.block_table, len(ctx), next_n, idx,
                                   layout.num_pages)
        got_out, got_lse = _static(mla, layout.block_table, len(ctx), next_n, idx,
                                   layout.num_pages)
        torch.cuda.synchronize()
        assert dsa.dsa_get_device_error() == 0
        assert (got_out.float() - ref_out.float()).abs().max().item() <= MLA_ATOL
        assert (got_lse - ref_lse).abs().max().item() <= LSE_ATOL
        assert torch.equal(got_out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(got_lse.view(torch.int32), ref_lse.view(torch.int32))


def test_static_scratch_covers_every_batch_shape():
    from deepseek_sparse_attention_02_gb300 import dsa
    # the largest split-K scratch any batch shape asks for fits the static
    # array, for selections from one token to the largest k
    cap = dsa.dsa_sparse_mla_static_scratch_bytes()
    for k in (1, 128, 2048, dsa.DSA_MAX_TOPK):
        worst = max(dsa.dsa_sparse_mla_workspace_size(R, k) for R in range(1, 400))
        assert worst <= cap, (k, worst, cap)
