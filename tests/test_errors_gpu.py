"""Device-side error paths with host-injected bad inputs: a selected index
outside its row's block table or outside the cache (sparse MLA), a row length
longer than the logits row (top-k), and a varlen entry whose row range runs
past the rows (indexer).  Each call must finish, set its error bit, skip only
the bad element, and leave every other result equal to the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from dsa_check import LSE_ATOL, MLA_ATOL, check_logits, gpu_mla, gpu_topk, ld_for, mla_oracle, np_
from deepseek_sparse_attention_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _dsa():
    from deepseek_sparse_attention_02_gb300 import dsa
    return dsa


@pytest.mark.parametrize("nreq,k", [(3, 512), (48, 2048)])
def test_mla_bad_index_is_reported_and_skipped(nreq, k):
    dsa = _dsa()
    dsa.dsa_get_device_error(clear=True)
    ctx = ([3000, 4000, 5000] * nreq)[:nreq]
    layout = W.make_layout(ctx, 21, device="cuda")
    mla = W.make_mla_case(nreq, layout.num_pages, seed=21, device="cuda")
    idx = W.random_indices(W.row_lengths(layout.ctx_len, 1).tolist(), k, seed=21, device="cuda")
    bt_stride = layout.block_table.shape[1]
    bad = idx.clone()
    bad[0, 7] = bt_stride * 64 + 5            # past the row's block-table entries
    bad[1, k - 3] = layout.num_pages * 64 + 1  # past the whole cache
    out, lse = gpu_mla(mla, layout.block_table, nreq, 1, bad, layout.num_pages)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error(clear=True) == dsa.DEVERR_BAD_INDEX
    # the bad selections are skipped exactly like -1: the oracle of the same
    # selection with -1 in their place matches every row
    skipped = bad.clone()
    skipped[0, 7] = -1
    skipped[1, k - 3] = -1
    rows = np.array(sorted({0, 1, 2, nreq - 1}), np.int32)
    o_ref, l_ref = mla_oracle(mla, layout.block_table, 1, skipped, rows=rows)
    assert np.abs(np_(out.float())[rows] - o_ref).max() <= MLA_ATOL
    assert np.abs(np_(lse)[rows] - l_ref).max() <= LSE_ATOL
    # and the rows without a bad index equal the call on valid indices
    out2, lse2 = gpu_mla(mla, layout.block_table, nreq, 1, idx, layout.num_pages)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error() == 0
    assert torch.equal(out[2:].view(torch.int16), out2[2:].view(torch.int16))


def test_topk_row_longer_than_logits_is_reported_and_clamped():
    dsa = _dsa()
    dsa.dsa_get_device_error(clear=True)
    g = torch.Generator(device="cuda").manual_seed(3)
    R, ld, k = 3, 20000, 1024
    logits = torch.randn((R, ld), generator=g, device="cuda")
    L = torch.tensor([15000, ld + 8, 19999], dtype=torch.int32, device="cuda")
    sel = gpu_topk(logits, ld, L, k)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error(clear=True) == dsa.DEVERR_BAD_INDEX
    want_L = np.array([15000, ld, 19999])
    ref = oracle.topk(np_(logits).astype(np.float64), want_L, k)
    got = np_(sel)
    for i in range(R):
        assert np.array_equal(np.sort(got[i]), np.sort(ref[i])), i


def test_varlen_indexer_entry_past_the_rows_is_reported_and_skipped():
    dsa = _dsa()
    dsa.dsa_get_device_error(clear=True)
    base = W.make_indexer_case([3000, 2000], next_n=1, seed=8, device="cuda")
    lay = base.layout
    qc, qs, w = W.make_index_queries(4, seed=81, device="cuda")
    ld = ld_for(3000)
    logits = torch.full((4, ld), float("nan"), device="cuda")
    # entry 0: rows [0, 2) of request 0; entry 1: rows [2, 9) -- past the 4 rows
    cu = torch.tensor([0, 2, 9], dtype=torch.int32, device="cuda")
    ctx_e = torch.tensor([3000, 2000], dtype=torch.int32, device="cuda")
    bt_rows = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    c = base.cache
    dsa.dsa_indexer_logits_varlen(qc, qs, w, c, W.FP8_PAGE_BYTES, c.data_ptr() + W.FP8_KEY_BYTES,
                                  W.FP8_PAGE_BYTES, lay.num_pages, lay.block_table, bt_rows, ctx_e,
                                  cu, 2, 7, 4, logits, ld)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error(clear=True) == dsa.DEVERR_BAD_INDEX
    got = np_(logits)
    assert np.all(np.isnan(got[2:]))  # the bad entry wrote nothing
    cache = np_(c).reshape(-1)
    ref, mag = oracle.indexer_logits(np_(qc[:2]), np_(qs[:2]), np_(w[:2]), cache,
                                     W.FP8_PAGE_BYTES, cache[W.FP8_KEY_BYTES:], W.FP8_PAGE_BYTES,
                                     64, np_(lay.block_table)[0:1],
                                     np.array([3000], np.int32), 2, ld=ld)
    check_logits(got[:2], ref, mag, [2999, 3000])
