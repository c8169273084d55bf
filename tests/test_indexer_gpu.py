"""Parity of dsa_indexer_logits (Eq. (1)) with the fp64 oracle."""
import numpy as np
import pytest
import torch

from dsa_check import check_logits, gpu_indexer, np_, oracle_indexer, row_lens
from deepseek_sparse_attention_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ctx,next_n", [
    ([1, 63, 64, 65, 127, 128, 129, 1000, 2500], 1),   # ragged tails, page and tile edges
    ([300, 4097], 2),                                   # MTP rows, N = 128
    ([700, 1], 3),                                      # N = 192, a row with no token
    ([1500], 7),                                        # prefill-style groups of 4 + a partial group
    ([0, 640, 0], 1),                                   # empty requests
])
def test_indexer_small(ctx, next_n):
    case = W.make_indexer_case(ctx, next_n=next_n, seed=3, device="cuda")
    logits, ld = gpu_indexer(case)
    torch.cuda.synchronize()
    from deepseek_sparse_attention_02_gb300 import dsa
    assert dsa.dsa_get_device_error() == 0
    ref, mag = oracle_indexer(case, ld=ld)
    L = np_(row_lens(case))
    check_logits(np_(logits), ref, mag, L)
    # nothing is written past a row's length
    for i, n in enumerate(L):
        assert np.all(np.isnan(np_(logits[i, n:])))


def test_indexer_contiguous_tiny_decode():
    """8192-token single-row decode on an identity block table."""
    case = W.make_indexer_case([8192], next_n=1, seed=0, device="cuda", shuffle=False)
    logits, ld = gpu_indexer(case)
    ref, mag = oracle_indexer(case, ld=ld)
    check_logits(np_(logits), ref, mag, [8192])


def test_indexer_repeatable():
    case = W.make_indexer_case([5000, 3000], next_n=2, seed=9, device="cuda")
    a, _ = gpu_indexer(case)
    b, _ = gpu_indexer(case)
    assert torch.equal(torch.nan_to_num(a, nan=7.0), torch.nan_to_num(b, nan=7.0))


def test_indexer_bad_page_is_reported_not_trapped():
    from deepseek_sparse_attention_02_gb300 import dsa
    case = W.make_indexer_case([500], next_n=1, seed=2, device="cuda")
    case.layout.block_table[0, 3] = case.layout.num_pages + 10
    gpu_indexer(case)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error(clear=True) & dsa.DEVERR_BAD_PAGE
    assert dsa.dsa_get_device_error() == 0
