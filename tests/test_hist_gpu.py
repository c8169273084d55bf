"""The top-k's first pass fused into the indexer (dsa_indexer_logits_hist +
dsa_topk_hist).

* The logits equal dsa_indexer_logits' bit for bit, and each row's histogram
  equals, count for count, the histogram of those logits computed here from
  its definition (bin = top 12 bits of the order-preserving key: sign bit
  set for positives, all bits flipped for negatives, -0.0 as +0.0).
* dsa_topk_hist selects exactly the oracle's full-sort set on the GPU's own
  fp32 logits (one CTA per row and the two-CTA pair, short rows, rows with
  L <= k), and leaves every histogram zero.
* A histogram that does not describe the row (garbage, or counts of another
  row) changes nothing in the result.
"""
import numpy as np
import pytest
import torch

import oracle
from dsa_check import gpu_indexer, host_hist, ld_for, np_, row_lens
from deepseek_sparse_attention_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu
BINS = 4096


def _dsa():
    from deepseek_sparse_attention_02_gb300 import dsa
    return dsa


def run_hist(case, ld=None, k=2048, force_path=0):
    dsa = _dsa()
    L = row_lens(case)
    ld = ld or ld_for(int(L.max()))
    R = case.rows
    logits = torch.full((R, ld), float("nan"), device="cuda")
    hist = torch.zeros((R, BINS), dtype=torch.int32, device="cuda")
    c = case.cache
    dsa.dsa_indexer_logits_hist(case.q, case.q_scale, case.w, c, W.FP8_PAGE_BYTES,
                                c.data_ptr() + W.FP8_KEY_BYTES, W.FP8_PAGE_BYTES,
                                case.layout.num_pages, case.layout.block_table,
                                case.layout.ctx_len, len(case.layout.ctx_len), case.next_n, logits,
                                ld, hist)
    torch.cuda.synchronize()
    h_after_indexer = np_(hist).astype(np.int64)
    sel = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_topk_hist(logits, ld, L, R, k, hist, sel, force_path=force_path)
    torch.cuda.synchronize()
    return logits, ld, L, sel, h_after_indexer, hist


@pytest.mark.parametrize("ctx,next_n", [
    ([131072] * 4, 2),                    # the 128K MTP rows: the two-CTA pair
    ([20000, 70000, 3000, 1500], 1),      # short rows (L <= k), staged and cutoff paths
    ([40000] * 100, 1),                   # more rows than half the SMs: one CTA per row
])
def test_hist_matches_definition_and_topk_is_exact(ctx, next_n):
    dsa = _dsa()
    dsa.dsa_get_device_error(clear=True)
    case = W.make_indexer_case(ctx, next_n=next_n, seed=31, device="cuda")
    logits, ld, L, sel, h, hist_left = run_hist(case)
    assert dsa.dsa_get_device_error() == 0
    # the same logits as the plain indexer, bit for bit
    ref_logits, _ = gpu_indexer(case, ld=ld)
    torch.cuda.synchronize()
    Ln = np_(L)
    lg, rl = np_(logits), np_(ref_logits)
    for r in range(case.rows):
        assert np.array_equal(lg[r, :Ln[r]].view(np.uint32), rl[r, :Ln[r]].view(np.uint32)), r
    # the histogram of exactly those logits
    assert np.array_equal(h, host_hist(lg, Ln))
    # exact selection, and every histogram cleared
    ref = oracle.topk(lg.astype(np.float64), Ln, 2048)
    got = np_(sel)
    for r in range(case.rows):
        assert np.array_equal(np.sort(got[r]), np.sort(ref[r])), r
    assert int(hist_left.abs().sum()) == 0


def test_topk_hist_ignores_a_histogram_of_something_else():
    dsa = _dsa()
    dsa.dsa_get_device_error(clear=True)
    g = torch.Generator(device="cuda").manual_seed(5)
    R, ld, k = 8, 131072, 2048
    logits = torch.randn((R, ld), generator=g, device="cuda") * 3
    L = torch.full((R,), ld, dtype=torch.int32, device="cuda")
    L[3] = ld - 1000
    ref = oracle.topk(np_(logits).astype(np.float64), np_(L), k)
    cases = {
        "garbage": torch.randint(0, 1 << 20, (R, BINS), generator=g, device="cuda",
                                 dtype=torch.int32),
        "another row's counts": torch.tensor(host_hist(np_(logits)[::-1].copy(), np_(L)[::-1]),
                                             dtype=torch.int32, device="cuda"),
        "all mass in one bin": torch.zeros((R, BINS), dtype=torch.int32, device="cuda"),
    }
    cases["all mass in one bin"][:, 3000] = L
    for name, hist in cases.items():
        sel = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
        dsa.dsa_topk_hist(logits, ld, L, R, k, hist, sel)
        torch.cuda.synchronize()
        dsa.dsa_get_device_error(clear=True)  # a missed cutoff is redone (capacity bit)
        got = np_(sel)
        for r in range(R):
            assert np.array_equal(np.sort(got[r]), np.sort(ref[r])), (name, r)
        assert int(hist.abs().sum()) == 0, name


def test_hist_rejects_prefill_shapes_and_null():
    dsa = _dsa()
    case = W.make_indexer_case([500], next_n=4, seed=2, device="cuda")
    hist = torch.zeros((4, BINS), dtype=torch.int32, device="cuda")
    logits = torch.empty((4, 512), device="cuda")
    c = case.cache
    with pytest.raises(dsa.DsaError, match="UNSUPPORTED"):
        dsa.dsa_indexer_logits_hist(case.q, case.q_scale, case.w, c, W.FP8_PAGE_BYTES,
                                    c.data_ptr() + W.FP8_KEY_BYTES, W.FP8_PAGE_BYTES,
                                    case.layout.num_pages, case.layout.block_table,
                                    case.layout.ctx_len, 1, 4, logits, 512, hist)
    with pytest.raises(dsa.DsaError, match="INVALID_ARG"):
        dsa.dsa_topk_hist(logits, 512, torch.ones(4, dtype=torch.int32, device="cuda"), 4, 8,
                          None, torch.empty((4, 8), dtype=torch.int32, device="cuda"))
