"""Parity of the candidate-block path (expansion, MXFP4 candidate logits,
top-k over candidate columns mapped to tokens) with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from dsa_check import check_logits, check_topk_vs_oracle_scores, gpu_topk, np_
from deepseek_sparse_attention_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def expand(cand, ctx_len, next_n, bs=64):
    from deepseek_sparse_attention_02_gb300 import dsa
    R, nb = cand.shape
    si = torch.empty_like(cand)
    end = torch.empty(R, dtype=torch.int32, device=cand.device)
    nbytes = dsa.dsa_candidate_schedule_size(R)
    sched = torch.zeros(nbytes // 4, dtype=torch.int32, device=cand.device)
    dsa.dsa_candidate_expand(cand, R, nb, bs, ctx_len, next_n, si, end, sched, nbytes)
    return si, end, sched, nbytes


def cand_logits(case, si, end, sched, nbytes, ld):
    from deepseek_sparse_attention_02_gb300 import dsa
    c = case.cache
    R, nb = si.shape
    logits = torch.full((R, ld), float("nan"), device=c.device)
    dsa.dsa_candidate_logits(case.q, case.q_scale, case.w, c, W.FP4_PAGE_BYTES,
                             c.data_ptr() + W.FP4_KEY_BYTES, W.FP4_PAGE_BYTES,
                             case.layout.num_pages, case.layout.block_table,
                             len(case.layout.ctx_len), case.next_n, si, nb, 64, end, sched, nbytes,
                             logits, ld)
    return logits


def oracle_cand(case, si, end, rows=None):
    cache = np_(case.cache).reshape(-1)
    return oracle.candidate_logits(np_(case.q), np_(case.q_scale), np_(case.w), cache,
                                   W.FP4_PAGE_BYTES, cache[W.FP4_KEY_BYTES:], W.FP4_PAGE_BYTES,
                                   64, np_(case.layout.block_table), case.next_n, np_(si), 64,
                                   np_(end), rows=rows)


def test_expand_matches_oracle():
    ctx = [640, 1000, 64 * 40 + 5, 130]
    cand = W.make_candidates(ctx, 1, 64, 8, seed=1, device="cuda")
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    si, end, sched, _ = expand(cand, ctx_t, 1)
    rsi, rend = oracle.candidate_expand(np_(cand), 64, np.array(ctx, np.int32), 1)
    assert np.array_equal(np_(si), rsi) and np.array_equal(np_(end), rend)
    chunks = [-(-(-(-e // 128)) // 4) for e in rend]
    assert np_(sched)[:len(ctx) + 1].tolist() == [0] + np.cumsum(chunks).tolist()


@pytest.mark.parametrize("ctx,next_n,nb", [
    ([64 * 30, 64 * 30 + 17, 500], 1, 12),
    ([64 * 50], 2, 16),
    ([9000, 12000], 1, 64),
])
def test_candidate_logits_and_topk(ctx, next_n, nb):
    case = W.make_indexer_case(ctx, next_n=next_n, seed=4, device="cuda", fmt="mxfp4")
    cand = W.make_candidates(ctx, next_n, 64, nb, seed=4, device="cuda")
    si, end, sched, nbytes = expand(cand, case.layout.ctx_len, next_n)
    ld = nb * 64
    logits = cand_logits(case, si, end, sched, nbytes, ld)
    torch.cuda.synchronize()
    from deepseek_sparse_attention_02_gb300 import dsa
    assert dsa.dsa_get_device_error() == 0
    ref, mag = oracle_cand(case, si, end)
    E = np_(end)
    check_logits(np_(logits), ref, mag, E)
    k = min(256, ld)
    sel = gpu_topk(logits, ld, end, k, col_blocks=si, bs=64)
    # exact on the GPU's own logits, mapped to tokens
    exact = oracle.topk(np_(logits).astype(np.float64), E, k, col_blocks=np_(si), bs=64)
    for i in range(len(E)):
        assert sorted(np_(sel)[i].tolist()) == sorted(exact[i].tolist())
