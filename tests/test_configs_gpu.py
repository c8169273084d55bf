"""Parity at the full workload sizes, in the launch configuration bench.py
times.  The CUDA path runs every row; the fp64 oracle checks sampled rows
(first, last and seeded middle rows) for the logits and the attention, and the
top-k is checked exactly on every row against the oracle's full sort of the
GPU's own fp32 logits, plus the 1e-3 tie-band rule against the oracle's fp64
scores on the sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from dsa_check import (LSE_ATOL, MLA_ATOL, check_logits, check_topk_vs_oracle_scores,
                       gpu_indexer, gpu_mla, gpu_topk, mla_oracle, np_, oracle_indexer, row_lens)
from deepseek_sparse_attention_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu
K = 2048


def sample_rows(R, n=4, seed=0):
    rng = np.random.default_rng(seed)
    rows = {0, R - 1} | set(rng.choice(R, size=min(R, n), replace=False).tolist())
    return np.array(sorted(rows), np.int32)


def exact_topk_all_rows(logits, L, sel, col_blocks=None, bs=0):
    got = np_(sel)
    ref = oracle.topk(np_(logits).astype(np.float64), np_(L), K,
                      col_blocks=None if col_blocks is None else np_(col_blocks), bs=bs)
    for i in range(got.shape[0]):
        assert np.array_equal(np.sort(got[i]), np.sort(ref[i])), f"top-k row {i}"


def run_dense(cfg, with_mla):
    spec = W.config_ctx(cfg)
    case = W.make_indexer_case(spec["ctx"], next_n=spec["next_n"], seed=cfg, device="cuda",
                               shuffle=spec["shuffle"])
    logits, ld = gpu_indexer(case)
    L = row_lens(case)
    sel = gpu_topk(logits, ld, L, K)
    torch.cuda.synchronize()
    from deepseek_sparse_attention_02_gb300 import dsa
    assert dsa.dsa_get_device_error() == 0
    rows = sample_rows(case.rows, seed=cfg)
    ref, mag = oracle_indexer(case, rows=rows, ld=ld)
    worst, worst_plain = check_logits(np_(logits)[rows], ref, mag, np_(L)[rows], plain=True)
    print(f"config {cfg}: worst logit error {worst:.3g} of max(|ref|, A); "
          f"plain relative error where |ref| >= A/8: {worst_plain:.3g}")
    check_topk_vs_oracle_scores(np_(sel)[rows], ref, mag, np_(L)[rows], K)
    exact_topk_all_rows(logits, L, sel)
    if with_mla:
        mla = W.make_mla_case(case.rows, case.layout.num_pages, seed=cfg, device="cuda")
        out, lse = gpu_mla(mla, case.layout.block_table, len(spec["ctx"]), spec["next_n"], sel,
                           case.layout.num_pages)
        torch.cuda.synchronize()
        o_ref, l_ref = mla_oracle(mla, case.layout.block_table, spec["next_n"], sel, rows=rows)
        assert np.abs(np_(out.float())[rows] - o_ref).max() <= MLA_ATOL
        assert np.abs(np_(lse)[rows] - l_ref).max() <= LSE_ATOL


def test_tiny_decode_full_path():
    run_dense(0, with_mla=True)


def test_batched_varlen_full_path():
    run_dense(1, with_mla=True)


def test_long_context_mtp_decode():
    run_dense(2, with_mla=True)


def test_chunked_prefill():
    run_dense(4, with_mla=True)


def test_candidate_block_indexer():
    from deepseek_sparse_attention_02_gb300 import dsa
    spec = W.config_ctx(3)
    ctx, nb = spec["ctx"], spec["candidate_topk_blocks"]
    cand = W.make_candidates(ctx, 1, 64, nb, seed=3, device="cuda")
    R = cand.shape[0]
    si = torch.empty_like(cand)
    end = torch.empty(R, dtype=torch.int32, device="cuda")
    nbytes = dsa.dsa_candidate_schedule_size(R)
    sched = torch.zeros(nbytes // 4, dtype=torch.int32, device="cuda")
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    dsa.dsa_candidate_expand(cand, R, nb, 64, ctx_t, 1, si, end, sched, nbytes)
    rsi, rend = oracle.candidate_expand(np_(cand), 64, np.array(ctx, np.int32), 1)
    assert np.array_equal(np_(si), rsi) and np.array_equal(np_(end), rend)
    ld = nb * 64
    rows = sample_rows(R, seed=3)
    for layer in (0, 3):  # consumer layers share the expansion
        case = W.make_indexer_case(ctx, next_n=1, seed=3 + layer, device="cuda", fmt="mxfp4")
        logits = torch.full((R, ld), float("nan"), device="cuda")
        c = case.cache
        dsa.dsa_candidate_logits(case.q, case.q_scale, case.w, c, W.FP4_PAGE_BYTES,
                                 c.data_ptr() + W.FP4_KEY_BYTES, W.FP4_PAGE_BYTES,
                                 case.layout.num_pages, case.layout.block_table, R, 1, si, nb, 64,
                                 end, sched, nbytes, logits, ld)
        sel = gpu_topk(logits, ld, end, K, col_blocks=si, bs=64)
        torch.cuda.synchronize()
        assert dsa.dsa_get_device_error() == 0
        cache = np_(c).reshape(-1)
        ref, mag = oracle.candidate_logits(np_(case.q), np_(case.q_scale), np_(case.w), cache,
                                           W.FP4_PAGE_BYTES, cache[W.FP4_KEY_BYTES:],
                                           W.FP4_PAGE_BYTES, 64, np_(case.layout.block_table), 1,
                                           rsi, 64, rend, rows=rows)
        check_logits(np_(logits)[rows], ref, mag, rend[rows])
        exact_topk_all_rows(logits, end, sel, col_blocks=si, bs=64)
