"""Prefill in chunks: the chunk plan (dsa_prefill_chunk_plan) against the
oracle's, and on the GPU a multi-request prefill run chunk by chunk through
the varlen entry points (dsa_indexer_logits_varlen, dsa_varlen_row_lengths,
dsa_topk, dsa_sparse_mla_decode_varlen), every row checked against the oracle
of its own request (logits on sampled rows, the exact top-k on the GPU's own
logits plus the tie band against the oracle's scores, the attention over the
GPU's selection)."""
import numpy as np
import pytest
import torch

import oracle
from dsa_check import (LSE_ATOL, MLA_ATOL, check_logits, check_topk_vs_oracle_scores, ld_for,
                       np_)
from deepseek_sparse_attention_02_gb300 import workloads as W


def _dsa():
    from deepseek_sparse_attention_02_gb300 import dsa
    return dsa


# --------------------------------------------------------------------- CPU --
def test_chunk_plan_matches_oracle():
    dsa = _dsa()
    rng = np.random.default_rng(41)
    for _ in range(300):
        nreq = int(rng.integers(1, 9))
        q = rng.integers(0, 50, nreq).tolist()
        ctx = rng.integers(1, 70000, nreq).tolist()
        mn = int(rng.choice([0, 64, 8192]))
        budget = int(rng.integers(64, 1 << 24))
        assert dsa.dsa_prefill_chunk_plan(q, ctx, budget, mn) == \
            oracle.prefill_chunk_plan(q, ctx, budget, mn)


def test_chunk_plan_host_checks():
    dsa = _dsa()
    with pytest.raises(dsa.DsaError, match="INVALID_ARG"):
        dsa.dsa_prefill_chunk_plan([3, -1], [10, 10], 1000)
    with pytest.raises(dsa.DsaError, match="INVALID_ARG"):
        dsa.dsa_prefill_chunk_plan([3], [10], 0)
    lib = dsa.lib()
    # varlen entry points reject a NULL cu_rows / row_bt before touching a device
    assert lib.dsa_indexer_logits_varlen(16, 16, 16, 16, 8448, 16, 8448, 1, 16, 1, 1, None, 16,
                                         None, 1, 1, 1, 16, 4, None) == 1
    assert lib.dsa_sparse_mla_decode_varlen(16, 16, 73728, 1, 16, 1, 1, None, 1, 16, 16, 0.1, 16,
                                            None, None, 0, None) == 1


# --------------------------------------------------------------------- GPU --
Q_LEN = [70, 30, 5]
CTX = [3000, 2500, 1200]
K = 1024


def _case():
    """One cache with the three requests' pages; every query row of the
    prefill (the last Q_LEN[b] positions of request b) has its own indexer and
    attention query."""
    base = W.make_indexer_case(CTX, next_n=1, seed=5, device="cuda")
    total = sum(Q_LEN)
    qc, qs, w = W.make_index_queries(total, seed=51, device="cuda")
    mla = W.make_mla_case(total, base.layout.num_pages, seed=52, device="cuda")
    return base, (qc, qs, w), mla


@pytest.mark.gpu
def test_prefill_in_chunks_matches_oracle():
    dsa = _dsa()
    base, (qc, qs, w), mla = _case()
    lay = base.layout
    total = sum(Q_LEN)
    first = np.concatenate([[0], np.cumsum(Q_LEN)])  # global first row of each request
    # a budget of ~40 rows of the widest request: several chunks, requests split
    budget = 40 * ld_for(max(CTX)) * 4
    pieces = dsa.dsa_prefill_chunk_plan(Q_LEN, CTX, budget)
    assert pieces == oracle.prefill_chunk_plan(Q_LEN, CTX, budget)
    assert len({p[0] for p in pieces}) >= 3
    logits_all = np.full((total, max(CTX)), np.nan, np.float32)
    sel_all = np.full((total, K), -9, np.int32)
    out_all = torch.empty((total, W.MLA_HEADS, W.MLA_DV), dtype=torch.bfloat16, device="cuda")
    lse_all = torch.empty((total, W.MLA_HEADS), device="cuda")
    for ch in sorted({p[0] for p in pieces}):
        ps = [p for p in pieces if p[0] == ch]
        rows = [first[b] + j for _, b, j0, j1 in ps for j in range(j0, j1)]
        n = len(rows)
        ld = ld_for(max(CTX[b] for _, b, _, _ in ps))
        assert n * ld * 4 <= budget or n == 1
        ridx = torch.tensor(rows, dtype=torch.long, device="cuda")
        cu = torch.tensor(np.concatenate([[0], np.cumsum([j1 - j0 for _, _, j0, j1 in ps])]),
                          dtype=torch.int32, device="cuda")
        ctx_e = torch.tensor([CTX[b] - (Q_LEN[b] - j1) for _, b, _, j1 in ps], dtype=torch.int32,
                             device="cuda")
        bt_rows = torch.tensor([b for _, b, _, _ in ps], dtype=torch.int32, device="cuda")
        q8, s8, w8 = qc[ridx].contiguous(), qs[ridx].contiguous(), w[ridx].contiguous()
        logits = torch.full((n, ld), float("nan"), device="cuda")
        c = base.cache
        dsa.dsa_indexer_logits_varlen(q8, s8, w8, c, W.FP8_PAGE_BYTES,
                                      c.data_ptr() + W.FP8_KEY_BYTES, W.FP8_PAGE_BYTES,
                                      lay.num_pages, lay.block_table, bt_rows, ctx_e, cu, len(ps),
                                      max(j1 - j0 for _, _, j0, j1 in ps), n, logits, ld)
        row_len = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        dsa.dsa_varlen_row_lengths(ctx_e, cu, len(ps), n, row_len)
        sel = torch.full((n, K), -7, dtype=torch.int32, device="cuda")
        dsa.dsa_topk(logits, ld, row_len, n, K, sel)
        row_bt = torch.repeat_interleave(bt_rows, torch.diff(cu).long())
        out = torch.empty((n, W.MLA_HEADS, W.MLA_DV), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((n, W.MLA_HEADS), device="cuda")
        wsb = dsa.dsa_sparse_mla_workspace_size(n, K)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
        dsa.dsa_sparse_mla_decode_varlen(mla.q[ridx].contiguous(), mla.kv, 64 * 576 * 2,
                                         lay.num_pages, lay.block_table, row_bt, n, sel, K,
                                         mla.scale, out, lse, ws, wsb)
        torch.cuda.synchronize()
        assert dsa.dsa_get_device_error() == 0
        # row lengths: row j of request b sees CTX[b] - (Q_LEN[b] - 1 - j) tokens
        want = [CTX[b] - (Q_LEN[b] - 1 - j) for _, b, j0, j1 in ps for j in range(j0, j1)]
        assert np_(row_len).tolist() == want
        lg = np_(logits)
        for i, r in enumerate(rows):
            logits_all[r, :ld] = lg[i, :ld] if ld <= logits_all.shape[1] else lg[i, :logits_all.shape[1]]
        sel_all[rows] = np_(sel)
        out_all[ridx] = out
        lse_all[ridx] = lse
    # every row against the oracle of its own request
    cache = np_(base.cache).reshape(-1)
    bt = np_(lay.block_table)
    for b in range(len(Q_LEN)):
        g = np.arange(first[b], first[b + 1])
        L = np.array([CTX[b] - (Q_LEN[b] - 1 - j) for j in range(Q_LEN[b])], np.int32)
        samp = np.unique([0, Q_LEN[b] - 1, Q_LEN[b] // 2]).astype(np.int32)
        ref, mag = oracle.indexer_logits(np_(qc[g]), np_(qs[g]), np_(w[g]), cache,
                                         W.FP8_PAGE_BYTES, cache[W.FP8_KEY_BYTES:],
                                         W.FP8_PAGE_BYTES, 64, bt[b:b + 1],
                                         np.array([CTX[b]], np.int32), Q_LEN[b], rows=samp,
                                         ld=max(CTX))
        check_logits(logits_all[g[samp]], ref, mag, L[samp])
        check_topk_vs_oracle_scores(sel_all[g[samp]], ref, mag, L[samp], K)
        # exact top-k on the GPU's own logits
        exact = oracle.topk(logits_all[g].astype(np.float64), L, K)
        for jj in range(Q_LEN[b]):
            assert sorted(sel_all[g[jj]].tolist()) == sorted(exact[jj].tolist()), (b, jj)
        o_ref, l_ref = oracle.sparse_mla(
            W.bf16_bits(mla.q[torch.as_tensor(g, device="cuda")]).cpu().numpy().view(np.uint16),
            W.bf16_bits(mla.kv).cpu().numpy().view(np.uint16), 64 * 576, 64, bt[b:b + 1],
            Q_LEN[b], sel_all[g], mla.scale, rows=samp)
        got = np_(out_all[torch.as_tensor(g[samp], device="cuda")].float())
        assert np.abs(got - o_ref).max() <= MLA_ATOL, b
        assert np.abs(np_(lse_all[torch.as_tensor(g[samp], device="cuda")]) - l_ref).max() <= LSE_ATOL
