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
    si = torch.empty((R, nb * (bs // 64)), dtype=torch.int32, device=cand.device)
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


@pytest.mark.parametrize("cbs", [128, 256])
def test_expand_larger_candidate_blocks_matches_oracle(cbs):
    """Candidate blocks of cbs tokens become cbs/64 sparse blocks of one page."""
    ctx = [cbs * 9 + 5, 3000, cbs * 3, 70]
    cand = W.make_candidates(ctx, 1, cbs, 8, seed=2, device="cuda")
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    si, end, sched, _ = expand(cand, ctx_t, 1, bs=cbs)
    rsi, rend = oracle.candidate_expand(np_(cand), cbs, np.array(ctx, np.int32), 1, sparse_bs=64)
    assert np.array_equal(np_(si), rsi) and np.array_equal(np_(end), rend)
    chunks = [-(-(-(-e // 128)) // 4) for e in rend]
    assert np_(sched)[:len(ctx) + 1].tolist() == [0] + np.cumsum(chunks).tolist()


def test_candidate_path_with_256_token_candidate_blocks():
    """The whole candidate path with candidate_block_size = 256 over 64-token
    sparse blocks (4 per candidate block): expansion, logits, top-k mapped to
    tokens, against the oracle."""
    ctx, next_n, nb, cbs = [256 * 40 + 3, 256 * 25], 2, 16, 256
    case = W.make_indexer_case(ctx, next_n=next_n, seed=6, device="cuda", fmt="mxfp4")
    cand = W.make_candidates(ctx, next_n, cbs, nb, seed=6, device="cuda")
    si, end, sched, nbytes = expand(cand, case.layout.ctx_len, next_n, bs=cbs)
    ns = si.shape[1]
    assert ns == nb * cbs // 64
    ld = ns * 64
    logits = cand_logits(case, si, end, sched, nbytes, ld)
    torch.cuda.synchronize()
    from deepseek_sparse_attention_02_gb300 import dsa
    assert dsa.dsa_get_device_error() == 0
    rsi, rend = oracle.candidate_expand(np_(cand), cbs, np_(case.layout.ctx_len), next_n,
                                        sparse_bs=64)
    assert np.array_equal(np_(si), rsi) and np.array_equal(np_(end), rend)
    ref, mag = oracle_cand(case, si, end)
    E = np_(end)
    check_logits(np_(logits), ref, mag, E)
    k = 512
    sel = gpu_topk(logits, ld, end, k, col_blocks=si, bs=64)
    exact = oracle.topk(np_(logits).astype(np.float64), E, k, col_blocks=np_(si), bs=64)
    for i in range(len(E)):
        assert sorted(np_(sel)[i].tolist()) == sorted(exact[i].tolist())
    check_topk_vs_oracle_scores_tokens(np_(sel), ref, mag, E, k, np_(si))


def check_topk_vs_oracle_scores_tokens(sel_tok, ref, mag, E, k, si):
    """The token selection against the oracle's fp64 scores of the columns:
    only tokens whose scores tie the k-th within 1e-3 may differ."""
    for i in range(len(E)):
        n = int(E[i])
        cols_tok = si[i][np.arange(n) // 64] * 64 + np.arange(n) % 64
        sel_cols = [int(np.flatnonzero(cols_tok == t)[0]) for t in sel_tok[i] if t >= 0]
        check_topk_vs_oracle_scores(np.array([sel_cols]), ref[i:i + 1], mag[i:i + 1],
                                    [n], k)


def test_candidate_bf16_logits_and_topk():
    """bf16 candidate logits: each is the f32 kernel's result rounded to nearest
    even, hence within 1e-3 (the f32 bound) plus one bf16 half-ulp (2^-8
    relative) of the oracle; the bf16 top-k over them, mapped to tokens, equals
    the oracle's full sort of the same bf16 values."""
    from deepseek_sparse_attention_02_gb300 import dsa
    ctx, next_n, nb = [9000, 12000, 64 * 31 + 9], 1, 64
    case = W.make_indexer_case(ctx, next_n=next_n, seed=9, device="cuda", fmt="mxfp4")
    cand = W.make_candidates(ctx, next_n, 64, nb, seed=9, device="cuda")
    si, end, sched, nbytes = expand(cand, case.layout.ctx_len, next_n)
    ld = nb * 64
    R = si.shape[0]
    f32 = cand_logits(case, si, end, sched, nbytes, ld)
    c = case.cache
    b16 = torch.zeros((R, ld), dtype=torch.bfloat16, device="cuda")
    dsa.dsa_candidate_logits_bf16(case.q, case.q_scale, case.w, c, W.FP4_PAGE_BYTES,
                                  c.data_ptr() + W.FP4_KEY_BYTES, W.FP4_PAGE_BYTES,
                                  case.layout.num_pages, case.layout.block_table,
                                  len(case.layout.ctx_len), case.next_n, si, nb, 64, end, sched,
                                  nbytes, b16, ld)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error() == 0
    E = np_(end)
    for i in range(R):
        n = int(E[i])
        assert torch.equal(b16[i, :n], f32[i, :n].to(torch.bfloat16)), f"row {i}"
    ref, mag = oracle_cand(case, si, end)
    got = np_(b16.float()).astype(np.float64)
    for i in range(R):
        n = int(E[i])
        tol = 1e-3 * np.maximum(np.abs(ref[i, :n]), mag[i, :n]) + 2.0 ** -8 * np.abs(ref[i, :n]) * 1.001
        assert np.all(np.abs(got[i, :n] - ref[i, :n]) <= tol), f"row {i}"
    k = 256
    sel = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_topk_bf16(b16, ld, end, R, k, sel, col_blocks=si, nb=nb, block_size=64)
    torch.cuda.synchronize()
    exact = oracle.topk(got, E, k, col_blocks=np_(si), bs=64)
    for i in range(R):
        assert sorted(np_(sel)[i].tolist()) == sorted(exact[i].tolist()), f"row {i}"


def test_candidate_logits_split_key_and_scale_buffers():
    """Keys and UE8M0 scales in two separate buffers (each with its own page
    stride) give the same logits, bit for bit, as the canonical page (scales
    right after the keys, fetched as one copy per page)."""
    from deepseek_sparse_attention_02_gb300 import dsa
    ctx, next_n, nb = [64 * 40 + 9, 5000], 1, 24
    case = W.make_indexer_case(ctx, next_n=next_n, seed=6, device="cuda", fmt="mxfp4")
    cand = W.make_candidates(ctx, next_n, 64, nb, seed=6, device="cuda")
    si, end, sched, nbytes = expand(cand, case.layout.ctx_len, next_n)
    ld = nb * 64
    ref = cand_logits(case, si, end, sched, nbytes, ld)
    c = case.cache.view(-1, W.FP4_PAGE_BYTES)
    keys = c[:, :W.FP4_KEY_BYTES].contiguous()
    scales = torch.zeros((c.shape[0], 512), dtype=torch.uint8, device="cuda")  # stride 512
    scales[:, :256] = c[:, W.FP4_KEY_BYTES:]
    got = torch.full((case.rows, ld), float("nan"), device="cuda")
    dsa.dsa_candidate_logits(case.q, case.q_scale, case.w, keys, W.FP4_KEY_BYTES, scales, 512,
                             case.layout.num_pages, case.layout.block_table,
                             len(case.layout.ctx_len), next_n, si, nb, 64, end, sched, nbytes,
                             got, ld)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error() == 0
    E = np_(end)
    g, r = np_(got), np_(ref)
    for i in range(case.rows):
        assert np.array_equal(g[i, :E[i]].view(np.uint32), r[i, :E[i]].view(np.uint32)), i


def test_candidate_logits_many_short_rows():
    """Many rows of one or two tiles each, so every CTA walks several row
    groups (the q slots are refilled after both MMA issuers and both epilogue
    warpgroups have let go of them) and some rows have a partial last page;
    MTP rows (next_n = 2) see different lengths of the same candidates."""
    from deepseek_sparse_attention_02_gb300 import dsa
    rng = np.random.default_rng(17)
    ctx = [int(x) for x in rng.integers(70, 1100, size=190)]
    next_n, nb = 2, 4
    case = W.make_indexer_case(ctx, next_n=next_n, seed=17, device="cuda", fmt="mxfp4")
    cand = W.make_candidates(ctx, next_n, 64, nb, seed=17, device="cuda")
    si, end, sched, nbytes = expand(cand, case.layout.ctx_len, next_n)
    ld = nb * 64
    logits = cand_logits(case, si, end, sched, nbytes, ld)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error() == 0
    assert case.rows > 2 * 152  # more row groups than CTAs
    ref, mag = oracle_cand(case, si, end)
    check_logits(np_(logits), ref, mag, np_(end))
