"""Shared helpers for the parity tests: run one step of the CUDA path through
the C ABI and the same step through the fp64 oracle, on the same seeded inputs,
and compare with the acceptance rules:

* logits: |gpu - ref| <= 1e-3 * max(|ref|, A) with A = sum_h |w_h| ReLU(q_h.k_t)
  (the condition scale of the sum; plain relative error is meaningless where
  mixed-sign head weights cancel);
* top-k: on the GPU's own fp32 logits the selected set must equal the oracle's
  (score descending, column ascending) exactly; against the oracle's fp64
  logits the sets may differ only by tokens whose oracle scores lie within
  1e-3 (same condition scale) of the k-th score;
* sparse MLA: max |out - ref| <= 1e-2 (bf16 output), lse within 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from deepseek_sparse_attention_02_gb300 import workloads as W

LOGIT_RTOL = 1e-3
HIST_BINS = 4096
MLA_ATOL = 1e-2
LSE_ATOL = 1e-3


def lib():
    from deepseek_sparse_attention_02_gb300 import dsa
    return dsa


def np_(t):
    return t.detach().cpu().numpy()


def bits16(t):
    return W.bf16_bits(t).cpu().numpy().view(np.uint16)


def row_lens(case):
    return W.row_lengths(case.layout.ctx_len, case.next_n).to(torch.int32)


def ld_for(n):
    return max(4, (int(n) + 3) // 4 * 4)


def gpu_indexer(case, ld=None):
    dsa = lib()
    L = row_lens(case)
    ld = ld or ld_for(int(L.max()) if L.numel() else 4)
    logits = torch.full((case.rows, ld), float("nan"), device=case.q.device)
    c = case.cache
    dsa.dsa_indexer_logits(case.q, case.q_scale, case.w, c, W.FP8_PAGE_BYTES,
                           c.data_ptr() + W.FP8_KEY_BYTES, W.FP8_PAGE_BYTES,
                           case.layout.num_pages, case.layout.block_table, case.layout.ctx_len,
                           len(case.layout.ctx_len), case.next_n, logits, ld)
    return logits, ld


def oracle_indexer(case, rows=None, ld=None):
    cache = np_(case.cache).reshape(-1)
    return oracle.indexer_logits(np_(case.q), np_(case.q_scale), np_(case.w), cache,
                                 W.FP8_PAGE_BYTES, cache[W.FP8_KEY_BYTES:], W.FP8_PAGE_BYTES, 64,
                                 np_(case.layout.block_table), np_(case.layout.ctx_len),
                                 case.next_n, rows=rows, ld=ld)


def check_logits(got, ref, mag, L, plain=False):
    """got/ref/mag: 2-D arrays over the same rows; L: per-row valid length.
    Returns the worst error scaled by max(|ref|, A).

    With plain=True it also checks the criterion as stated, plain relative
    error |gpu - ref| / |ref| <= 1e-3, on every logit whose sum is not
    cancelled, |ref| >= A / 8 (there the condition-scaled bound alone would
    allow up to 8e-3), and returns (worst scaled, worst plain)."""
    worst = worst_plain = 0.0
    for i in range(len(L)):
        n = int(L[i])
        g, r, a = got[i, :n].astype(np.float64), ref[i, :n], mag[i, :n]
        assert np.all(np.isfinite(g)), f"row {i}: non-finite logits"
        err = np.abs(g - r) / np.maximum(np.maximum(np.abs(r), a), 1e-300)
        if n:
            worst = max(worst, float(err.max()))
        bad = np.flatnonzero(err > LOGIT_RTOL)
        assert bad.size == 0, f"row {i}: {bad.size} logits off, first t={bad[0]} got {g[bad[0]]} ref {r[bad[0]]}"
        if plain:
            m = (np.abs(r) >= a / 8) & (np.abs(r) > 0)
            if m.any():
                pe = np.abs(g[m] - r[m]) / np.abs(r[m])
                worst_plain = max(worst_plain, float(pe.max()))
                assert pe.max() <= LOGIT_RTOL, f"row {i}: plain relative error {pe.max()}"
    return (worst, worst_plain) if plain else worst


def check_topk_vs_oracle_scores(sel, ref, mag, L, k):
    """sel: [n, k] GPU selection (tokens, -1 pad); ref/mag: oracle fp64 scores."""
    for i in range(len(L)):
        n = int(L[i])
        s = sel[i]
        if n <= k:
            assert sorted(s[:n].tolist()) == list(range(n)) and np.all(s[n:] == -1)
            continue
        exact = oracle.topk(ref[i:i + 1, :n], n, k)[0]
        kth = ref[i, exact[-1]]
        band = LOGIT_RTOL * max(abs(kth), mag[i, exact[-1]])
        gs, es = set(s.tolist()), set(exact.tolist())
        assert len(gs) == k and -1 not in gs
        for t in gs ^ es:
            assert abs(ref[i, t] - kth) <= band, f"row {i}: token {t} differs beyond the tie band"


def gpu_topk(logits, ld, L, k, force_path=0, col_blocks=None, bs=0):
    dsa = lib()
    R = L.shape[0]
    out = torch.full((R, k), -7, dtype=torch.int32, device=logits.device)
    nb = 0 if col_blocks is None else col_blocks.shape[1]
    dsa.dsa_topk(logits, ld, L, R, k, out, col_blocks=col_blocks, nb=nb, block_size=bs,
                 force_path=force_path)
    return out


def mla_oracle(mla, bt, next_n, idx, rows=None):
    return oracle.sparse_mla(bits16(mla.q), bits16(mla.kv), 64 * 576, 64, np_(bt), next_n,
                             np_(idx), mla.scale, rows=rows)


def gpu_mla(mla, bt, num_req, next_n, idx, num_pages):
    dsa = lib()
    R, k = idx.shape
    dev = idx.device
    out = torch.full((R, W.MLA_HEADS, W.MLA_DV), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((R, W.MLA_HEADS), float("nan"), dtype=torch.float32, device=dev)
    wsb = dsa.dsa_sparse_mla_workspace_size(R, k)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    dsa.dsa_sparse_mla_decode(mla.q, mla.kv, 64 * 576 * 2, num_pages, bt, num_req, next_n, idx, k,
                              mla.scale, out, lse, ws, wsb)
    return out, lse


def host_hist(logits, L):
    """[R, 4096] counts of the 12-bit order-key prefix of logits[r, :L[r]]."""
    out = np.zeros((len(L), HIST_BINS), np.int64)
    for r, n in enumerate(L):
        u = np.ascontiguousarray(logits[r, :int(n)], dtype=np.float32).view(np.uint32).copy()
        u[(u << np.uint32(1)) == 0] = 0                       # -0.0 ranks as +0.0
        neg = (u & np.uint32(0x80000000)) != 0
        key = np.where(neg, ~u, u | np.uint32(0x80000000))
        out[r] = np.bincount((key >> np.uint32(20)).astype(np.int64), minlength=HIST_BINS)
    return out
