"""The multi-layer decode step with the IndexCache / Multi-layer Indexer (MLI)
selection schedules (dsa_decode_layers; the MLI abstract of the "JEV Paper
Radar" efficiency digest, 2026-11-04).

CPU: the library's schedule (dsa_layer_sources) equals the oracle's, and bad
arguments are rejected on the host.  GPU: every layer's output equals the
single calls made in the schedule's order, on one stream and on two, within
the sparse MLA bound (the top-k returns its set in no fixed order, and the
attention's running max and f32 sums follow the order of the selected
tokens, which moves results by a few bf16 ulps); and on sampled rows the
attention of each layer matches the oracle's sparse MLA over the selection of
the layer the oracle's schedule names, that selection itself agreeing with the
oracle's indexer scores."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from dsa_check import (LSE_ATOL, MLA_ATOL, check_topk_vs_oracle_scores, gpu_indexer, gpu_mla,
                       gpu_topk, ld_for, mla_oracle, np_, oracle_indexer, row_lens)
from deepseek_sparse_attention_02_gb300 import workloads as W

CTX = [3000, 4500, 6100]
NEXT_N = 2
K = 512
N_LAYERS = 5


def _dsa():
    from deepseek_sparse_attention_02_gb300 import dsa
    return dsa


# --------------------------------------------------------------------- CPU --
def test_layer_sources_matches_oracle():
    dsa = _dsa()
    rng = np.random.default_rng(21)
    for _ in range(300):
        n = int(rng.integers(1, 40))
        keep = rng.integers(0, 2, n)
        keep[0] = 1
        for mli in (False, True):
            assert dsa.dsa_layer_sources(keep.tolist(), mli) == oracle.layer_sources(keep, mli)


def test_decode_layers_host_validation():
    dsa = _dsa()
    lib = dsa.lib()
    rec = (dsa.DsaLayer * 2)()
    for r in rec:
        for f, _ in dsa.DsaLayer._fields_:
            setattr(r, f, 256)
    keep = (ctypes.c_uint8 * 2)(1, 1)
    args = dict(k_page_stride=8448, s_page_stride=8448, kv_page_stride=73728, num_pages=4,
                block_table=256, bt_stride=4, ctx_len=256, row_len=256, num_req=1, next_n=2,
                k=16, sm_scale=0.1, ld=64, workspace=256, workspace_bytes=1 << 30)

    def call(rec_=rec, keep_=keep, **over):
        a = dict(args, **over)
        return lib.dsa_decode_layers(ctypes.cast(rec_, ctypes.c_void_p), 2,
                                     ctypes.cast(keep_, ctypes.c_void_p), 1, a["k_page_stride"],
                                     a["s_page_stride"], a["kv_page_stride"], a["num_pages"],
                                     a["block_table"], a["bt_stride"], a["ctx_len"], a["row_len"],
                                     a["num_req"], a["next_n"], a["k"], a["sm_scale"], a["ld"],
                                     a["workspace"], a["workspace_bytes"], None, None)

    assert call(keep_=(ctypes.c_uint8 * 2)(0, 1)) == 1
    assert "layer 0" in dsa.dsa_last_error()
    assert call(kv_page_stride=1000) == 1
    assert call(k=0) == 1
    assert call(ld=63) == 1
    assert call(workspace_bytes=16) == 3
    rec2 = (dsa.DsaLayer * 2)()
    ctypes.memmove(rec2, rec, ctypes.sizeof(rec))
    rec2[1].q = 258  # misaligned attention query of layer 1
    assert call(rec_=rec2) == 1
    assert "layer 1" in dsa.dsa_last_error()
    rec3 = (dsa.DsaLayer * 2)()
    ctypes.memmove(rec3, rec, ctypes.sizeof(rec))
    rec3[1].k_cache = None  # layer 1 keeps an indexer but has no key cache
    assert call(rec_=rec3) == 1
    assert dsa.dsa_decode_layers_workspace_size(6, 6104, 512) >= 6 * 6104 * 4 + 2 * 6 * 512 * 4
    with pytest.raises(dsa.DsaError):
        dsa.dsa_layer_sources([0, 1], False)


# --------------------------------------------------------------------- GPU --
def _model(seed=0):
    """N_LAYERS layers sharing one page layout and block table, each with its
    own indexer query, FP8 key cache, attention query and latent cache."""
    base = W.make_indexer_case(CTX, next_n=NEXT_N, seed=seed, device="cuda")
    layout = base.layout
    idx_cases, mla_cases = [], []
    for l in range(N_LAYERS):
        idx_cases.append(base if l == 0 else
                         W.make_indexer_case(CTX, next_n=NEXT_N, seed=seed + 10 + l,
                                             device="cuda", layout=layout))
        mla_cases.append(W.make_mla_case(base.rows, layout.num_pages, seed=seed + 20 + l,
                                         device="cuda"))
    return layout, idx_cases, mla_cases


def _run_schedule(layout, idx_cases, mla_cases, keep, mli, side):
    dsa = _dsa()
    R = idx_cases[0].rows
    L = row_lens(idx_cases[0])
    ld = ld_for(int(L.max()))
    layers, outs = [], []
    for c, m in zip(idx_cases, mla_cases):
        out = torch.full((R, W.MLA_HEADS, W.MLA_DV), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        lse = torch.full((R, W.MLA_HEADS), float("nan"), device="cuda")
        outs.append((out, lse))
        layers.append(dict(q_fp8=c.q, q_scale=c.q_scale, weights=c.w, k_cache=c.cache,
                           k_scale=c.cache.data_ptr() + W.FP8_KEY_BYTES, q=m.q, kv_cache=m.kv,
                           out=out, lse=lse))
    wsb = dsa.dsa_decode_layers_workspace_size(R, ld, K)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    side_stream = torch.cuda.Stream() if side else None
    dsa.dsa_decode_layers(layers, keep, mli, W.FP8_PAGE_BYTES, W.FP8_PAGE_BYTES, 64 * 576 * 2,
                          layout.num_pages, layout.block_table, layout.ctx_len, L, len(CTX),
                          NEXT_N, K, mla_cases[0].scale, ld, ws, wsb,
                          side_stream=side_stream)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error() == 0
    return outs


def _replay(layout, idx_cases, mla_cases, keep, mli):
    """The same step as single calls: each kept layer's indexer and top-k, then
    every layer's attention over the selection the oracle's schedule names."""
    L = row_lens(idx_cases[0])
    ld = ld_for(int(L.max()))
    sels = {}
    for j, kept in enumerate(keep):
        if kept:
            logits, _ = gpu_indexer(idx_cases[j], ld)
            sels[j] = gpu_topk(logits, ld, L, K)
    src = oracle.layer_sources(keep, mli)
    outs = [gpu_mla(mla_cases[l], layout.block_table, len(CTX), NEXT_N, sels[src[l]],
                    layout.num_pages) for l in range(len(keep))]
    torch.cuda.synchronize()
    return outs, sels, src


@pytest.mark.gpu
@pytest.mark.parametrize("keep", [[1, 1, 1, 1, 1], [1, 0, 1, 0, 1], [1, 0, 0, 1, 1]])
@pytest.mark.parametrize("mli", [False, True])
@pytest.mark.parametrize("side", [False, True])
def test_decode_layers_equals_single_calls(keep, mli, side):
    layout, idx_cases, mla_cases = _model()
    got = _run_schedule(layout, idx_cases, mla_cases, keep, mli, side)
    ref, _, _ = _replay(layout, idx_cases, mla_cases, keep, mli)
    for l in range(N_LAYERS):
        # same selected set, maybe in another order (so another running max and
        # bf16 P): the results agree to a few bf16 ulps, within the sparse MLA
        # acceptance bound and a tenth of what another layer's selection changes
        # (the sampled-row test asserts that gap)
        assert (got[l][0].float() - ref[l][0].float()).abs().max() <= MLA_ATOL, f"layer {l} out"
        assert (got[l][1] - ref[l][1]).abs().max() <= LSE_ATOL, f"layer {l} lse"


@pytest.mark.gpu
def test_decode_layers_oracle_sampled_rows():
    keep, mli = [1, 0, 1, 1, 0], True
    layout, idx_cases, mla_cases = _model(seed=3)
    got = _run_schedule(layout, idx_cases, mla_cases, keep, mli, side=True)
    _, sels, src = _replay(layout, idx_cases, mla_cases, keep, mli)
    rows = np.array([0, 3, 5], np.int32)
    L = np_(row_lens(idx_cases[0]))
    # each source layer's selection agrees with the oracle's indexer scores
    for j in sorted(set(src)):
        ref, mag = oracle_indexer(idx_cases[j], rows=rows)
        check_topk_vs_oracle_scores(np_(sels[j])[rows], ref, mag, L[rows], K)
    # each layer attended the selection of the layer the oracle's schedule names
    for l in range(N_LAYERS):
        o_ref, l_ref = mla_oracle(mla_cases[l], layout.block_table, NEXT_N, sels[src[l]],
                                  rows=rows)
        assert np.abs(np_(got[l][0].float())[rows] - o_ref).max() <= MLA_ATOL, f"layer {l}"
        assert np.abs(np_(got[l][1])[rows] - l_ref).max() <= LSE_ATOL, f"layer {l}"
        if src[l] != l and keep[l]:
            # the check can tell: the layer's own selection gives another result
            o_own, _ = mla_oracle(mla_cases[l], layout.block_table, NEXT_N, sels[l], rows=rows)
            assert np.abs(np_(got[l][0].float())[rows] - o_own).max() > 10 * MLA_ATOL
