"""fp64 CPU oracle for the DeepSeek Sparse Attention decode path.

TEST INFRASTRUCTURE ONLY: the slow, plain reference that the CUDA library is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
product package never does, and the two share no code.

The arithmetic lives in ``dsa_oracle.cpp`` (plain C++17, double precision, one
row per task on ``std::thread``); this module only compiles it with g++ and
marshals numpy arrays through ctypes.  Each wrapper cites the passage it
follows:

* ``indexer_logits`` -- Eq. (1), "DeepSeek V3.2-Exp support", section
  "1. Architecture" (lightning indexer), with FP8 keys and a per-token key
  scale (the "128-element k_s value for each token" cache of the same issue).
* ``candidate_expand`` / ``candidate_logits`` -- the vLLM ``sparse_indexer``
  API page (candidate consumers "score only the candidate blocks"; MXFP4 cache
  with "UE8M0-packed granularity-32 scales"; ``sparse_indices`` / ``end``).
* ``topk`` -- the fine-grained token selection of Eq. (2) context: Top-k of the
  index scores (worked example [0.8, 0.3, 0.9, 0.5], k=2 in the issue's cheat
  sheet), by full sort.
* ``sparse_mla`` -- Eq. (2): attention over the selected latents only.

Where the pages leave a step open this module takes the plainest reading:
ties in the top-k go to the lower index; the next_n rows of a request are
consecutive positions, row j seeing ctx_len - (next_n - 1 - j) tokens; packed
e2m1 element 2i is the low nibble of byte i; the per-head q scale multiplies
q inside the ReLU (it is positive, so it may equally be folded into w).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile dsa_oracle.cpp into oracle/_build/liboracle.so with g++."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
        return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def hardware_threads() -> int:
    return int(_load().orc_hardware_threads())


def _threads(n):
    return hardware_threads() if n is None else int(n)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().orc_decode_e4m3(_p(codes), ctypes.c_int64(codes.size), _p(out))
    return out


def decode_e2m1(packed: np.ndarray, n_elems: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    assert packed.size * 2 >= n_elems
    out = np.empty(n_elems, np.float64)
    _load().orc_decode_e2m1(_p(packed), ctypes.c_int64(n_elems), _p(out))
    return out


def decode_ue8m0(codes: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().orc_decode_ue8m0(_p(codes), ctypes.c_int64(codes.size), _p(out))
    return out


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, np.float64)
    _load().orc_decode_bf16(_p(bits), ctypes.c_int64(bits.size), _p(out))
    return out


def row_lengths(ctx_len: np.ndarray, next_n: int) -> np.ndarray:
    """L_r for the flattened rows r = req*next_n + j: row j of a request sees
    ctx_len - (next_n - 1 - j) tokens (its own position included)."""
    ctx = np.asarray(ctx_len, np.int64)
    j = np.arange(next_n, dtype=np.int64)
    L = ctx[:, None] - (next_n - 1 - j)[None, :]
    return np.maximum(L, 0).reshape(-1)


def indexer_logits(q, q_scale, w, k_cache, k_page_stride, k_scale_bytes,
                   s_page_stride, page_tokens, block_table, ctx_len, next_n,
                   rows=None, ld=None, nthreads=None):
    """Eq. (1) over a paged FP8 cache.  Returns (logits, mag), both [nrows, ld]
    float64, NaN where t >= L_r.

    ``k_cache`` / ``k_scale_bytes`` are uint8 views of the cache; the scale of
    slot i of page p is the little-endian f32 at byte p*s_page_stride + 4*i of
    ``k_scale_bytes``."""
    q = np.ascontiguousarray(q, np.uint8)
    R, H, D = q.shape
    q_scale = np.ascontiguousarray(q_scale, np.float32).reshape(R, H)
    w = np.ascontiguousarray(w, np.float32).reshape(R, H)
    bt = np.ascontiguousarray(block_table, np.int32)
    ctx = np.ascontiguousarray(ctx_len, np.int32)
    Ls = row_lengths(ctx, next_n)
    rows = np.arange(R, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    if ld is None:
        ld = int(max(1, Ls.max(initial=1)))
    out = np.full((len(rows), ld), np.nan)
    mag = np.full((len(rows), ld), np.nan)
    bad = _load().orc_indexer_logits(
        _p(q), _p(q_scale), _p(w), _p(np.ascontiguousarray(k_cache)),
        ctypes.c_int64(k_page_stride), _p(np.ascontiguousarray(k_scale_bytes)),
        ctypes.c_int64(s_page_stride), ctypes.c_int(page_tokens), _p(bt),
        ctypes.c_int64(bt.shape[1]), _p(ctx), ctypes.c_int(len(ctx)),
        ctypes.c_int(next_n), ctypes.c_int(H), ctypes.c_int(D), _p(rows),
        ctypes.c_int(len(rows)), _p(out), _p(mag), ctypes.c_int64(ld),
        ctypes.c_int(_threads(nthreads)))
    if bad:
        raise ValueError("oracle: NaN FP8 code in the indexer inputs")
    return out, mag


def candidate_expand(cand, bs, ctx_len, next_n, sparse_bs=None):
    """Sorted candidate blocks and the valid sparse-column count per row.

    With sparse_bs (a divisor of bs; the vLLM ``sparse_indexer`` builder's
    ``sparse_block_kv``, which makes ``num_sparse_blocks = candidate_topk_blocks
    * (candidate_block_size // sparse_block_kv)``), candidate block b of bs
    tokens is first written as its m = bs / sparse_bs consecutive sparse blocks
    b*m .. b*m+m-1 of sparse_bs tokens; the result is then over those."""
    cand = np.ascontiguousarray(cand, np.int32)
    if sparse_bs is not None and sparse_bs != bs:
        if sparse_bs <= 0 or bs % sparse_bs:
            raise ValueError("sparse_bs must divide the candidate block size")
        m = bs // sparse_bs
        R0, nb0 = cand.shape
        cand = (cand.astype(np.int64)[:, :, None] * m + np.arange(m)).reshape(R0, nb0 * m)
        cand = np.ascontiguousarray(cand, np.int32)
        bs = sparse_bs
    R, nb = cand.shape
    ctx = np.ascontiguousarray(ctx_len, np.int32)
    si = np.empty_like(cand)
    end = np.empty(R, np.int32)
    _load().orc_candidate_expand(_p(cand), ctypes.c_int(R), ctypes.c_int(nb),
                                 ctypes.c_int(bs), _p(ctx), ctypes.c_int(next_n),
                                 _p(si), _p(end))
    return si, end


def candidate_logits(q, q_scale, w, k_fp4, k_page_stride, k_sf, sf_page_stride,
                     page_tokens, block_table, next_n, sparse_indices, bs, end,
                     rows=None, ld=None, nthreads=None):
    """Scores of the candidate columns c < end[r] over MXFP4 keys.  Returns
    (logits, mag) [nrows, ld] float64, NaN past end[r]."""
    q = np.ascontiguousarray(q, np.uint8)
    R, H, D = q.shape
    q_scale = np.ascontiguousarray(q_scale, np.float32).reshape(R, H)
    w = np.ascontiguousarray(w, np.float32).reshape(R, H)
    bt = np.ascontiguousarray(block_table, np.int32)
    si = np.ascontiguousarray(sparse_indices, np.int32)
    nb = si.shape[1]
    end = np.ascontiguousarray(end, np.int32)
    rows = np.arange(R, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    if ld is None:
        ld = nb * bs
    out = np.full((len(rows), ld), np.nan)
    mag = np.full((len(rows), ld), np.nan)
    bad = _load().orc_candidate_logits(
        _p(q), _p(q_scale), _p(w), _p(np.ascontiguousarray(k_fp4)),
        ctypes.c_int64(k_page_stride), _p(np.ascontiguousarray(k_sf)),
        ctypes.c_int64(sf_page_stride), ctypes.c_int(page_tokens), _p(bt),
        ctypes.c_int64(bt.shape[1]), ctypes.c_int(next_n), ctypes.c_int(H),
        ctypes.c_int(D), _p(si), ctypes.c_int(nb), ctypes.c_int(bs), _p(end),
        _p(rows), ctypes.c_int(len(rows)), _p(out), _p(mag), ctypes.c_int64(ld),
        ctypes.c_int(_threads(nthreads)))
    if bad:
        raise ValueError("oracle: NaN code in the candidate-path inputs")
    return out, mag


def topk(scores, lengths, k, col_blocks=None, bs=0, nthreads=None):
    """Top-k column (or token) indices per row by full sort: score descending,
    index ascending; -1 pads rows shorter than k."""
    s = np.ascontiguousarray(scores, np.float64)
    if s.ndim == 1:
        s = s[None, :]
    n = s.shape[0]
    L = np.ascontiguousarray(np.broadcast_to(np.asarray(lengths, np.int32), (n,)))
    out = np.empty((n, k), np.int32)
    cb = None if col_blocks is None else np.ascontiguousarray(col_blocks, np.int32)
    nb = 0 if cb is None else cb.shape[1]
    _load().orc_topk(_p(s), ctypes.c_int64(s.shape[1]), _p(L), ctypes.c_int(n),
                     ctypes.c_int(k), _p(cb), ctypes.c_int(nb), ctypes.c_int(bs),
                     _p(out), ctypes.c_int(_threads(nthreads)))
    return out


def sparse_mla(q_bits, kv_bits, kv_page_stride, page_tokens, block_table, next_n,
               idx, scale, dv=512, rows=None, nthreads=None):
    """Eq. (2) over the selected latents.  q_bits [R, Hq, Dqk] and kv_bits
    (pages of page_tokens x Dqk) are bf16 bit patterns (uint16).  Returns
    (out [nrows, Hq, dv], lse [nrows, Hq]) float64."""
    q = np.ascontiguousarray(q_bits, np.uint16)
    R, Hq, Dqk = q.shape
    kv = np.ascontiguousarray(kv_bits, np.uint16)
    bt = np.ascontiguousarray(block_table, np.int32)
    idx = np.ascontiguousarray(idx, np.int32)
    k = idx.shape[1]
    rows = np.arange(R, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    out = np.empty((len(rows), Hq, dv), np.float64)
    lse = np.empty((len(rows), Hq), np.float64)
    _load().orc_sparse_mla(_p(q), _p(kv), ctypes.c_int64(kv_page_stride),
                           ctypes.c_int(page_tokens), _p(bt), ctypes.c_int64(bt.shape[1]),
                           ctypes.c_int(next_n), _p(idx), ctypes.c_int(k),
                           ctypes.c_int(Hq), ctypes.c_int(Dqk), ctypes.c_int(dv),
                           ctypes.c_double(scale), _p(rows), ctypes.c_int(len(rows)),
                           _p(out), _p(lse), ctypes.c_int(_threads(nthreads)))
    return out, lse


def layer_sources(keep, mli):
    """For each layer of a decode step, the layer whose indexer selection its
    attention uses, following the Multi-layer Indexer abstract of the "JEV
    Paper Radar" efficiency digest (2026-11-04):

    * IndexCache: only the layers with keep[l] set run an indexer; a layer
      without one reuses the selection of the latest earlier indexer layer;
    * MLI (mli true): a layer attends the selection of the previous indexer
      layer instead of its own, so its own indexer (if it keeps one) can run
      concurrently with its attention.

    Readings: "previous" means the latest indexer layer strictly before the
    layer; the first layer has no previous one, so it must keep its indexer
    and attends its own selection (the abstract does not say).  Plain Python
    over a few layers: this is a schedule, not arithmetic."""
    keep = [bool(x) for x in keep]
    if not keep or not keep[0]:
        raise ValueError("layer 0 must keep its indexer")
    out = []
    latest = -1  # the latest indexer layer before the current one
    for layer, kept in enumerate(keep):
        if mli and layer > 0:
            out.append(latest)
        else:
            out.append(layer if kept else latest)
        if kept:
            latest = layer
    return out


def prefill_chunk_plan(q_lens, ctx_lens, budget_bytes, min_cols=0):
    """Splits a batch of prefill queries into chunks whose f32 logits scratch
    [rows, ld] fits budget_bytes, as the vLLM ``sparse_indexer`` builder's
    prefill chunker does ("budgets fp32 [rows, seq_len]"; ``min_split_seq_len``
    makes it "size chunks as if every row were this wide").

    Readings: the rows are taken in order (request by request, position by
    position); a row of request b needs a logits row of max(ctx_lens[b],
    min_cols) columns, rounded up to a multiple of 4; a chunk's scratch is
    rows x (its widest row) x 4 bytes; rows are added to the current chunk
    while that stays within the budget, and a row that alone exceeds it is a
    chunk by itself.  Returns pieces (chunk, request, row_begin, row_end):
    each chunk is a run of consecutive pieces, each piece a run of one
    request's rows."""
    pieces = []
    chunk, rows, width = 0, 0, 0
    for b, (n, c) in enumerate(zip(q_lens, ctx_lens)):
        w = (max(int(c), int(min_cols)) + 3) // 4 * 4
        for j in range(int(n)):
            if rows > 0 and (rows + 1) * max(width, w) * 4 > budget_bytes:
                chunk += 1
                rows, width = 0, 0
            if pieces and pieces[-1][0] == chunk and pieces[-1][1] == b:
                pieces[-1][3] = j + 1
            else:
                pieces.append([chunk, b, j, j + 1])
            rows += 1
            width = max(width, w)
    return [tuple(p) for p in pieces]
