"""Thin Python binding of the C ABI in include/dsa.h (ctypes).

Every function here has the name of the C entry point it wraps and does
argument marshalling only: tensors become device pointers, the stream defaults
to torch's current stream, a non-zero status raises DsaError with the library's
message.  All arithmetic runs in the CUDA kernels of libdsa.so; there is no
other code path.  Importing this module raises ImportError if libdsa.so has not
been built (``deepseek_sparse_attention_02_gb300._build.build()``).

Pointer arguments accept a torch tensor (its data_ptr()), a plain int (a raw
device address, e.g. ``cache.data_ptr() + 8192`` for the scale block of the
canonical FP8 page) or None (NULL).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float

_SIGS = {
    "dsa_version": ([], _I),
    "dsa_last_error": ([], ctypes.c_char_p),
    "dsa_get_device_error": ([_P, ctypes.POINTER(ctypes.c_uint32), _I], _I),
    "dsa_indexer_logits": ([_P, _P, _P, _P, _I64, _P, _I64, _I, _P, _I64, _P, _I, _I, _P, _I64,
                            _P], _I),
    "dsa_topk": ([_P, _I64, _P, _I, _I, _P, _I, _I, _P, _I, _P], _I),
    "dsa_score_hist_size": ([_I], _SZ),
    "dsa_indexer_logits_hist": ([_P, _P, _P, _P, _I64, _P, _I64, _I, _P, _I64, _P, _I, _I, _P,
                                 _I64, _P, _P], _I),
    "dsa_topk_hist": ([_P, _I64, _P, _I, _I, _P, _P, _I, _P], _I),
    "dsa_sparse_mla_workspace_size": ([_I, _I], _SZ),
    "dsa_sparse_mla_decode": ([_P, _P, _I64, _I, _P, _I64, _I, _I, _P, _I, _F, _P, _P, _P, _SZ,
                               _P], _I),
    "dsa_sparse_mla_static_scratch_bytes": ([], _SZ),
    "dsa_sparse_mla_decode_static": ([_P, _P, _I64, _I, _P, _I64, _I, _I, _P, _I, _F, _P, _P, _P],
                                     _I),
    "dsa_candidate_schedule_size": ([_I], _SZ),
    "dsa_candidate_expand": ([_P, _I, _I, _I, _P, _I, _P, _P, _P, _SZ, _P], _I),
    "dsa_candidate_logits": ([_P, _P, _P, _P, _I64, _P, _I64, _I, _P, _I64, _I, _I, _P, _I, _I,
                              _P, _P, _SZ, _P, _I64, _P], _I),
    "dsa_topk_bf16": ([_P, _I64, _P, _I, _I, _P, _I, _I, _P, _I, _P], _I),
    "dsa_candidate_logits_bf16": ([_P, _P, _P, _P, _I64, _P, _I64, _I, _P, _I64, _I, _I, _P, _I,
                                   _I, _P, _P, _SZ, _P, _I64, _P], _I),
    "dsa_prefill_chunk_plan": ([_P, _P, _I, _I64, _I64, _P, _I, _P], _I),
    "dsa_indexer_logits_varlen": ([_P, _P, _P, _P, _I64, _P, _I64, _I, _P, _I64, _I, _P, _P, _P,
                                   _I, _I, _I, _P, _I64, _P], _I),
    "dsa_varlen_row_lengths": ([_P, _P, _I, _I, _P, _P], _I),
    "dsa_sparse_mla_decode_varlen": ([_P, _P, _I64, _I, _P, _I64, _I, _P, _I, _P, _I, _F, _P, _P,
                                      _P, _SZ, _P], _I),
    "dsa_layer_sources": ([_P, _I, _I, _P], _I),
    "dsa_decode_layers_workspace_size": ([_I, _I64, _I], _SZ),
    "dsa_decode_layers": ([_P, _I, _P, _I, _I64, _I64, _I64, _I, _P, _I64, _P, _P, _I, _I, _I, _F,
                           _I64, _P, _SZ, _P, _P], _I),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res

EXPORTED = tuple(_SIGS)

STATUS = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED", 3: "DSA_ERR_WORKSPACE",
          4: "DSA_ERR_CUDA", 5: "DSA_ERR_DEVICE"}
DEVERR_TIMEOUT, DEVERR_BAD_PAGE, DEVERR_BAD_INDEX, DEVERR_CAPACITY = 1, 2, 4, 8
DSA_MAX_TOPK = 8192  # include/dsa.h
DSA_HIST_BINS = 4096


class DsaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return None
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int):
    if st != 0:
        raise DsaError(st, dsa_last_error())


def lib() -> ctypes.CDLL:
    return _lib


def dsa_version() -> int:
    return _lib.dsa_version()


def dsa_last_error() -> str:
    return (_lib.dsa_last_error() or b"").decode()


def dsa_get_device_error(stream=None, clear: bool = True) -> int:
    bits = ctypes.c_uint32(0)
    _check(_lib.dsa_get_device_error(_stream(stream), ctypes.byref(bits), int(clear)))
    return bits.value


def dsa_indexer_logits(q_fp8, q_scale, weights, k_cache, k_page_stride, k_scale, s_page_stride,
                       num_pages, block_table, ctx_len, num_req, next_n, logits, ld,
                       stream=None):
    """Eq. (1) logits; see include/dsa.h.  block_table is [num_req, bt_stride]."""
    bt_stride = block_table.shape[1]
    _check(_lib.dsa_indexer_logits(_ptr(q_fp8), _ptr(q_scale), _ptr(weights), _ptr(k_cache),
                                   k_page_stride, _ptr(k_scale), s_page_stride, num_pages,
                                   _ptr(block_table), bt_stride, _ptr(ctx_len), num_req, next_n,
                                   _ptr(logits), ld, _stream(stream)))


def dsa_topk(logits, ld, row_len, R, k, out_idx, col_blocks=None, nb=0, block_size=0,
             force_path=0, stream=None):
    _check(_lib.dsa_topk(_ptr(logits), ld, _ptr(row_len), R, k, _ptr(col_blocks), nb, block_size,
                         _ptr(out_idx), force_path, _stream(stream)))


def dsa_score_hist_size(R: int) -> int:
    return _lib.dsa_score_hist_size(R)


def dsa_indexer_logits_hist(q_fp8, q_scale, weights, k_cache, k_page_stride, k_scale,
                            s_page_stride, num_pages, block_table, ctx_len, num_req, next_n, logits,
                            ld, hist, stream=None):
    """dsa_indexer_logits that also adds per-row score histograms into hist."""
    bt_stride = block_table.shape[1]
    _check(_lib.dsa_indexer_logits_hist(_ptr(q_fp8), _ptr(q_scale), _ptr(weights), _ptr(k_cache),
                                        k_page_stride, _ptr(k_scale), s_page_stride, num_pages,
                                        _ptr(block_table), bt_stride, _ptr(ctx_len), num_req,
                                        next_n, _ptr(logits), ld, _ptr(hist), _stream(stream)))


def dsa_topk_hist(logits, ld, row_len, R, k, hist, out_idx, force_path=0, stream=None):
    """dsa_topk placing its cutoff from the histograms (and clearing them)."""
    _check(_lib.dsa_topk_hist(_ptr(logits), ld, _ptr(row_len), R, k, _ptr(hist), _ptr(out_idx),
                              force_path, _stream(stream)))


def dsa_topk_bf16(logits, ld, row_len, R, k, out_idx, col_blocks=None, nb=0, block_size=0,
                  force_path=0, stream=None):
    _check(_lib.dsa_topk_bf16(_ptr(logits), ld, _ptr(row_len), R, k, _ptr(col_blocks), nb,
                              block_size, _ptr(out_idx), force_path, _stream(stream)))


def dsa_sparse_mla_workspace_size(R: int, k: int) -> int:
    return int(_lib.dsa_sparse_mla_workspace_size(R, k))


def dsa_sparse_mla_decode(q, kv_cache, kv_page_stride, num_pages, block_table, num_req, next_n,
                          idx, k, sm_scale, out, lse=None, workspace=None, workspace_bytes=0,
                          stream=None):
    bt_stride = block_table.shape[1]
    _check(_lib.dsa_sparse_mla_decode(_ptr(q), _ptr(kv_cache), kv_page_stride, num_pages,
                                      _ptr(block_table), bt_stride, num_req, next_n, _ptr(idx), k,
                                      float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                      workspace_bytes, _stream(stream)))


def dsa_sparse_mla_static_scratch_bytes() -> int:
    return int(_lib.dsa_sparse_mla_static_scratch_bytes())


def dsa_sparse_mla_decode_static(q, kv_cache, kv_page_stride, num_pages, block_table, num_req,
                                 next_n, idx, k, sm_scale, out, lse=None, stream=None):
    """dsa_sparse_mla_decode without a workspace, for callers that cannot
    allocate device memory; its split-K scratch is a static array inside the
    library (see include/dsa.h)."""
    bt_stride = block_table.shape[1]
    _check(_lib.dsa_sparse_mla_decode_static(_ptr(q), _ptr(kv_cache), kv_page_stride, num_pages,
                                             _ptr(block_table), bt_stride, num_req, next_n,
                                             _ptr(idx), k, float(sm_scale), _ptr(out), _ptr(lse),
                                             _stream(stream)))


def dsa_candidate_schedule_size(R: int) -> int:
    return int(_lib.dsa_candidate_schedule_size(R))


def dsa_candidate_expand(cand, R, nb, block_size, ctx_len, next_n, sparse_indices, end,
                         schedule, schedule_bytes, stream=None):
    _check(_lib.dsa_candidate_expand(_ptr(cand), R, nb, block_size, _ptr(ctx_len), next_n,
                                     _ptr(sparse_indices), _ptr(end), _ptr(schedule),
                                     schedule_bytes, _stream(stream)))


def dsa_candidate_logits(q_fp8, q_scale, weights, k_fp4, k_page_stride, k_sf, sf_page_stride,
                         num_pages, block_table, num_req, next_n, sparse_indices, nb, block_size,
                         end, schedule, schedule_bytes, logits, ld, stream=None):
    bt_stride = block_table.shape[1]
    _check(_lib.dsa_candidate_logits(_ptr(q_fp8), _ptr(q_scale), _ptr(weights), _ptr(k_fp4),
                                     k_page_stride, _ptr(k_sf), sf_page_stride, num_pages,
                                     _ptr(block_table), bt_stride, num_req, next_n,
                                     _ptr(sparse_indices), nb, block_size, _ptr(end),
                                     _ptr(schedule), schedule_bytes, _ptr(logits), ld,
                                     _stream(stream)))



class DsaLayer(ctypes.Structure):
    """One record of dsa_decode_layers (struct dsa_layer of include/dsa.h)."""
    _fields_ = [("q_fp8", _P), ("q_scale", _P), ("weights", _P), ("k_cache", _P),
                ("k_scale", _P), ("q", _P), ("kv_cache", _P), ("out", _P), ("lse", _P)]


def dsa_layer_sources(keep_indexer, mli: bool) -> list:
    """Host-only: the layer whose selection each layer attends."""
    n = len(keep_indexer)
    keep = (ctypes.c_uint8 * n)(*[1 if x else 0 for x in keep_indexer])
    src = (ctypes.c_int32 * n)()
    _check(_lib.dsa_layer_sources(ctypes.cast(keep, _P), n, int(bool(mli)), ctypes.cast(src, _P)))
    return list(src)


def dsa_decode_layers_workspace_size(R: int, ld: int, k: int) -> int:
    return int(_lib.dsa_decode_layers_workspace_size(R, ld, k))


def dsa_decode_layers(layers, keep_indexer, mli, k_page_stride, s_page_stride, kv_page_stride,
                      num_pages, block_table, ctx_len, row_len, num_req, next_n, k, sm_scale,
                      ld, workspace, workspace_bytes, stream=None, side_stream=None):
    """layers: a sequence of dicts with the dsa_layer fields (tensors, ints or
    None); keep_indexer: a sequence of bools."""
    n = len(layers)
    recs = (DsaLayer * n)()
    for i, L in enumerate(layers):
        for f, _ in DsaLayer._fields_:
            setattr(recs[i], f, _ptr(L.get(f)))
    keep = (ctypes.c_uint8 * n)(*[1 if x else 0 for x in keep_indexer])
    bt_stride = block_table.shape[1]
    side = None if side_stream is None else _stream(side_stream)
    _check(_lib.dsa_decode_layers(ctypes.cast(recs, _P), n, ctypes.cast(keep, _P), int(bool(mli)),
                                  k_page_stride, s_page_stride, kv_page_stride, num_pages,
                                  _ptr(block_table), bt_stride, _ptr(ctx_len), _ptr(row_len),
                                  num_req, next_n, k, float(sm_scale), ld, _ptr(workspace),
                                  workspace_bytes, _stream(stream), side))


def dsa_candidate_logits_bf16(q_fp8, q_scale, weights, k_fp4, k_page_stride, k_sf,
                              sf_page_stride, num_pages, block_table, num_req, next_n,
                              sparse_indices, nb, block_size, end, schedule, schedule_bytes,
                              logits, ld, stream=None):
    bt_stride = block_table.shape[1]
    _check(_lib.dsa_candidate_logits_bf16(_ptr(q_fp8), _ptr(q_scale), _ptr(weights), _ptr(k_fp4),
                                          k_page_stride, _ptr(k_sf), sf_page_stride, num_pages,
                                          _ptr(block_table), bt_stride, num_req, next_n,
                                          _ptr(sparse_indices), nb, block_size, _ptr(end),
                                          _ptr(schedule), schedule_bytes, _ptr(logits), ld,
                                          _stream(stream)))


def dsa_prefill_chunk_plan(q_len, ctx_len, budget_bytes: int, min_cols: int = 0) -> list:
    """Host-only: [(chunk, request, row_begin, row_end), ...]."""
    n = len(q_len)
    ql = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in q_len])
    cl = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in ctx_len])
    cap = sum(int(x) for x in q_len) + 1
    out = (ctypes.c_int32 * (4 * cap))()
    npc = ctypes.c_int(0)
    _check(_lib.dsa_prefill_chunk_plan(ctypes.cast(ql, _P), ctypes.cast(cl, _P), n, budget_bytes,
                                       min_cols, ctypes.cast(out, _P), cap, ctypes.byref(npc)))
    return [tuple(out[4 * i:4 * i + 4]) for i in range(npc.value)]


def dsa_indexer_logits_varlen(q_fp8, q_scale, weights, k_cache, k_page_stride, k_scale,
                              s_page_stride, num_pages, block_table, bt_rows, ctx_len, cu_rows,
                              num_entries, max_rows, total_rows, logits, ld, stream=None):
    bt_num_rows, bt_stride = block_table.shape
    _check(_lib.dsa_indexer_logits_varlen(_ptr(q_fp8), _ptr(q_scale), _ptr(weights),
                                          _ptr(k_cache), k_page_stride, _ptr(k_scale),
                                          s_page_stride, num_pages, _ptr(block_table), bt_stride,
                                          bt_num_rows, _ptr(bt_rows), _ptr(ctx_len),
                                          _ptr(cu_rows), num_entries, max_rows, total_rows,
                                          _ptr(logits), ld, _stream(stream)))


def dsa_varlen_row_lengths(ctx_len, cu_rows, num_entries, total_rows, row_len, stream=None):
    _check(_lib.dsa_varlen_row_lengths(_ptr(ctx_len), _ptr(cu_rows), num_entries, total_rows,
                                       _ptr(row_len), _stream(stream)))


def dsa_sparse_mla_decode_varlen(q, kv_cache, kv_page_stride, num_pages, block_table, row_bt, R,
                                 idx, k, sm_scale, out, lse, workspace, workspace_bytes,
                                 stream=None):
    bt_num_rows, bt_stride = block_table.shape
    _check(_lib.dsa_sparse_mla_decode_varlen(_ptr(q), _ptr(kv_cache), kv_page_stride, num_pages,
                                             _ptr(block_table), bt_stride, bt_num_rows,
                                             _ptr(row_bt), R, _ptr(idx), k, float(sm_scale),
                                             _ptr(out), _ptr(lse), _ptr(workspace),
                                             workspace_bytes, _stream(stream)))
