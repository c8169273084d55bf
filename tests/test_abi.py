"""The C-ABI library loads without a GPU, exports every entry point that
include/dsa.h declares, and rejects bad arguments on the host (no kernel is
launched by these tests)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__ as g
    from deepseek_sparse_attention_02_gb300 import _build
    _build.build()
    from deepseek_sparse_attention_02_gb300 import dsa as mod
    return mod


def declared():
    src = open(os.path.join(ROOT, "include", "dsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(dsa):
    names = declared()
    assert len(names) >= 10
    lib = ctypes.CDLL(dsa.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dsa.EXPORTED)


def test_version_and_sizes(dsa):
    assert dsa.dsa_version() == 200
    assert dsa.dsa_score_hist_size(64) == 64 * 4096 * 4
    assert dsa.dsa_score_hist_size(0) == 0
    assert dsa.dsa_sparse_mla_workspace_size(64, 2048) == 0          # one wave, no split
    assert dsa.dsa_sparse_mla_workspace_size(1, 2048) > 0            # split-K partials
    assert dsa.dsa_candidate_schedule_size(64) >= 65 * 4
    assert dsa.dsa_candidate_schedule_size(0) == 0


def test_host_validation_without_gpu(dsa):
    with pytest.raises(dsa.DsaError, match="INVALID_ARG"):
        dsa.dsa_topk(None, 2048, None, 1, 16, None)
    lib = dsa.lib()
    # k out of range, misaligned logits: rejected before any device call
    assert lib.dsa_topk(16, 2048, 16, 1, 0, None, 0, 0, 16, 0, None) == 1
    assert lib.dsa_topk(18, 2048, 16, 1, 8, None, 0, 0, 16, 0, None) == 1
    assert "16-byte" in dsa.dsa_last_error()
    # indexer: NULL pointers, then a bad page stride
    assert lib.dsa_indexer_logits(None, 16, 16, 16, 8448, 16, 8448, 1, 16, 1, 16, 1, 1, 16, 4,
                                  None) == 1
    assert lib.dsa_indexer_logits(16, 16, 16, 16, 100, 16, 8448, 1, 16, 1, 16, 1, 1, 16, 4,
                                  None) == 1
    # candidate block size must be the 64-token page
    assert lib.dsa_candidate_expand(16, 1, 4, 32, 16, 1, 16, 16, 16, 64, None) == 2
    # an empty batch is a no-op that needs no device
    assert lib.dsa_indexer_logits(16, 16, 16, 16, 8448, 16, 8448, 1, 16, 1, 16, 0, 1, 16, 4,
                                  None) == 0

    # candidate logits read the MXFP4 keys with a 4-bit tensor copy: k_fp4 must
    # be 32-byte aligned and the key page stride a multiple of 32
    cand = lambda k_fp4, stride: lib.dsa_candidate_logits(  # noqa: E731
        64, 64, 64, k_fp4, stride, 64, 4352, 1, 64, 1, 0, 1, 64, 8, 64, 64, 64, 16, 64, 512, None)
    assert cand(48, 4352) == 1
    assert "32-byte" in dsa.dsa_last_error()
    assert cand(64, 4368) == 1
    assert cand(64, 4352) == 0  # no rows: nothing to do, no device needed

    # fused-histogram pair: hist is required and 16-byte aligned; the indexer
    # builds histograms for decode shapes only (next_n <= 2)
    assert lib.dsa_topk_hist(16, 2048, 16, 1, 8, None, 16, 0, None) == 1
    assert lib.dsa_topk_hist(16, 2048, 16, 1, 8, 20, 16, 0, None) == 1
    assert lib.dsa_indexer_logits_hist(16, 16, 16, 16, 8448, 16, 8448, 1, 16, 1, 16, 1, 1, 16, 4,
                                       None, None) == 1
    assert lib.dsa_indexer_logits_hist(16, 16, 16, 16, 8448, 16, 8448, 1, 16, 1, 16, 1, 3, 16, 4,
                                       16, None) == 2
    assert lib.dsa_indexer_logits_hist(16, 16, 16, 16, 8448, 16, 8448, 1, 16, 1, 16, 0, 2, 16, 4,
                                       16, None) == 0
