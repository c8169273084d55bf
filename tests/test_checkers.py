"""The acceptance checks of the GPU parity tests accept what the rules allow
and reject what they do not (CPU, on constructed results)."""
from __future__ import annotations

import numpy as np
import pytest

from dsa_check import LOGIT_RTOL, check_logits, check_topk_vs_oracle_scores, host_hist


def _logit_case(seed=0, n=200):
    rng = np.random.default_rng(seed)
    ref = rng.normal(size=(2, n))
    mag = np.abs(ref) + rng.uniform(0.0, 1.0, size=(2, n))  # A >= |ref|
    return ref, mag, np.array([n, n - 37])


def test_logits_accepts_the_reference_and_errors_inside_the_bound():
    ref, mag, L = _logit_case()
    check_logits(ref.astype(np.float32), ref, mag, L)
    scale = np.maximum(np.abs(ref), mag)
    check_logits(ref + 0.9 * LOGIT_RTOL * scale, ref, mag, L)


def test_logits_rejects_one_element_outside_the_bound():
    ref, mag, L = _logit_case()
    got = ref.copy()
    got[1, 5] += 1.1 * LOGIT_RTOL * max(abs(ref[1, 5]), mag[1, 5])
    with pytest.raises(AssertionError, match="row 1"):
        check_logits(got, ref, mag, L)


def test_logits_judges_a_cancelled_sum_by_its_condition_scale():
    # mixed-sign head weights cancel to ~0: the error is judged against A
    ref = np.array([[1e-9, 2.0]])
    mag = np.array([[5.0, 2.0]])
    check_logits(np.array([[1e-9 + 4e-3, 2.0]]), ref, mag, [2])
    with pytest.raises(AssertionError):
        check_logits(np.array([[1e-9 + 6e-3, 2.0]]), ref, mag, [2])


def test_logits_plain_mode_holds_the_stated_relative_bound_where_nothing_cancels():
    # |ref| >= A/8: the plain 1e-3 relative error applies there; a cancelled
    # sum (|ref| < A/8) is still judged by its condition scale only
    ref = np.array([[2.0, 1e-6]])
    mag = np.array([[8.0, 5.0]])
    worst, plain = check_logits(np.array([[2.0 * (1 + 0.5e-3), 1e-6 + 4e-3]]), ref, mag, [2],
                                plain=True)
    assert 0.4e-3 < plain < 0.6e-3 and worst > 0.7e-3
    with pytest.raises(AssertionError, match="plain relative"):
        check_logits(np.array([[2.0 * (1 + 2e-3), 1e-6]]), ref, mag, [2], plain=True)


def test_logits_rejects_non_finite_and_ignores_columns_past_the_row():
    ref, mag, L = _logit_case()
    got = ref.copy()
    got[1, int(L[1]) + 3] = np.nan  # past the row: not compared
    check_logits(got, ref, mag, L)
    got[0, 0] = np.nan
    with pytest.raises(AssertionError, match="non-finite"):
        check_logits(got, ref, mag, L)


def _topk_case():
    n, k = 50, 8
    # tokens 0-6 well above, token 7 the k-th largest (3.0), the rest below it
    ref = np.concatenate([np.linspace(10.0, 4.0, 7), [3.0], np.linspace(2.9, 0.1, n - 8)])[None, :]
    ref[0, 20] = 3.0 - 1e-4            # within 1e-3 of the k-th score: a tie
    mag = np.abs(ref)
    assert sorted(np.argsort(-ref[0], kind="stable")[:k].tolist()) == list(range(k))
    return ref, mag, n, k


def test_topk_accepts_the_exact_set_in_any_order_and_swaps_in_the_tie_band():
    ref, mag, n, k = _topk_case()
    exact = np.argsort(-ref[0], kind="stable")[:k]
    check_topk_vs_oracle_scores(exact[::-1][None, :].copy(), ref, mag, [n], k)
    swapped = exact.copy()
    swapped[swapped == 7] = 20          # the near-tie instead of the k-th
    check_topk_vs_oracle_scores(swapped[None, :], ref, mag, [n], k)


def test_topk_rejects_a_token_outside_the_band_and_duplicates():
    ref, mag, n, k = _topk_case()
    exact = np.argsort(-ref[0], kind="stable")[:k]
    wrong = exact.copy()
    wrong[wrong == 7] = 30              # far below the k-th score
    with pytest.raises(AssertionError, match="tie band"):
        check_topk_vs_oracle_scores(wrong[None, :], ref, mag, [n], k)
    dup = exact.copy()
    dup[0] = dup[1]
    with pytest.raises(AssertionError):
        check_topk_vs_oracle_scores(dup[None, :], ref, mag, [n], k)


def test_topk_short_rows_need_every_token_then_padding():
    ref = np.arange(5.0)[None, :]
    mag = np.abs(ref)
    check_topk_vs_oracle_scores(np.array([[4, 0, 2, 1, 3, -1, -1, -1]]), ref, mag, [5], 8)
    with pytest.raises(AssertionError):
        check_topk_vs_oracle_scores(np.array([[4, 0, 2, 1, 3, 0, -1, -1]]), ref, mag, [5], 8)
    with pytest.raises(AssertionError):
        check_topk_vs_oracle_scores(np.array([[4, 0, 2, 1, -1, -1, -1, -1]]), ref, mag, [5], 8)


def test_host_histogram_bins_follow_the_score_order():
    # the reference histogram of the indexer's fused top-k pass: bins ordered
    # like the scores, -0.0 with +0.0, 1.0 in bin 0xBF8 (sign flipped:
    # 0xBF800000 >> 20), -1.0 in bin 0x407 (all bits flipped: 0x407FFFFF >> 20)
    vals = np.array([-np.inf, -3e38, -2.0, -1.0, -1e-30, -0.0, 0.0, 1e-30, 1.0, 1.0625, 2.0,
                     3e38, np.inf], np.float32)
    bins = [int(np.argmax(host_hist(np.array([[v]], np.float32), [1])[0])) for v in vals]
    assert bins == sorted(bins)
    assert bins[5] == bins[6] == 0x800
    assert bins[8] == 0xBF8 and bins[3] == 0x407
    assert bins[9] == bins[8]  # 1.0625 shares 1.0's three leading mantissa bits
    rng = np.random.default_rng(0)
    x = rng.normal(size=(3, 5000)).astype(np.float32) * 10
    h = host_hist(x, [5000, 4000, 10])
    assert h.sum(axis=1).tolist() == [5000, 4000, 10]
