"""The comparison rules the GPU parity tests apply (tests/helpers.py), checked on
the CPU with crafted rows: identical outputs pass; a selected position whose
oracle score lies within the tolerance of the K-th score may replace another
one (counted); any other difference, an order that contradicts the oracle
scores by more than the tolerance, a wrong physical slot or a wrong short row
fails; the score bound follows its formula."""
from types import SimpleNamespace

import numpy as np
import pytest

from tests import helpers as H

K = 4


def _problem(length):
    return SimpleNamespace(topk=K, row_req=np.array([0], np.int32),
                           row_start=np.array([0], np.int32),
                           row_end=np.array([length], np.int32),
                           page_table=np.array([[5, 9]], np.int32))


def _phys(p, raw):
    return np.where(raw >= 0, p.page_table[0, np.maximum(raw, 0) // 64] * 64 + raw % 64, -1)


SCORES = np.array([0.5, 3.0, 1.0, 2.0, 0.25, 2.5, 1.0 + 5e-6, 0.1, -1.0, 0.0])
ORACLE = np.array([1, 5, 3, 6])          # top 4; the K-th score is 1.0 + 5e-6


def _cmp(p, g_raw, o_raw=ORACLE, g_phys=None):
    g_raw = np.asarray(g_raw)
    g_phys = _phys(p, g_raw) if g_phys is None else np.asarray(g_phys)
    return H.compare_rows(p, [0], g_raw[None], g_phys[None], o_raw[None], _phys(p, o_raw)[None],
                          {0: SCORES})


def test_identical_rows_pass():
    assert _cmp(_problem(10), ORACLE) == 0


def test_boundary_swap_within_tolerance_is_counted():
    # position 2 (score 1.0) is within 1e-5 relative of the K-th score 1.0 + 5e-6
    assert _cmp(_problem(10), np.array([1, 5, 3, 2])) == 1


def test_swap_outside_tolerance_fails():
    with pytest.raises(AssertionError):
        _cmp(_problem(10), np.array([1, 5, 3, 0]))      # score 0.5, far below


def test_wrong_physical_slot_fails():
    p = _problem(10)
    bad = _phys(p, ORACLE).copy()
    bad[0] += 1
    with pytest.raises(AssertionError):
        _cmp(p, ORACLE, g_phys=bad)


def test_short_row_must_match_exactly():
    p = _problem(3)                                      # length 3 <= K: 0, 1, 2, -1
    want = np.array([0, 1, 2, -1])
    assert _cmp(p, want, o_raw=want) == 0
    with pytest.raises(AssertionError):
        _cmp(p, np.array([0, 2, 1, -1]), o_raw=want)


def test_score_bound_formula():
    logits = np.array([[1.0, -2.0, 4.0] + [0.0] * 61])
    w = np.zeros(64, np.float32)
    w[:3] = [2.0, -3.0, -0.5]
    # 1e-6 + 1e-5 * (|2| * 1 + |-3| * 0 + |-0.5| * 4)
    assert H.score_bound(logits, w)[0] == pytest.approx(1e-6 + 1e-5 * 4.0)


def test_same_set_in_wrong_order_fails():
    # the oracle's set, but scores 3.0 and 2.5 swapped: far outside tolerance
    with pytest.raises(AssertionError):
        _cmp(_problem(10), np.array([5, 1, 3, 6]))


def test_same_set_order_swap_within_tolerance_passes():
    # positions 2 (1.0) and 6 (1.0 + 5e-6) lie within 1e-5 relative of each
    # other: fp32 rounding may order them either way
    assert _cmp(_problem(10), np.array([1, 5, 3, 2]), o_raw=np.array([1, 5, 3, 6])) == 1
    assert H.order_follows_oracle(np.array([1, 5, 3, 2, 6]), SCORES, 0)
    assert H.order_follows_oracle(np.array([1, 5, 3, 6, 2]), SCORES, 0)


def test_equal_scores_must_come_in_position_order():
    sc = np.array([2.0, 1.0, 2.0, 1.0])
    assert H.order_follows_oracle(np.array([0, 2, 1, 3]), sc, 0)
    assert not H.order_follows_oracle(np.array([2, 0, 1, 3]), sc, 0)


def test_selected_scores_pure_bar_and_counted_waiver():
    w = np.zeros(64, np.float32)
    w[:2] = [1.0, -1.0]
    lg = np.zeros((3, 64))
    lg[:, 0] = [10.0, 10.0, 10.0]
    lg[:, 1] = [0.0, 0.0, 9.9999]
    want = np.array([10.0, 10.0, 1e-4])              # the third sum cancels 2e5-fold
    # within 1e-5 relative: passes with no waiver
    assert H.check_selected_scores(want * (1 + 5e-6), want, lg, w) == 0
    # the cancelling sum off by 1e-5 absolute: within the conditioned bound, waived
    assert H.check_selected_scores(want + np.array([0, 0, 1e-5]), want, lg, w) == 1
    # a well-conditioned score off by 2e-5 relative fails
    with pytest.raises(AssertionError):
        H.check_selected_scores(want * np.array([1 + 2e-5, 1, 1]), want, lg, w)
