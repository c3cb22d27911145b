"""CPU checks of the parity-rule helper itself (it must reject the mistakes it exists for)."""
import numpy as np

from parity import check_topk_row


def test_exact_set_required_when_gap_is_clear():
    s = np.array([5.0, 4.0, 3.0, 1.0, 0.5])
    assert check_topk_row(np.array([0, 1, 2]), s, 3) is None
    assert check_topk_row(np.array([1, 0, 2]), s, 3) is not None      # rows are sorted ascending
    assert check_topk_row(np.array([0, 1, 3]), s, 3) is not None


def test_near_tie_accepts_either_choice_but_not_a_low_score():
    s = np.array([5.0, 3.0, 3.0 - 1e-6, 1.0])
    assert check_topk_row(np.array([0, 1]), s, 2) is None
    assert check_topk_row(np.array([0, 2]), s, 2) is None
    assert check_topk_row(np.array([0, 3]), s, 2) is not None
    assert check_topk_row(np.array([1, 2]), s, 2) is not None     # drops the clear winner


def test_count_padding_and_duplicates():
    s = np.arange(10, dtype=float)
    assert check_topk_row(np.array([9, 8, -1]), s, 3) is not None
    assert check_topk_row(np.array([9, -1, 8]), s, 3) is not None
    assert check_topk_row(np.array([9, 9, 8]), s, 3) is not None
    assert check_topk_row(np.array([0, 1, 2, -1, -1]), np.array([1.0, 2.0, 3.0]), 5) is None
    assert check_topk_row(np.array([0, 1, 3, -1, -1]), np.array([1.0, 2.0, 3.0]), 5) is not None
