"""The parity rule's own logic (CPU): exact-tie order, gap segments."""
import numpy as np

from tests import parity


def test_tied_pair_keeps_relative_order_even_if_a_close_expert_moves():
    # oracle: 252 just above the tied pair (29, 203); fp32 may merge 252 into the tie
    idx_r = np.array([252, 29, 203, 168, 104, 110])
    gaps = np.array([2.2e-9, 0.0, 8.8e-5, 3.3e-5, 0.0, 7.9e-5])
    assert not parity.tie_broken_wrong(np.array([29, 203, 252, 168, 104, 110]), idx_r, gaps)
    assert parity.tie_broken_wrong(np.array([203, 29, 252, 168, 104, 110]), idx_r, gaps)
    assert parity.tie_broken_wrong(np.array([252, 29, 203, 168, 110, 104]), idx_r, gaps)


def test_no_tie_no_error():
    idx_r = np.array([1, 2, 3, 4, 5, 6])
    gaps = np.array([0.1, 0.1, 0.1, 0.1, 0.1, 0.1])
    assert not parity.tie_broken_wrong(np.array([6, 5, 4, 3, 2, 1]), idx_r, gaps)
