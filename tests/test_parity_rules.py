"""The comparison rules of the GPU parity tests, checked on the CPU with hand-made rows.

compare_selection accepts a selection that differs from the oracle's only where the differing
pages' oracle scores lie within 1e-6 relative of the cutoff score, logs every such near tie, and
rejects anything else (a clear loss, a missing forced page, bad padding, a wrong count).
"""
import numpy as np

import parity


def _row(ids, b_max=6):
    return np.array(list(ids) + [-1] * (b_max - len(ids)), dtype=np.int32)


def test_exact_selection_is_accepted_and_counted():
    s = np.array([5.0, 1.0, 4.0, 3.0, 2.0, 0.0])
    n0 = parity.SELECTION_LOG["units"]
    ok, near, got, ref = parity.compare_selection(_row([0, 2, 3, 5]), s, 4)
    assert ok and not near and got == ref == [0, 2, 3, 5]
    assert parity.SELECTION_LOG["units"] == n0 + 1


def test_near_tie_at_the_cutoff_is_accepted_and_logged():
    # pages 3 and 4 differ by 1e-9 relative at the cutoff: either may be chosen
    s = np.array([5.0, 1.0, 4.0, 3.0, 3.0 * (1 - 1e-9), 0.0])
    n0 = len(parity.SELECTION_LOG["near_ties"])
    ok, near, got, ref = parity.compare_selection(_row([0, 2, 4, 5]), s, 4)
    assert ref == [0, 2, 3, 5] and ok and near
    assert len(parity.SELECTION_LOG["near_ties"]) == n0 + 1
    assert parity.SELECTION_LOG["near_ties"][-1]["pages"] == [3, 4]


def test_clear_loss_missing_forced_page_and_bad_padding_are_rejected():
    s = np.array([5.0, 1.0, 4.0, 3.0, 2.9, 0.0])
    assert not parity.compare_selection(_row([0, 2, 4, 5]), s, 4)[0]   # 2.9 vs 3.0: not a near tie
    s = np.array([5.0, 1.0, 4.0, 3.0, 3.0, 0.0])
    assert not parity.compare_selection(_row([0, 2, 3, 4]), s, 4)[0]   # tail page 5 missing
    bad = _row([0, 2, 3, 5])
    bad[5] = 1
    assert not parity.compare_selection(bad, s, 4)[0]                   # junk after the valid ids
    assert not parity.compare_selection(_row([0, 2, 5]), s, 4)[0]      # one page short
