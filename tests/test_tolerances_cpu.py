"""The parity metric: both forms must hold, and the element-wise one sees what the
norm-wise one hides."""
import numpy as np

from tests.tolerances import elem_rel_err, max_rel_err, norm_rel_err


def test_small_entry_error_is_seen_element_wise():
    ref = np.ones(100)
    ref[0] = 100.0
    got = ref.copy()
    got[1] = 1.5  # 50% off on a small entry, 0.5% of the largest (rms ~ 10)
    assert norm_rel_err(got, ref) <= 0.01
    assert elem_rel_err(got, ref) > 0.01
    assert max_rel_err(got, ref) == elem_rel_err(got, ref)


def test_rms_floor_keeps_entries_near_zero_from_failing():
    ref = np.array([1.0, -1.0, 1e-9, 1.0])
    got = ref + np.array([0.0, 0.0, 1e-3, 0.0])  # absolute error well below the terms' scale
    assert elem_rel_err(got, ref) < 2e-3


def test_exact_and_empty():
    a = np.arange(6.0).reshape(2, 3)
    assert max_rel_err(a, a) == 0.0
    assert max_rel_err(np.zeros(0), np.zeros(0)) == 0.0
    assert max_rel_err(np.zeros(3), np.zeros(3)) == 0.0
