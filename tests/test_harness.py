"""Host logic of the parity harness (CPU): the index rule that the GPU tests apply is the contract's,
no looser. Planted selections show that each way of breaking it is caught."""
import numpy as np

from harness import INDEX_GAP, index_parity, oracle_order


def _case():
    # 8 experts, top-3. Oracle ranking: 5 (3.0), 1 (2.0), {2, 6} exactly tied at 1.5 (2 before 6), then
    # 0 at 1.5 - INDEX_GAP / 2 (near the k-th), 3, 4, 7.
    keys = np.array([1.5 - INDEX_GAP / 2, 2.0, 1.5, -1.0, -2.0, 3.0, 1.5, -3.0])
    return keys[None, :], np.array([[5, 1, 2]])


def test_oracle_order_breaks_ties_by_lower_id():
    keys, _ = _case()
    assert oracle_order(keys[0]).tolist() == [5, 1, 2, 6, 0, 3, 4, 7]


def test_exact_selection_passes():
    keys, ref = _case()
    ok, near, msg = index_parity(ref, ref, keys, 3)
    assert ok and near == [] and msg is None


def test_exact_tie_across_kth_place_gets_no_excuse():
    keys, ref = _case()
    ok, _, msg = index_parity(np.array([[5, 1, 6]]), ref, keys, 3)  # 6 ties 2 exactly: lower id wins
    assert not ok and "sets differ" in msg


def test_exact_tie_order_inside_selection_gets_no_excuse():
    keys = np.array([[3.0, 2.0, 2.0, 1.0, 0.0]])
    ref = np.array([[0, 1, 2]])
    assert index_parity(ref, ref, keys, 3)[0]
    ok, _, msg = index_parity(np.array([[0, 2, 1]]), ref, keys, 3)
    assert not ok and "out of the oracle's order" in msg


def test_near_tie_exchange_only_of_kth_and_next():
    # k-th (2, 1.5) and (k+1)-th (0, 1.5 - INDEX_GAP/2) are near, not equal: that exchange is allowed
    keys = np.array([[1.5 - INDEX_GAP / 2, 2.0, 1.5, -1.0, -2.0, 3.0, -0.5, -3.0]])
    ref = np.array([[5, 1, 2]])
    ok, near, _ = index_parity(np.array([[5, 1, 0]]), ref, keys, 3)
    assert ok and near == [0]
    # any other member in its place is a failure
    ok, _, msg = index_parity(np.array([[5, 1, 6]]), ref, keys, 3)
    assert not ok and "sets differ" in msg
    ok, _, _ = index_parity(np.array([[5, 0, 2]]), ref, keys, 3)  # dropped the 2nd, not the k-th
    assert not ok


def test_near_reorder_allowed_far_reorder_not():
    keys = np.array([[3.0, 3.0 - INDEX_GAP / 4, 1.0, 0.0]])
    ref = np.array([[0, 1, 2]])
    assert index_parity(np.array([[1, 0, 2]]), ref, keys, 3)[0]
    assert not index_parity(np.array([[0, 2, 1]]), ref, keys, 3)[0]


def test_duplicate_or_out_of_range_ids_fail():
    keys = np.array([[3.0, 2.0, 1.0, 0.0]])
    ref = np.array([[0, 1, 2]])
    assert not index_parity(np.array([[0, 0, 1]]), ref, keys, 3)[0]
    assert not index_parity(np.array([[0, 1, 4]]), ref, keys, 3)[0]
    assert not index_parity(np.array([[0, 1, -1]]), ref, keys, 3)[0]
