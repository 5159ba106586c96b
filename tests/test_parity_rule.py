"""The acceptance rule that every GPU parity test applies (oracle/parity.py), checked on the CPU
with hand-made inputs: it accepts what the rule allows and rejects the mistakes it exists to
catch."""
import numpy as np
import pytest

from oracle import parity
from oracle import zipage_oracle as O


def test_tolerance_band_and_infinities():
    parity.assert_close("x", [1.0, 0.0, np.inf], [1.0009, 9e-7, np.inf])
    with pytest.raises(AssertionError):
        parity.assert_close("x", [1.0], [1.0011])           # 1.1e-3 relative: outside
    with pytest.raises(AssertionError):
        parity.assert_close("x", [2e-6], [0.0])              # above the absolute floor
    with pytest.raises(AssertionError):
        parity.assert_close("x", [np.inf], [5.0])             # a protected token must match
    with pytest.raises(AssertionError):
        parity.assert_close("x", [5.0], [np.inf])             # ... in both directions
    with pytest.raises(AssertionError):
        parity.assert_close("x", [-np.inf], [np.inf])
    with pytest.raises(AssertionError):
        parity.assert_close("x", [np.nan], [1.0])


def _scores():
    # 12 tokens, k = 8: the keep/evict boundary lies between S = 0.50 (kept) and 0.40 (evicted)
    return np.array([0.9, 0.1, 0.8, 0.5, 0.7, 0.2, 0.6, 0.3, 0.95, 0.4, 0.85, 0.75])


def _keep_mask(src, n):
    m = np.zeros(n, dtype=np.int32)
    m[src] = 1
    return m


def test_selection_equal_to_the_oracle_is_accepted():
    S = _scores()
    src = O.select_keep(S, 8)
    parity.check_selection(_keep_mask(src, 12), S.astype(np.float32), S, 8)


def test_wrong_kept_count_is_rejected():
    S = _scores()
    src = O.select_keep(S, 8)
    with pytest.raises(AssertionError):
        parity.check_selection(_keep_mask(src[:-1], 12), S.astype(np.float32), S, 8)


def test_selection_inconsistent_with_the_kernel_scores_is_rejected():
    # the kernel's own scores say token 9 (0.40) is below the boundary, yet it is kept
    S = _scores()
    src = O.select_keep(S, 8)
    bad = np.sort(np.r_[np.setdiff1d(src, [3]), 9])
    with pytest.raises(AssertionError):
        parity.check_selection(_keep_mask(bad, 12), S.astype(np.float32), S, 8)


def test_swap_at_the_boundary_within_tolerance_is_accepted():
    # two tokens at the boundary within the tolerance of each other: the kernel's fp32 scores
    # order them the other way, and its kept set follows its own scores
    S_ref = _scores()
    S_ref[9] = 0.5 - 1e-4                                  # just below token 3 (0.50)
    S_gpu = S_ref.copy()
    S_gpu[9] = 0.5 + 1e-4                                  # the kernel sees it just above
    src_gpu = O.select_keep(S_gpu.astype(np.float32).astype(np.float64), 8)
    assert 9 in src_gpu and 3 not in src_gpu
    parity.check_selection(_keep_mask(src_gpu, 12), S_gpu.astype(np.float32), S_ref, 8)


def test_swap_far_from_the_boundary_is_rejected():
    # the kernel's score of token 1 is far off (0.1 -> 0.99): its selection follows its own
    # scores, but token 1 lies far below the oracle's boundary
    S_ref = _scores()
    S_gpu = S_ref.copy()
    S_gpu[1] = 0.99
    src_gpu = O.select_keep(S_gpu.astype(np.float32).astype(np.float64), 8)
    with pytest.raises(AssertionError):
        parity.check_selection(_keep_mask(src_gpu, 12), S_gpu.astype(np.float32), S_ref, 8)


def test_expected_pool_moves_rows_through_both_tables():
    # one layer, 3 blocks of b = 2, one head, d = 1: logical tokens 0..3 in blocks [2, 0];
    # keep tokens 1 and 3 into the destination table [1, ...]
    b = 2
    pool = np.zeros((1, 3, 2, 1, b, 1), dtype=np.uint16)
    for blk in range(3):
        for row in range(b):
            pool[0, blk, :, 0, row, 0] = 10 * blk + row     # K and V rows carry their address
    tables = np.array([[2, 0]])
    dst = np.array([[1, 0]])
    out = parity.expected_pool(pool, tables, dst, {(0, 0, 0): [1, 3]}, b)
    # slot 0 <- token 1 (block 2, row 1); slot 1 <- token 3 (block 0, row 1); both land in block 1
    assert out[0, 1, 0, 0, 0, 0] == 21 and out[0, 1, 0, 0, 1, 0] == 1
    assert out[0, 1, 1, 0, 0, 0] == 21 and out[0, 1, 1, 0, 1, 0] == 1
    assert np.array_equal(out[0, [0, 2]], pool[0, [0, 2]])  # the source blocks are untouched
