"""The index-set comparison rule of the parity tests (helpers.py), on CPU:
well-separated top-k sets must match exactly, near ties may differ only
within 1e-4 of the k-th score, and a Block-Sparse row that breaks the layout
contract (order, diagonal, padding) is caught."""
import numpy as np
import pytest

from helpers import check_block_index, check_topk_set, topk_margin


def test_margin_of_separated_and_tied_scores():
    s = np.array([5.0, 4.0, 3.0, 2.0, 1.0])
    assert topk_margin(s, 2) == pytest.approx(0.25)
    assert topk_margin(s, 5) == float("inf") and topk_margin(s, 0) == float("inf")
    assert topk_margin(np.array([3.0, 2.0, 2.0, 1.0]), 2) == 0.0


def test_separated_sets_must_be_equal():
    s = np.array([5.0, 4.0, 3.0, 2.0, 1.0])
    assert check_topk_set([1, 0], [0, 1], s, 2, "same") == 0
    with pytest.raises(AssertionError, match="separated"):
        check_topk_set([0, 2], [0, 1], s, 2, "swapped")


def test_near_ties_within_the_rule_are_accepted():
    s = np.array([5.0, 4.0, 4.0 * (1 - 1e-5), 1.0])
    assert check_topk_set([0, 2], [0, 1], s, 2, "near tie") == 2
    s = np.array([5.0, 4.0, 4.0 * (1 - 5e-4), 1.0])   # within the margin, outside 1e-4
    with pytest.raises(AssertionError, match="member"):
        check_topk_set([0, 2], [0, 1], s, 2, "not close enough")
    with pytest.raises(AssertionError, match="members"):
        check_topk_set([0], [0, 1], s, 2, "short")


def _bs_case():
    rng = np.random.default_rng(3)
    nb, d, topk = 6, 4, 3
    qb, kb = rng.standard_normal((nb, d)), rng.standard_normal((nb, d))
    J = -np.ones((nb, topk), np.int32)
    cnt = np.zeros(nb, np.int32)
    for u in range(nb):
        sc = qb[u] @ kb[:u].T
        pick = sorted(np.argsort(-sc, kind="stable")[:topk - 1].tolist()) + [u]
        J[u, :len(pick)] = pick
        cnt[u] = len(pick)
    return J, cnt, qb, kb, topk


def test_block_rows_equal_pass_and_broken_rows_fail():
    J, cnt, qb, kb, topk = _bs_case()
    assert check_block_index(J, cnt, J, cnt, qb, kb, topk, "same") == 0
    bad = J.copy()
    bad[4, :2] = bad[4, 1::-1]            # not ascending
    with pytest.raises(AssertionError, match="ascending"):
        check_block_index(bad, cnt, J, cnt, qb, kb, topk, "order")
    bad2 = J.copy()
    bad2[2, cnt[2] - 1] = 1               # diagonal replaced
    with pytest.raises(AssertionError):
        check_block_index(bad2, cnt, J, cnt, qb, kb, topk, "diagonal")
    swapped = J.copy()
    u = 5
    others = [v for v in range(u) if v not in J[u, :cnt[u]]]
    swapped[u, 0] = others[0]
    swapped[u, :cnt[u]] = np.sort(swapped[u, :cnt[u]])
    with pytest.raises(AssertionError):
        check_block_index(swapped, cnt, J, cnt, qb, kb, topk, "wrong member")


def test_output_tolerance_allows_bf16_storage_rounding_only():
    """compare_rows: a bf16 output may sit half a bf16 step from the exact
    value on top of the arithmetic tolerance, and no more."""
    from helpers import BF16_U, O_MAX_ABS, compare_rows
    import torch
    ref = np.full((1, 16), 0.5, dtype=np.float64)
    ref[0, 0] = 4.0 + 0.0155                                     # rounds to 4.0 in bf16: error 0.0155
    got = torch.tensor(ref).to(torch.bfloat16).double().numpy()
    assert np.abs(got - ref).max() > O_MAX_ABS
    compare_rows(got, None, ref, None, "bf16 rounding of 4.0155")
    bad = ref.copy()
    bad[0, 0] += O_MAX_ABS + BF16_U * abs(ref[0, 0]) + 1e-4
    with pytest.raises(AssertionError, match="exceeds"):
        compare_rows(bad, None, ref, None, "beyond the storage rounding")
