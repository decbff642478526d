"""The parity bar's exclusion rule, checked on hand-made routing results (no
GPU): ids compare as sets, an order swap inside the selection is not an
exclusion, and only a token whose 8th/9th logit gap is below 1e-4 may hold a
different set of experts (and is then left out of the y comparison)."""
import numpy as np
import pytest

from tests import parity


def _logits(rows):
    """Per token: 9 leading logits in ranked order, the rest far below."""
    out = np.full((len(rows), 32), -10.0)
    for t, lead in enumerate(rows):
        out[t, : len(lead)] = lead
    return out


CLEAR = [5.0, 4.0, 3.0, 2.9999, 2.0, 1.5, 1.0, 0.5, 0.0]    # 8th/9th gap 0.5; a near tie inside the top 8
NEAR89 = [5.0, 4.0, 3.0, 2.5, 2.0, 1.5, 1.0, 0.50005, 0.5]  # 8th/9th gap 5e-5


def test_order_swap_is_compared_not_excluded():
    logits = _logits([CLEAR] * 2)
    ref = np.tile(np.arange(8), (2, 1))
    gpu = ref.copy()
    gpu[0, [2, 3]] = gpu[0, [3, 2]]  # experts 2 and 3 swapped (logit gap 1e-4 inside the top 8)
    excl = parity.check_ids(gpu, ref, logits, 8)
    assert not excl.any()


def test_near_tie_at_the_boundary_may_differ_and_is_excluded():
    logits = _logits([NEAR89] + [CLEAR] * 1999)
    ref = np.tile(np.arange(8), (2000, 1))
    gpu = ref.copy()
    gpu[0, 7] = 8  # the 9th expert chosen instead of the 8th across a 5e-5 gap
    excl = parity.check_ids(gpu, ref, logits, 8)
    assert excl.tolist() == [True] + [False] * 1999


def test_set_difference_with_a_clear_boundary_fails():
    logits = _logits([CLEAR] * 4)
    ref = np.tile(np.arange(8), (4, 1))
    gpu = ref.copy()
    gpu[1, 3] = 8  # a different set although the 8th/9th gap is 0.5
    with pytest.raises(AssertionError):
        parity.check_ids(gpu, ref, logits, 8)


def test_excluded_tokens_are_capped_at_a_thousandth():
    logits = _logits([NEAR89] * 3 + [CLEAR] * 997)
    ref = np.tile(np.arange(8), (1000, 1))
    gpu = ref.copy()
    gpu[:2, 7] = 8  # two of 1000 tokens differ: above the 0.1 % cap
    with pytest.raises(AssertionError):
        parity.check_ids(gpu, ref, logits, 8)


def test_weights_compare_per_expert_not_per_slot():
    ids_ref = np.array([[0, 1, 2]])
    w_ref = np.array([[0.5, 0.3, 0.2]])
    ids_gpu = np.array([[0, 2, 1]])
    w_gpu = np.array([[0.5, 0.2, 0.3]])
    parity.check_weights(ids_gpu, w_gpu, ids_ref, w_ref, np.array([True]))
    with pytest.raises(AssertionError):
        parity.check_weights(ids_gpu, w_ref, ids_ref, w_ref, np.array([True]))
