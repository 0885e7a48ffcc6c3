"""CPU checks of the parity rule itself: it accepts the oracle's own answer and
any valid near-tie substitution, and rejects plausible wrong answers."""

import numpy as np
import pytest

import oracle
from tests.parity import check_query, check_scores_row


def _ref(n=200, seed=0):
    return np.random.default_rng(seed).standard_normal(n)


def test_accepts_exact():
    I = _ref()
    gi, gs = oracle.topk_sorted(I, 20)
    check_query(I, gi, gs.astype(np.float32), 20)


def test_accepts_near_tie_swap():
    I = _ref()
    gi, gs = oracle.topk_sorted(I, 20)
    nxt = np.argsort(-I, kind="stable")[20]
    I2 = I.copy()
    I2[nxt] = I[gi[19]] - 1e-9          # the 21st is within tol of the 20th
    gi2 = gi.copy(); gi2[19] = nxt
    gs2 = gs.copy(); gs2[19] = I2[nxt]
    check_query(I2, gi2, gs2, 20)


@pytest.mark.parametrize("mutate", ["drop_best", "duplicate", "bad_order", "bad_score", "bad_pad", "swap_far"])
def test_rejects(mutate):
    I = _ref()
    k = 20
    gi, gs = oracle.topk_sorted(I, k)
    gi, gs = gi.copy(), gs.copy()
    if mutate == "drop_best":
        gi[0] = np.argsort(I)[0]; gs[0] = I[gi[0]]
    elif mutate == "duplicate":
        gi[5] = gi[4]; gs[5] = gs[4]
    elif mutate == "bad_order":
        gi[[2, 3]] = gi[[3, 2]]; gs[[2, 3]] = gs[[3, 2]]
    elif mutate == "bad_score":
        gs[7] += 1.0
    elif mutate == "bad_pad":
        gi, gs = oracle.topk_sorted(I[:10], k)
        gi = gi.copy(); gi[15] = 3
        I = I[:10]
    elif mutate == "swap_far":
        far = np.argsort(-I)[100]
        gi[19] = far; gs[19] = I[far]
    with pytest.raises(AssertionError):
        check_query(I, gi, gs, k)


def test_scores_row_rule():
    I = _ref(50)
    I[3] = -np.inf
    check_scores_row(I, I.astype(np.float32))
    bad = I.copy(); bad[4] += 0.1
    with pytest.raises(AssertionError):
        check_scores_row(I, bad)
    bad = I.copy(); bad[3] = 0.0
    with pytest.raises(AssertionError):
        check_scores_row(I, bad)
