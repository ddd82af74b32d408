"""CPU checks of the acceptance validity checker used by the GPU parity test:
it admits the fp64 decision, admits the alternatives that rounding can
produce on near ties, and rejects plausible wrong decisions (a row skipped, a
row too many, a less confident row taken, nothing taken)."""

import numpy as np

import oracle.acceptance as acc
from acceptance_validity import check_accept, check_converge, clear_accept


def _canvas(seed, n=64):
    rng = np.random.default_rng(seed)
    H = rng.uniform(0.0, 2.0, n)
    c = rng.uniform(0.05, 1.0, n)
    open_ = rng.uniform(size=n) > 0.25
    return H, c, open_


def test_fp64_decision_is_valid_and_mostly_clear():
    n_clear = 0
    for seed in range(40):
        H, c, open_ = _canvas(seed)
        for budget in (0.0, 0.7, 3.0, 1e6):
            dec = acc.accept(H, c, ~open_, budget) & open_
            ok, why = check_accept(dec, open_, H, c, budget)
            assert ok, (seed, budget, why)
            d2, clear = clear_accept(open_, H, c, budget)
            assert np.array_equal(d2, dec)
            n_clear += clear
    assert n_clear >= 120  # of 160: random statistics are rarely near a tie


def test_wrong_decisions_are_rejected():
    for seed in range(40):
        H, c, open_ = _canvas(seed)
        budget = 3.0
        dec, clear = clear_accept(open_, H, c, budget)
        if not clear:
            continue
        order = acc.confidence_order(c, open_)
        k = int(dec.sum())
        # one row too many / one too few / the last taken swapped for the next
        if k < len(order):
            more = dec.copy()
            more[order[k]] = True
            assert not check_accept(more, open_, H, c, budget)[0]
            swap = dec.copy()
            swap[order[k - 1]] = False
            swap[order[k]] = True
            assert not check_accept(swap, open_, H, c, budget)[0]
        if k > 1:
            fewer = dec.copy()
            fewer[order[k - 1]] = False
            assert not check_accept(fewer, open_, H, c, budget)[0]
        assert not check_accept(np.zeros_like(dec), open_, H, c, budget)[0]
        closed = dec.copy()
        closed[np.flatnonzero(~open_)[:1]] = True
        if (~open_).any():
            assert not check_accept(closed, open_, H, c, budget)[0]


def test_near_ties_admit_both_orders():
    # rows 0 and 1 tie within the confidence tolerance; the budget takes one
    H = np.array([0.5, 0.6, 0.1])
    c = np.array([0.80000, 0.80002, 0.1])
    open_ = np.ones(3, dtype=bool)
    a = np.array([True, False, False])
    b = np.array([False, True, False])
    assert check_accept(a, open_, H, c, 0.55)[0]
    assert check_accept(b, open_, H, c, 0.55)[0]
    assert not clear_accept(open_, H, c, 0.55)[1]
    # the running entropy at the cut sits on the budget: both cuts are correct
    H = np.array([0.5, 0.50001, 0.1])
    c = np.array([0.9, 0.5, 0.1])
    assert check_accept(np.array([True, True, False]), open_, H, c, 1.0)[0]
    assert check_accept(np.array([True, False, False]), open_, H, c, 1.0)[0]
    assert not clear_accept(open_, H, c, 1.0)[1]


def test_convergence_checker():
    H = np.full(8, 0.25)
    a = np.arange(8)
    ok, clear, _ = check_converge(True, 3, a, a, 2, H, 0.5, 3, 0, 48)
    assert ok and clear
    assert not check_converge(False, 3, a, a, 2, H, 0.5, 3, 0, 48)[0]
    assert not check_converge(True, 2, a, a, 2, H, 0.5, 3, 0, 48)[0]      # stable counter wrong
    ok, clear, _ = check_converge(False, 3, a, a, 2, H, 0.25 + 1e-6, 3, 0, 48)
    assert ok and not clear                                              # mean on the threshold
    assert check_converge(True, 0, a, a + 1, 2, H, 0.0, 3, 47, 48)[0]    # step limit
