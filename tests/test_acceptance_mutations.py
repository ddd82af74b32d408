"""Plant plausible mistakes in the acceptance oracle and check the pins catch them."""

import numpy as np
import pytest

import oracle.acceptance as acc
import test_acceptance_oracle as pins

_ORIG = {n: getattr(acc, n) for n in ("row_stats", "confidence_order", "accept", "converge")}


def _stats_log2(logits):
    H, c, a = _ORIG["row_stats"](logits)
    return H / np.log(2.0), c, a


def _stats_argmax_last(logits):
    H, c, a = _ORIG["row_stats"](logits)
    x = np.asarray(logits)
    return H, c, x.shape[1] - 1 - np.argmax(x[:, ::-1], axis=1)


def _stats_no_shift_sign(logits):
    H, c, a = _ORIG["row_stats"](logits)
    return -H, c, a


def _order_ascending(c, candidates):
    idx = np.flatnonzero(candidates)
    return idx[np.argsort(np.asarray(c)[idx], kind="stable")]


def _order_unstable_ties(c, candidates):
    idx = np.flatnonzero(candidates)[::-1]
    return idx[np.argsort(-np.asarray(c)[idx], kind="stable")]


def _accept_includes_overflow(H, c, before, budget):
    out = _ORIG["accept"](H, c, before, budget)
    order = acc.confidence_order(c, ~np.asarray(before, dtype=bool))
    k = int((out & ~np.asarray(before, dtype=bool)).sum())
    if k < len(order):
        out[order[k]] = True
    return out


def _accept_no_progress(H, c, before, budget):
    before = np.asarray(before, dtype=bool)
    order = acc.confidence_order(c, ~before)
    out = before.copy()
    run = 0.0
    for i in order:
        run += H[i]
        if run > budget:
            break
        out[i] = True
    return out


def _converge_no_reset(a_now, a_prev, stable_before, H, tau, patience, step, max_steps):
    cv, st = _ORIG["converge"](a_now, a_prev, stable_before, H, tau, patience, step, max_steps)
    if st == 0:
        st = stable_before + 1
        cv = (st >= patience and float(np.mean(H)) < tau) or (step + 1 >= max_steps)
    return cv, st


def _converge_le(a_now, a_prev, stable_before, H, tau, patience, step, max_steps):
    same = bool(np.array_equal(a_now, a_prev))
    st = stable_before + 1 if same else 0
    return bool((st >= patience and float(np.mean(H)) <= tau) or (step + 1 >= max_steps)), st


MUTANTS = [
    ("row_stats", _stats_log2), ("row_stats", _stats_argmax_last), ("row_stats", _stats_no_shift_sign),
    ("confidence_order", _order_ascending), ("confidence_order", _order_unstable_ties),
    ("accept", _accept_includes_overflow), ("accept", _accept_no_progress),
    ("converge", _converge_no_reset), ("converge", _converge_le),
]

PINS = [pins.test_uniform_logits_entropy_is_log_vocab, pins.test_two_level_closed_form,
        pins.test_entropy_matches_scipy, pins.test_acceptance_golden,
        pins.test_acceptance_properties_random, pins.test_convergence_truth_table]


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[f.__name__ for _, f in MUTANTS])
def test_pins_catch_planted_mistake(monkeypatch, name, fn):
    monkeypatch.setattr(acc, name, fn)
    caught = False
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            caught = True
            break
    assert caught, f"planted mistake {fn.__name__} in {name} went unnoticed"
