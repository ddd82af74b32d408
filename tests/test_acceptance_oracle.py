"""Pins of the entropy-bounded acceptance oracle (CPU only): closed forms of the
entropy, a library cross-check, argmax tie-breaking, the acceptance rule on a
hand-worked example and as properties on random data, and the convergence test."""

import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle.acceptance as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_uniform_logits_entropy_is_log_vocab():
    for V in (2, 7, 1000, 65536):
        H, c, a = acc.row_stats(np.full((3, V), 1.25))
        np.testing.assert_allclose(H, math.log(V), rtol=1e-13)
        np.testing.assert_allclose(c, 1.0 / V, rtol=1e-13)
        assert np.all(a == 0)


def test_two_level_closed_form():
    V, k, alpha = 5000, 7, 3.0
    x = np.zeros((1, V))
    x[0, 100:100 + k] = alpha
    Z = k * math.exp(alpha) + (V - k)
    ph, pl = math.exp(alpha) / Z, 1.0 / Z
    H_ref = -(k * ph * math.log(ph) + (V - k) * pl * math.log(pl))
    H, c, a = acc.row_stats(x)
    assert abs(H[0] - H_ref) < 1e-12
    assert abs(c[0] - ph) < 1e-15
    assert a[0] == 100  # lowest index among the k tied maxima


def test_entropy_matches_scipy():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 3000)) * 2.5
    H, c, a = acc.row_stats(x)
    p = scipy.special.softmax(x, axis=1)
    np.testing.assert_allclose(H, scipy.stats.entropy(p, axis=1), rtol=1e-12)
    np.testing.assert_allclose(c, p.max(axis=1), rtol=1e-12)
    np.testing.assert_array_equal(a, np.argmax(p, axis=1))


def test_near_one_hot():
    x = np.zeros((1, 100))
    x[0, 42] = 60.0
    H, c, a = acc.row_stats(x)
    assert 0.0 <= H[0] < 1e-20
    assert abs(c[0] - 1.0) < 1e-15 and a[0] == 42


def _golden():
    rows = []
    with open(os.path.join(GOLDEN, "acceptance_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_acceptance_golden():
    H = np.array([0.125, 0.5, 0.25, 0.375])
    c = np.array([0.9, 0.6, 0.8, 0.7])
    rows = _golden()
    assert len(rows) == 7
    for budget, before, after in rows:
        prev = np.zeros(4, dtype=bool)
        if before != "-":
            prev[[int(x) for x in before.split(",")]] = True
        got = acc.accept(H, c, prev, float(budget))
        exp = np.zeros(4, dtype=bool)
        exp[[int(x) for x in after.split(",")]] = True
        np.testing.assert_array_equal(got, exp, err_msg=f"budget {budget} before {before}")


def test_acceptance_properties_random():
    rng = np.random.default_rng(11)
    for trial in range(200):
        n = int(rng.integers(1, 40))
        H = rng.uniform(0, 2, n)
        c = rng.uniform(0, 1, n)
        c[rng.integers(0, n, 3)] = c[0]  # some ties
        prev = rng.uniform(size=n) < 0.3
        budget = float(rng.uniform(0, 5))
        out = acc.accept(H, c, prev, budget)
        assert np.all(out[prev])                      # accepted stays accepted
        new = out & ~prev
        order = acc.confidence_order(c, ~prev)
        k = int(new.sum())
        if (~prev).any():
            assert k >= 1                             # progress
            assert set(np.flatnonzero(new)) == set(order[:k])   # a prefix of the ranking
            if k > 1:
                assert H[order[:k]].sum() <= budget + 1e-12
            if k < len(order):
                assert H[order[:k + 1]].sum() > budget   # the next one would pass the budget
        else:
            assert k == 0
        # ranking: confidence descending, ties by position
        cs = c[order]
        assert np.all(np.diff(cs) <= 0)
        for i in range(len(order) - 1):
            if cs[i] == cs[i + 1]:
                assert order[i] < order[i + 1]


def test_convergence_truth_table():
    a = np.array([1, 2, 3])
    H_low, H_high = np.full(3, 0.1), np.full(3, 2.0)
    assert acc.converge(a, a, 2, H_low, 0.5, 3, 4, 100) == (True, 3)
    assert acc.converge(a, a, 1, H_low, 0.5, 3, 4, 100) == (False, 2)     # not stable long enough
    assert acc.converge(a, a, 5, H_high, 0.5, 3, 4, 100) == (False, 6)    # entropy too high
    assert acc.converge(a, a + 1, 9, H_low, 0.5, 3, 4, 100) == (False, 0)  # argmax changed: reset
    assert acc.converge(a, a + 1, 0, H_high, 0.5, 3, 99, 100) == (True, 0)  # step limit
    assert acc.converge(a, a, 2, np.array([0.4, 0.6, 0.5]), 0.5, 3, 1, 100) == (False, 3)  # mean = 0.5, not < 0.5


def test_batch_step_matches_per_canvas_calls():
    rng = np.random.default_rng(5)
    cu = np.array([0, 5, 12, 20])
    x = rng.standard_normal((20, 300)) * 3
    prev_acc = rng.uniform(size=20) < 0.2
    prev_arg = rng.integers(0, 300, 20)
    res = acc.denoise_step(x, cu, prev_acc, prev_arg, np.array([1, 0, 4]), 1.5, 3.0, 2, 7, 48)
    H, c, a = acc.row_stats(x)
    for b in range(3):
        r0, r1 = cu[b], cu[b + 1]
        np.testing.assert_array_equal(res["accepted"][r0:r1], acc.accept(H[r0:r1], c[r0:r1], prev_acc[r0:r1], 1.5))
        assert (res["converged"][b], res["stable"][b]) == acc.converge(a[r0:r1], prev_arg[r0:r1], [1, 0, 4][b], H[r0:r1], 3.0, 2, 7, 48)
