"""Pins of the self-conditioning oracle (``oracle/selfcond.py``) against facts
that do not come from the oracle itself: a hand-worked dyadic example, closed
forms (one dominant token, uniform logits, two-level logits), invariance under
a per-row shift, and the convex-combination bounds."""

import os

import numpy as np

import oracle.selfcond as sc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "selfcond_example.txt")


def load_golden():
    g = {"logit_exp": [], "E": [], "Y": []}
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if line:
            g[line[0]].append([float(x) for x in line[1:]])
    return np.log(np.array(g["logit_exp"])), np.array(g["E"]), np.array(g["Y"])


def test_golden_dyadic_example():
    x, E, Y = load_golden()
    np.testing.assert_allclose(sc.self_conditioning(x, E), Y, rtol=0, atol=1e-12)


def test_dominant_token_gives_its_embedding():
    rng = np.random.default_rng(0)
    V, d = 50, 7
    E = rng.standard_normal((V, d))
    x = rng.standard_normal((3, V))
    tok = [4, 0, V - 1]
    for r, t in enumerate(tok):
        x[r, t] = 1000.0          # exp(-1000 + O(1)) underflows: a one-hot distribution
    np.testing.assert_array_equal(sc.self_conditioning(x, E), E[tok])


def test_uniform_logits_give_the_mean_embedding():
    rng = np.random.default_rng(1)
    E = rng.standard_normal((64, 5))
    x = np.full((2, 64), -3.25)
    np.testing.assert_allclose(sc.self_conditioning(x, E), np.tile(E.mean(axis=0), (2, 1)),
                               rtol=0, atol=1e-14)


def test_two_level_logits_closed_form():
    """a on k tokens, b on the rest: weight w = e^a / (k e^a + (V-k) e^b) on
    the k tokens, (1 - k w) / (V - k) on the others."""
    rng = np.random.default_rng(2)
    V, d, k, a, b = 40, 6, 5, 2.0, -1.0
    E = rng.standard_normal((V, d))
    hot = rng.choice(V, size=k, replace=False)
    x = np.full((1, V), b)
    x[0, hot] = a
    w_hot = np.exp(a) / (k * np.exp(a) + (V - k) * np.exp(b))
    w_cold = (1.0 - k * w_hot) / (V - k)
    cold = np.setdiff1d(np.arange(V), hot)
    want = w_hot * E[hot].sum(axis=0) + w_cold * E[cold].sum(axis=0)
    np.testing.assert_allclose(sc.self_conditioning(x, E)[0], want, rtol=1e-13, atol=1e-14)


def test_shift_invariance_and_convex_bounds():
    rng = np.random.default_rng(3)
    V, d = 300, 9
    E = rng.standard_normal((V, d))
    x = 3.0 * rng.standard_normal((4, V))
    y = sc.self_conditioning(x, E)
    shifted = x + np.array([[700.0], [-700.0], [0.5], [1e-3]])
    np.testing.assert_allclose(sc.self_conditioning(shifted, E), y, rtol=1e-12, atol=1e-13)
    # a convex combination of the rows of E: inside their coordinate-wise range
    assert (y <= E.max(axis=0) + 1e-12).all() and (y >= E.min(axis=0) - 1e-12).all()


def test_row_order_and_token_relabelling():
    """Permuting rows permutes the outputs; relabelling tokens (the same
    permutation on the logits' columns and on E's rows) changes nothing."""
    rng = np.random.default_rng(4)
    V, d = 33, 4
    E = rng.standard_normal((V, d))
    x = rng.standard_normal((5, V))
    y = sc.self_conditioning(x, E)
    pr = rng.permutation(5)
    pv = rng.permutation(V)
    np.testing.assert_allclose(sc.self_conditioning(x[pr], E), y[pr], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(sc.self_conditioning(x[:, pv], E[pv]), y, rtol=1e-13, atol=1e-15)
