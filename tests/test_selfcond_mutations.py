"""Plant plausible mistakes in the self-conditioning oracle (on the CPU, one at
a time) and check that the pins in ``test_selfcond_oracle.py`` catch each."""

import numpy as np
import pytest

import oracle.selfcond as sc
import test_selfcond_oracle as pins

_ORIG = {name: getattr(sc, name) for name in ("softmax_rows", "weighted_embedding")}


def _softmax_no_shift(logits):
    e = np.exp(np.asarray(logits, dtype=np.float64))
    return e / e.sum(axis=1, keepdims=True)


def _softmax_columns(logits):
    x = np.asarray(logits, dtype=np.float64)
    e = np.exp(x - x.max(axis=0, keepdims=True))
    return e / e.sum(axis=0, keepdims=True)


def _softmax_unnormalised(logits):
    x = np.asarray(logits, dtype=np.float64)
    return np.exp(x - x.max(axis=1, keepdims=True))


def _softmax_temperature_two(logits):
    return _ORIG["softmax_rows"](np.asarray(logits, dtype=np.float64) / 2.0)


def _embedding_token_shift(p, E):
    return _ORIG["weighted_embedding"](p, np.roll(np.asarray(E), 1, axis=0))


def _embedding_mean_not_weighted(p, E):
    p = np.asarray(p)
    return np.tile(np.asarray(E, dtype=np.float64).mean(axis=0), (p.shape[0], 1))


def _embedding_dims_reversed(p, E):
    return _ORIG["weighted_embedding"](p, E)[:, ::-1].copy()


MUTANTS = [
    ("softmax_rows", _softmax_no_shift),
    ("softmax_rows", _softmax_columns),
    ("softmax_rows", _softmax_unnormalised),
    ("softmax_rows", _softmax_temperature_two),
    ("weighted_embedding", _embedding_token_shift),
    ("weighted_embedding", _embedding_mean_not_weighted),
    ("weighted_embedding", _embedding_dims_reversed),
]

PIN_CALLS = [
    pins.test_golden_dyadic_example,
    pins.test_dominant_token_gives_its_embedding,
    pins.test_uniform_logits_give_the_mean_embedding,
    pins.test_two_level_logits_closed_form,
    pins.test_shift_invariance_and_convex_bounds,
    pins.test_row_order_and_token_relabelling,
]


def _caught(monkeypatch, name, fn):
    monkeypatch.setattr(sc, name, fn)
    for call in PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                call()
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            return True
    return False


def test_unmutated_oracle_passes_every_pin():
    for call in PIN_CALLS:
        call()


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[f.__name__ for _, f in MUTANTS])
def test_pins_catch_planted_mistake(monkeypatch, name, fn):
    assert _caught(monkeypatch, name, fn), f"no pin caught the mutant {fn.__name__} of {name}"
