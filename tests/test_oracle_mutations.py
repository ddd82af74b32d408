"""Plant plausible mistakes in the CPU oracle (one step at a time, on the CPU)
and check that the pins in ``test_oracle_pins.py`` catch every one of them.
This is what makes the pins worth trusting: a dropped term, a wrong sign or
index, or a transposed operand anywhere in the oracle fails at least one pin.
"""

import importlib

import numpy as np
import pytest

import test_oracle_pins as pins

orc = importlib.import_module("oracle.attention")


def _mask_no_diagonal(ctx_len, n_q, causal, window, t_begin=0, t_end=None):
    m = _ORIG["visible_mask"](ctx_len, n_q, causal, window, t_begin, t_end)
    if causal:
        L = ctx_len + n_q
        for r, t in enumerate(range(t_begin, t_end if t_end is not None else n_q)):
            i = ctx_len + t
            if i < L and r < m.shape[0] and m[r, :i].any():
                m[r, i] = False
    return m


def _mask_bidir_window_short(ctx_len, n_q, causal, window, t_begin=0, t_end=None):
    m = _ORIG["visible_mask"](ctx_len, n_q, causal, window, t_begin, t_end)
    if not causal and window > 0:
        for r, t in enumerate(range(t_begin, t_end if t_end is not None else n_q)):
            i = ctx_len + t
            if i + window < m.shape[1]:
                m[r, i + window] = False
    return m


def _mask_left_window_long(ctx_len, n_q, causal, window, t_begin=0, t_end=None):
    return _ORIG["visible_mask"](ctx_len, n_q, causal, window + 1 if window >= 0 else window,
                                 t_begin, t_end)


def _mask_positions_ignore_context(ctx_len, n_q, causal, window, t_begin=0, t_end=None):
    # query positions counted from 0 instead of from ctx_len, keys shifted to match
    m = _ORIG["visible_mask"](0, ctx_len + n_q, causal, window)
    te = n_q if t_end is None else t_end
    return m[t_begin:te]


def _mask_causal_for_everyone(ctx_len, n_q, causal, window, t_begin=0, t_end=None):
    return _ORIG["visible_mask"](ctx_len, n_q, True, window, t_begin, t_end)


def _gqa_modulo(h, num_q_heads, num_kv_heads):
    return h % num_kv_heads


def _scores_no_scale(q_rows, k_rows, scale):
    return q_rows @ k_rows.T


def _scores_sign(q_rows, k_rows, scale):
    return -scale * (q_rows @ k_rows.T)


def _softmax_unmasked_sum(z, mask):
    zm = np.where(mask, z, -np.inf)
    m = zm.max(axis=1)
    l = np.exp(z - m[:, None]).sum(axis=1)          # masked entries leak into l
    e = np.where(mask, np.exp(zm - m[:, None]), 0.0)
    return e / l[:, None], m, l


def _softmax_no_normalise(z, mask):
    w, m, l = _ORIG["masked_softmax"](z, mask)
    return w * l[:, None], m, l


def _lse_drop_max(m, l):
    return np.log(l)


def _values_shifted(w, v_rows):
    return w @ np.roll(v_rows, 1, axis=0)


def _values_transposed_features(w, v_rows):
    out = w @ v_rows
    return out[:, ::-1].copy()


_ORIG = {name: getattr(orc, name) for name in
         ("visible_mask", "kv_head_of", "scores", "masked_softmax", "log_sum_exp", "weighted_values")}

MUTANTS = [
    ("visible_mask", _mask_no_diagonal),
    ("visible_mask", _mask_bidir_window_short),
    ("visible_mask", _mask_left_window_long),
    ("visible_mask", _mask_positions_ignore_context),
    ("visible_mask", _mask_causal_for_everyone),
    ("kv_head_of", _gqa_modulo),
    ("scores", _scores_no_scale),
    ("scores", _scores_sign),
    ("masked_softmax", _softmax_unmasked_sum),
    ("masked_softmax", _softmax_no_normalise),
    ("log_sum_exp", _lse_drop_max),
    ("weighted_values", _values_shifted),
    ("weighted_values", _values_transposed_features),
]

PIN_CALLS = [
    lambda: [pins.test_causal_rows_match_bruteforce_triangular(c, n, W)
             for c, n, W in [(0, 7, -1), (5, 6, -1), (4, 9, 2), (0, 5, 0), (3, 4, 10)]],
    lambda: [pins.test_bidirectional_window_rows_match_bruteforce(c, n, W)
             for c, n, W in [(3, 6, 1), (0, 8, 2), (6, 4, 3), (2, 5, 0)]],
    lambda: [pins.test_bidirectional_wide_window_equals_unmasked_sdpa(W) for W in (-1, 64)],
    pins.test_causal_without_context_equals_sdpa_is_causal,
    pins.test_window_counts_golden,
    pins.test_window_counts_edge_clipping,
    pins.test_q_zero_gives_mean_of_visible_values,
    pins.test_single_visible_key_returns_its_value_exactly,
    pins.test_worked_example_golden,
    pins.test_bidirectional_permutation_equivariance,
    pins.test_causal_output_ignores_future_tokens,
]


def _caught(monkeypatch, name, fn):
    monkeypatch.setattr(orc, name, fn)
    for call in PIN_CALLS:
        try:
            call()
        except (AssertionError, ValueError, IndexError):
            return True
    return False


def test_unmutated_oracle_passes_every_pin():
    for call in PIN_CALLS:
        call()


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[f.__name__ for _, f in MUTANTS])
def test_pins_catch_planted_mistake(monkeypatch, name, fn):
    assert _caught(monkeypatch, name, fn), f"planted mistake {fn.__name__} in {name} went unnoticed"


def test_gqa_mistake_caught_by_head_pin(monkeypatch):
    monkeypatch.setattr(orc, "kv_head_of", _gqa_modulo)
    with pytest.raises(AssertionError):
        pins.test_gqa_mapping_and_head_duplication()
