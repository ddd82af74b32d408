"""Plant plausible mistakes in the e4m3 decoder of the FP8 oracle (on the
CPU, one at a time) and check that the pins in ``test_fp8_oracle.py`` catch
every one."""

import numpy as np
import pytest

import oracle.fp8 as f8
import test_fp8_oracle as pins

_ORIG = f8.e4m3_to_float


def _bias_8(codes):
    return _ORIG(codes) / 2.0


def _no_subnormals(codes):
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    out = _ORIG(codes)
    e = (b >> 3) & 0xF
    m = b & 7
    return np.where((e == 0) & (m > 0), np.sign(out) * (1 + m / 8.0) * 2.0 ** -7, out)


def _unsigned(codes):
    return np.abs(_ORIG(codes))


def _mantissa_sixteenths(codes):
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    e = (b >> 3) & 0xF
    m = b & 7
    out = _ORIG(codes)
    alt = np.sign(out) * (1 + m / 16.0) * np.exp2(e - 7.0)
    return np.where((e > 0) & ~np.isnan(out), alt, out)


def _top_binade_is_nan(codes):
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return np.where(((b >> 3) & 0xF) == 15, np.nan, _ORIG(codes))


MUTANTS = [_bias_8, _no_subnormals, _unsigned, _mantissa_sixteenths, _top_binade_is_nan]

PIN_CALLS = [pins.test_golden_codes, pins.test_every_code_matches_the_library_type,
             pins.test_unit_scales_equal_the_attention_of_the_decoded_values,
             pins.test_scales_act_as_the_algebra_says]


def test_unmutated_oracle_passes_every_pin():
    for call in PIN_CALLS:
        call()


@pytest.mark.parametrize("fn", MUTANTS, ids=[f.__name__ for f in MUTANTS])
def test_pins_catch_planted_mistake(monkeypatch, fn):
    monkeypatch.setattr(f8, "e4m3_to_float", fn)
    caught = False
    for call in PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                call()
        except (AssertionError, ValueError):
            caught = True
            break
    assert caught, fn.__name__
