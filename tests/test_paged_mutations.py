"""Plant plausible mistakes in the paged-cache oracle (on the CPU, one at a
time) and check that the pins in ``test_paged_oracle.py`` catch every one."""

import numpy as np
import pytest

import oracle.paged as pg
import test_paged_oracle as pins

_ORIG = {name: getattr(pg, name) for name in ("page_slot", "append_kv", "gather_kv")}


def _slot_swapped(block_table_row, pos, page_size):
    # page from the row within the page and vice versa
    return int(block_table_row[pos % page_size]), pos // page_size


def _slot_logical_page(block_table_row, pos, page_size):
    # forgets the table: logical page used as the physical page
    return pos // page_size, pos % page_size


def _append_one_late(cache, block_table, page_size, cu_q, ctx_len, new):
    return _ORIG["append_kv"](cache, block_table, page_size, cu_q, np.asarray(ctx_len) + 1, new)


def _append_first_table_row(cache, block_table, page_size, cu_q, ctx_len, new):
    bt = np.repeat(np.asarray(block_table)[:1], len(block_table), axis=0)
    return _ORIG["append_kv"](cache, bt, page_size, cu_q, ctx_len, new)


def _append_reversed_tokens(cache, block_table, page_size, cu_q, ctx_len, new):
    new = np.array(new, copy=True)
    for s in range(len(ctx_len)):
        new[cu_q[s]:cu_q[s + 1]] = new[cu_q[s]:cu_q[s + 1]][::-1]
    return _ORIG["append_kv"](cache, block_table, page_size, cu_q, ctx_len, new)


def _append_nothing(cache, block_table, page_size, cu_q, ctx_len, new):
    return np.array(cache, copy=True)


def _gather_skip_first(cache, block_table_row, L, page_size):
    rows = _ORIG["gather_kv"](cache, block_table_row, L + 1, page_size) if L else \
        _ORIG["gather_kv"](cache, block_table_row, L, page_size)
    return rows[1:] if L else rows


def _gather_page_reversed(cache, block_table_row, L, page_size):
    rows = _ORIG["gather_kv"](cache, block_table_row, L, page_size)
    out = rows.copy()
    for p0 in range(0, L, page_size):
        out[p0:p0 + page_size] = rows[p0:p0 + page_size][::-1]
    return out


MUTANTS = [
    ("page_slot", _slot_swapped),
    ("page_slot", _slot_logical_page),
    ("append_kv", _append_one_late),
    ("append_kv", _append_first_table_row),
    ("append_kv", _append_reversed_tokens),
    ("append_kv", _append_nothing),
    ("gather_kv", _gather_skip_first),
    ("gather_kv", _gather_page_reversed),
]

PIN_CALLS = [
    pins.test_golden_append_and_gather,
    lambda: [pins.test_in_order_pages_equal_the_contiguous_layout(P) for P in (1, 2, 4, 16)],
    pins.test_relabelling_physical_pages_changes_nothing,
    pins.test_append_writes_exactly_the_query_positions,
    pins.test_canvas_rewrite_overwrites_the_previous_step,
    pins.test_without_new_rows_the_cache_is_read_as_is,
]


def _caught(monkeypatch, name, fn):
    monkeypatch.setattr(pg, name, fn)
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
    assert _caught(monkeypatch, name, fn), f"no pin caught the mutant {fn.__name__} of {name}"
