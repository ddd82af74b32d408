"""Plain CPU oracle of the paged KV cache: the append of a batch's new K/V rows
and the dual-mode attention read through the page table.

TEST INFRASTRUCTURE ONLY: only the tests, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` use it; it shares no code with the CUDA library.

What the pages fix (DiffusionGemma, agentlenshq page, "dual-mode operation"
and "sampling loop and entropy-bounded denoising"; developer guide
(molayo1419), "block autoregressive denoising", the prefill item):

* the encoder (causal) pass writes finished blocks into the KV cache, and each
  committed 256-token canvas is appended to that cache before the next canvas
  is denoised;
* vLLM's automatic prefix caching works unchanged, i.e. the cache is vLLM's
  block-based one.

Readings where the pages are silent (stated as assumptions):

* the cache is a pool of ``num_pages`` pages of ``page_size`` token rows, one
  pool for K and one for V, each ``[num_pages, page_size, Hkv, D]``;
* ``block_table[s, p]`` is the physical page holding positions
  ``p*page_size .. (p+1)*page_size - 1`` of sequence ``s``; entries past the
  sequence's last page are not read;
* a call first writes the K/V rows of its query tokens (``k_new``/``v_new``,
  packed like ``q``) at positions ``ctx_len[s] .. ctx_len[s]+n_s-1`` of their
  sequence (the commit block of a prefill / commit pass, or this step's
  canvas, which overwrites the previous step's canvas rows), then attends over
  positions ``0 .. ctx_len[s]+n_s-1`` read through the table, with the same
  masks as the contiguous layout;
* pages written by the append are owned by one sequence of the batch (shared
  prefix pages are only read).
"""

from __future__ import annotations

import numpy as np

from .attention import attention


def page_slot(block_table_row, pos: int, page_size: int):
    """(physical page, row within the page) of sequence position ``pos``."""
    return int(block_table_row[pos // page_size]), pos % page_size


def append_kv(cache, block_table, page_size: int, cu_q, ctx_len, new):
    """Copy of ``cache`` [num_pages, page_size, Hkv, D] with row ``r`` of
    ``new`` [total_q, Hkv, D] (query token ``t`` of sequence ``s``) written at
    position ``ctx_len[s] + t`` of sequence ``s``."""
    out = np.array(cache, copy=True)
    for s in range(len(ctx_len)):
        for t in range(int(cu_q[s + 1]) - int(cu_q[s])):
            page, row = page_slot(block_table[s], int(ctx_len[s]) + t, page_size)
            out[page, row] = new[int(cu_q[s]) + t]
    return out


def gather_kv(cache, block_table_row, L: int, page_size: int):
    """Positions ``0 .. L-1`` of one sequence, ``[L, Hkv, D]``, read through
    its page-table row."""
    rows = []
    for j in range(L):
        page, row = page_slot(block_table_row, j, page_size)
        rows.append(cache[page, row])
    return np.stack(rows) if rows else np.zeros((0,) + tuple(cache.shape[2:]), cache.dtype)


def paged_attention(q, k_new, v_new, k_cache, v_cache, block_table, page_size: int, cu_q,
                    ctx_len, mode, window: int, scale: float, query_rows=None, heads=None):
    """Append (when ``k_new``/``v_new`` are given), then attention over each
    sequence's positions read through the page table.  Returns
    ``(out, lse, k_cache_after, v_cache_after)``; ``query_rows`` / ``heads``
    restrict the attention output as in ``oracle.attention.attention``."""
    if k_new is not None:
        k_cache = append_kv(k_cache, block_table, page_size, cu_q, ctx_len, k_new)
        v_cache = append_kv(v_cache, block_table, page_size, cu_q, ctx_len, v_new)
    # the packed contiguous layout of the same keys: sequence after sequence
    ks, vs = [], []
    for s in range(len(ctx_len)):
        L = int(ctx_len[s]) + int(cu_q[s + 1]) - int(cu_q[s])
        ks.append(gather_kv(k_cache, block_table[s], L, page_size))
        vs.append(gather_kv(v_cache, block_table[s], L, page_size))
    k = np.concatenate(ks, axis=0)
    v = np.concatenate(vs, axis=0)
    out, lse = attention(q, k, v, cu_q, ctx_len, mode, window, scale, query_rows=query_rows,
                         heads=heads)
    return out, lse, k_cache, v_cache
