"""Plain fp64 CPU oracle of the dual-mode attention forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may call it.  It shares no code with the CUDA library.

What it computes (the plain definition, written out; no blocking, no online
softmax, no split-KV):

* A batch holds ``B`` sequences.  Sequence ``s`` has ``ctx_len[s]`` cached
  tokens at absolute positions ``0 .. c-1`` and ``n = cu_q[s+1]-cu_q[s]``
  query tokens at positions ``c .. c+n-1``.  Its key/value rows are the ``c``
  cached rows followed by the ``n`` rows of its own query tokens, so it owns
  ``L = c + n`` KV rows, stored contiguously after the previous sequences'.
* Encoder mode (prefill / incremental prefill / commit) is causal: a query at
  position ``i`` sees keys ``j <= i``.  DiffusionGemma page (agentlenshq):
  section "dual-mode operation" (encoder mode uses causal attention) and the
  developer guide (molayo1419), section "block autoregressive denoising",
  prefill item.
* Decoder (denoise) mode is bidirectional: every canvas query sees every
  cached key and every canvas key.  Same two pages: "dual-mode operation"
  (decoder mode, bidirectional) and the denoising item of "block
  autoregressive denoising" (a canvas query attends to all canvas tokens and
  the KV cache).
* The causal / bidirectional choice is made per sequence inside one batch.
  agentlenshq page, section "dynamic per-sequence causal attention";
  24-ai.news page, section "integration into vLLM" (mixed batches).
* On a sliding-window layer a causal query sees the ``W`` preceding tokens
  (plus itself, ``W+1`` keys), a bidirectional query sees ``W`` tokens on each
  side (``2W+1`` keys).  agentlenshq page, section "symmetric sliding-window
  attention"; 24-ai.news page, "why diffusion differs" (windows of +-W).
* Readings where the pages are silent (stated as assumptions): a causal query
  sees itself; windows are measured in absolute positions over context plus
  canvas and are clipped at ``0`` and ``L-1``; ``window < 0`` means a full
  layer and ``window == 0`` means "self only"; query head ``h`` reads KV head
  ``h // (Hq // Hkv)``; scores are ``scale * q.k`` with no soft-capping, bias
  or sinks; ``lse`` is the natural log of the sum of ``exp(score)`` over the
  visible keys.

Every step is its own small function so a test can plant a mistake in exactly
one of them and check that the pins notice.
"""

from __future__ import annotations

import numpy as np

MODE_CAUSAL = 0
MODE_BIDIRECTIONAL = 1


def visible_mask(ctx_len: int, n_q: int, causal: bool, window: int,
                 t_begin: int = 0, t_end: int | None = None) -> np.ndarray:
    """Boolean mask ``[t_end-t_begin, ctx_len+n_q]``: row ``t`` (query token
    ``t_begin+t`` of the sequence, absolute position ``i = ctx_len + t``),
    column ``j`` (key position) is True when the query may attend to the key.

    Rules (agentlenshq page, "dual-mode operation" and "symmetric
    sliding-window attention"):
      key exists:            j < L                (L = ctx_len + n_q)
      window, left side:     j >= i - W           (only when W >= 0)
      causal:                j <= i
      bidirectional window:  j <= i + W           (only when W >= 0)
    """
    if t_end is None:
        t_end = n_q
    L = ctx_len + n_q
    i = ctx_len + np.arange(t_begin, t_end, dtype=np.int64)[:, None]
    j = np.arange(L, dtype=np.int64)[None, :]
    vis = np.broadcast_to(j < L, (t_end - t_begin, L)).copy()
    if window >= 0:
        vis &= j >= i - window
    if causal:
        vis &= j <= i
    elif window >= 0:
        vis &= j <= i + window
    return vis


def kv_head_of(h: int, num_q_heads: int, num_kv_heads: int) -> int:
    """GQA: consecutive query heads share one KV head (an assumption; the
    pages do not describe the head layout)."""
    return h // (num_q_heads // num_kv_heads)


def scores(q_rows: np.ndarray, k_rows: np.ndarray, scale: float) -> np.ndarray:
    """``scale * q . k`` for every (query row, key row) pair, fp64."""
    return scale * (q_rows @ k_rows.T)


def masked_softmax(z: np.ndarray, mask: np.ndarray):
    """Row-wise softmax of ``z`` restricted to ``mask``.  Returns the weights
    (zero where masked), the row maximum ``m`` over visible entries and the
    row sum ``l = sum exp(z - m)`` over visible entries."""
    if not np.all(mask.any(axis=1)):
        raise ValueError("a query row has no visible key")
    zm = np.where(mask, z, -np.inf)
    m = zm.max(axis=1)
    e = np.where(mask, np.exp(zm - m[:, None]), 0.0)
    l = e.sum(axis=1)
    return e / l[:, None], m, l


def log_sum_exp(m: np.ndarray, l: np.ndarray) -> np.ndarray:
    """Natural-log LSE of the visible scores from the max and the shifted sum."""
    return m + np.log(l)


def weighted_values(w: np.ndarray, v_rows: np.ndarray) -> np.ndarray:
    """Softmax weights times the value rows."""
    return w @ v_rows


def _check_batch(cu_q, ctx_len, mode, total_q, total_kv, num_q_heads, num_kv_heads):
    B = len(ctx_len)
    if len(cu_q) != B + 1 or len(mode) != B:
        raise ValueError("cu_q must have num_seqs+1 entries and mode num_seqs")
    if cu_q[0] != 0 or cu_q[-1] != total_q or np.any(np.diff(cu_q) < 0):
        raise ValueError("cu_q must start at 0, end at total_q and not decrease")
    if np.any(np.asarray(ctx_len) < 0):
        raise ValueError("ctx_len must be >= 0")
    if int(np.sum(ctx_len)) + total_q > total_kv:
        raise ValueError("KV buffer shorter than sum(ctx_len + n_q)")
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    for md in mode:
        if int(md) not in (MODE_CAUSAL, MODE_BIDIRECTIONAL):
            raise ValueError("mode must be 0 (causal) or 1 (bidirectional)")


def attention(q, k, v, cu_q, ctx_len, mode, window, scale,
              query_rows=None, heads=None, chunk=64):
    """Dual-mode attention forward, fp64.

    q:        [total_q, Hq, D]   query rows, sequences packed back to back
    k, v:     [total_kv, Hkv, D] key/value rows; sequence s owns rows
              ``kv_off[s] .. kv_off[s] + ctx_len[s] + n_s - 1`` where
              ``kv_off[s] = sum_{r<s} (ctx_len[r] + n_r)``
    cu_q:     [B+1] query offsets;  ctx_len: [B];  mode: [B] (0 causal, 1 bidir)
    window:   -1 for a full layer, W >= 0 for a sliding-window layer
    scale:    softmax scale applied to q.k
    query_rows: optional iterable of global query rows to evaluate (others
              are left NaN); default all rows
    heads:    optional iterable of query heads to evaluate; default all

    Returns ``(out [total_q, Hq, D] float64, lse [total_q, Hq] float64)``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    cu_q = np.asarray(cu_q, dtype=np.int64)
    ctx_len = np.asarray(ctx_len, dtype=np.int64)
    mode = np.asarray(mode, dtype=np.int64)
    total_q, Hq, D = q.shape
    total_kv, Hkv, _ = k.shape
    _check_batch(cu_q, ctx_len, mode, total_q, total_kv, Hq, Hkv)

    out = np.full((total_q, Hq, D), np.nan)
    lse = np.full((total_q, Hq), np.nan)
    want = None if query_rows is None else np.zeros(total_q, dtype=bool)
    if want is not None:
        want[np.asarray(list(query_rows), dtype=np.int64)] = True
    head_list = range(Hq) if heads is None else list(heads)

    kv_off = 0
    for s in range(len(ctx_len)):
        c = int(ctx_len[s])
        q0, q1 = int(cu_q[s]), int(cu_q[s + 1])
        n = q1 - q0
        L = c + n
        causal = int(mode[s]) == MODE_CAUSAL
        for t0 in range(0, n, chunk):
            t1 = min(n, t0 + chunk)
            rows = np.arange(q0 + t0, q0 + t1)
            sel = np.ones(t1 - t0, dtype=bool) if want is None else want[rows]
            if not sel.any():
                continue
            rows = rows[sel]
            mask = visible_mask(c, n, causal, window, t0, t1)[sel]
            for h in head_list:
                g = kv_head_of(h, Hq, Hkv)
                z = scores(q[rows, h, :], k[kv_off:kv_off + L, g, :], scale)
                w, m, l = masked_softmax(z, mask)
                out[rows, h, :] = weighted_values(w, v[kv_off:kv_off + L, g, :])
                lse[rows, h] = log_sum_exp(m, l)
        kv_off += L
    return out, lse

