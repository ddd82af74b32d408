"""Plain CPU oracle of the self-conditioning input of a denoise step: the
probability-weighted average of the token embeddings under the previous
step's softmax distribution.

TEST INFRASTRUCTURE ONLY: only the tests, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` use it; it shares no code with the CUDA library.

What the pages fix (DiffusionGemma, agentlenshq page, "self-conditioning for
stability"; 24-ai.news page, the passage on the self-conditioning signal
between iterations): between denoise steps the model takes the full softmax
distribution of its previous prediction at every canvas position, turns it
into the probability-weighted average of the token embeddings, and feeds that
vector back in (through a gated MLP, which needs trained weights and is not
part of this path).

Readings where the pages are silent (stated as assumptions): the distribution
is softmax(logits) at temperature 1 over the whole vocabulary, the same one the
acceptance step uses; the embedding table is the input embedding
``E [vocab, d_model]``; the average is ``sum_v p_v E[v, :]`` with no extra
scaling.
"""

from __future__ import annotations

import numpy as np


def softmax_rows(logits):
    """Row-wise softmax of ``logits`` [rows, V] in fp64 (max-shifted)."""
    x = np.asarray(logits, dtype=np.float64)
    m = x.max(axis=1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=1, keepdims=True)


def weighted_embedding(p, E):
    """``p`` [rows, V] times ``E`` [V, d] in fp64: row r is sum_v p[r, v] E[v]."""
    return np.asarray(p, dtype=np.float64) @ np.asarray(E, dtype=np.float64)


def self_conditioning(logits, E):
    """The self-conditioning vector of every row: ``softmax(logits) @ E``,
    ``[rows, d_model]`` fp64."""
    return weighted_embedding(softmax_rows(logits), E)
