"""Plain CPU oracle of the entropy-bounded acceptance step of a denoise step.

TEST INFRASTRUCTURE ONLY: only the tests, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` use it; it shares no code with the CUDA library.

What one denoise step decides after the LM head (DiffusionGemma, agentlenshq
page, section "sampling loop and entropy-bounded denoising"; 24-ai.news page,
section "the mechanism for deciding finished tokens"):

* every canvas position gets a probability distribution over the vocabulary,
  a confidence and an entropy;
* positions are accepted from the most to the least confident until the
  accumulated entropy passes a fixed budget;
* a canvas has converged when its argmax predictions stayed the same for
  several steps and the mean per-token entropy is under a threshold, or when a
  step limit is reached.

Readings where the pages are silent (stated as assumptions):

* the distribution is softmax(logits) at temperature 1; confidence is its
  largest probability; the candidate token is its argmax, the lowest index on
  ties; entropy is in nats;
* only positions not accepted in earlier steps take part in the ranking; ties
  in confidence go to the lower position;
* a position is accepted while the running entropy sum, including it, stays
  within the budget; the most confident position is always accepted, so every
  step makes progress; the position that would push the sum past the budget
  and every later one stay open;
* "argmax stable" means the argmax of every position of the canvas equals the
  previous step's; ``stable`` counts consecutive such steps; "mean per-token
  entropy" averages over all positions of the canvas.
"""

from __future__ import annotations

import numpy as np


def row_stats(logits):
    """Per row of ``logits`` [rows, V]: entropy H (nats), confidence c (max
    probability) and argmax a (lowest index on ties), in fp64."""
    x = np.asarray(logits, dtype=np.float64)
    m = x.max(axis=1, keepdims=True)
    e = np.exp(x - m)
    z = e.sum(axis=1, keepdims=True)
    p = e / z
    with np.errstate(divide="ignore", invalid="ignore"):
        plogp = np.where(p > 0, p * np.log(p), 0.0)
    H = -plogp.sum(axis=1)
    c = p.max(axis=1)
    a = np.argmax(x, axis=1)  # numpy returns the first (lowest) index of the maximum
    return H, c, a.astype(np.int64)


def confidence_order(c, candidates):
    """Indices of the candidate rows, most confident first (ties: lower index)."""
    idx = np.flatnonzero(candidates)
    # stable sort on -c keeps equal confidences in increasing index order
    return idx[np.argsort(-np.asarray(c)[idx], kind="stable")]


def accept(H, c, accepted_before, budget):
    """New accepted flags of one canvas (running entropy sum in fp64)."""
    accepted_before = np.asarray(accepted_before, dtype=bool)
    order = confidence_order(c, ~accepted_before)
    out = accepted_before.copy()
    run = 0.0
    H = np.asarray(H, dtype=np.float64)
    for k, i in enumerate(order):
        run += float(H[i])
        if k > 0 and run > budget:
            break
        out[i] = True
    return out


def converge(argmax_now, argmax_prev, stable_before, H, tau, patience, step, max_steps):
    """(converged, stable) of one canvas after this step (mean entropy in fp64)."""
    same = bool(np.array_equal(np.asarray(argmax_now), np.asarray(argmax_prev)))
    stable = stable_before + 1 if same else 0
    mean_h = float(np.sum(np.asarray(H, dtype=np.float64))) / len(H)
    converged = (stable >= patience and mean_h < tau) or (step + 1 >= max_steps)
    return bool(converged), int(stable)


def denoise_step(logits, cu_rows, accepted_before, argmax_prev, stable_before, budget, tau,
                 patience, step, max_steps):
    """Whole step for a batch of canvases (rows cu_rows[b] .. cu_rows[b+1]-1 of
    ``logits`` belong to canvas b).  Returns a dict with H, c, argmax, the new
    accepted flags, and per canvas the converged flag and stable counter."""
    H, c, a = row_stats(logits)
    acc = np.zeros(len(H), dtype=bool)
    conv, stab = [], []
    for b in range(len(cu_rows) - 1):
        r0, r1 = int(cu_rows[b]), int(cu_rows[b + 1])
        acc[r0:r1] = accept(H[r0:r1], c[r0:r1], accepted_before[r0:r1], budget)
        cv, st = converge(a[r0:r1], argmax_prev[r0:r1], int(stable_before[b]), H[r0:r1], tau,
                          patience, step, max_steps)
        conv.append(cv)
        stab.append(st)
    return dict(H=H, c=c, argmax=a, accepted=acc, converged=np.array(conv),
                stable=np.array(stab, dtype=np.int64))
