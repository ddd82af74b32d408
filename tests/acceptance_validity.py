"""Which acceptance decisions are correct when the statistics carry rounding.

The acceptance rule of a denoise step (DiffusionGemma, agentlenshq page,
"sampling loop and entropy-bounded denoising"; 24-ai.news page, "the mechanism
for deciding finished tokens") ranks a canvas's open positions by confidence
and accepts them, most confident first, while the running entropy stays
within the budget (the first is always accepted).  A GPU computes entropy and
confidence in fp32; they agree with the fp64 oracle only within a tolerance.
Where two confidences lie within that tolerance of each other, or the running
entropy at the cut lies within it of the budget, more than one decision is
correct.  This module states exactly which ones, from the fp64 statistics
alone (no GPU value enters it):

* the accepted set is a prefix of some ranking consistent with the tolerance:
  no open row left out is clearly more confident than a row taken;
* the entropies taken (beyond the first row) sum to at most the budget, within
  the tolerance;
* no further row could have been taken: some row that may come next in such a
  ranking would push the sum past the budget, within the tolerance.

When the fp64 decision is "clear" (the taken rows are separated from the rest
by more than the tolerance and both budget margins exceed it) these three
conditions admit exactly that decision, so callers compare it bit for bit.
"""

from __future__ import annotations

import numpy as np

import oracle.acceptance as acc

# the statistics tolerance the GPU parity tests hold entropy and confidence to
H_RTOL, H_ATOL = 1e-4, 1e-4
C_RTOL, C_ATOL = 1e-4, 1e-7
FP32_EPS = 2.0 ** -23


def tolerances(H0, c0):
    H0 = np.asarray(H0, dtype=np.float64)
    c0 = np.asarray(c0, dtype=np.float64)
    return H_ATOL + H_RTOL * np.abs(H0), C_ATOL + C_RTOL * np.abs(c0)


def _sum_tol(eH, idx, total, budget):
    """Tolerance of an fp32 running sum over rows ``idx``: each term's own
    tolerance plus one fp32 rounding of the running value per term."""
    return float(eH[idx].sum()) + len(idx) * FP32_EPS * (abs(total) + abs(budget))


def _next_candidates(c0, ec, rest):
    """Rows of ``rest`` that may come first among them in a consistent ranking:
    no other row of ``rest`` is clearly more confident."""
    if len(rest) == 0:
        return rest
    top = np.max(c0[rest] - ec[rest])
    return rest[c0[rest] + ec[rest] >= top]


def check_accept(new, open_, H0, c0, budget):
    """(ok, reason) for ``new`` (bool, rows taken this step) of one canvas whose
    open rows are ``open_``, against the fp64 statistics ``H0``, ``c0``."""
    new = np.asarray(new, dtype=bool)
    open_ = np.asarray(open_, dtype=bool)
    H0 = np.asarray(H0, dtype=np.float64)
    c0 = np.asarray(c0, dtype=np.float64)
    eH, ec = tolerances(H0, c0)
    if (new & ~open_).any():
        return False, "a row taken that was not open"
    taken = np.flatnonzero(new)
    rest = np.flatnonzero(open_ & ~new)
    if not open_.any():
        return True, "no open row"
    if len(taken) == 0:
        return False, "no row taken although rows were open"
    if len(rest) and np.max(c0[rest] - ec[rest]) > np.min(c0[taken] + ec[taken]):
        return False, "a row left out is clearly more confident than a row taken"
    S = float(H0[taken].sum())
    eS = _sum_tol(eH, taken, S, budget)
    if len(taken) > 1 and S - eS > budget:
        return False, f"entropy taken {S:.6g} exceeds the budget {budget:.6g}"
    cand = _next_candidates(c0, ec, rest)
    if len(cand) and all(S + H0[j] + eS + eH[j] <= budget for j in cand):
        return False, "another row fits within the budget"
    return True, "valid"


def clear_accept(open_, H0, c0, budget):
    """The fp64 decision of one canvas and whether it is clear (the only
    decision ``check_accept`` admits)."""
    open_ = np.asarray(open_, dtype=bool)
    H0 = np.asarray(H0, dtype=np.float64)
    c0 = np.asarray(c0, dtype=np.float64)
    eH, ec = tolerances(H0, c0)
    dec = acc.accept(H0, c0, ~open_, budget) & open_
    taken = np.flatnonzero(dec)
    rest = np.flatnonzero(open_ & ~dec)
    if len(taken) == 0:
        return dec, True
    if len(rest) and np.min(c0[taken] - ec[taken]) <= np.max(c0[rest] + ec[rest]):
        return dec, False
    S = float(H0[taken].sum())
    eS = _sum_tol(eH, taken, S, budget)
    if len(taken) > 1 and S + eS >= budget:
        return dec, False
    cand = _next_candidates(c0, ec, rest)
    if any(S + H0[j] - eS - eH[j] <= budget for j in cand):
        return dec, False
    return dec, True


def check_converge(converged, stable, argmax_now, argmax_prev, stable_before, H0, tau, patience,
                   step, max_steps):
    """(ok, clear, reason) for one canvas's convergence outputs.  The stable
    counter depends only on the argmax (exact); the mean-entropy test is
    ambiguous only when the fp64 mean lies within the tolerance of tau."""
    cv0, st0 = acc.converge(argmax_now, argmax_prev, stable_before, H0, tau, patience, step,
                            max_steps)
    if int(stable) != st0:
        return False, True, f"stable {stable} != {st0}"
    H0 = np.asarray(H0, dtype=np.float64)
    eH, _ = tolerances(H0, np.zeros_like(H0))
    mean = float(H0.sum()) / len(H0)
    e_mean = float(eH.mean()) + len(H0) * FP32_EPS * (abs(mean) + abs(tau))
    forced = step + 1 >= max_steps
    ambiguous = (not forced) and st0 >= patience and abs(mean - tau) <= e_mean
    if ambiguous:
        return True, False, "mean entropy within the tolerance of tau: either answer"
    return bool(converged) == cv0, True, f"converged {bool(converged)} != {cv0}"
