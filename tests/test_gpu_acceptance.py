"""GPU parity of the entropy-bounded acceptance step (called through the C ABI)
against the CPU fp64 oracle on the same seeded bf16 logits.

Entropy and confidence are compared with the fp64 oracle within a tolerance;
the argmax is compared exactly (both sides see the same bf16 values; ties go to
the lower index).  The decisions (ranking, budget cut, convergence) are
compared with the fp64 oracle's own decisions, made from the fp64 statistics:
bit for bit on every canvas where that decision is clear, and, where a near
tie or a sum on the budget lets rounding pick another correct answer, through
a complete validity checker that uses only the fp64 statistics.  No GPU value
is passed into the oracle.
"""

import numpy as np
import pytest
import torch

import oracle.acceptance as acc
from acceptance_validity import check_accept, check_converge, clear_accept
from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    assert binding.status() == binding.DG_OK


def run_and_check(wl, budget, tau, patience, step, max_steps, seed=0):
    """Runs one step; returns (result, canvases whose decision was clear)."""
    x, cu = wls.make_logits(wl, device="cuda")
    rows = wl.rows
    rng = np.random.default_rng(seed)
    acc_in = torch.from_numpy((rng.uniform(size=rows) < 0.25).astype(np.uint8)).cuda()
    prev = torch.from_numpy(rng.integers(0, wl.vocab, rows).astype(np.int32))
    H0, c0, a0 = acc.row_stats(x.float().cpu().numpy())
    # half of the canvases keep every argmax of the previous step
    nb = len(wl.canvases)
    cu_h = cu.numpy()
    for b in range(0, nb, 2):
        prev[cu_h[b]:cu_h[b + 1]] = torch.from_numpy(a0[cu_h[b]:cu_h[b + 1]].astype(np.int32))
    stable_in = torch.from_numpy(rng.integers(0, 4, nb).astype(np.int32)).cuda()
    res = binding.accept_step(x, cu.cuda(), acc_in, prev.cuda(), stable_in, budget, tau, patience,
                              step, max_steps)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    np.testing.assert_allclose(res["entropy"].cpu().numpy(), H0, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(res["confidence"].cpu().numpy(), c0, rtol=1e-4, atol=1e-7)
    np.testing.assert_array_equal(res["argmax"].cpu().numpy(), a0)
    acc_np = acc_in.cpu().numpy().astype(bool)
    got_acc = res["accepted"].cpu().numpy().astype(bool)
    prev_np = prev.numpy()
    st = stable_in.cpu().numpy()
    clear = 0
    for b in range(nb):
        r0, r1 = cu_h[b], cu_h[b + 1]
        before = acc_np[r0:r1]
        got = got_acc[r0:r1]
        assert (got | ~before).all(), f"canvas {b}: an earlier acceptance was dropped"
        new = got & ~before
        ok, why = check_accept(new, ~before, H0[r0:r1], c0[r0:r1], budget)
        assert ok, f"canvas {b}: {why}"
        dec, is_clear = clear_accept(~before, H0[r0:r1], c0[r0:r1], budget)
        if is_clear:
            np.testing.assert_array_equal(new, dec, err_msg=f"canvas {b}")
        ok, c_clear, why = check_converge(res["converged"][b].item(), res["stable"][b].item(),
                                          a0[r0:r1], prev_np[r0:r1], int(st[b]), H0[r0:r1], tau,
                                          patience, step, max_steps)
        assert ok, f"canvas {b}: {why}"
        clear += int(is_clear and c_clear)
    return res, clear


@pytest.mark.parametrize("budget", [0.0, 0.5, 4.0, 1e6])
def test_ragged_canvases_unaligned_vocab(budget):
    _, clear = run_and_check(wls.LOGITS_WORKLOADS["accept_small"], budget, 3.0, 2, 5, 48)
    assert clear >= 1  # at least one canvas compared bit for bit with the fp64 decision


def test_step_limit_and_threshold():
    wl = wls.LOGITS_WORKLOADS["accept_small"]
    run_and_check(wl, 1.0, 100.0, 1, 47, 48, seed=3)   # step limit reached
    run_and_check(wl, 1.0, 0.0, 0, 0, 48, seed=4)      # threshold never met


def test_full_vocab_four_canvases():
    _, clear = run_and_check(wls.LOGITS_WORKLOADS["accept_step"], 2.0, 4.0, 3, 10, 48, seed=5)
    assert clear >= 2


def test_tiny_vocab_and_ties():
    wl = wls.LogitsWorkload("ties", (5, 3), 9, 30)
    x = torch.zeros((8, 9), dtype=torch.bfloat16, device="cuda")
    x[1, 4] = x[1, 7] = 2.0                            # tie: lowest index wins
    x[2, :] = 1.0                                      # all equal: index 0, entropy ln 9
    x[3, 8] = 5.0
    cu = torch.tensor([0, 5, 8], dtype=torch.int32, device="cuda")
    z8 = torch.zeros(8, dtype=torch.uint8, device="cuda")
    z32 = torch.zeros(8, dtype=torch.int32, device="cuda")
    res = binding.accept_step(x, cu, z8, z32, torch.zeros(2, dtype=torch.int32, device="cuda"),
                              0.1, 1.0, 1, 0, 10)
    torch.cuda.synchronize()
    a = res["argmax"].cpu().numpy()
    assert a[1] == 4 and a[2] == 0 and a[3] == 8
    assert abs(res["entropy"][2].item() - np.log(9)) < 1e-5
    # at least one position of each canvas is accepted even with a tiny budget
    got = res["accepted"].cpu().numpy()
    assert got[:5].sum() >= 1 and got[5:].sum() >= 1


def test_oversized_canvas_sets_status():
    x = torch.zeros((1100, 16), dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 1100], dtype=torch.int32, device="cuda")
    z8 = torch.zeros(1100, dtype=torch.uint8, device="cuda")
    z32 = torch.zeros(1100, dtype=torch.int32, device="cuda")
    binding.accept_step(x, cu, z8, z32, torch.zeros(1, dtype=torch.int32, device="cuda"), 1.0, 1.0, 1, 0, 4)
    assert binding.status() == binding.DG_ERR_INVALID_ARG


@pytest.mark.parametrize("vocab", [16383, 16385, 32771, 40000])
def test_chunk_edges_ties_and_masked_logits(vocab):
    """Vocabularies on both sides of a chunk multiple (rows start at every
    misalignment), maxima at the first / last position, ties across chunks
    and rows with -inf (masked) logits; statistics against the oracle."""
    g = torch.Generator().manual_seed(vocab)
    rows = 9
    x = (torch.randn(rows, vocab, generator=g) * 2).to(torch.bfloat16)
    x[0, vocab - 1] = 30.0                         # max at the last position
    x[1, 0] = 30.0                                 # max at the first position
    p_tie = min(16383, vocab // 2)
    x[2, p_tie] = x[2, vocab - 2] = 30.0           # tie across chunks: the lower wins
    x[3, 5] = x[3, 16390 % vocab] = x[3, vocab - 1] = 25.0
    x[4, vocab // 2:] = float("-inf")              # upper half masked
    x[5, :] = float("-inf")
    x[5, [3, vocab // 3, vocab - 4]] = torch.tensor([1.0, 2.0, 2.0], dtype=torch.bfloat16)
    x[6, :] = 0.0                                  # uniform: entropy ln V, argmax 0
    xd = x.cuda()
    cu = torch.tensor([0, rows], dtype=torch.int32, device="cuda")
    z8 = torch.zeros(rows, dtype=torch.uint8, device="cuda")
    z32 = torch.zeros(rows, dtype=torch.int32, device="cuda")
    res = binding.accept_step(xd, cu, z8, z32, torch.zeros(1, dtype=torch.int32, device="cuda"),
                              1.0, 1.0, 1, 0, 10)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    H0, c0, a0 = acc.row_stats(x.float().numpy())
    np.testing.assert_allclose(res["entropy"].cpu().numpy(), H0, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(res["confidence"].cpu().numpy(), c0, rtol=1e-4, atol=1e-7)
    np.testing.assert_array_equal(res["argmax"].cpu().numpy(), a0)
    assert a0[2] == p_tie and a0[5] == vocab // 3 and a0[6] == 0
