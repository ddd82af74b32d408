"""The two ways a call gets its work list, through the C ABI.

Batches of at most 256 query tiles with contiguous K/V have no work-list
grid: every CTA of the attention grid builds the list for itself, from the
same helpers as the work-list grid.  The tiles, unit ranges, KV visiting
order and merge contributors are the same either way, so the outputs must be
bit-identical to those of the separate grid (DG_ATTN_FUSED_WL=0).  Larger
batches take the separate grid; one such batch is checked against the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
LSE_ABS = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    assert binding.status() == binding.DG_OK


def to_dev(batch):
    return {k: batch[k].cuda().contiguous() for k in ("q", "k", "v", "cu_q", "ctx_len", "mode")}


def run(dev, window, scale):
    out, lse = binding.forward(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["ctx_len"], dev["mode"],
                               window, scale)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    return out, lse


CASES = [
    # (seed, seqs (ctx, n, mode), Hq, Hkv, D, windows)
    (90, ((300, 256, 1), (0, 333, 0), (1000, 200, 1)), 8, 4, 128, (-1, 50)),
    (91, ((700, 256, 1), (5, 100, 0)), 16, 2, 256, (-1, 129)),
    (92, ((0, 1, 0), (5, 1, 1), (0, 77, 1), (130, 3, 0), (200, 129, 1)), 2, 1, 64, (-1, 0, 127)),
]


@pytest.mark.parametrize("ctas", [None, "7"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_in_grid_work_list_is_bit_identical(case, ctas, monkeypatch):
    seed, seqs, Hq, Hkv, D, windows = CASES[case]
    if ctas is not None:
        monkeypatch.setenv("DG_ATTN_NUM_CTAS", ctas)
    wl, batch = wls.random_batch(seed, seqs, Hq, Hkv, D, -1)
    dev = to_dev(batch)
    for W in windows:
        monkeypatch.delenv("DG_ATTN_FUSED_WL", raising=False)
        out_a, lse_a = run(dev, W, wl.scale)
        monkeypatch.setenv("DG_ATTN_FUSED_WL", "0")
        out_b, lse_b = run(dev, W, wl.scale)
        assert torch.equal(out_a, out_b), f"case {case} W={W}: outputs differ"
        assert torch.equal(lse_a, lse_b), f"case {case} W={W}: LSEs differ"


def test_in_grid_work_list_is_bit_identical_e4m3(monkeypatch):
    b = wls.make_fp8_batch(wls.Workload("fp8", ((700, 256, 1), (5, 100, 0)), 16, 2, 256, -1, 93))
    d = {k: b[k].cuda() for k in ("q8", "k8", "v8", "cu_q", "ctx_len", "mode")}

    def go():
        out, lse = binding.forward_fp8(d["q8"], d["k8"], d["v8"], d["cu_q"], d["ctx_len"], d["mode"], -1,
                                       b["scale"], b["q_scale"], b["k_scale"], b["v_scale"])
        torch.cuda.synchronize()
        assert binding.status() == binding.DG_OK
        return out, lse

    monkeypatch.delenv("DG_ATTN_FUSED_WL", raising=False)
    out_a, lse_a = go()
    monkeypatch.setenv("DG_ATTN_FUSED_WL", "0")
    out_b, lse_b = go()
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)


@pytest.mark.parametrize("fused", [None, "0"])
def test_bad_metadata_either_way(fused, monkeypatch):
    """Device-side metadata checks run in whichever grid builds the list."""
    if fused is not None:
        monkeypatch.setenv("DG_ATTN_FUSED_WL", fused)
    wl, batch = wls.random_batch(94, ((10, 20, 1), (0, 12, 0)), 2, 1, 64, -1)
    dev = to_dev(batch)
    bad = dev["cu_q"].clone()
    bad[2] = 31  # cu_q[B] != total_q
    binding.forward(dev["q"], dev["k"], dev["v"], bad, dev["ctx_len"], dev["mode"], -1, wl.scale)
    assert binding.status() == binding.DG_ERR_INVALID_ARG
    neg = dev["ctx_len"].clone()
    neg[1] = -3
    binding.forward(dev["q"], dev["k"], dev["v"], dev["cu_q"], neg, dev["mode"], -1, wl.scale)
    assert binding.status() == binding.DG_ERR_INVALID_ARG
    out, lse = run(dev, -1, wl.scale)  # a good call afterwards
    ref_o, ref_l = oracle.attention(batch["q"].double().numpy(), batch["k"].double().numpy(),
                                    batch["v"].double().numpy(), batch["cu_q"].numpy(),
                                    batch["ctx_len"].numpy(), batch["mode"].numpy(), -1, wl.scale)
    assert np.abs(out.double().cpu().numpy() - ref_o).max() <= MAX_ABS


def test_batch_past_the_in_grid_limit():
    """48 sequences x 8 KV heads x 3 tiles = 1152 query tiles: the separate
    work-list grid, against the oracle."""
    rng = np.random.default_rng(95)
    seqs = tuple((int(rng.integers(0, 60)), int(rng.integers(130, 190)), int(rng.integers(0, 2)))
                 for _ in range(48))
    wl, batch = wls.random_batch(95, seqs, 16, 8, 64, -1)
    dev = to_dev(batch)
    for W in (-1, 33):
        out, lse = run(dev, W, wl.scale)
        ref_o, ref_l = oracle.attention(batch["q"].double().numpy(), batch["k"].double().numpy(),
                                        batch["v"].double().numpy(), batch["cu_q"].numpy(),
                                        batch["ctx_len"].numpy(), batch["mode"].numpy(), W, wl.scale)
        d = np.abs(out.double().cpu().numpy() - ref_o)
        assert d.max() <= MAX_ABS, f"W={W}: max|dout|={d.max():.3g}"
        assert np.abs(lse.double().cpu().numpy() - ref_l).max() <= LSE_ABS
