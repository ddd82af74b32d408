"""GPU edge cases of every entry point: empty batches, sequences with no
queries in the middle of a batch, the GQA extremes (one KV head for 128
query heads, i.e. one token per 128-row tile), and empty acceptance steps.
Compared with the oracles under the same bars as the main parity tests."""

import numpy as np
import pytest
import torch

import oracle
import oracle.acceptance as oacc
import oracle.paged as pg
from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls
from test_gpu_parity import EDGE_REL, check, f64, run_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    assert binding.status() == binding.DG_OK


def test_empty_batches_are_no_ops():
    lib = binding.load_library()
    dummy = torch.zeros(64, dtype=torch.uint8, device="cuda")
    ptr = dummy.data_ptr()
    stream = torch.cuda.current_stream().cuda_stream
    # no sequences, no queries: nothing is read or launched
    assert lib.dg_attn_forward(ptr, ptr, ptr, ptr, ptr, ptr, 0, 0, 0, 4, 2, 128, -1, 0.1, ptr, None,
                               None, 0, stream) == binding.DG_OK
    assert lib.dg_attn_forward_fp8(ptr, ptr, ptr, ptr, ptr, ptr, 0, 0, 0, 4, 2, 128, -1, 0.1, 1.0, 1.0, 1.0,
                                   ptr, None, None, 0, stream) == binding.DG_OK
    # sequences without queries
    cu = torch.zeros(3, dtype=torch.int32, device="cuda")
    ctx = torch.tensor([5, 9], dtype=torch.int32, device="cuda")
    mode = torch.ones(2, dtype=torch.uint8, device="cuda")
    assert lib.dg_attn_forward(ptr, ptr, ptr, cu.data_ptr(), ctx.data_ptr(), mode.data_ptr(), 2, 0, 14,
                               4, 2, 128, -1, 0.1, ptr, None, None, 0, stream) == binding.DG_OK
    # an acceptance step over no rows
    assert lib.dg_accept_step(ptr, 0, 16, cu.data_ptr(), 2, ptr, ptr, ptr, 1.0, 1.0, 1, 0, 4, ptr, ptr,
                              ptr, ptr, ptr, ptr, ptr, 0, stream) == binding.DG_OK
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK


@pytest.mark.parametrize("D", [64, 128, 256])
def test_sequences_without_queries(D):
    """Pure-context sequences (no queries this call) at the start, middle and
    end of a batch: they produce no tiles and shift the KV offsets only."""
    seqs = ((100, 0, 1), (50, 64, 1), (0, 0, 0), (30, 17, 0), (7, 0, 1))
    wl, b = wls.random_batch(300 + D, seqs, 4, 2, D, -1)
    dev = to_dev(b)
    for W in (-1, 20):
        out, lse = run_gpu(dev, W, wl.scale)
        ro, rl = oracle.attention(f64(b["q"]), f64(b["k"]), f64(b["v"]), b["cu_q"].numpy(),
                                  b["ctx_len"].numpy(), b["mode"].numpy(), W, wl.scale)
        check(f64(out), f64(lse), ro, rl, f"D={D} W={W}", rel=EDGE_REL)


@pytest.mark.parametrize("Hq,Hkv,D", [(128, 1, 64), (128, 1, 128), (16, 1, 256), (64, 2, 128)])
def test_gqa_extremes(Hq, Hkv, D):
    """G = Hq / Hkv up to 128: a 128-row tile then holds one token's heads."""
    seqs = ((40, 3, 1), (0, 5, 0), (300, 20, 1))
    wl, b = wls.random_batch(400 + Hq + D, seqs, Hq, Hkv, D, -1)
    dev = to_dev(b)
    for W in (-1, 7):
        out, lse = run_gpu(dev, W, wl.scale)
        ro, rl = oracle.attention(f64(b["q"]), f64(b["k"]), f64(b["v"]), b["cu_q"].numpy(),
                                  b["ctx_len"].numpy(), b["mode"].numpy(), W, wl.scale)
        check(f64(out), f64(lse), ro, rl, f"G={Hq // Hkv} D={D} W={W}", rel=EDGE_REL)


def test_paged_with_query_free_sequences():
    """The paged path with a pure-context sequence (its pages are read by no
    one, its table row still exists) between two sequences that append."""
    wl = wls.Workload("paged_edges", ((64, 32, 1), (200, 0, 1), (0, 40, 0)), 4, 2, 128, -1, 501)
    b = wls.make_paged_batch(wl, 16, device="cuda")
    kc, vc = b["k_cache"].clone(), b["v_cache"].clone()
    out, lse = binding.forward_paged(b["q"], b["k_new"], b["v_new"], kc, vc, b["block_table"].cuda(),
                                     b["cu_q"].cuda(), b["ctx_len"].cuda(), b["mode"].cuda(), -1, wl.scale)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    ro, rl, ka, va = pg.paged_attention(f64(b["q"]), f64(b["k_new"]), f64(b["v_new"]), f64(b["k_cache"]),
                                        f64(b["v_cache"]), b["block_table"].numpy(), 16, b["cu_q"].numpy(),
                                        b["ctx_len"].numpy(), b["mode"].numpy(), -1, wl.scale)
    check(f64(out), f64(lse), ro, rl, "paged edges", rel=EDGE_REL)
    np.testing.assert_array_equal(f64(kc), ka)


def test_acceptance_single_row_canvases():
    """Canvases of one row (always accepted: the most confident open row is),
    and a canvas with every row accepted before (nothing to rank)."""
    V = 1000
    g = torch.Generator(device="cuda").manual_seed(77)
    x = (2.0 * torch.randn(4, V, generator=g, device="cuda")).to(torch.bfloat16)
    cu = torch.tensor([0, 1, 2, 4], dtype=torch.int32, device="cuda")
    acc_in = torch.tensor([0, 0, 1, 1], dtype=torch.uint8, device="cuda")
    prev = torch.zeros(4, dtype=torch.int32, device="cuda")
    res = binding.accept_step(x, cu, acc_in, prev, torch.zeros(3, dtype=torch.int32, device="cuda"),
                              0.0, 1.0, 1, 0, 10)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    H, c, a = oacc.row_stats(f64(x))
    np.testing.assert_allclose(res["entropy"].cpu().numpy(), H, rtol=1e-4, atol=1e-4)
    assert res["accepted"].cpu().numpy().tolist() == [1, 1, 1, 1]
