"""Failure detection without a GPU fault: every wait inside the attention
kernel is bounded.  With DG_ATTN_DEBUG_SKIP_K_LOAD the K loader skips one TMA
load, so nothing ever completes the barrier the MMA warp waits on; the wait
expires (250 ms), the kernel records DG_ERR_DEVICE_TIMEOUT, every role drains
its own work in flight, TMEM is freed and the kernel returns.  The status word
reports it, and the next call on the same context computes correct results."""

import os

import numpy as np
import pytest
import torch

import oracle
from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_stays_usable():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    wl, b = wls.random_batch(61, ((300, 256, 1), (0, 200, 0)), 4, 2, 128, -1)
    dev = {k: b[k].cuda() for k in ("q", "k", "v", "cu_q", "ctx_len", "mode")}
    args = (dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["ctx_len"], dev["mode"], -1, wl.scale)
    assert binding.status() == binding.DG_OK
    os.environ["DG_ATTN_DEBUG_SKIP_K_LOAD"] = "0"
    os.environ["DG_ATTN_NUM_CTAS"] = "2"
    try:
        binding.forward(*args)
        torch.cuda.synchronize()
    finally:
        del os.environ["DG_ATTN_DEBUG_SKIP_K_LOAD"]
        del os.environ["DG_ATTN_NUM_CTAS"]
    assert binding.status() == binding.DG_ERR_DEVICE_TIMEOUT
    out, lse = binding.forward(*args)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    ref_o, ref_l = oracle.attention(f64(b["q"]), f64(b["k"]), f64(b["v"]), b["cu_q"].numpy(),
                                    b["ctx_len"].numpy(), b["mode"].numpy(), -1, wl.scale)
    assert np.abs(f64(out) - ref_o).max() <= 1e-2
    assert np.abs(f64(lse) - ref_l).max() <= 1e-3


def test_selfcond_expired_wait_reports_timeout_and_context_stays_usable():
    """The self-conditioning GEMM's waits are bounded the same way: with
    DG_SELFCOND_DEBUG_SKIP_E_LOAD the E loader skips one TMA load, the MMA
    warp's wait for that stage expires, the kernel records
    DG_ERR_DEVICE_TIMEOUT and returns; the next call is correct."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle.selfcond as osc
    binding.load_library()
    lw = wls.LogitsWorkload("sc_timeout", (300,), 5000, 62)
    x, _ = wls.make_logits(lw, device="cuda")
    E = wls.make_embedding(lw.vocab, 320, 63, device="cuda")
    assert binding.status() == binding.DG_OK
    os.environ["DG_SELFCOND_DEBUG_SKIP_E_LOAD"] = "0"
    try:
        binding.self_conditioning(x, E)
        torch.cuda.synchronize()
    finally:
        del os.environ["DG_SELFCOND_DEBUG_SKIP_E_LOAD"]
    assert binding.status() == binding.DG_ERR_DEVICE_TIMEOUT
    y = binding.self_conditioning(x, E)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    assert np.abs(f64(y) - osc.self_conditioning(f64(x), f64(E))).max() <= 1e-2
