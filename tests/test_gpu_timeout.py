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
