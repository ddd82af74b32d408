"""The bounds-checking build (``lib/libdg_attn_debug.so``, compiled with
DG_ATTN_DEBUG): every TMA coordinate, shared-memory destination, TMEM column
and global index of the kernels is checked before the access, and a failed
check is reported as DG_ERR_DEVICE_BOUNDS in the status word (the access is
skipped, the kernel returns; nothing traps).

Small ragged shapes of every path must pass every check (status DG_OK) and
still match the oracles.  A planted coordinate past the K tensor (a debug-only
knob; the TMA load it would have issued is skipped, and a TMA load past a
tensor only reads the fill value anyway) must be caught, and the next call on
the same context must be correct again.
"""

import os

import numpy as np
import pytest
import torch

import oracle
import oracle.paged as opg
import oracle.selfcond as osc
from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls
from test_gpu_parity import EDGE, EDGE_REL, check, f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _debug_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    with binding.debug_library():
        assert binding.status() == binding.DG_OK
        yield
        assert binding.status() == binding.DG_OK


def _attention_against_oracle(wl, batch, window, rel=EDGE_REL):
    dev = to_dev(batch)
    out, lse = binding.forward(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["ctx_len"], dev["mode"],
                               window, wl.scale)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    ref_o, ref_l = oracle.attention(f64(batch["q"]), f64(batch["k"]), f64(batch["v"]),
                                    batch["cu_q"].numpy(), batch["ctx_len"].numpy(),
                                    batch["mode"].numpy(), window, wl.scale)
    check(f64(out), f64(lse), ref_o, ref_l, f"{wl.seqs} W={window}", rel=rel)


@pytest.mark.parametrize("case", range(len(EDGE)))
def test_ragged_shapes_pass_every_check(case):
    seqs, Hq, Hkv, D, windows = EDGE[case]
    wl, batch = wls.random_batch(300 + case, seqs, Hq, Hkv, D, -1)
    for W in windows[:3]:
        _attention_against_oracle(wl, batch, W)


def test_split_tiles_pass_every_check():
    """A 3-CTA grid: tiles cut between CTAs write partial slots and the merge
    reads them back."""
    wl, batch = wls.random_batch(310, ((3000, 256, 1), (1000, 300, 0)), 8, 2, 128, -1)
    os.environ["DG_ATTN_NUM_CTAS"] = "3"
    try:
        _attention_against_oracle(wl, batch, -1)
        _attention_against_oracle(wl, batch, 200)
    finally:
        del os.environ["DG_ATTN_NUM_CTAS"]


@pytest.mark.parametrize("P", [8, 16, 128])
def test_paged_cache_passes_every_check(P):
    wl = wls.Workload("dbg_paged", ((200, 130, 1), (0, 77, 0), (33, 1, 1)), 8, 2, 256, -1, 311)
    b = wls.make_paged_batch(wl, P, device="cuda")
    kc, vc = b["k_cache"].clone(), b["v_cache"].clone()
    out, lse = binding.forward_paged(b["q"], b["k_new"], b["v_new"], kc, vc, b["block_table"].cuda(),
                                     b["cu_q"].cuda(), b["ctx_len"].cuda(), b["mode"].cuda(), -1, wl.scale)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    ro, rl, _, _ = opg.paged_attention(f64(b["q"]), f64(b["k_new"]), f64(b["v_new"]), f64(b["k_cache"]),
                                       f64(b["v_cache"]), b["block_table"].numpy(), P, b["cu_q"].numpy(),
                                       b["ctx_len"].numpy(), b["mode"].numpy(), -1, wl.scale)
    check(f64(out), f64(lse), ro, rl, f"paged P={P}", rel=EDGE_REL)


def test_e4m3_passes_every_check():
    fb = wls.make_fp8_batch(wls.Workload("dbg_fp8", ((300, 200, 1), (0, 77, 0)), 8, 2, 128, -1, 312))
    d = {k: fb[k].cuda() for k in ("q8", "k8", "v8", "cu_q", "ctx_len", "mode")}
    binding.forward_fp8(d["q8"], d["k8"], d["v8"], d["cu_q"], d["ctx_len"], d["mode"], 64, fb["scale"],
                        fb["q_scale"], fb["k_scale"], fb["v_scale"])
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK


@pytest.mark.parametrize("rows,vocab,d", [(300, 5000, 320), (130, 40000, 256)])
def test_self_conditioning_passes_every_check(rows, vocab, d):
    lw = wls.LogitsWorkload("dbg_sc", (rows,), vocab, 313)
    x, _ = wls.make_logits(lw, device="cuda")
    E = wls.make_embedding(vocab, d, 314, device="cuda")
    y = binding.self_conditioning(x, E)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    ref = osc.self_conditioning(f64(x), f64(E))
    assert np.abs(f64(y) - ref).max() <= 1e-2


def test_planted_bad_row_is_caught_and_the_context_stays_usable():
    wl, batch = wls.random_batch(315, ((300, 256, 1), (0, 200, 0)), 4, 2, 128, -1)
    dev = to_dev(batch)
    args = (dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["ctx_len"], dev["mode"], -1, wl.scale)
    os.environ["DG_ATTN_DEBUG_BAD_KV_ROW"] = "1"
    try:
        binding.forward(*args)
        torch.cuda.synchronize()
    finally:
        del os.environ["DG_ATTN_DEBUG_BAD_KV_ROW"]
    assert binding.status() == binding.DG_ERR_DEVICE_BOUNDS
    _attention_against_oracle(wl, batch, -1)
