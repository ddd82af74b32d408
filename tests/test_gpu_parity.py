"""GPU parity of the CUDA path (called through the C ABI) against the fp64 CPU
oracle on the same seeded bf16 inputs.

Bar (from the method's accuracy target): max |out - oracle| <= 1e-2,
mean |out - oracle| <= 1e-3, max |lse - oracle| <= 1e-3.  Small workloads are
compared element by element; the full-size ones on sampled rows the oracle
computes one by one, plus properties that hold at any size.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
LSE_ABS = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    assert binding.status() == binding.DG_OK


def to_dev(batch):
    d = {}
    for key in ("q", "k", "v"):
        d[key] = batch[key].cuda().contiguous()
    d["cu_q"] = batch["cu_q"].cuda()
    d["ctx_len"] = batch["ctx_len"].cuda()
    d["mode"] = batch["mode"].cuda()
    return d


def run_gpu(dev, window, scale):
    out, lse = binding.forward(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["ctx_len"], dev["mode"],
                               window, scale)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    return out, lse


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


# Rows whose softmax mass sits on a handful of keys (windows of 0-1, the first
# rows of a prefill) have |out| up to ~4.  There the bf16 output rounding alone
# is up to 2^-8 |out| and the bf16 weights the PV MMA multiplies add up to 2^-8
# of the value spread, so the edge-case tests allow 1e-2 + 2^-7 |ref| per
# element; every configured workload is held to the plain 1e-2.
EDGE_REL = 2.0 ** -7


def check(out_gpu, lse_gpu, out_ref, lse_ref, what="", rel=0.0):
    d = np.abs(out_gpu - out_ref)
    dl = np.abs(lse_gpu - lse_ref)
    assert np.isfinite(out_gpu).all() and np.isfinite(lse_gpu).all(), what
    excess = d - (MAX_ABS + rel * np.abs(out_ref))
    assert excess.max() <= 0, f"{what} max|dout|={d.max():.3g} (worst excess {excess.max():.3g})"
    assert d.mean() <= MEAN_ABS, f"{what} mean|dout|={d.mean():.3g}"
    assert dl.max() <= LSE_ABS, f"{what} max|dlse|={dl.max():.3g}"


def full_check(wl, batch, window=None, dev=None, rel=0.0):
    window = wl.window if window is None else window
    dev = to_dev(batch) if dev is None else dev
    out, lse = run_gpu(dev, window, wl.scale)
    ref_o, ref_l = oracle.attention(f64(batch["q"]), f64(batch["k"]), f64(batch["v"]),
                                    batch["cu_q"].numpy(), batch["ctx_len"].numpy(),
                                    batch["mode"].numpy(), window, wl.scale)
    check(f64(out), f64(lse), ref_o, ref_l, f"{wl.name} W={window}", rel=rel)
    return out, lse


# ------------------------------------------------------------ small workloads

def test_tiny_bidirectional_head_dim_64():
    wl = wls.WORKLOADS["tiny"]
    full_check(wl, wls.make_batch(wl))


@pytest.mark.parametrize("name", ["mixed_full", "mixed_w512"])
def test_mixed_batch(name):
    wl = wls.WORKLOADS[name]
    full_check(wl, wls.make_batch(wl))


# ragged batches: contexts of 0, lengths that are not tile multiples, windows at
# and around the tile size, every supported head_dim, group sizes 1/2/3/8
EDGE = [
    # (seqs, Hq, Hkv, D, windows)
    (((0, 1, 0), (5, 1, 1), (0, 77, 1), (130, 3, 0), (200, 129, 1)), 2, 1, 64, (-1, 0, 1, 127, 128, 129, 5000)),
    (((17, 300, 1), (0, 255, 0), (1, 1, 1), (300, 64, 0)), 6, 2, 128, (-1, 0, 63, 64, 200)),
    (((129, 40, 1), (0, 190, 0), (64, 64, 0)), 8, 1, 256, (-1, 1, 100)),
    (((250, 100, 1), (3, 70, 0)), 4, 4, 128, (-1, 31)),
]


@pytest.mark.parametrize("case", range(len(EDGE)))
def test_ragged_edge_cases(case):
    seqs, Hq, Hkv, D, windows = EDGE[case]
    wl, batch = wls.random_batch(100 + case, seqs, Hq, Hkv, D, -1)
    dev = to_dev(batch)
    for W in windows:
        full_check(wl, batch, window=W, dev=dev, rel=EDGE_REL)


@pytest.mark.parametrize("ctas", ["1", "3", "37"])
def test_grid_sizes(ctas):
    """Persistent grids of 1, 3 and 37 CTAs cut the (tile, KV tile) units at
    other places than the full grid: every grid gives the oracle's result,
    with windowed ranges that differ per tile and tiles merged from several
    CTAs' partials."""
    os.environ["DG_ATTN_NUM_CTAS"] = ctas
    try:
        for seed, seqs, Hq, Hkv, D, windows in (
                (41, ((300, 256, 1), (0, 333, 0), (1000, 200, 1)), 8, 4, 128, (-1, 50)),
                (42, ((700, 256, 1), (5, 100, 0)), 16, 2, 256, (-1, 129)),
                (43, ((64, 500, 1), (0, 260, 0)), 2, 2, 64, (-1, 0, 200))):
            wl, batch = wls.random_batch(seed, seqs, Hq, Hkv, D, -1)
            dev = to_dev(batch)
            for W in windows:
                full_check(wl, batch, window=W, dev=dev, rel=EDGE_REL)
    finally:
        del os.environ["DG_ATTN_NUM_CTAS"]


@pytest.mark.parametrize("weight", ["0", "3", "40"])
def test_segment_weights(weight, monkeypatch):
    """The work split's segment weight moves every CTA boundary (0: KV
    tiles only; 40: a tile start outweighs most of its KV tiles): each split
    gives the oracle's result, at head_dim 128 and 256."""
    monkeypatch.setenv("DG_ATTN_SEG_WEIGHT", weight)
    for seed, seqs, Hq, Hkv, D in ((44, ((300, 256, 1), (0, 333, 0), (1000, 200, 1)), 8, 4, 128),
                                   (45, ((700, 256, 1), (5, 100, 0)), 16, 2, 256)):
        wl, batch = wls.random_batch(seed, seqs, Hq, Hkv, D, -1)
        dev = to_dev(batch)
        for W in (-1, 129):
            full_check(wl, batch, window=W, dev=dev, rel=EDGE_REL)


@pytest.mark.parametrize("D", [128, 256])
def test_large_logits(D):
    """A large softmax scale spreads the scores over hundreds of units: the row
    maximum keeps growing across KV tiles (lazy O rescale) and many exponents
    fall far below the bf16 range."""
    wl, batch = wls.random_batch(50 + D, ((3000, 256, 1), (0, 400, 0)), 8, 2, D, -1)
    dev = to_dev(batch)
    out, lse = run_gpu(dev, -1, 1.5)
    ref_o, ref_l = oracle.attention(f64(batch["q"]), f64(batch["k"]), f64(batch["v"]),
                                    batch["cu_q"].numpy(), batch["ctx_len"].numpy(),
                                    batch["mode"].numpy(), -1, 1.5)
    check(f64(out), f64(lse), ref_o, ref_l, f"large logits D={D}", rel=EDGE_REL)


def test_single_visible_key_is_exact():
    """W = 0, bidirectional: every query sees only itself, so out == v (bf16)."""
    wl, batch = wls.random_batch(7, ((40, 200, 1), (0, 129, 1)), 4, 2, 128, 0)
    dev = to_dev(batch)
    out, lse = run_gpu(dev, 0, wl.scale)
    rows = []
    off = 0
    for c, n, _ in wl.seqs:
        rows.append(torch.arange(off + c, off + c + n))
        off += c + n
    rows = torch.cat(rows).cuda()
    vq = dev["v"][rows].repeat_interleave(2, dim=1)
    assert torch.equal(out, vq)


def test_causal_row0_without_context_is_exact():
    wl, batch = wls.random_batch(8, ((0, 300, 0),), 2, 2, 128, -1)
    dev = to_dev(batch)
    out, _ = run_gpu(dev, -1, wl.scale)
    assert torch.equal(out[0], dev["v"][0])


# keys per KV tile of the bf16 kernel by head_dim (the LSE bounds below count tiles)
KV_TILE_ROWS = {64: 128, 128: 128, 256: 64}


def lse_order_bound(lse_a, lse_b, max_keys, bn=64):
    """How far two LSEs of the same rows may differ when the kernel visits the
    KV tiles in another order or cuts them elsewhere.  The row sum l runs over
    T = ceil(keys / BN) tiles: each tile adds one fp32 rounding (2^-24) and,
    when its maximum grows, one rescale by an ex2 approximation (2^-22
    relative), so each side's l is within T (2^-22 + 2^-24) of the exact sum;
    the LSE adds ln l and a few ulps of its own value."""
    T = -(-max_keys // bn)
    ulp = torch.maximum(lse_a.abs(), lse_b.abs()) * 2.0 ** -23
    return 2 * T * (2.0 ** -22 + 2.0 ** -24) + 4 * ulp


def test_split_kv_matches_single_cta():
    """The LSE merge of split tiles equals the unsplit result (fp32 rounding)."""
    wl, batch = wls.random_batch(9, ((3000, 256, 1), (1000, 300, 0)), 8, 2, 128, -1)
    dev = to_dev(batch)
    out_split, lse_split = run_gpu(dev, -1, wl.scale)
    os.environ["DG_ATTN_NUM_CTAS"] = "1"
    try:
        out_one, lse_one = run_gpu(dev, -1, wl.scale)
    finally:
        del os.environ["DG_ATTN_NUM_CTAS"]
    assert (out_split.float() - out_one.float()).abs().max().item() <= 2 ** -7
    assert ((lse_split - lse_one).abs() <= lse_order_bound(lse_split, lse_one, 3256, KV_TILE_ROWS[128])).all()


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("ctas", ["152", "10"])
def test_rotated_kv_order_matches_ascending(ctas, D):
    """Visiting each tile's KV tiles from a rotated start (the default) gives
    the ascending-order result up to fp32 rounding, with the cut points of the
    full grid and of a 10-CTA grid (many cuts inside each tile); head_dim 256
    runs with the softmax-side stage release, 128 with the MMA warp's."""
    wl, batch = wls.random_batch(10 + D, ((3000, 256, 1), (1000, 300, 0), (500, 64, 1)), 8, 2, D, -1)
    dev = to_dev(batch)
    os.environ["DG_ATTN_NUM_CTAS"] = ctas
    try:
        for W in (-1, 700):
            out_rot, lse_rot = run_gpu(dev, W, wl.scale)
            os.environ["DG_ATTN_KV_ORDER"] = "linear"
            try:
                out_lin, lse_lin = run_gpu(dev, W, wl.scale)
            finally:
                del os.environ["DG_ATTN_KV_ORDER"]
            assert (out_rot.float() - out_lin.float()).abs().max().item() <= 2 ** -7, W
            assert ((lse_rot - lse_lin).abs() <= lse_order_bound(lse_rot, lse_lin, 3256, KV_TILE_ROWS[D])).all(), W
    finally:
        del os.environ["DG_ATTN_NUM_CTAS"]


def test_device_detected_bad_metadata_sets_status():
    """cu_q contents are only visible on the device: the call is enqueued, the
    kernels skip the work and the status word reports the error."""
    wl, batch = wls.random_batch(10, ((10, 20, 1), (0, 12, 0)), 2, 1, 64, -1)
    dev = to_dev(batch)
    bad = dev["cu_q"].clone()
    bad[1] = 25  # second sequence would have a negative length... and totals mismatch
    bad[2] = 31
    binding.forward(dev["q"], dev["k"], dev["v"], bad, dev["ctx_len"], dev["mode"], -1, wl.scale)
    assert binding.status() == binding.DG_ERR_INVALID_ARG
    assert binding.status() == binding.DG_OK  # cleared by the read
    bad_mode = dev["mode"].clone()
    bad_mode[0] = 7
    binding.forward(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["ctx_len"], bad_mode, -1, wl.scale)
    assert binding.status() == binding.DG_ERR_INVALID_ARG


def test_workspace_checks():
    wl, batch = wls.random_batch(11, ((10, 20, 1),), 2, 1, 64, -1)
    dev = to_dev(batch)
    need = binding.workspace_size(1, 20, 2, 1, 64)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    lib = binding.load_library()
    out = torch.empty_like(dev["q"])
    rc = lib.dg_attn_forward(dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(),
                             dev["cu_q"].data_ptr(), dev["ctx_len"].data_ptr(), dev["mode"].data_ptr(),
                             1, 20, 30, 2, 1, 64, -1, 0.125, out.data_ptr(), None, small.data_ptr(),
                             need - 256, None)
    assert rc == binding.DG_ERR_WORKSPACE
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    rc = lib.dg_attn_forward(dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(),
                             dev["cu_q"].data_ptr(), dev["ctx_len"].data_ptr(), dev["mode"].data_ptr(),
                             1, 20, 30, 2, 1, 64, -1, 0.125, out.data_ptr(), None, ws.data_ptr() + 16,
                             need, None)
    assert rc == binding.DG_ERR_WORKSPACE


# ------------------------------------------------------- full-size workloads

def sampled_check(wl, dev, out, lse, rng, kv_heads=2, tokens=16, window=None):
    """Oracle on sampled (sequence, KV head, token) rows, all query heads of the
    sampled KV heads; each sequence is evaluated alone on its own KV rows
    (sequences are independent, pinned by the oracle's mixed-batch test)."""
    window = wl.window if window is None else window
    G = wl.num_q_heads // wl.num_kv_heads
    off = 0
    cu = [0]
    for _, n, _ in wl.seqs:
        cu.append(cu[-1] + n)
    for s, (c, n, md) in enumerate(wl.seqs):
        L = c + n
        for g in rng.choice(wl.num_kv_heads, size=min(kv_heads, wl.num_kv_heads), replace=False):
            toks = np.unique(np.concatenate([[0, n - 1], rng.choice(n, size=min(tokens, n), replace=False)]))
            hs = slice(g * G, (g + 1) * G)
            qs = f64(dev["q"][cu[s]:cu[s + 1], hs])
            ks = f64(dev["k"][off:off + L, g:g + 1])
            vs = f64(dev["v"][off:off + L, g:g + 1])
            ro, rl = oracle.attention(qs, ks, vs, [0, n], [c], [md], window, wl.scale, query_rows=toks)
            go = f64(out[cu[s]:cu[s + 1], hs])[toks]
            gl = f64(lse[cu[s]:cu[s + 1], hs])[toks]
            check(go, gl, ro[toks], rl[toks], f"{wl.name} seq {s} kvh {g}")
        off += L


def any_size_properties(dev, out, lse):
    """Each output is a convex combination of value rows: finite and within the
    value range; lse finite."""
    assert torch.isfinite(out.float()).all()
    assert torch.isfinite(lse).all()
    assert out.float().abs().max().item() <= dev["v"].float().abs().max().item() + 1e-2


def test_denoise_loop_two_steps():
    wl = wls.WORKLOADS["denoise_loop"]
    batch = wls.make_batch(wl, device="cuda")
    dev = to_dev(batch)
    rng = np.random.default_rng(0)
    out, lse = run_gpu(dev, wl.window, wl.scale)
    any_size_properties(dev, out, lse)
    sampled_check(wl, dev, out, lse, rng)
    # step 1: fresh canvas q and canvas K/V rows, context reused
    q1, kc, vc = wls.denoise_step_inputs(wl, 1, device="cuda")
    (r0, r1), = wls.canvas_rows(wl)
    dev["q"].copy_(q1)
    dev["k"][r0:r1].copy_(kc)
    dev["v"][r0:r1].copy_(vc)
    out, lse = run_gpu(dev, wl.window, wl.scale)
    any_size_properties(dev, out, lse)
    sampled_check(wl, dev, out, lse, rng)


@pytest.mark.parametrize("name", ["maxmix_full", "maxmix_w1024"])
def test_maxmix(name):
    wl = wls.WORKLOADS[name]
    batch = wls.make_batch(wl, device="cuda")
    dev = to_dev(batch)
    out, lse = run_gpu(dev, wl.window, wl.scale)
    any_size_properties(dev, out, lse)
    sampled_check(wl, dev, out, lse, np.random.default_rng(1), kv_heads=2, tokens=12)
