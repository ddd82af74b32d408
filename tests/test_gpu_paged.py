"""GPU parity of the paged-KV-cache path (``dg_attn_forward_paged``, called
through the C ABI) against the CPU oracle of the paged cache on the same
seeded inputs: attention outputs within the attention bar, the cache after the
append bit for bit, and the paged result bit-identical to the contiguous path
on the same keys."""


import numpy as np
import pytest
import torch

import oracle
import oracle.paged as pg
from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls
from test_gpu_parity import EDGE_REL, any_size_properties, check, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    assert binding.status() == binding.DG_OK


def to_dev(b):
    d = {key: b[key].cuda().clone() for key in ("q", "k_new", "v_new", "k_cache", "v_cache")}
    for key in ("block_table", "cu_q", "ctx_len", "mode"):
        d[key] = b[key].cuda()
    return d


def run_paged(d, window, scale, append=True):
    out, lse = binding.forward_paged(d["q"], d["k_new"] if append else None,
                                     d["v_new"] if append else None, d["k_cache"], d["v_cache"],
                                     d["block_table"], d["cu_q"], d["ctx_len"], d["mode"], window,
                                     scale)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    return out, lse


def oracle_paged(b, window, scale):
    return pg.paged_attention(f64(b["q"]), f64(b["k_new"]), f64(b["v_new"]), f64(b["k_cache"]),
                              f64(b["v_cache"]), b["block_table"].numpy(), b["page_size"],
                              b["cu_q"].numpy(), b["ctx_len"].numpy(), b["mode"].numpy(), window,
                              scale)


# (seqs, Hq, Hkv, D, page sizes, windows): page sizes below, at and above the
# KV tile (one TMA box per page and per lane of the loader warp, up to 32
# boxes per tile), contexts that end mid-page, a sequence of one token
CASES = [
    (((0, 300, 0), (257, 129, 1), (1000, 256, 1), (37, 1, 0)), 8, 2, 128, (8, 16, 64, 256), (-1, 100)),
    (((130, 77, 1), (0, 200, 0)), 2, 1, 64, (8, 16, 128), (-1, 0, 129)),
    (((700, 256, 1), (5, 100, 0)), 16, 2, 256, (8, 16, 32, 1024), (-1, 129)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_paged_matches_oracle(case):
    seqs, Hq, Hkv, D, pages, windows = CASES[case]
    wl = wls.Workload("paged", seqs, Hq, Hkv, D, -1, 200 + case)
    for P in pages:
        b = wls.make_paged_batch(wl, P, device="cuda")
        for W in windows:
            d = to_dev(b)
            out, lse = run_paged(d, W, wl.scale)
            ro, rl, ka, va = oracle_paged(b, W, wl.scale)
            check(f64(out), f64(lse), ro, rl, f"P={P} W={W}", rel=EDGE_REL)
            np.testing.assert_array_equal(f64(d["k_cache"]), ka)
            np.testing.assert_array_equal(f64(d["v_cache"]), va)


@pytest.mark.parametrize("name", ["mixed_full", "mixed_w512"])
@pytest.mark.parametrize("P", [16, 64])
def test_configured_mixed_batches_at_the_plain_bar(name, P):
    """The configured mixed batches (causal prefills and canvases over cached
    contexts, GQA 16/8, head_dim 128, full and W=512 layers) through the paged
    cache, every element against the oracle at the stated bar (max 1e-2, mean
    1e-3, LSE 1e-3): the plain bar, not the edge-case one."""
    wl = wls.WORKLOADS[name]
    b = wls.make_paged_batch(wl, P, device="cuda")
    d = to_dev(b)
    out, lse = run_paged(d, wl.window, wl.scale)
    ro, rl, ka, va = oracle_paged(b, wl.window, wl.scale)
    check(f64(out), f64(lse), ro, rl, f"{name} P={P}")
    np.testing.assert_array_equal(f64(d["k_cache"]), ka)
    np.testing.assert_array_equal(f64(d["v_cache"]), va)


def _bits(t):
    return t.cpu().view(torch.int16).numpy()


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("P", [8, 16, 64])
def test_paged_equals_contiguous_bit_for_bit(P, D):
    """The same keys laid out contiguously (gathered through the page table by
    the oracle's gather) give bit-identical outputs through dg_attn_forward:
    both calls split the work the same way and differ only in where each TMA
    box of a KV tile comes from (16-row pages: one V box per page, read by P.V
    with the page's column-block stride)."""
    Hq, Hkv = (8, 4) if D == 128 else (16, 2)
    wl = wls.Workload("paged", ((300, 256, 1), (0, 333, 0), (1000, 200, 1)), Hq, Hkv, D, -1, 77)
    b = wls.make_paged_batch(wl, P, device="cuda")
    d = to_dev(b)
    out_p, lse_p = run_paged(d, -1, wl.scale)
    kb, vb = _bits(d["k_cache"]), _bits(d["v_cache"])
    bt = b["block_table"].numpy()
    ks, vs = [], []
    for s, (c, n, _) in enumerate(wl.seqs):
        ks.append(pg.gather_kv(kb, bt[s], c + n, P))
        vs.append(pg.gather_kv(vb, bt[s], c + n, P))
    k = torch.from_numpy(np.concatenate(ks)).view(torch.bfloat16).cuda()
    v = torch.from_numpy(np.concatenate(vs)).view(torch.bfloat16).cuda()
    out_c, lse_c = binding.forward(d["q"], k, v, d["cu_q"], d["ctx_len"], d["mode"], -1, wl.scale)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    assert torch.equal(out_p, out_c)
    assert torch.equal(lse_p, lse_c)


@pytest.mark.parametrize("knob", ["DG_ATTN_V_PAGE_BOX", "DG_ATTN_K_PAGE_BOX", "DG_ATTN_K_SPLIT"])
@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("P", [8, 16])
def test_box_layouts_give_the_same_bits(P, D, knob, monkeypatch):
    """8- and 16-row pages: the default loads (V as one box per page, read
    with a page stride between 8-row groups when a page is half a K step; K as
    one box per 8-row page, its 8-row groups a page apart; a K tile's boxes
    issued by two warps) and the plain ones (a box per page and 128-byte column
    block; one K warp) give the same bits."""
    Hq, Hkv = (8, 4) if D == 128 else (16, 2)
    wl = wls.Workload("vbox", ((700, 256, 1), (0, 190, 0)), Hq, Hkv, D, -1, 78)
    b = wls.make_paged_batch(wl, P, device="cuda")
    d = to_dev(b)
    out_a, lse_a = run_paged(d, -1, wl.scale, append=False)
    monkeypatch.setenv(knob, "0")
    out_b, lse_b = run_paged(d, -1, wl.scale, append=False)
    assert torch.equal(out_a, out_b)
    assert torch.equal(lse_a, lse_b)


def test_rows_already_in_the_cache():
    """Without k_new / v_new the cache is read as it is: a second call after
    the append gives the same result bit for bit and leaves the cache alone."""
    wl = wls.Workload("paged", ((129, 256, 1), (40, 70, 0)), 4, 2, 128, -1, 78)
    b = wls.make_paged_batch(wl, 32, device="cuda")
    d = to_dev(b)
    out1, lse1 = run_paged(d, 50, wl.scale)
    k_after = d["k_cache"].clone()
    out2, lse2 = run_paged(d, 50, wl.scale, append=False)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    assert torch.equal(k_after, d["k_cache"])


def test_denoise_loop_paged_two_steps():
    """The denoise-loop geometry (one canvas of 256 over 32768 cached tokens,
    32/4 heads, head_dim 256) on pages of 16 rows: step 0, then step 1 with a
    fresh canvas appended over the previous one; sampled rows vs the oracle."""
    wl = wls.WORKLOADS["denoise_loop"]
    P = 16
    b = wls.make_paged_batch(wl, P, device="cuda")
    d = to_dev(b)
    rng = np.random.default_rng(5)
    bt = b["block_table"].numpy()
    (c, n, md), = wl.seqs
    G = wl.num_q_heads // wl.num_kv_heads
    for step in (0, 1):
        if step:
            q1, kc, vc = wls.denoise_step_inputs(wl, 1, device="cuda")
            d["q"].copy_(q1)
            d["k_new"].copy_(kc)
            d["v_new"].copy_(vc)
        out, lse = run_paged(d, wl.window, wl.scale)
        any_size_properties({"v": d["v_cache"]}, out, lse)
        for g in rng.choice(wl.num_kv_heads, size=2, replace=False):
            toks = np.unique(np.concatenate([[0, n - 1], rng.choice(n, size=14, replace=False)]))
            hs = slice(g * G, (g + 1) * G)
            kk = pg.gather_kv(f64(d["k_cache"][:, :, g:g + 1]), bt[0], c + n, P)
            vv = pg.gather_kv(f64(d["v_cache"][:, :, g:g + 1]), bt[0], c + n, P)
            # the canvas rows in the cache are this step's new rows
            np.testing.assert_array_equal(kk[c:], f64(d["k_new"][:, g:g + 1]))
            ro, rl = oracle.attention(f64(d["q"][:, hs]), kk, vv, [0, n], [c], [md], wl.window,
                                      wl.scale, query_rows=toks)
            check(f64(out[:, hs])[toks], f64(lse[:, hs])[toks], ro[toks], rl[toks],
                  f"step {step} kvh {g}")


def test_bad_page_table_is_reported():
    wl = wls.Workload("paged", ((100, 60, 1), (0, 90, 0)), 4, 2, 64, -1, 79)
    b = wls.make_paged_batch(wl, 16, device="cuda")
    num_pages = b["k_cache"].shape[0]
    # an entry outside the pool in a page the attention reads
    d = to_dev(b)
    d["block_table"][0, 1] = num_pages
    binding.forward_paged(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                          d["block_table"], d["cu_q"], d["ctx_len"], d["mode"], -1, wl.scale)
    assert binding.status() == binding.DG_ERR_INVALID_ARG
    # a page table too short for the sequence (its appended rows included)
    d = to_dev(b)
    short = d["block_table"][:, :5].contiguous()
    binding.forward_paged(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], short,
                          d["cu_q"], d["ctx_len"], d["mode"], -1, wl.scale)
    assert binding.status() == binding.DG_ERR_INVALID_ARG
    # host-checked: page sizes that are not a power of two >= 8
    kc = torch.zeros((4, 12, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.DgAttnError):
        binding.forward_paged(d["q"], None, None, kc, kc.clone(), d["block_table"], d["cu_q"],
                              d["ctx_len"], d["mode"], -1, wl.scale)
    # a valid call afterwards is unaffected
    d = to_dev(b)
    out, lse = run_paged(d, -1, wl.scale)
    ro, rl, _, _ = oracle_paged(b, -1, wl.scale)
    check(f64(out), f64(lse), ro, rl, "after errors")
