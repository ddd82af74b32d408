"""GPU parity of the FP8 (e4m3) attention variant (``dg_attn_forward_fp8``,
called through the C ABI) against the fp64 oracle of the dequantised inputs.

Tolerance, derived from the variant's arithmetic.  Q.K and P.V accumulate in
fp32 from the exact e4m3 products; the one lossy step is rounding the
probabilities, scaled by 2^5, to e4m3 before P.V.  With p'_j the scaled
probability and l its fp32 sum (at least 2^5 times the oracle's max-shifted
sum), |round(p') - p'| <= max(2^-4 p', 2^-10) gives, per output element,

    |out - ref| <= 2^-4 sum_j w_j |v_j| + 2^-15 sum_j |v_j| / l_ref
                   + 2^-8 |ref| (bf16 output) + 1e-4,

w the oracle's attention weights.  The LSE sees no rounding: within 1e-3.
"""

import os

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8 as f8
from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

LSE_ABS = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    assert binding.status() == binding.DG_OK


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def dequant(b):
    return (f8.e4m3_to_float(b["q8"].cpu().numpy()) * b["q_scale"],
            f8.e4m3_to_float(b["k8"].cpu().numpy()) * b["k_scale"],
            f8.e4m3_to_float(b["v8"].cpu().numpy()) * b["v_scale"])


def run_fp8(b, window):
    d = {k: b[k].cuda() for k in ("q8", "k8", "v8", "cu_q", "ctx_len", "mode")}
    out, lse = binding.forward_fp8(d["q8"], d["k8"], d["v8"], d["cu_q"], d["ctx_len"], d["mode"], window,
                                   b["scale"], b["q_scale"], b["k_scale"], b["v_scale"])
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    return f64(out), f64(lse)


def bound(q, k, v, cu, ctx, mode, window, scale, ref, rows=None):
    """The per-element bound above, for every query row (or ``rows`` of a
    one-sequence batch)."""
    wv, _ = oracle.attention(q, k, np.abs(v), cu, ctx, mode, window, scale, query_rows=rows)
    t2 = np.zeros_like(ref)
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    off = 0
    for s in range(len(ctx)):
        c, n = int(ctx[s]), int(cu[s + 1] - cu[s])
        L = c + n
        toks = np.arange(n) if rows is None else np.asarray(rows) - int(cu[s])
        mask = oracle.visible_mask(c, n, int(mode[s]) == 0, window)[toks]
        for h in range(Hq):
            g = h // G
            z = scale * (q[int(cu[s]) + toks, h] @ k[off:off + L, g].T)
            z = np.where(mask, z, -np.inf)
            lsum = np.exp(z - z.max(axis=1, keepdims=True)).sum(axis=1)
            t2[int(cu[s]) + toks, h] = 2.0 ** -15 * (mask @ np.abs(v[off:off + L, g])) / lsum[:, None]
        off += L
    return 2.0 ** -4 * wv + t2 + 2.0 ** -8 * np.abs(ref) + 1e-4


def check(out, lse, b, window, what, rows=None):
    q, k, v = dequant(b)
    cu, ctx, mode = b["cu_q"].numpy(), b["ctx_len"].numpy(), b["mode"].numpy()
    ref_o, ref_l = oracle.attention(q, k, v, cu, ctx, mode, window, b["scale"], query_rows=rows)
    sel = slice(None) if rows is None else np.asarray(rows)
    bnd = bound(q, k, v, cu, ctx, mode, window, b["scale"], ref_o, rows=rows)[sel]
    d = np.abs(out[sel] - ref_o[sel])
    assert np.isfinite(out[sel]).all() and np.isfinite(lse[sel]).all(), what
    excess = d - bnd
    assert excess.max() <= 0, f"{what}: max|d|={d.max():.3g}, worst excess over the bound {excess.max():.3g}"
    dl = np.abs(lse[sel] - ref_l[sel])
    assert dl.max() <= LSE_ABS, f"{what}: max|dlse|={dl.max():.3g}"


def test_mixed_batch_head_dim_128():
    wl = wls.WORKLOADS["mixed_full"]
    b = wls.make_fp8_batch(wl)
    for W in (-1, 512):
        out, lse = run_fp8(b, W)
        check(out, lse, b, W, f"mixed W={W}")


CASES = [
    # (seed, seqs, Hq, Hkv, D, windows)
    (71, ((700, 256, 1), (5, 100, 0)), 16, 2, 256, (-1, 129)),
    (72, ((0, 1, 0), (5, 1, 1), (130, 3, 0), (200, 129, 1)), 2, 1, 128, (-1, 0, 1, 127)),
    (73, ((300, 256, 1), (0, 333, 0), (1000, 200, 1)), 8, 4, 128, (-1, 50)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_ragged_batches(case):
    seed, seqs, Hq, Hkv, D, windows = CASES[case]
    b = wls.make_fp8_batch(wls.Workload("fp8", seqs, Hq, Hkv, D, -1, seed))
    for W in windows:
        out, lse = run_fp8(b, W)
        check(out, lse, b, W, f"case {case} W={W}")


@pytest.mark.parametrize("ctas", ["1", "5"])
def test_grid_sizes(ctas):
    os.environ["DG_ATTN_NUM_CTAS"] = ctas
    try:
        b = wls.make_fp8_batch(wls.Workload("fp8", ((300, 256, 1), (0, 333, 0)), 8, 4, 256, -1, 74))
        out, lse = run_fp8(b, -1)
        check(out, lse, b, -1, f"{ctas} CTAs")
    finally:
        del os.environ["DG_ATTN_NUM_CTAS"]


@pytest.mark.parametrize("weight", ["0", "40"])
def test_segment_weights(weight, monkeypatch):
    """The work split's segment weight moves every CTA boundary, so CTAs
    switch tiles mid-range: each segment's query tile is loaded into shared
    memory (head_dim 256) at its start, and each split gives the oracle's
    result."""
    monkeypatch.setenv("DG_ATTN_SEG_WEIGHT", weight)
    b = wls.make_fp8_batch(wls.Workload("fp8", ((700, 256, 1), (5, 100, 0)), 16, 2, 256, -1, 77))
    for W in (-1, 129):
        out, lse = run_fp8(b, W)
        check(out, lse, b, W, f"weight {weight} W={W}")


@pytest.mark.parametrize("D", [128, 256])
def test_large_logits(D):
    """A large softmax scale spreads the scores over hundreds of units: the
    running maximum keeps growing across KV tiles, so the lazy O rescale
    (every 2^3 of growth in e4m3) and the recomputed exponentials of rows
    whose maximum moved run many times."""
    b = wls.make_fp8_batch(wls.Workload("fp8", ((3000, 256, 1), (0, 400, 0)), 8, 2, D, -1, 76 + D))
    b["scale"] = 1.5
    out, lse = run_fp8(b, -1)
    check(out, lse, b, -1, f"large logits D={D}")


def test_denoise_loop_sampled():
    """One 256-query canvas over 32768 cached tokens, 32 / 4 heads, head_dim
    256: sampled rows against the oracle."""
    wl = wls.WORKLOADS["denoise_loop"]
    b = wls.make_fp8_batch(wl, device="cuda")
    out, lse = run_fp8(b, wl.window)
    b = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in b.items()}
    rows = np.unique(np.concatenate([[0, 255], np.random.default_rng(3).choice(256, 10, replace=False)]))
    check(out, lse, b, wl.window, "denoise", rows=rows)


def test_host_checks():
    b = wls.make_fp8_batch(wls.Workload("fp8", ((10, 20, 1),), 2, 1, 64, -1, 75))
    d = {k: b[k].cuda() for k in ("q8", "k8", "v8", "cu_q", "ctx_len", "mode")}
    with pytest.raises(binding.DgAttnError):   # head_dim 64 is not supported in e4m3
        binding.forward_fp8(d["q8"], d["k8"], d["v8"], d["cu_q"], d["ctx_len"], d["mode"], -1, 0.1,
                            1.0, 1.0, 1.0)
    b = wls.make_fp8_batch(wls.Workload("fp8", ((10, 20, 1),), 2, 1, 128, -1, 76))
    d = {k: b[k].cuda() for k in ("q8", "k8", "v8", "cu_q", "ctx_len", "mode")}
    with pytest.raises(binding.DgAttnError):   # scales must be positive
        binding.forward_fp8(d["q8"], d["k8"], d["v8"], d["cu_q"], d["ctx_len"], d["mode"], -1, 0.1,
                            0.0, 1.0, 1.0)
