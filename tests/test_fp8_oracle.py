"""Pins of the FP8 attention oracle (``oracle/fp8.py``): the e4m3 decoder
against hand-worked codes and, for all 256 codes, against PyTorch's e4m3
type (a library routine); the attention of the dequantised values against the
pinned bf16/fp64 oracle and against the scales' exact algebra."""

import os

import numpy as np
import torch

import oracle
import oracle.fp8 as f8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_codes.txt")


def test_golden_codes():
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if not line:
            continue
        code, want = int(line[0], 16), float(line[1])
        got = f8.e4m3_to_float(np.array([code], dtype=np.uint8))[0]
        if np.isnan(want):
            assert np.isnan(got), hex(code)
        else:
            assert got == want and np.signbit(got) == np.signbit(want), (hex(code), got, want)


def test_every_code_matches_the_library_type():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = f8.e4m3_to_float(codes)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), codes[~same]


def _codes(rng, shape):
    """Random finite e4m3 codes (NaN codes excluded)."""
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    return np.where((c & 0x7F) == 0x7F, np.uint8(0x38), c)


SEQS = ((5, 7, 1), (0, 9, 0), (11, 4, 1))


def _batch(seed, Hq=4, Hkv=2, D=8):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum([n for _, n, _ in SEQS])])
    ctx = np.array([c for c, _, _ in SEQS])
    mode = np.array([m for _, _, m in SEQS])
    tq = int(cu[-1])
    tk = int(sum(c + n for c, n, _ in SEQS))
    return (_codes(rng, (tq, Hq, D)), _codes(rng, (tk, Hkv, D)), _codes(rng, (tk, Hkv, D)), cu, ctx,
            mode)


def test_unit_scales_equal_the_attention_of_the_decoded_values():
    q8, k8, v8, cu, ctx, mode = _batch(1)
    o, l = f8.attention_fp8(q8, k8, v8, 1.0, 1.0, 1.0, cu, ctx, mode, 3, 0.01)
    qf = torch.from_numpy(q8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    kf = torch.from_numpy(k8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    vf = torch.from_numpy(v8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ro, rl = oracle.attention(qf, kf, vf, cu, ctx, mode, 3, 0.01)
    np.testing.assert_array_equal(o, ro)
    np.testing.assert_array_equal(l, rl)


def test_scales_act_as_the_algebra_says():
    """q and k scales multiply the scores (the same as multiplying the softmax
    scale), the v scale multiplies the output and leaves the LSE alone."""
    q8, k8, v8, cu, ctx, mode = _batch(2)
    o1, l1 = f8.attention_fp8(q8, k8, v8, 0.5, 0.25, 1.0, cu, ctx, mode, -1, 0.02)
    o2, l2 = f8.attention_fp8(q8, k8, v8, 1.0, 1.0, 1.0, cu, ctx, mode, -1, 0.02 * 0.125)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-12)
    o3, l3 = f8.attention_fp8(q8, k8, v8, 0.5, 0.25, 3.0, cu, ctx, mode, -1, 0.02)
    np.testing.assert_allclose(o3, 3.0 * o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(l3, l1)
