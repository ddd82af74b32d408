"""Plain CPU oracle of the FP8 (e4m3) variant of the dual-mode attention.

TEST INFRASTRUCTURE ONLY: only the tests, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` use it; it shares no code with the CUDA library.

The pages serve DiffusionGemma from FP8 checkpoints (agentlenshq page,
"quantised checkpoints": FP8 weights with fully dynamic activations; the
throughput results are FP8 runs on H200 / H100).  They do not say that
attention runs in FP8; this variant is an assumption of the build: Q, K and V
arrive as e4m3 bytes, each tensor with one fp32 scale, and the attention is
exactly that of the dequantised values,

    attention(q_scale * e4m3(q), k_scale * e4m3(k), v_scale * e4m3(v)),

with the same masks, windows, GQA mapping and LSE definition as
``oracle.attention``.

e4m3 (the OCP 8-bit floating-point format E4M3): 1 sign bit, 4 exponent bits
with bias 7, 3 mantissa bits; exponent 0 encodes subnormals
``m/8 * 2^-6``; the all-ones exponent is an ordinary binade except for
mantissa 7, which is NaN (there are no infinities); largest finite 448.
"""

from __future__ import annotations

import numpy as np

from .attention import attention


def e4m3_to_float(codes):
    """float64 value of every e4m3 byte in ``codes`` (any shape, uint8)."""
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def attention_fp8(q8, k8, v8, q_scale, k_scale, v_scale, cu_q, ctx_len, mode, window, scale,
                  query_rows=None, heads=None):
    """Dual-mode attention of the dequantised e4m3 tensors (fp64).  ``q8``
    [total_q, Hq, D], ``k8`` / ``v8`` [total_kv, Hkv, D] uint8 codes; the
    scales are per tensor.  Returns ``(out, lse)`` like ``oracle.attention``."""
    q = e4m3_to_float(q8) * float(q_scale)
    k = e4m3_to_float(k8) * float(k_scale)
    v = e4m3_to_float(v8) * float(v_scale)
    return attention(q, k, v, cu_q, ctx_len, mode, window, scale, query_rows=query_rows, heads=heads)
