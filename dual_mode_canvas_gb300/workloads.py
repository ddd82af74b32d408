"""Seeded synthetic inputs for the dual-mode attention workloads.

This module only describes batch shapes and draws random numbers; it holds
none of the attention arithmetic, so both the CUDA path and the CPU oracle can
be fed from it without sharing any of the method.

Recipe: every tensor is drawn i.i.d. N(0, 1) in fp32 from one
``torch.Generator`` seeded with the workload's seed, in the fixed order
q, k, v, on the device that will hold it, then rounded to bf16 (the library's
input type).  The denoise loop redraws its canvas (q, then the canvas rows of
k, then those of v) for step ``s > 0`` from seed ``seed + s``; the cached
context rows of k/v are drawn once (step 0) and reused by every step.

Shapes follow the DiffusionGemma pages: a 256-token canvas (agentlenshq page,
"architecture and decoding"), per-sequence causal (prefill / commit) or
bidirectional (denoise) mode in one batch ("dynamic per-sequence causal
attention"), up to 4 sequences with contexts up to 262144 tokens (the developer
guide's ``vllm serve --max-model-len 262144 --max-num-seqs 4`` example), and
full or symmetric sliding-window layers.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

CAUSAL = 0
BIDIRECTIONAL = 1


@dataclass(frozen=True)
class Workload:
    name: str
    seqs: tuple            # ((ctx_len, n_q, mode), ...)
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    window: int            # -1 full layer, W >= 0 sliding window
    seed: int
    steps: int = 1         # denoise steps (the loop redraws the canvas)
    draw_dtype: str = "bf16"   # "fp32": the oracle may also use the unrounded draw

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def total_q(self) -> int:
        return sum(n for _, n, _ in self.seqs)

    @property
    def total_kv(self) -> int:
        return sum(c + n for c, n, _ in self.seqs)


_MIX = ((0, 512, CAUSAL), (0, 1000, CAUSAL), (2048, 256, BIDIRECTIONAL), (4096, 256, BIDIRECTIONAL))
_MAX = ((65536, 256, BIDIRECTIONAL), (131072, 256, BIDIRECTIONAL),
        (262144, 256, BIDIRECTIONAL), (131072, 256, CAUSAL))

WORKLOADS = {
    # one bidirectional canvas of 256 queries over 128 cached tokens, 1 head, D=64
    "tiny": Workload("tiny", ((128, 256, BIDIRECTIONAL),), 1, 1, 64, -1, 0, draw_dtype="fp32"),
    # 2 causal prefills (512, 1000) + 2 canvases over 2048 / 4096 cached tokens
    "mixed_full": Workload("mixed_full", _MIX, 16, 8, 128, -1, 1),
    "mixed_w512": Workload("mixed_w512", _MIX, 16, 8, 128, 512, 2),
    # batch-1 denoise loop: 48 steps of one canvas over a 32768-token context
    "denoise_loop": Workload("denoise_loop", ((32768, 256, BIDIRECTIONAL),), 32, 4, 256, -1, 3,
                             steps=48),
    # 3 canvases over 64k/128k/256k contexts + a causal commit block over 128k
    "maxmix_full": Workload("maxmix_full", _MAX, 16, 8, 128, -1, 4),
    "maxmix_w1024": Workload("maxmix_w1024", _MAX, 16, 8, 128, 1024, 4),
}

_CHUNK = 1 << 24


def _randn(gen: torch.Generator, shape, device) -> torch.Tensor:
    """fp32 N(0,1) of ``shape`` drawn in chunks of 2^24 elements (bounded
    temporary memory on the host)."""
    numel = 1
    for d in shape:
        numel *= d
    out = torch.empty(numel, dtype=torch.float32, device=device)
    for o in range(0, numel, _CHUNK):
        e = min(numel, o + _CHUNK)
        out[o:e] = torch.randn(e - o, generator=gen, dtype=torch.float32, device=device)
    return out.view(*shape)


def metadata(wl: Workload):
    """Host int32 ``cu_q`` [B+1], int32 ``ctx_len`` [B], uint8 ``mode`` [B]."""
    cu = [0]
    for _, n, _ in wl.seqs:
        cu.append(cu[-1] + n)
    cu_q = torch.tensor(cu, dtype=torch.int32)
    ctx_len = torch.tensor([c for c, _, _ in wl.seqs], dtype=torch.int32)
    mode = torch.tensor([m for _, _, m in wl.seqs], dtype=torch.uint8)
    return cu_q, ctx_len, mode


def make_batch(wl: Workload, device="cpu", dtype=torch.bfloat16):
    """Step-0 inputs of ``wl``: dict with q [total_q,Hq,D], k/v [total_kv,Hkv,D]
    (``dtype``; fp32 keeps the unrounded draw) and the host metadata."""
    gen = torch.Generator(device=device).manual_seed(wl.seed)
    q = _randn(gen, (wl.total_q, wl.num_q_heads, wl.head_dim), device)
    k = _randn(gen, (wl.total_kv, wl.num_kv_heads, wl.head_dim), device)
    v = _randn(gen, (wl.total_kv, wl.num_kv_heads, wl.head_dim), device)
    cu_q, ctx_len, mode = metadata(wl)
    return dict(q=q.to(dtype), k=k.to(dtype), v=v.to(dtype), cu_q=cu_q, ctx_len=ctx_len,
                mode=mode, window=wl.window, scale=wl.scale)


def canvas_rows(wl: Workload):
    """KV row indices (within the packed KV buffer) of each sequence's query
    block, i.e. the rows a denoise step rewrites."""
    rows, off = [], 0
    for c, n, _ in wl.seqs:
        rows.append((off + c, off + c + n))
        off += c + n
    return rows


def denoise_step_inputs(wl: Workload, step: int, device="cpu", dtype=torch.bfloat16):
    """Fresh canvas tensors of denoise step ``step >= 1``: q [total_q,Hq,D] and
    the canvas rows of k and v [total_q,Hkv,D], drawn from seed ``seed+step``."""
    gen = torch.Generator(device=device).manual_seed(wl.seed + step)
    q = _randn(gen, (wl.total_q, wl.num_q_heads, wl.head_dim), device)
    kc = _randn(gen, (wl.total_q, wl.num_kv_heads, wl.head_dim), device)
    vc = _randn(gen, (wl.total_q, wl.num_kv_heads, wl.head_dim), device)
    return q.to(dtype), kc.to(dtype), vc.to(dtype)


def random_batch(seed: int, seqs, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 window: int, device="cpu", dtype=torch.bfloat16):
    """Ad-hoc batch for edge-case tests: same recipe, caller-chosen shapes."""
    wl = Workload("adhoc", tuple(seqs), num_q_heads, num_kv_heads, head_dim, window, seed)
    return wl, make_batch(wl, device=device, dtype=dtype)


# ---------------------------------------------------------------- sampler step
@dataclass(frozen=True)
class LogitsWorkload:
    """LM-head logits of the canvases of one denoise step."""
    name: str
    canvases: tuple        # rows per canvas
    vocab: int
    seed: int
    sigma: float = 2.0     # spread of the background logits
    peak: float = 14.0     # largest bump added to one token per row

    @property
    def rows(self) -> int:
        return sum(self.canvases)


# 4 canvases of 256 positions (max-num-seqs 4); a 262144-token vocabulary is an
# assumption (the pages do not give the vocabulary size)
LOGITS_WORKLOADS = {
    "accept_small": LogitsWorkload("accept_small", (256, 100, 37), 50001, 20),
    "accept_step": LogitsWorkload("accept_step", (256, 256, 256, 256), 262144, 21),
}


def make_logits(wl: LogitsWorkload, device="cpu", dtype=torch.bfloat16):
    """logits [rows, vocab]: sigma * N(0,1) background plus, per row, one token
    raised by U(0, peak) (so confidences and entropies spread out), drawn in the
    order background, bump tokens, bump heights; and cu_rows [canvases+1]."""
    gen = torch.Generator(device=device).manual_seed(wl.seed)
    x = _randn(gen, (wl.rows, wl.vocab), device) * wl.sigma
    tok = torch.randint(0, wl.vocab, (wl.rows,), generator=gen, device=device)
    bump = torch.rand(wl.rows, generator=gen, device=device) * wl.peak
    x[torch.arange(wl.rows, device=device), tok] += bump
    cu = [0]
    for n in wl.canvases:
        cu.append(cu[-1] + n)
    return x.to(dtype), torch.tensor(cu, dtype=torch.int32)


# ------------------------------------------------------------ paged KV cache
def make_paged_batch(wl: Workload, page_size: int, device="cpu", spare_pages: int = 7,
                     dtype=torch.bfloat16):
    """Inputs of ``wl`` over a paged KV cache.  Drawn from seed ``wl.seed``
    in the order q, k_new, v_new (the query tokens' K/V, [total_q, Hkv, D]),
    the whole K pool, the whole V pool ([num_pages, page_size, Hkv, D], every
    row N(0, 1)), then a random permutation of the physical pages: sequence s
    owns pages ``perm[o_s : o_s + ceil(L_s / page_size)]`` in order, and
    ``spare_pages`` pages belong to no sequence.  Page-table entries past a
    sequence's last page are -1.  The metadata (cu_q, ctx_len, mode,
    block_table) stays on the host."""
    gen = torch.Generator(device=device).manual_seed(wl.seed)
    Hq, Hkv, D = wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    q = _randn(gen, (wl.total_q, Hq, D), device)
    k_new = _randn(gen, (wl.total_q, Hkv, D), device)
    v_new = _randn(gen, (wl.total_q, Hkv, D), device)
    need = [-(-(c + n) // page_size) for c, n, _ in wl.seqs]
    num_pages = sum(need) + spare_pages
    k_cache = _randn(gen, (num_pages, page_size, Hkv, D), device)
    v_cache = _randn(gen, (num_pages, page_size, Hkv, D), device)
    perm = torch.randperm(num_pages, generator=gen, device=device).cpu()
    table = torch.full((len(wl.seqs), max(need)), -1, dtype=torch.int32)
    o = 0
    for s, k in enumerate(need):
        table[s, :k] = perm[o:o + k].to(torch.int32)
        o += k
    cu_q, ctx_len, mode = metadata(wl)
    return dict(q=q.to(dtype), k_new=k_new.to(dtype), v_new=v_new.to(dtype),
                k_cache=k_cache.to(dtype), v_cache=v_cache.to(dtype), block_table=table,
                page_size=page_size, cu_q=cu_q, ctx_len=ctx_len, mode=mode, window=wl.window,
                scale=wl.scale)


# ------------------------------------------------------------ self-conditioning
@dataclass(frozen=True)
class SelfCondWorkload:
    """LM-head logits of one denoise step and the token-embedding table."""
    name: str
    logits: LogitsWorkload
    d_model: int
    seed: int


# The pages give neither the model width nor the vocabulary size: d_model 2560
# and the 262144-token vocabulary of the acceptance workload are assumptions.
SELFCOND_WORKLOADS = {
    "selfcond_small": SelfCondWorkload("selfcond_small", LogitsWorkload("sc_small", (256, 44), 5000, 30),
                                       320, 31),
    "selfcond_step": SelfCondWorkload("selfcond_step", LOGITS_WORKLOADS["accept_step"], 2560, 32),
    # the same step over a quarter of the vocabulary: a profiling-sized case
    # (about 0.5 GB on the device, still larger than L2)
    "selfcond_v64k": SelfCondWorkload("selfcond_v64k",
                                      LogitsWorkload("v64k", (256, 256, 256, 256), 65536, 33), 2560, 34),
}


def make_embedding(vocab: int, d_model: int, seed: int, device="cpu", dtype=torch.bfloat16):
    """Token-embedding table [vocab, d_model]: N(0, 1) from ``seed``, rounded to
    ``dtype``."""
    gen = torch.Generator(device=device).manual_seed(seed)
    return _randn(gen, (vocab, d_model), device).to(dtype)


# ------------------------------------------------------------------ e4m3 inputs
def quantize_e4m3(x: torch.Tensor, scale: float) -> torch.Tensor:
    """e4m3 codes (uint8) of x / scale, clamped to the finite range +-448."""
    return (x / scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def to_e4m3(x: torch.Tensor):
    """(codes uint8, scale): x / scale rounded to e4m3, scale = max|x| / 448
    (one scale per tensor, so the largest magnitude maps to the largest e4m3)."""
    amax = float(x.abs().max())
    scale = amax / 448.0 if amax > 0 else 1.0
    return quantize_e4m3(x, scale), scale


def make_fp8_batch(wl: Workload, device="cpu"):
    """Step-0 inputs of ``wl`` for the FP8 variant: the same fp32 N(0, 1) draws
    as ``make_batch`` (seed, order q, k, v), each tensor quantised to e4m3
    with its own scale.  Keys q8/k8/v8 (uint8), q_scale/k_scale/v_scale and
    the host metadata."""
    gen = torch.Generator(device=device).manual_seed(wl.seed)
    q = _randn(gen, (wl.total_q, wl.num_q_heads, wl.head_dim), device)
    k = _randn(gen, (wl.total_kv, wl.num_kv_heads, wl.head_dim), device)
    v = _randn(gen, (wl.total_kv, wl.num_kv_heads, wl.head_dim), device)
    q8, qs = to_e4m3(q)
    k8, ks = to_e4m3(k)
    v8, vs = to_e4m3(v)
    cu_q, ctx_len, mode = metadata(wl)
    return dict(q8=q8, k8=k8, v8=v8, q_scale=qs, k_scale=ks, v_scale=vs, cu_q=cu_q,
                ctx_len=ctx_len, mode=mode, window=wl.window, scale=wl.scale)
