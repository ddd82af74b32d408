"""ctypes binding of the dg_attn C ABI (``include/dg_attn.h``).

Argument marshalling only: every step of the forward pass runs in the CUDA
library.  PyTorch supplies device memory and the current stream.  There is no
fallback: if the library is missing or the GPU is not an sm_103 part, calls
raise.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

import torch

from . import build as _build

DG_OK = 0
DG_ERR_INVALID_ARG = 1
DG_ERR_UNSUPPORTED = 2
DG_ERR_CUDA = 3
DG_ERR_WORKSPACE = 4
DG_ERR_DEVICE_TIMEOUT = 5
DG_ERR_DEVICE_BOUNDS = 6

DG_MODE_CAUSAL = 0
DG_MODE_BIDIRECTIONAL = 1

# capacity of dg_attn_forward_noalloc's static scratch (DG_ATTN_NOALLOC_SCRATCH_BYTES)
NOALLOC_SCRATCH_BYTES = 48 << 20

EXPORTED = ("dg_attn_workspace_size", "dg_attn_launches_per_call", "dg_attn_forward", "dg_attn_forward_profiled",
            "dg_attn_forward_noalloc", "dg_attn_forward_paged", "dg_attn_forward_paged_profiled",
            "dg_attn_forward_fp8", "dg_attn_forward_fp8_profiled",
            "dg_selfcond_workspace_size", "dg_selfcond_forward", "dg_selfcond_forward_profiled",
            "dg_accept_workspace_size", "dg_accept_step", "dg_sampler_workspace_size",
            "dg_sampler_step",
            "dg_attn_status", "dg_attn_error_string", "dg_attn_version")

_libs = {}        # loaded libraries: False -> the library, True -> the checking build
_use_debug = False


class DgAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} (status {code})")


def library_path(debug: bool = False) -> str:
    return _build.lib_path(debug)


def load_library(debug: bool | None = None):
    """Loads ``lib/libdg_attn.so`` (built by ``build.build_all()``); raises if
    absent.  ``debug=True`` loads the bounds-checking build
    ``lib/libdg_attn_debug.so`` instead; by default the one selected by
    ``debug_library()`` (the library itself outside it)."""
    dbg = _use_debug if debug is None else bool(debug)
    if dbg in _libs:
        return _libs[dbg]
    path = library_path(dbg)
    if not os.path.exists(path):
        raise RuntimeError(f"dg_attn CUDA library not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.dg_attn_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.dg_attn_workspace_size.restype = sz
    lib.dg_attn_launches_per_call.argtypes = [i32] * 7
    lib.dg_attn_launches_per_call.restype = i32
    lib.dg_attn_forward.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                    ctypes.c_float, vp, vp, vp, sz, vp]
    lib.dg_attn_forward.restype = ctypes.c_int
    lib.dg_attn_forward_profiled.argtypes = lib.dg_attn_forward.argtypes + [vp, vp]
    lib.dg_attn_forward_profiled.restype = ctypes.c_int
    lib.dg_attn_forward_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                            i32, ctypes.c_float, vp, vp, vp]
    lib.dg_attn_forward_noalloc.restype = ctypes.c_int
    lib.dg_attn_forward_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                        ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                        ctypes.c_float, vp, vp, vp, sz, vp]
    lib.dg_attn_forward_fp8.restype = ctypes.c_int
    lib.dg_attn_forward_fp8_profiled.argtypes = lib.dg_attn_forward_fp8.argtypes + [vp, vp]
    lib.dg_attn_forward_fp8_profiled.restype = ctypes.c_int
    lib.dg_attn_forward_paged.argtypes = [vp, vp, vp, vp, vp, i32, i32, vp, i32, vp, vp, vp, i32,
                                          i32, i32, i32, i32, i32, ctypes.c_float, vp, vp, vp, sz,
                                          vp]
    lib.dg_attn_forward_paged.restype = ctypes.c_int
    lib.dg_attn_forward_paged_profiled.argtypes = lib.dg_attn_forward_paged.argtypes + [vp, vp]
    lib.dg_attn_forward_paged_profiled.restype = ctypes.c_int
    lib.dg_selfcond_workspace_size.argtypes = [i32, i32, i32]
    lib.dg_selfcond_workspace_size.restype = sz
    lib.dg_selfcond_forward.argtypes = [vp, i32, i32, vp, i32, vp, vp, sz, vp]
    lib.dg_selfcond_forward.restype = ctypes.c_int
    lib.dg_selfcond_forward_profiled.argtypes = lib.dg_selfcond_forward.argtypes + [vp, vp]
    lib.dg_selfcond_forward_profiled.restype = ctypes.c_int
    lib.dg_accept_workspace_size.argtypes = [i32, i32]
    lib.dg_accept_workspace_size.restype = sz
    f32 = ctypes.c_float
    lib.dg_accept_step.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, f32, f32, i32, i32, i32,
                                   vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.dg_accept_step.restype = ctypes.c_int
    lib.dg_sampler_workspace_size.argtypes = [i32, i32, i32]
    lib.dg_sampler_workspace_size.restype = sz
    lib.dg_sampler_step.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, f32, f32, i32, i32, i32, vp, i32,
                                    vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.dg_sampler_step.restype = ctypes.c_int
    lib.dg_attn_status.argtypes = [vp]
    lib.dg_attn_status.restype = ctypes.c_int
    lib.dg_attn_error_string.argtypes = [i32]
    lib.dg_attn_error_string.restype = ctypes.c_char_p
    lib.dg_attn_version.argtypes = []
    lib.dg_attn_version.restype = i32
    _libs[dbg] = lib
    return lib


@contextlib.contextmanager
def debug_library():
    """Within the block every call of this module goes to the bounds-checking
    build (its own status word included)."""
    global _use_debug
    prev = _use_debug
    _use_debug = True
    try:
        yield load_library()
    finally:
        _use_debug = prev


def error_string(code: int) -> str:
    return load_library().dg_attn_error_string(int(code)).decode()


def version() -> int:
    return int(load_library().dg_attn_version())


def workspace_size(num_seqs: int, total_q: int, num_q_heads: int, num_kv_heads: int,
                   head_dim: int) -> int:
    return int(load_library().dg_attn_workspace_size(num_seqs, total_q, num_q_heads, num_kv_heads,
                                                     head_dim))


def launches_per_call(num_seqs: int, total_q: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                      paged: bool = False, e4m3: bool = False) -> int:
    """Kernels one forward call with these sizes launches (2 or 3)."""
    return int(load_library().dg_attn_launches_per_call(num_seqs, total_q, num_q_heads, num_kv_heads,
                                                        head_dim, int(paged), int(e4m3)))


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def status(stream=None) -> int:
    """Synchronises the stream and returns (then clears) the device status word."""
    return int(load_library().dg_attn_status(_stream_handle(stream)))


def forward(q, k, v, cu_q, ctx_len, mode, window: int, scale: float, *, out=None, lse=None,
            workspace=None, stream=None, return_lse: bool = True, events=None):
    """Dual-mode attention forward through ``dg_attn_forward``.

    q [total_q, Hq, D] bf16, k/v [total_kv, Hkv, D] bf16, cu_q [B+1] int32,
    ctx_len [B] int32, mode [B] uint8 (0 causal, 1 bidirectional), all on the
    same CUDA device.  Returns ``(out, lse)`` (``lse`` None unless requested).
    ``events=(begin, end)`` (torch.cuda.Event) goes through
    ``dg_attn_forward_profiled``: the events bracket the main attention kernel.
    """
    lib = load_library()
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
                        ("cu_q", cu_q, torch.int32), ("ctx_len", ctx_len, torch.int32),
                        ("mode", mode, torch.uint8)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    total_q, Hq, D = q.shape
    total_kv, Hkv, Dk = k.shape
    if tuple(v.shape) != (total_kv, Hkv, Dk) or Dk != D:
        raise ValueError("k and v must both be [total_kv, Hkv, D]")
    B = ctx_len.numel()
    if cu_q.numel() != B + 1 or mode.numel() != B:
        raise ValueError("cu_q must have num_seqs+1 entries and mode num_seqs")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    need = lib.dg_attn_workspace_size(B, total_q, Hq, Hkv, D)
    if need == 0:
        raise DgAttnError(DG_ERR_INVALID_ARG, "dg_attn_workspace_size")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(cu_q), _ptr(ctx_len), _ptr(mode), B, total_q, total_kv,
            Hq, Hkv, D, int(window), float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if events is None:
        rc = lib.dg_attn_forward(*args)
    else:
        rc = lib.dg_attn_forward_profiled(*args, events[0].cuda_event, events[1].cuda_event)
    if rc != DG_OK:
        raise DgAttnError(rc, "dg_attn_forward")
    return out, lse


def forward_fp8(q8, k8, v8, cu_q, ctx_len, mode, window: int, scale: float, q_scale: float,
                k_scale: float, v_scale: float, *, out=None, lse=None, workspace=None, stream=None,
                events=None):
    """FP8 variant through ``dg_attn_forward_fp8``: q8 / k8 / v8 are e4m3 codes
    (uint8 or torch.float8_e4m3fn) shaped like the bf16 inputs, with one fp32
    scale per tensor.  Returns ``(out bf16, lse fp32)``."""
    lib = load_library()
    q8, k8, v8 = (t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t for t in (q8, k8, v8))
    for name, t, dt in (("q8", q8, torch.uint8), ("k8", k8, torch.uint8), ("v8", v8, torch.uint8),
                        ("cu_q", cu_q, torch.int32), ("ctx_len", ctx_len, torch.int32),
                        ("mode", mode, torch.uint8)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    total_q, Hq, D = q8.shape
    total_kv, Hkv, Dk = k8.shape
    if tuple(v8.shape) != (total_kv, Hkv, Dk) or Dk != D:
        raise ValueError("k8 and v8 must both be [total_kv, Hkv, D]")
    B = ctx_len.numel()
    if out is None:
        out = torch.empty((total_q, Hq, D), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q8.device)
    need = lib.dg_attn_workspace_size(B, total_q, Hq, Hkv, D)
    if need == 0:
        raise DgAttnError(DG_ERR_INVALID_ARG, "dg_attn_workspace_size")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q8.device)
    args = (_ptr(q8), _ptr(k8), _ptr(v8), _ptr(cu_q), _ptr(ctx_len), _ptr(mode), B, total_q, total_kv,
            Hq, Hkv, D, int(window), float(scale), float(q_scale), float(k_scale), float(v_scale),
            _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream_handle(stream))
    if events is None:
        rc = lib.dg_attn_forward_fp8(*args)
    else:
        rc = lib.dg_attn_forward_fp8_profiled(*args, events[0].cuda_event, events[1].cuda_event)
    if rc != DG_OK:
        raise DgAttnError(rc, "dg_attn_forward_fp8")
    return out, lse


def forward_paged(q, k_new, v_new, k_cache, v_cache, block_table, cu_q, ctx_len, mode,
                  window: int, scale: float, *, out=None, lse=None, workspace=None, stream=None,
                  return_lse: bool = True, events=None):
    """Dual-mode attention over a paged KV cache through ``dg_attn_forward_paged``.

    k_cache / v_cache [num_pages, page_size, Hkv, D] bf16, block_table
    [B, max_pages_per_seq] int32; k_new / v_new [total_q, Hkv, D] bf16 (or
    both None) are written into the cache at the query tokens' positions
    first.  Other arguments as for ``forward``.  Returns ``(out, lse)``.
    """
    lib = load_library()
    checks = [("q", q, torch.bfloat16), ("k_cache", k_cache, torch.bfloat16),
              ("v_cache", v_cache, torch.bfloat16), ("block_table", block_table, torch.int32),
              ("cu_q", cu_q, torch.int32), ("ctx_len", ctx_len, torch.int32),
              ("mode", mode, torch.uint8)]
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new must both be given or both be None")
    if k_new is not None:
        checks += [("k_new", k_new, torch.bfloat16), ("v_new", v_new, torch.bfloat16)]
    for name, t, dt in checks:
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    total_q, Hq, D = q.shape
    num_pages, page_size, Hkv, Dk = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape) or Dk != D:
        raise ValueError("k_cache and v_cache must both be [num_pages, page_size, Hkv, D]")
    if k_new is not None and (tuple(k_new.shape) != (total_q, Hkv, D) or
                              tuple(v_new.shape) != (total_q, Hkv, D)):
        raise ValueError("k_new and v_new must be [total_q, Hkv, D]")
    B = ctx_len.numel()
    if cu_q.numel() != B + 1 or mode.numel() != B or block_table.dim() != 2 or \
            block_table.shape[0] != B:
        raise ValueError("cu_q [B+1], mode [B] and block_table [B, max_pages] required")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    need = lib.dg_attn_workspace_size(B, total_q, Hq, Hkv, D)
    if need == 0:
        raise DgAttnError(DG_ERR_INVALID_ARG, "dg_attn_workspace_size")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    args = (_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), num_pages, page_size,
            _ptr(block_table), block_table.shape[1], _ptr(cu_q), _ptr(ctx_len), _ptr(mode), B,
            total_q, Hq, Hkv, D, int(window), float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if events is None:
        rc = lib.dg_attn_forward_paged(*args)
    else:
        rc = lib.dg_attn_forward_paged_profiled(*args, events[0].cuda_event, events[1].cuda_event)
    if rc != DG_OK:
        raise DgAttnError(rc, "dg_attn_forward_paged")
    return out, lse


def self_conditioning(logits, embedding, *, out=None, workspace=None, stream=None, events=None):
    """Probability-weighted embedding average through ``dg_selfcond_forward``.

    logits [rows, vocab] bf16, embedding [vocab, d_model] bf16 (CUDA).  Returns
    ``out`` [rows, d_model] fp32.  ``events=(begin, end)`` goes through
    ``dg_selfcond_forward_profiled``: the events bracket the tensor-core kernel.
    """
    lib = load_library()
    for name, t in (("logits", logits), ("embedding", embedding)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 2:
            raise ValueError(f"{name} must be a contiguous 2-D CUDA bfloat16 tensor")
    rows, vocab = logits.shape
    if embedding.shape[0] != vocab:
        raise ValueError("embedding must be [vocab, d_model]")
    d = embedding.shape[1]
    if out is None:
        out = torch.empty((rows, d), dtype=torch.float32, device=logits.device)
    need = lib.dg_selfcond_workspace_size(rows, vocab, d)
    if need == 0:
        raise DgAttnError(DG_ERR_INVALID_ARG, "dg_selfcond_workspace_size")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=logits.device)
    args = (_ptr(logits), rows, vocab, _ptr(embedding), d, _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if events is None:
        rc = lib.dg_selfcond_forward(*args)
    else:
        rc = lib.dg_selfcond_forward_profiled(*args, events[0].cuda_event, events[1].cuda_event)
    if rc != DG_OK:
        raise DgAttnError(rc, "dg_selfcond_forward")
    return out


def accept_step(logits, cu_rows, accepted_in, argmax_prev, stable_in, entropy_budget: float,
                entropy_threshold: float, patience: int, step: int, max_steps: int, *,
                workspace=None, stream=None, events=None):
    """Entropy-bounded acceptance of one denoise step through ``dg_accept_step``.

    logits [rows, vocab] bf16, cu_rows [canvases+1] int32, accepted_in [rows]
    uint8, argmax_prev [rows] int32, stable_in [canvases] int32 (CUDA).  Returns
    a dict of entropy, confidence, argmax, accepted, stable, converged tensors.
    ``events=(begin, end)`` are recorded around the call on the stream.
    """
    lib = load_library()
    for name, t, dt in (("logits", logits, torch.bfloat16), ("cu_rows", cu_rows, torch.int32),
                        ("accepted_in", accepted_in, torch.uint8),
                        ("argmax_prev", argmax_prev, torch.int32), ("stable_in", stable_in, torch.int32)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    rows, vocab = logits.shape
    nb = cu_rows.numel() - 1
    dev = logits.device
    res = dict(entropy=torch.empty(rows, dtype=torch.float32, device=dev),
               confidence=torch.empty(rows, dtype=torch.float32, device=dev),
               argmax=torch.empty(rows, dtype=torch.int32, device=dev),
               accepted=torch.empty(rows, dtype=torch.uint8, device=dev),
               stable=torch.empty(nb, dtype=torch.int32, device=dev),
               converged=torch.empty(nb, dtype=torch.uint8, device=dev))
    need = lib.dg_accept_workspace_size(rows, vocab)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    sh = _stream_handle(stream)
    if events is not None:
        events[0].record(torch.cuda.current_stream() if stream is None else stream)
    rc = lib.dg_accept_step(_ptr(logits), rows, vocab, _ptr(cu_rows), nb, _ptr(accepted_in),
                            _ptr(argmax_prev), _ptr(stable_in), float(entropy_budget),
                            float(entropy_threshold), int(patience), int(step), int(max_steps),
                            _ptr(res["entropy"]), _ptr(res["confidence"]), _ptr(res["argmax"]),
                            _ptr(res["accepted"]), _ptr(res["stable"]), _ptr(res["converged"]),
                            _ptr(workspace), workspace.numel() * workspace.element_size(), sh)
    if events is not None:
        events[1].record(torch.cuda.current_stream() if stream is None else stream)
    if rc != DG_OK:
        raise DgAttnError(rc, "dg_accept_step")
    return res


def sampler_step(logits, cu_rows, accepted_in, argmax_prev, stable_in, entropy_budget: float,
                 entropy_threshold: float, patience: int, step: int, max_steps: int, embedding, *,
                 workspace=None, stream=None, events=None):
    """Acceptance step and self-conditioning average of one step's logits
    through ``dg_sampler_step`` (one pass of row statistics for both).
    Returns the ``accept_step`` dict plus ``selfcond`` [rows, d_model] fp32.
    ``events=(begin, end)`` are recorded around the call on the stream."""
    lib = load_library()
    for name, t, dt in (("logits", logits, torch.bfloat16), ("cu_rows", cu_rows, torch.int32),
                        ("accepted_in", accepted_in, torch.uint8),
                        ("argmax_prev", argmax_prev, torch.int32), ("stable_in", stable_in, torch.int32),
                        ("embedding", embedding, torch.bfloat16)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    rows, vocab = logits.shape
    d = embedding.shape[1]
    if embedding.shape[0] != vocab:
        raise ValueError("embedding must be [vocab, d_model]")
    nb = cu_rows.numel() - 1
    dev = logits.device
    res = dict(entropy=torch.empty(rows, dtype=torch.float32, device=dev),
               confidence=torch.empty(rows, dtype=torch.float32, device=dev),
               argmax=torch.empty(rows, dtype=torch.int32, device=dev),
               accepted=torch.empty(rows, dtype=torch.uint8, device=dev),
               stable=torch.empty(nb, dtype=torch.int32, device=dev),
               converged=torch.empty(nb, dtype=torch.uint8, device=dev),
               selfcond=torch.empty((rows, d), dtype=torch.float32, device=dev))
    need = lib.dg_sampler_workspace_size(rows, vocab, d)
    if need == 0:
        raise DgAttnError(DG_ERR_INVALID_ARG, "dg_sampler_workspace_size")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    sh = _stream_handle(stream)
    if events is not None:
        events[0].record(torch.cuda.current_stream() if stream is None else stream)
    rc = lib.dg_sampler_step(_ptr(logits), rows, vocab, _ptr(cu_rows), nb, _ptr(accepted_in),
                             _ptr(argmax_prev), _ptr(stable_in), float(entropy_budget),
                             float(entropy_threshold), int(patience), int(step), int(max_steps),
                             _ptr(embedding), d, _ptr(res["entropy"]), _ptr(res["confidence"]),
                             _ptr(res["argmax"]), _ptr(res["accepted"]), _ptr(res["stable"]),
                             _ptr(res["converged"]), _ptr(res["selfcond"]), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), sh)
    if events is not None:
        events[1].record(torch.cuda.current_stream() if stream is None else stream)
    if rc != DG_OK:
        raise DgAttnError(rc, "dg_sampler_step")
    return res
