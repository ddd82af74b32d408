"""Host-only checks of the C ABI: the library builds and loads, exports every
function ``include/dg_attn.h`` declares, and returns the documented error
codes for arguments the host can reject without touching a GPU."""

import ctypes
import os
import re

import pytest

from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import build as dg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dg_attn.h")


@pytest.fixture(scope="module")
def lib():
    dg_build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_(?:attn|accept|selfcond|sampler)_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("dg_attn_forward", "dg_attn_workspace_size", "dg_attn_status", "dg_attn_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(binding.EXPORTED) <= set(declared_functions())


def test_error_strings_and_version(lib):
    assert binding.error_string(0) == "ok"
    assert "timed out" in binding.error_string(binding.DG_ERR_DEVICE_TIMEOUT)
    assert binding.error_string(999) == "unknown status"
    assert binding.version() >= 100


FAKE = 0x10000  # 64 KiB-aligned non-null address; never dereferenced by these calls


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, cu_q=FAKE, ctx_len=FAKE, mode=FAKE, B=2, total_q=10,
             total_kv=30, Hq=4, Hkv=2, D=128, window=-1, scale=0.1, out=FAKE, lse=None,
             ws=FAKE, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.dg_attn_forward(a["q"], a["k"], a["v"], a["cu_q"], a["ctx_len"], a["mode"], a["B"],
                               a["total_q"], a["total_kv"], a["Hq"], a["Hkv"], a["D"], a["window"],
                               ctypes.c_float(a["scale"]), a["out"], a["lse"], a["ws"], a["ws_bytes"],
                               a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), binding.DG_ERR_INVALID_ARG),
    (dict(k=None), binding.DG_ERR_INVALID_ARG),
    (dict(out=None), binding.DG_ERR_INVALID_ARG),
    (dict(cu_q=None), binding.DG_ERR_INVALID_ARG),
    (dict(Hq=5, Hkv=2), binding.DG_ERR_INVALID_ARG),
    (dict(Hkv=0), binding.DG_ERR_INVALID_ARG),
    (dict(D=96), binding.DG_ERR_UNSUPPORTED),
    (dict(D=100), binding.DG_ERR_INVALID_ARG),
    (dict(Hq=512, Hkv=2), binding.DG_ERR_UNSUPPORTED),
    (dict(window=-2), binding.DG_ERR_INVALID_ARG),
    (dict(scale=0.0), binding.DG_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.DG_ERR_INVALID_ARG),
    (dict(total_kv=5), binding.DG_ERR_INVALID_ARG),
    (dict(q=FAKE + 2), binding.DG_ERR_INVALID_ARG),
    (dict(out=FAKE + 8), binding.DG_ERR_INVALID_ARG),
    (dict(B=-1), binding.DG_ERR_INVALID_ARG),
    (dict(B=0), binding.DG_ERR_INVALID_ARG),
])
def test_host_checked_errors(lib, kw, code):
    assert _fwd(lib, **kw) == code


def test_launches_per_call(lib, monkeypatch):
    """The host-side rule for the launch chain: small contiguous batches have
    no work-list grid (2 kernels), a batch past the per-CTA table bound, a
    paged cache and the e4m3 head_dim-128 shape have one (3)."""
    lp = binding.launches_per_call
    assert lp(1, 256, 32, 4, 256) == 2                      # denoise loop: 4 x (16 + 1) tile bound
    assert lp(4, 1024, 16, 8, 128) == 2                     # max mix: 160
    assert lp(4, 2024, 16, 8, 128) == 3                     # mixed batch: 288 > 256
    assert lp(1, 256, 32, 4, 256, paged=True) == 3          # the work-list grid appends the new rows
    assert lp(4, 1024, 16, 8, 128, e4m3=True) == 3
    assert lp(1, 256, 32, 4, 256, e4m3=True) == 2
    assert lp(1, 256, 32, 5, 256) == 0                      # Hq % Hkv != 0
    monkeypatch.setenv("DG_ATTN_FUSED_WL", "0")
    assert lp(1, 256, 32, 4, 256) == 3


def test_empty_batch_is_a_no_op(lib):
    assert _fwd(lib, B=0, total_q=0) == binding.DG_OK
    assert _fwd(lib, total_q=0) == binding.DG_OK


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "dual_mode_canvas_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, flags=re.M), f
                assert "oracle/" not in text, f


def _noalloc(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, cu_q=FAKE, ctx_len=FAKE, mode=FAKE, B=1, total_q=1 << 22,
             total_kv=1 << 22, Hq=32, Hkv=1, D=256, window=-1, scale=0.0625, out=FAKE, lse=None,
             stream=None)
    a.update(kw)
    return lib.dg_attn_forward_noalloc(a["q"], a["k"], a["v"], a["cu_q"], a["ctx_len"], a["mode"],
                                       a["B"], a["total_q"], a["total_kv"], a["Hq"], a["Hkv"], a["D"],
                                       a["window"], ctypes.c_float(a["scale"]), a["out"], a["lse"],
                                       a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), binding.DG_ERR_INVALID_ARG),
    (dict(out=FAKE + 8), binding.DG_ERR_INVALID_ARG),
    (dict(window=-2), binding.DG_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.DG_ERR_INVALID_ARG),
    (dict(total_kv=5), binding.DG_ERR_INVALID_ARG),
    (dict(D=96), binding.DG_ERR_UNSUPPORTED),
])
def test_noalloc_checks_arguments_before_its_scratch_size(lib, kw, code):
    """Sizes far beyond the static scratch with one bad argument: the argument
    error is reported (as dg_attn_forward reports it), not a workspace error,
    and nothing reaches a GPU."""
    assert _noalloc(lib, **kw) == code


def test_no_cluster_multicast_in_sources():
    """Every kernel loads its operands from this GPU's memory into its own
    shared memory: no TMA load or tcgen05 commit names a cluster multicast."""
    for d in (os.path.join(ROOT, "dual_mode_canvas_gb300", "csrc"), os.path.join(ROOT, "include")):
        for f in os.listdir(d):
            text = open(os.path.join(d, f)).read()
            assert "multicast" not in text, f


def test_bounds_checking_build_exports_the_same_symbols():
    dg_build.build(debug=True)
    dbg = binding.load_library(debug=True)
    for name in declared_functions():
        assert hasattr(dbg, name), name
    assert binding.load_library(debug=False) is not dbg
