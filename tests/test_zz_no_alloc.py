"""The allocation-free entry point, for callers that cannot call cudaMalloc
(a host framework that owns every device allocation, or a decode loop that
cannot take cudaMalloc's device-wide synchronisation between steps).

``dg_attn_forward_noalloc`` runs the same kernels as ``dg_attn_forward`` on
the same inputs, with its scratch in a static array inside the library
instead of a caller workspace, so its results must equal the workspace entry
point's bit for bit.  The array keeps the previous call's contents: the cases
below alternate (a split-KV-heavy batch with many partial slots, then a
windowed batch of another shape, then the first again, ...), so every call
after the first finds the other case's work list and partials in the array.
The file is named to be collected last; it also passes when run alone in a
fresh process.
"""

import pytest
import torch

from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


def _dev(batch):
    return {k: batch[k].cuda().contiguous() for k in ("q", "k", "v", "cu_q", "ctx_len", "mode")}


def _noalloc(lib, d, window, scale, out, lse):
    total_q, Hq, D = d["q"].shape
    total_kv, Hkv, _ = d["k"].shape
    return lib.dg_attn_forward_noalloc(
        d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["cu_q"].data_ptr(),
        d["ctx_len"].data_ptr(), d["mode"].data_ptr(), d["ctx_len"].numel(), total_q, total_kv,
        Hq, Hkv, D, window, scale, out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return binding.load_library()


CASES = [
    # (seed, sequences (ctx, n, mode), Hq, Hkv, D, window)
    # few query tiles over long contexts: every tile is cut between CTAs
    (31, ((8192, 256, 1), (0, 700, 0), (4096, 256, 1)), 16, 8, 128, -1),
    (32, ((1500, 256, 1), (300, 129, 0)), 32, 4, 256, 300),
]


def test_noalloc_equals_workspace_entry_point_bit_for_bit(lib):
    prepared = []
    for seed, seqs, Hq, Hkv, D, W in CASES:
        wl, batch = wls.random_batch(seed, seqs, Hq, Hkv, D, W)
        d = _dev(batch)
        ref_out, ref_lse = binding.forward(d["q"], d["k"], d["v"], d["cu_q"], d["ctx_len"],
                                           d["mode"], W, wl.scale)
        torch.cuda.synchronize()
        assert binding.status() == binding.DG_OK
        prepared.append((wl, d, W, ref_out, ref_lse))
    # two calls of each case in a row, interleaved with the other case
    for rnd in range(2):
        for wl, d, W, ref_out, ref_lse in prepared:
            out = torch.full_like(d["q"], float("nan"))
            lse = torch.full((wl.total_q, wl.num_q_heads), float("nan"), dtype=torch.float32,
                             device="cuda")
            rc = _noalloc(lib, d, W, wl.scale, out, lse)
            assert rc == binding.DG_OK, binding.error_string(rc)
            torch.cuda.synchronize()
            assert binding.status() == binding.DG_OK
            assert torch.equal(out, ref_out), (rnd, wl.seqs)
            assert torch.equal(lse, ref_lse), (rnd, wl.seqs)


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    need = binding.workspace_size(1, 1 << 22, 32, 1, 256)
    assert need > binding.NOALLOC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the size check fails before anything is enqueued
    rc = lib.dg_attn_forward_noalloc(fake, fake, fake, fake, fake, fake, 1, 1 << 22, 1 << 22,
                                     32, 1, 256, -1, 0.0625, fake, None, None)
    assert rc == binding.DG_ERR_WORKSPACE
