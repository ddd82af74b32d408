"""Out-of-bounds write detection without a memory checker: every output and
workspace of every entry point is a window into a larger buffer filled with
a sentinel byte, and the bytes around the window must be untouched after the
call (the workspaces are passed with exactly the size the library asks for)."""

import pytest
import torch

from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

GUARD = 4096
SENT = 0x5A


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    assert binding.status() == binding.DG_OK


class Guarded:
    """A window of ``nbytes`` between two guard regions of sentinel bytes."""

    def __init__(self, nbytes):
        self.n = nbytes
        self.big = torch.full((2 * GUARD + nbytes,), SENT, dtype=torch.uint8, device="cuda")

    def view(self, dtype, shape):
        return self.big[GUARD:GUARD + self.n].view(dtype).view(shape)

    def bytes(self):
        return self.big[GUARD:GUARD + self.n]

    def check(self, what):
        torch.cuda.synchronize()
        assert bool((self.big[:GUARD] == SENT).all()), f"{what}: write before the buffer"
        assert bool((self.big[GUARD + self.n:] == SENT).all()), f"{what}: write past the buffer"


def attention_outputs(total_q, Hq, D, B, Hkv):
    o = Guarded(total_q * Hq * D * 2)
    l = Guarded(total_q * Hq * 4)
    w = Guarded(binding.workspace_size(B, total_q, Hq, Hkv, D))
    return o, l, w


@pytest.mark.parametrize("D", [64, 128, 256])
def test_attention_writes_stay_in_bounds(D):
    seqs = ((300, 256, 1), (0, 333, 0), (1000, 200, 1), (17, 1, 0))
    wl, b = wls.random_batch(900 + D, seqs, 8, 4, D, -1)
    dev = {k: b[k].cuda() for k in ("q", "k", "v", "cu_q", "ctx_len", "mode")}
    o, l, w = attention_outputs(wl.total_q, 8, D, len(seqs), 4)
    for W in (-1, 33):
        binding.forward(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["ctx_len"], dev["mode"], W, wl.scale,
                        out=o.view(torch.bfloat16, (wl.total_q, 8, D)), lse=l.view(torch.float32, (wl.total_q, 8)),
                        workspace=w.bytes())
        assert binding.status() == binding.DG_OK
        for g, name in ((o, "out"), (l, "lse"), (w, "workspace")):
            g.check(f"D={D} W={W} {name}")


def test_fp8_and_paged_writes_stay_in_bounds():
    wl = wls.Workload("canary", ((300, 256, 1), (0, 100, 0)), 8, 2, 256, -1, 910)
    fb = wls.make_fp8_batch(wl, device="cuda")
    o, l, w = attention_outputs(wl.total_q, 8, 256, 2, 2)
    binding.forward_fp8(fb["q8"], fb["k8"], fb["v8"], fb["cu_q"].cuda(), fb["ctx_len"].cuda(), fb["mode"].cuda(),
                        -1, wl.scale, fb["q_scale"], fb["k_scale"], fb["v_scale"],
                        out=o.view(torch.bfloat16, (wl.total_q, 8, 256)),
                        lse=l.view(torch.float32, (wl.total_q, 8)), workspace=w.bytes())
    assert binding.status() == binding.DG_OK
    for g, name in ((o, "out"), (l, "lse"), (w, "workspace")):
        g.check(f"fp8 {name}")
    pb = wls.make_paged_batch(wl, 16, device="cuda")
    o, l, w = attention_outputs(wl.total_q, 8, 256, 2, 2)
    binding.forward_paged(pb["q"], pb["k_new"], pb["v_new"], pb["k_cache"], pb["v_cache"],
                          pb["block_table"].cuda(), pb["cu_q"].cuda(), pb["ctx_len"].cuda(), pb["mode"].cuda(),
                          -1, wl.scale, out=o.view(torch.bfloat16, (wl.total_q, 8, 256)),
                          lse=l.view(torch.float32, (wl.total_q, 8)), workspace=w.bytes())
    assert binding.status() == binding.DG_OK
    for g, name in ((o, "out"), (l, "lse"), (w, "workspace")):
        g.check(f"paged {name}")


def test_selfcond_and_sampler_writes_stay_in_bounds():
    wl = wls.SELFCOND_WORKLOADS["selfcond_small"]
    x, cu = wls.make_logits(wl.logits, device="cuda")
    E = wls.make_embedding(wl.logits.vocab, wl.d_model, wl.seed, device="cuda")
    rows, V, d = wl.logits.rows, wl.logits.vocab, wl.d_model
    lib = binding.load_library()
    o = Guarded(rows * d * 4)
    w = Guarded(lib.dg_selfcond_workspace_size(rows, V, d))
    binding.self_conditioning(x, E, out=o.view(torch.float32, (rows, d)), workspace=w.bytes())
    assert binding.status() == binding.DG_OK
    o.check("selfcond out")
    w.check("selfcond workspace")
    nb = len(wl.logits.canvases)
    outs = {"entropy": Guarded(rows * 4), "confidence": Guarded(rows * 4), "argmax": Guarded(rows * 4),
            "accepted": Guarded(rows), "stable": Guarded(nb * 4), "converged": Guarded(nb),
            "selfcond": Guarded(rows * d * 4)}
    w = Guarded(lib.dg_sampler_workspace_size(rows, V, d))
    z8 = torch.zeros(rows, dtype=torch.uint8, device="cuda")
    z32 = torch.zeros(rows, dtype=torch.int32, device="cuda")
    st = torch.zeros(nb, dtype=torch.int32, device="cuda")
    rc = lib.dg_sampler_step(x.data_ptr(), rows, V, cu.cuda().data_ptr(), nb, z8.data_ptr(), z32.data_ptr(),
                             st.data_ptr(), 2.0, 3.0, 2, 0, 48, E.data_ptr(), d,
                             *[outs[k].bytes().data_ptr() for k in ("entropy", "confidence", "argmax", "accepted",
                                                                    "stable", "converged", "selfcond")],
                             w.bytes().data_ptr(), w.n, torch.cuda.current_stream().cuda_stream)
    assert rc == binding.DG_OK
    assert binding.status() == binding.DG_OK
    for k, g in outs.items():
        g.check(f"sampler {k}")
    w.check("sampler workspace")
