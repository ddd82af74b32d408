"""The combined sampler call (``dg_sampler_step``: acceptance step and
self-conditioning average sharing one pass of row statistics) gives exactly
the outputs of the two separate calls, and those outputs match the oracles."""

import numpy as np
import pytest
import torch

import oracle.acceptance as oacc
import oracle.selfcond as osc
from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    assert binding.status() == binding.DG_OK


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", ["selfcond_small", "selfcond_step"])
def test_sampler_step_equals_the_separate_calls(name):
    wl = wls.SELFCOND_WORKLOADS[name]
    x, cu = wls.make_logits(wl.logits, device="cuda")
    E = wls.make_embedding(wl.logits.vocab, wl.d_model, wl.seed, device="cuda")
    rows, nb = wl.logits.rows, len(wl.logits.canvases)
    rng = np.random.default_rng(7)
    acc_in = torch.from_numpy((rng.uniform(size=rows) < 0.3).astype(np.uint8)).cuda()
    prev = torch.from_numpy(rng.integers(0, wl.logits.vocab, rows).astype(np.int32)).cuda()
    stable = torch.from_numpy(rng.integers(0, 3, nb).astype(np.int32)).cuda()
    cu = cu.cuda()
    args = (x, cu, acc_in, prev, stable, 2.0, 3.0, 2, 5, 48)
    both = binding.sampler_step(*args, E)
    sep = binding.accept_step(*args)
    y = binding.self_conditioning(x, E)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    for k in ("entropy", "confidence", "argmax", "accepted", "stable", "converged"):
        assert torch.equal(both[k], sep[k]), k
    assert torch.equal(both["selfcond"], y)
    # and the shared statistics are right: entropy, argmax and (on sampled
    # rows) the self-conditioning vector against the oracles
    sample = np.unique(np.concatenate([[0, rows - 1], rng.choice(rows, 6, replace=False)]))
    xs = f64(x[torch.from_numpy(sample).cuda()])
    H, c, a = oacc.row_stats(xs)
    np.testing.assert_allclose(both["entropy"].cpu().numpy()[sample], H, rtol=1e-4, atol=1e-4)
    np.testing.assert_array_equal(both["argmax"].cpu().numpy()[sample], a)
    cols = np.arange(min(wl.d_model, 128))
    ref = osc.self_conditioning(xs, f64(E[:, torch.from_numpy(cols).cuda()]))
    assert np.abs(f64(both["selfcond"])[np.ix_(sample, cols)] - ref).max() <= 1e-2
