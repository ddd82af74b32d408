"""GPU parity of the self-conditioning embedding average (``dg_selfcond_forward``,
called through the C ABI) against the fp64 CPU oracle on the same seeded bf16
logits and embeddings.

Bar: max |out - oracle| <= 1e-2 and mean |out - oracle| <= 1e-3 (the
embeddings are N(0, 1); the kernel rounds the probabilities to bf16, a
relative error of at most 2^-9 per term of a convex combination).  Small
shapes are compared element by element; the full-size step on sampled rows and
column blocks, which the oracle computes independently of the rest.
"""

import numpy as np
import pytest
import torch

import oracle.selfcond as sc
from dual_mode_canvas_gb300 import binding
from dual_mode_canvas_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
MEAN_ABS = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    assert binding.status() == binding.DG_OK


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check(got, ref, what=""):
    assert np.isfinite(got).all(), what
    d = np.abs(got - ref)
    assert d.max() <= MAX_ABS, f"{what} max|d|={d.max():.3g}"
    assert d.mean() <= MEAN_ABS, f"{what} mean|d|={d.mean():.3g}"


def check_bound(got, x, E, what=""):
    """Small vocabularies: a handful of large probabilities, whose bf16
    rounding (relative error <= 2^-9 each) does not average out.  The error
    of every element is then bounded by 2^-9 * sum_v p_v |E[v, c]|; the test
    allows twice that (ex2.approx and fp32 sums) plus 1e-4, and 1e-2 overall."""
    ref = sc.self_conditioning(x, E)
    bound = 2.0 ** -8 * (sc.softmax_rows(x) @ np.abs(E)) + 1e-4
    d = np.abs(got - ref)
    assert np.isfinite(got).all(), what
    assert d.max() <= MAX_ABS, f"{what} max|d|={d.max():.3g}"
    excess = d - bound
    assert excess.max() <= 0, f"{what} worst excess over the rounding bound {excess.max():.3g}"


def run(x, E):
    y = binding.self_conditioning(x, E)
    torch.cuda.synchronize()
    assert binding.status() == binding.DG_OK
    return y


def test_small_step_matches_oracle():
    """300 rows (a ragged row tile), vocabulary 5000 (a partial last block,
    several vocabulary splits), d_model 320 (a ragged column tile)."""
    wl = wls.SELFCOND_WORKLOADS["selfcond_small"]
    x, _ = wls.make_logits(wl.logits, device="cuda")
    E = wls.make_embedding(wl.logits.vocab, wl.d_model, wl.seed, device="cuda")
    y = run(x, E)
    check(f64(y), sc.self_conditioning(f64(x), f64(E)), "selfcond_small")


@pytest.mark.parametrize("rows,vocab,d", [(1, 8, 8), (130, 64, 264), (129, 4096, 256), (2, 72, 520)])
def test_shapes(rows, vocab, d):
    """One row, a single vocabulary block (one split, direct writes), vocab
    8 / 72 (partial blocks), d_model not a multiple of the 256-column tile."""
    g = torch.Generator(device="cuda").manual_seed(rows * 7 + vocab + d)
    x = (2.0 * torch.randn(rows, vocab, generator=g, device="cuda")).to(torch.bfloat16)
    E = torch.randn(vocab, d, generator=g, device="cuda").to(torch.bfloat16)
    y = run(x, E)
    check_bound(f64(y), f64(x), f64(E), f"{rows}x{vocab}x{d}")


def test_closed_form_rows():
    """A dominant token returns its embedding; uniform logits the mean
    embedding; masked (-inf) tokens carry no weight."""
    V, d = 1000, 128
    g = torch.Generator(device="cuda").manual_seed(7)
    E = torch.randn(V, d, generator=g, device="cuda").to(torch.bfloat16)
    x = torch.randn(6, V, generator=g, device="cuda")
    x[0, 17] = 60.0                      # one-hot up to exp(-55)
    x[1, V - 1] = 60.0
    x[2] = 0.0                           # uniform
    x[3, 500:] = float("-inf")           # upper half masked
    x[4, :] = float("-inf")
    x[4, [3, 900]] = 0.0                 # two tokens, equal weight
    x = x.to(torch.bfloat16)
    y = f64(run(x, E))
    Ef = f64(E)
    check_bound(y, f64(x), Ef, "closed forms vs oracle")
    np.testing.assert_allclose(y[0], Ef[17], atol=2e-2)
    np.testing.assert_allclose(y[1], Ef[V - 1], atol=2e-2)
    np.testing.assert_allclose(y[2], Ef.mean(axis=0), atol=2e-3)
    np.testing.assert_allclose(y[4], 0.5 * (Ef[3] + Ef[900]), atol=2e-2)


def test_full_step_sampled():
    """4 canvases x 256 positions, vocabulary 262144, d_model 2560: sampled
    rows and column blocks against the oracle; every output finite and inside
    the embeddings' column range (a convex combination)."""
    wl = wls.SELFCOND_WORKLOADS["selfcond_step"]
    x, _ = wls.make_logits(wl.logits, device="cuda")
    E = wls.make_embedding(wl.logits.vocab, wl.d_model, wl.seed, device="cuda")
    y = run(x, E)
    assert torch.isfinite(y).all()
    Ef = E.float()
    assert (y <= Ef.max(dim=0).values + 1e-2).all() and (y >= Ef.min(dim=0).values - 1e-2).all()
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, wl.logits.rows - 1], rng.choice(wl.logits.rows, 10, replace=False)]))
    blocks = [0, wl.d_model // 64 - 1] + list(rng.choice(np.arange(1, wl.d_model // 64 - 1), 2, replace=False))
    cols = np.concatenate([np.arange(b * 64, b * 64 + 64) for b in blocks])
    xr = f64(x[torch.from_numpy(rows).cuda()])
    Ec = f64(E[:, torch.from_numpy(cols).cuda()])
    check(f64(y)[np.ix_(rows, cols)], sc.self_conditioning(xr, Ec), "selfcond_step sampled")


def test_host_checks():
    x = torch.zeros((4, 12), dtype=torch.bfloat16, device="cuda")       # vocab not a multiple of 8
    E = torch.zeros((12, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.DgAttnError):
        binding.self_conditioning(x, E)
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    E = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    lib = binding.load_library()
    out = torch.empty((4, 64), dtype=torch.float32, device="cuda")
    rc = lib.dg_selfcond_forward(x.data_ptr(), 4, 64, E.data_ptr(), 64, out.data_ptr(), small.data_ptr(),
                                 16, torch.cuda.current_stream().cuda_stream)
    assert rc == binding.DG_ERR_WORKSPACE
