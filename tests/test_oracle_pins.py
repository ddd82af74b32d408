"""Pins of the CPU oracle against facts that do not come from the oracle itself:
brute force on tiny inputs, a library routine in the special cases where the
method reduces to it, closed forms, invariants, and a hand-worked example.

Rules being pinned: encoder (prefill/commit) mode is causal, decoder (denoise)
mode bidirectional and chosen per sequence (DiffusionGemma, agentlenshq page,
"dual-mode operation" and "dynamic per-sequence causal attention"); sliding
windows see W preceding tokens (causal) or W on each side, 2W+1 in total
(same page, "symmetric sliding-window attention").
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import MODE_BIDIRECTIONAL as BID
from oracle import MODE_CAUSAL as CAU

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _batch(rng, seqs, Hq, Hkv, D):
    total_q = sum(n for _, n, _ in seqs)
    total_kv = sum(c + n for c, n, _ in seqs)
    q = rng.standard_normal((total_q, Hq, D))
    k = rng.standard_normal((total_kv, Hkv, D))
    v = rng.standard_normal((total_kv, Hkv, D))
    cu = np.concatenate([[0], np.cumsum([n for _, n, _ in seqs])])
    ctx = np.array([c for c, _, _ in seqs])
    mode = np.array([m for _, _, m in seqs])
    return q, k, v, cu, ctx, mode


# ---------------------------------------------------------------- brute force

def _brute_causal(q, k, v, c, scale, W):
    """Nested loops over j <= i (and j >= i-W), math.exp, no masks, no numpy
    reductions: the textbook lower-triangular softmax for one head."""
    n, D = q.shape
    out = [[0.0] * D for _ in range(n)]
    lse = [0.0] * n
    for t in range(n):
        i = c + t
        j0 = 0 if W < 0 else max(0, i - W)
        sc = []
        for j in range(j0, i + 1):
            s = 0.0
            for d in range(D):
                s += float(q[t, d]) * float(k[j, d])
            sc.append(scale * s)
        mx = max(sc)
        ex = [math.exp(x - mx) for x in sc]
        tot = sum(ex)
        for d in range(D):
            acc = 0.0
            for jj, e in enumerate(ex):
                acc += e * float(v[j0 + jj, d])
            out[t][d] = acc / tot
        lse[t] = mx + math.log(tot)
    return np.array(out), np.array(lse)


def _brute_bidir(q, k, v, c, scale, W):
    n, D = q.shape
    L = c + n
    out = np.zeros((n, D))
    lse = np.zeros(n)
    for t in range(n):
        i = c + t
        j0 = 0 if W < 0 else max(0, i - W)
        j1 = L - 1 if W < 0 else min(L - 1, i + W)
        sc = [scale * sum(float(q[t, d]) * float(k[j, d]) for d in range(D)) for j in range(j0, j1 + 1)]
        mx = max(sc)
        ex = [math.exp(x - mx) for x in sc]
        tot = sum(ex)
        for d in range(D):
            out[t, d] = sum(e * float(v[j0 + jj, d]) for jj, e in enumerate(ex)) / tot
        lse[t] = mx + math.log(tot)
    return out, lse


@pytest.mark.parametrize("c,n,W", [(0, 7, -1), (5, 6, -1), (4, 9, 2), (0, 5, 0), (3, 4, 10)])
def test_causal_rows_match_bruteforce_triangular(c, n, W):
    rng = np.random.default_rng(11 + c + n)
    D = 5
    q, k, v, cu, ctx, mode = _batch(rng, [(c, n, CAU)], 1, 1, D)
    out, lse = oracle.attention(q, k, v, cu, ctx, mode, W, 0.7)
    bo, bl = _brute_causal(q[:, 0], k[:, 0], v[:, 0], c, 0.7, W)
    np.testing.assert_allclose(out[:, 0], bo, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse[:, 0], bl, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("c,n,W", [(3, 6, 1), (0, 8, 2), (6, 4, 3), (2, 5, 0)])
def test_bidirectional_window_rows_match_bruteforce(c, n, W):
    rng = np.random.default_rng(23 + c * n)
    q, k, v, cu, ctx, mode = _batch(rng, [(c, n, BID)], 1, 1, 4)
    out, lse = oracle.attention(q, k, v, cu, ctx, mode, W, 0.5)
    bo, bl = _brute_bidir(q[:, 0], k[:, 0], v[:, 0], c, 0.5, W)
    np.testing.assert_allclose(out[:, 0], bo, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse[:, 0], bl, rtol=1e-12, atol=1e-12)


# ------------------------------------------------- library special cases (SDPA)

@pytest.mark.parametrize("W", [-1, 64, 10**6])
def test_bidirectional_wide_window_equals_unmasked_sdpa(W):
    """A bidirectional query with W >= L sees every key: plain attention.
    Cross-checked with torch's SDPA (fp64, CPU, GQA by repeating KV heads)."""
    rng = np.random.default_rng(5)
    c, n, Hq, Hkv, D = 40, 24, 4, 2, 16
    q, k, v, cu, ctx, mode = _batch(rng, [(c, n, BID)], Hq, Hkv, D)
    scale = 1 / math.sqrt(D)
    out, lse = oracle.attention(q, k, v, cu, ctx, mode, W, scale)
    qt = torch.from_numpy(q).permute(1, 0, 2)                 # [Hq, n, D]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)
    ref_lse = torch.logsumexp(scale * qt @ kt.transpose(1, 2), dim=-1).T.numpy()
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_causal_without_context_equals_sdpa_is_causal():
    rng = np.random.default_rng(6)
    n, Hq, D = 33, 2, 8
    q, k, v, cu, ctx, mode = _batch(rng, [(0, n, CAU)], Hq, Hq, D)
    out, _ = oracle.attention(q, k, v, cu, ctx, mode, -1, 0.3)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).permute(1, 0, 2), torch.from_numpy(k).permute(1, 0, 2),
        torch.from_numpy(v).permute(1, 0, 2), is_causal=True, scale=0.3)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- closed forms

def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_window_counts_golden():
    rows = _read_golden("window_counts.txt")
    assert len(rows) >= 10
    for c, n, md, W, t, cnt in rows:
        m = oracle.visible_mask(int(c), int(n), md == "C", int(W))
        assert int(m[int(t)].sum()) == int(cnt), (c, n, md, W, t)


@pytest.mark.parametrize("W", [0, 1, 3, 17])
def test_window_counts_away_from_edges(W):
    c, n = 200, 120
    for causal, expect in ((True, W + 1), (False, 2 * W + 1)):
        m = oracle.visible_mask(c, n, causal, W)
        # rows whose window is clipped by neither edge
        for t in range(W, n - W - 1):
            assert m[t].sum() == expect
            i = c + t
            idx = np.flatnonzero(m[t])
            assert idx[0] == i - W and idx[-1] == (i if causal else i + W)


def test_window_counts_edge_clipping():
    """Clipped counts: bidirectional min(L-1, i+W) - max(0, i-W) + 1,
    causal i - max(0, i-W) + 1, for every row of several geometries."""
    for c, n, W in ((0, 50, 7), (3, 20, 30), (100, 256, 64), (10, 5, 0)):
        L = c + n
        for causal in (True, False):
            m = oracle.visible_mask(c, n, causal, W)
            for t in range(n):
                i = c + t
                hi = i if causal else min(L - 1, i + W)
                assert m[t].sum() == hi - max(0, i - W) + 1


def test_q_zero_gives_mean_of_visible_values():
    """q = 0 makes every visible score 0: out = mean of visible V rows and
    lse = ln(number of visible keys)."""
    rng = np.random.default_rng(9)
    seqs = [(7, 9, CAU), (0, 6, BID), (12, 5, BID)]
    for W in (-1, 2, 4):
        q, k, v, cu, ctx, mode = _batch(rng, seqs, 2, 1, 3)
        q[:] = 0.0
        out, lse = oracle.attention(q, k, v, cu, ctx, mode, W, 1.0)
        off = 0
        for s, (c, n, md) in enumerate(seqs):
            L = c + n
            for t in range(n):
                i = c + t
                lo = 0 if W < 0 else max(0, i - W)
                hi = i if md == CAU else (L - 1 if W < 0 else min(L - 1, i + W))
                exp_out = v[off + lo:off + hi + 1, 0].mean(axis=0)
                r = cu[s] + t
                for h in range(2):
                    np.testing.assert_allclose(out[r, h], exp_out, rtol=1e-13, atol=1e-13)
                    assert abs(lse[r, h] - math.log(hi - lo + 1)) < 1e-13
            off += L


def test_single_visible_key_returns_its_value_exactly():
    rng = np.random.default_rng(3)
    # W = 0 bidirectional: self only
    q, k, v, cu, ctx, mode = _batch(rng, [(5, 8, BID)], 2, 2, 6)
    out, lse = oracle.attention(q, k, v, cu, ctx, mode, 0, 0.25)
    for t in range(8):
        for h in range(2):
            assert np.array_equal(out[t, h], v[5 + t, h])
            assert abs(lse[t, h] - 0.25 * q[t, h] @ k[5 + t, h]) < 1e-13
    # causal row 0 with no context sees key 0 only
    q, k, v, cu, ctx, mode = _batch(rng, [(0, 4, CAU)], 1, 1, 6)
    out, _ = oracle.attention(q, k, v, cu, ctx, mode, -1, 0.25)
    assert np.array_equal(out[0, 0], v[0, 0])


def test_worked_example_golden():
    rows = _read_golden("worked_example.txt")
    q = np.array([[[1.0]], [[1.0]]])
    k = np.array([[[0.0]], [[math.log(2)]], [[math.log(3)]]])
    v = np.array([[[6.0]], [[0.0]], [[12.0]]])
    for md, W, t, o, l in rows:
        mode = [CAU if md == "causal" else BID]
        out, lse = oracle.attention(q, k, v, [0, 2], [1], mode, int(W), 1.0)
        assert abs(out[int(t), 0, 0] - float(o)) < 1e-12, (md, W, t)
        assert abs(lse[int(t), 0] - math.log(float(l[2:]))) < 1e-12, (md, W, t)


# ---------------------------------------------------------------- invariants

def test_bidirectional_permutation_equivariance():
    """Full window: permuting canvas keys+values leaves every output row
    unchanged; permuting canvas q,k,v jointly permutes the canvas outputs."""
    rng = np.random.default_rng(21)
    c, n = 17, 13
    q, k, v, cu, ctx, mode = _batch(rng, [(c, n, BID)], 2, 1, 8)
    out, lse = oracle.attention(q, k, v, cu, ctx, mode, -1, 0.4)
    perm = rng.permutation(n)
    k2, v2 = k.copy(), v.copy()
    k2[c:] = k[c + perm]
    v2[c:] = v[c + perm]
    o2, l2 = oracle.attention(q, k2, v2, cu, ctx, mode, -1, 0.4)
    np.testing.assert_allclose(o2, out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l2, lse, rtol=1e-12, atol=1e-12)
    o3, l3 = oracle.attention(q[perm], k2, v2, cu, ctx, mode, -1, 0.4)
    np.testing.assert_allclose(o3, out[perm], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l3, lse[perm], rtol=1e-12, atol=1e-12)
    # the causal mode is NOT permutation invariant (sanity: the test can fail)
    mode_c = np.array([CAU])
    oc, _ = oracle.attention(q, k, v, cu, ctx, mode_c, -1, 0.4)
    oc2, _ = oracle.attention(q, k2, v2, cu, ctx, mode_c, -1, 0.4)
    assert not np.allclose(oc, oc2)


def test_causal_output_ignores_future_tokens():
    rng = np.random.default_rng(4)
    c, n = 6, 10
    q, k, v, cu, ctx, mode = _batch(rng, [(c, n, CAU)], 1, 1, 4)
    out, _ = oracle.attention(q, k, v, cu, ctx, mode, -1, 0.5)
    k2, v2 = k.copy(), v.copy()
    k2[c + 6:] += 3.0
    v2[c + 6:] -= 2.0
    out2, _ = oracle.attention(q, k2, v2, cu, ctx, mode, -1, 0.5)
    np.testing.assert_array_equal(out2[:6], out[:6])
    assert not np.allclose(out2[6:], out[6:])


def test_gqa_mapping_and_head_duplication():
    """Query head h reads KV head h // (Hq/Hkv); duplicating each KV head
    (Hkv -> Hq) reproduces the grouped result, and heads are independent."""
    rng = np.random.default_rng(8)
    seqs = [(4, 6, CAU), (9, 5, BID)]
    Hq, Hkv = 6, 2
    q, k, v, cu, ctx, mode = _batch(rng, seqs, Hq, Hkv, 4)
    out, lse = oracle.attention(q, k, v, cu, ctx, mode, 3, 0.6)
    kd = np.repeat(k, Hq // Hkv, axis=1)
    vd = np.repeat(v, Hq // Hkv, axis=1)
    od, ld = oracle.attention(q, kd, vd, cu, ctx, mode, 3, 0.6)
    np.testing.assert_allclose(out, od, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, ld, rtol=1e-13, atol=1e-13)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        o1, l1 = oracle.attention(q[:, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], cu, ctx, mode, 3, 0.6)
        np.testing.assert_allclose(out[:, h:h + 1], o1, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lse[:, h:h + 1], l1, rtol=1e-13, atol=1e-13)


def test_mixed_batch_equals_each_sequence_alone():
    """Per-sequence mode: the packed mixed batch gives the same rows as each
    sequence run on its own (its own KV rows only)."""
    rng = np.random.default_rng(10)
    seqs = [(0, 7, CAU), (5, 6, BID), (3, 4, CAU), (8, 5, BID)]
    q, k, v, cu, ctx, mode = _batch(rng, seqs, 2, 1, 4)
    for W in (-1, 2):
        out, lse = oracle.attention(q, k, v, cu, ctx, mode, W, 0.5)
        off = 0
        for s, (c, n, md) in enumerate(seqs):
            qs = q[cu[s]:cu[s + 1]]
            ks, vs = k[off:off + c + n], v[off:off + c + n]
            o1, l1 = oracle.attention(qs, ks, vs, [0, n], [c], [md], W, 0.5)
            np.testing.assert_allclose(out[cu[s]:cu[s + 1]], o1, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(lse[cu[s]:cu[s + 1]], l1, rtol=1e-13, atol=1e-13)
            off += c + n


def test_selected_rows_and_heads_match_full_evaluation():
    rng = np.random.default_rng(12)
    seqs = [(30, 70, BID), (0, 65, CAU)]
    q, k, v, cu, ctx, mode = _batch(rng, seqs, 4, 2, 8)
    out, lse = oracle.attention(q, k, v, cu, ctx, mode, 5, 0.3, chunk=16)
    rows = [0, 17, 69, 70, 100, 134]
    o2, l2 = oracle.attention(q, k, v, cu, ctx, mode, 5, 0.3, query_rows=rows, heads=[1, 3])
    for r in rows:
        for h in (1, 3):
            np.testing.assert_allclose(o2[r, h], out[r, h], rtol=1e-13, atol=1e-13)
            assert abs(l2[r, h] - lse[r, h]) < 1e-13
    assert np.isnan(o2[1, 1, 0]) and np.isnan(o2[0, 0, 0])


def test_fp64_tolerance_is_far_below_the_parity_bound():
    """The oracle runs in fp64: rounding differences from reordering the
    reduction (here: chunk sizes) are many orders below the bf16 parity bound."""
    rng = np.random.default_rng(13)
    q, k, v, cu, ctx, mode = _batch(rng, [(300, 200, BID)], 2, 1, 32)
    a, la = oracle.attention(q, k, v, cu, ctx, mode, -1, 0.2, chunk=7)
    b, lb = oracle.attention(q, k, v, cu, ctx, mode, -1, 0.2, chunk=200)
    assert np.abs(a - b).max() < 1e-13 and np.abs(la - lb).max() < 1e-13


def test_rejects_invalid_batches():
    q = np.zeros((4, 2, 2))
    k = np.zeros((6, 1, 2))
    with pytest.raises(ValueError):
        oracle.attention(q, k, k, [0, 3], [2], [1], -1, 1.0)      # cu_q end != total_q
    with pytest.raises(ValueError):
        oracle.attention(q, k, k, [0, 4], [3], [1], -1, 1.0)      # KV too short
    with pytest.raises(ValueError):
        oracle.attention(q, k, k, [0, 4], [2], [2], -1, 1.0)      # bad mode
    with pytest.raises(ValueError):
        oracle.attention(np.zeros((4, 3, 2)), np.zeros((6, 2, 2)), np.zeros((6, 2, 2)),
                         [0, 4], [2], [1], -1, 1.0)               # Hq % Hkv
