"""Pins of the paged-KV-cache oracle (``oracle/paged.py``) against facts that
do not come from the oracle itself: a hand-worked example, the contiguous
layout as a special case, invariance under a relabelling of physical pages,
and the append's exact footprint."""

import os

import numpy as np
import pytest

import oracle
import oracle.paged as pg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "paged_example.txt")


def load_golden():
    g = {"table": {}, "seq": {}, "after": {}, "gather": {}}
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if not line:
            continue
        key, vals = line[0], line[1:]
        if key in ("page_size", "num_pages"):
            g[key] = int(vals[0])
        elif key == "table":
            g["table"][int(vals[0])] = [int(x) for x in vals[1:]]
        elif key == "seq":
            g["seq"][int(vals[0])] = (int(vals[1]), [float(x) for x in vals[2:]])
        elif key == "after":
            g["after"][(int(vals[0]), int(vals[1]))] = float(vals[2])
        elif key == "gather":
            g["gather"][int(vals[0])] = [float(x) for x in vals[1:]]
    return g


def test_golden_append_and_gather():
    g = load_golden()
    P, npg = g["page_size"], g["num_pages"]
    cache = np.zeros((npg, P, 1, 1))
    for pgi in range(npg):
        for r in range(P):
            cache[pgi, r, 0, 0] = 10 * pgi + r
    B = len(g["seq"])
    table = np.array([g["table"][s] for s in range(B)], dtype=np.int64)
    ctx = np.array([g["seq"][s][0] for s in range(B)])
    news = [g["seq"][s][1] for s in range(B)]
    cu = np.concatenate([[0], np.cumsum([len(n) for n in news])])
    new = np.array([x for n in news for x in n]).reshape(-1, 1, 1)
    after = pg.append_kv(cache, table, P, cu, ctx, new)
    for (pgi, r), val in g["after"].items():
        assert after[pgi, r, 0, 0] == val, (pgi, r)
    assert len(g["after"]) == npg * P
    for s in range(B):
        L = int(ctx[s]) + len(news[s])
        got = pg.gather_kv(after, table[s], L, P)[:, 0, 0]
        np.testing.assert_array_equal(got, g["gather"][s])
    # the input pool is not modified
    assert cache[1, 1, 0, 0] == 11


def _batch(seed, seqs, Hq, Hkv, D):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum([n for _, n, _ in seqs])])
    ctx = np.array([c for c, _, _ in seqs])
    mode = np.array([m for _, _, m in seqs])
    tq = int(cu[-1])
    q = rng.standard_normal((tq, Hq, D))
    k_new = rng.standard_normal((tq, Hkv, D))
    v_new = rng.standard_normal((tq, Hkv, D))
    return rng, cu, ctx, mode, q, k_new, v_new


def _random_pool(rng, seqs, P, Hkv, D, spare=5):
    """Pages of every sequence at random physical places of a pool with
    ``spare`` junk pages; table entries past a sequence's last page are -1."""
    need = [-(-(c + n) // P) for c, n, _ in seqs]
    npg = sum(need) + spare
    perm = rng.permutation(npg)
    maxp = max(need) + 2
    table = np.full((len(seqs), maxp), -1, dtype=np.int64)
    o = 0
    for s, k in enumerate(need):
        table[s, :k] = perm[o:o + k]
        o += k
    kc = rng.standard_normal((npg, P, Hkv, D))
    vc = rng.standard_normal((npg, P, Hkv, D))
    return table, kc, vc


SEQS = ((5, 7, 1), (0, 9, 0), (11, 4, 1), (3, 1, 0))


@pytest.mark.parametrize("P", [1, 2, 4, 16])
def test_in_order_pages_equal_the_contiguous_layout(P):
    """Pages allocated in order make the pool the packed contiguous buffer of
    the contiguous oracle, so both give the same numbers bit for bit."""
    rng, cu, ctx, mode, q, k_new, v_new = _batch(1, SEQS, 4, 2, 8)
    Ls = [c + n for c, n, _ in SEQS]
    pages = [-(-L // P) for L in Ls]
    table = np.full((len(SEQS), max(pages)), -1, dtype=np.int64)
    first = np.concatenate([[0], np.cumsum(pages)])
    for s in range(len(SEQS)):
        table[s, :pages[s]] = np.arange(first[s], first[s + 1])
    kc = rng.standard_normal((first[-1], P, 2, 8))
    vc = rng.standard_normal((first[-1], P, 2, 8))
    out, lse, ka, va = pg.paged_attention(q, k_new, v_new, kc, vc, table, P, cu, ctx, mode, -1, 0.3)
    # contiguous buffers: each sequence's context rows from its pages, then its new rows
    ks, vs = [], []
    for s, (c, n, _) in enumerate(SEQS):
        flat_k = kc[first[s]:first[s + 1]].reshape(-1, 2, 8)
        flat_v = vc[first[s]:first[s + 1]].reshape(-1, 2, 8)
        ks += [flat_k[:c], k_new[cu[s]:cu[s + 1]]]
        vs += [flat_v[:c], v_new[cu[s]:cu[s + 1]]]
    ref_o, ref_l = oracle.attention(q, np.concatenate(ks), np.concatenate(vs), cu, ctx, mode, -1, 0.3)
    np.testing.assert_array_equal(out, ref_o)
    np.testing.assert_array_equal(lse, ref_l)


def test_relabelling_physical_pages_changes_nothing():
    rng, cu, ctx, mode, q, k_new, v_new = _batch(2, SEQS, 4, 2, 8)
    P = 4
    table, kc, vc = _random_pool(rng, SEQS, P, 2, 8)
    o1, l1, ka1, va1 = pg.paged_attention(q, k_new, v_new, kc, vc, table, P, cu, ctx, mode, 3, 0.25)
    pi = rng.permutation(kc.shape[0])          # physical page p moves to pi[p]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    table2 = np.where(table >= 0, pi[np.maximum(table, 0)], -1)
    o2, l2, ka2, va2 = pg.paged_attention(q, k_new, v_new, kc2, vc2, table2, P, cu, ctx, mode, 3, 0.25)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    np.testing.assert_array_equal(ka2[pi], ka1)
    np.testing.assert_array_equal(va2[pi], va1)


def test_append_writes_exactly_the_query_positions():
    rng, cu, ctx, mode, q, k_new, v_new = _batch(3, SEQS, 4, 2, 8)
    P = 4
    table, kc, vc = _random_pool(rng, SEQS, P, 2, 8)
    ka = pg.append_kv(kc, table, P, cu, ctx, k_new)
    written = np.zeros(kc.shape[:2], dtype=bool)
    for s, (c, n, _) in enumerate(SEQS):
        for t in range(n):
            pos = c + t
            page, row = table[s, pos // P], pos % P
            np.testing.assert_array_equal(ka[page, row], k_new[cu[s] + t])
            written[page, row] = True
    assert written.sum() == cu[-1]
    np.testing.assert_array_equal(ka[~written], kc[~written])


def test_canvas_rewrite_overwrites_the_previous_step():
    """Two denoise steps at the same positions: the second step's result is
    that of attention over the context plus the second canvas only."""
    seqs = ((6, 5, 1),)
    rng, cu, ctx, mode, q, k1, v1 = _batch(4, seqs, 2, 1, 4)
    P = 2
    table, kc, vc = _random_pool(rng, seqs, P, 1, 4)
    _, _, ka, va = pg.paged_attention(q, k1, v1, kc, vc, table, P, cu, ctx, mode, -1, 0.5)
    k2 = rng.standard_normal(k1.shape)
    v2 = rng.standard_normal(v1.shape)
    o2, l2, _, _ = pg.paged_attention(q, k2, v2, ka, va, table, P, cu, ctx, mode, -1, 0.5)
    ctx_k = pg.gather_kv(kc, table[0], 6, P)
    ctx_v = pg.gather_kv(vc, table[0], 6, P)
    ref_o, ref_l = oracle.attention(q, np.concatenate([ctx_k, k2]), np.concatenate([ctx_v, v2]), cu,
                                    ctx, mode, -1, 0.5)
    np.testing.assert_array_equal(o2, ref_o)
    np.testing.assert_array_equal(l2, ref_l)


def test_without_new_rows_the_cache_is_read_as_is():
    rng, cu, ctx, mode, q, k_new, v_new = _batch(5, SEQS, 4, 2, 8)
    P = 4
    table, kc, vc = _random_pool(rng, SEQS, P, 2, 8)
    ka = pg.append_kv(kc, table, P, cu, ctx, k_new)
    va = pg.append_kv(vc, table, P, cu, ctx, v_new)
    o1, l1, _, _ = pg.paged_attention(q, k_new, v_new, kc, vc, table, P, cu, ctx, mode, -1, 0.2)
    o2, l2, kb, vb = pg.paged_attention(q, None, None, ka, va, table, P, cu, ctx, mode, -1, 0.2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    np.testing.assert_array_equal(kb, ka)
