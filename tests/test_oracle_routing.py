"""Pins for the oracle's routing and permutation (no GPU).

Each check is independent of the oracle's own code path: brute force over all
K-subsets with Python floats, closed forms, constructed exact ties and the
permutation rebuilt with plain loops.
"""
import itertools
import math

import numpy as np
import pytest

from oracle import pw_oracle as O
from synth import get_config, make_router, make_tokens


def _brute_route(x16, wr16, bias, K, renorm):
    T, d = x16.shape
    E = wr16.shape[0]
    idx = np.zeros((T, K), dtype=np.int64)
    w = np.zeros((T, K))
    for t in range(T):
        l = []
        for e in range(E):
            acc = math.fsum(float(x16[t, j]) * float(wr16[e, j]) for j in range(d))
            if bias is not None:
                acc += float(bias[e])
            l.append(acc)
        m = max(l)
        z = math.fsum(math.exp(v - m) for v in l)
        p = [math.exp(v - m) / z for v in l]
        best = None
        for comb in itertools.combinations(range(E), K):
            mass = math.fsum(p[e] for e in comb)
            if best is None or mass > best[0] + 1e-15:
                best = (mass, comb)
        chosen = sorted(best[1], key=lambda e: (-p[e], e))
        idx[t] = chosen
        ws = [p[e] for e in chosen]
        if renorm:
            s = math.fsum(ws)
            ws = [v / s for v in ws]
        w[t] = ws
    return idx, w


def test_route_matches_bruteforce_tiny():
    cfg = get_config("tiny", d=64)
    wr, _ = make_router(cfg, seed=3)
    x = make_tokens(cfg, 12, seed=3)
    bias = np.linspace(-0.3, 0.2, cfg.E).astype(np.float32)
    for renorm in (0, 1):
        idx, w, _ = O.route_topk(x, wr, bias, cfg.K, renorm)
        bi, bw = _brute_route(x, wr, bias, cfg.K, renorm)
        assert np.array_equal(idx, bi)
        np.testing.assert_allclose(w, bw, rtol=1e-12, atol=1e-15)


def test_route_K3_bruteforce():
    cfg = get_config("tiny", d=64, E=6, K=3)
    wr, _ = make_router(cfg, seed=5)
    x = make_tokens(cfg, 9, seed=5)
    idx, w, _ = O.route_topk(x, wr, None, 3, 1)
    bi, bw = _brute_route(x, wr, None, 3, 1)
    assert np.array_equal(idx, bi)
    np.testing.assert_allclose(w, bw, rtol=1e-12)


def test_softmax_two_expert_closed_form():
    l = np.array([[0.3, -1.1], [2.0, 2.0], [-5.0, 4.0]])
    p = O.softmax(l)
    p0 = 1.0 / (1.0 + np.exp(l[:, 1] - l[:, 0]))
    np.testing.assert_allclose(p[:, 0], p0, rtol=1e-14)
    np.testing.assert_allclose(p.sum(1), 1.0, rtol=1e-14)


def test_exact_ties_go_to_lower_index():
    E, d, K = 8, 16, 3
    wr = np.tile(np.linspace(-1, 1, d, dtype=np.float16), (E, 1))
    x = np.ones((4, d), dtype=np.float16)
    idx, w, _ = O.route_topk(x, wr, None, K, 0)
    assert np.array_equal(idx, np.tile(np.arange(K), (4, 1)))
    np.testing.assert_allclose(w, 1.0 / E)
    idx, w, _ = O.route_topk(x, wr, None, K, 1)
    np.testing.assert_allclose(w, 1.0 / K)
    # a partial tie at the K boundary: experts 2 and 5 equal, 2 wins
    bias = np.array([5, 4, 1, -3, -3, 1, -9, -9], dtype=np.float32)
    idx, _, _ = O.route_topk(x, wr, bias, 3, 0)
    assert np.array_equal(idx[0], [0, 1, 2])


def test_renormalized_equals_softmax_over_topk_logits():
    cfg = get_config("e128", d=128)
    wr, bias = make_router(cfg, seed=1)
    x = make_tokens(cfg, 20, seed=1)
    idx, w, l = O.route_topk(x, wr, bias, cfg.K, 1)
    sel = np.take_along_axis(l, idx.astype(np.int64), 1)
    ref = np.exp(sel - sel.max(1, keepdims=True))
    ref /= ref.sum(1, keepdims=True)
    np.testing.assert_allclose(w, ref, rtol=1e-12)
    assert (w >= 0).all() and (w <= 1).all()
    # descending order of weights, indices distinct
    assert (np.diff(w, axis=1) <= 1e-15).all()
    for row in idx:
        assert len(set(row.tolist())) == cfg.K


def test_zipf_bias_skews_routing():
    cfg = get_config("qwen", d=256)
    wr, bias = make_router(cfg, seed=0)
    x = make_tokens(cfg, 512, seed=0)
    idx, _, _ = O.route_topk(x, wr, bias, cfg.K, 0)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
    top = np.argmax(bias)
    assert counts[top] == counts.max()
    assert counts[top] > 4 * np.median(counts)


def test_near_tie_detection():
    l = np.array([[1.0, 0.99999, 0.2], [1.0, 0.5, 0.2], [3.0, 2.0, 1.99999]])
    nt = O.near_tie_tokens(l, 1)
    assert nt.tolist() == [True, False, False]
    nt = O.near_tie_tokens(l, 2)
    assert nt.tolist() == [False, False, True]


def _brute_perm(idx, E):
    T, K = idx.shape
    perm_src, inv_slot = [], [0] * (T * K)
    offsets = [0]
    for e in range(E):
        for t in range(T):
            for k in range(K):
                if idx[t, k] == e:
                    inv_slot[t * K + k] = len(perm_src)
                    perm_src.append(t)
        offsets.append(len(perm_src))
    return np.array(offsets), np.array(perm_src), np.array(inv_slot)


@pytest.mark.parametrize("T,E,K", [(1, 8, 2), (16, 8, 2), (37, 60, 4), (50, 128, 8), (9, 4, 4)])
def test_permute_matches_loops(T, E, K):
    rng = np.random.default_rng(T * 1000 + E)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    off, ps, inv = O.permute(idx, E)
    bo, bp, bi = _brute_perm(idx, E)
    assert np.array_equal(off, bo) and np.array_equal(ps, bp) and np.array_equal(inv, bi)
    # invariants
    assert off[-1] == T * K and (np.diff(off) >= 0).all()
    assert sorted(inv.tolist()) == list(range(T * K))
    flat = idx.reshape(-1)
    for e in range(E):
        slots = [s for s in range(T * K) if flat[s] == e]
        assert [inv[s] for s in slots] == list(range(off[e], off[e + 1]))


def test_permute_empty():
    off, ps, inv = O.permute(np.zeros((0, 2), dtype=np.int32), 8)
    assert off.tolist() == [0] * 9 and ps.size == 0 and inv.size == 0
