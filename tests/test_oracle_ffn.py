"""Pins for the oracle's expert FFN, combine and whole-layer composition (no GPU)."""
import math

import numpy as np

from oracle import pw_oracle as O
from synth import bits_plan, get_config, make_expert, make_router, make_shared, make_tokens


def _brute_ffn(Wg, Wu, Wd, x):
    f, d = Wg.shape
    h = []
    for r in range(f):
        g = math.fsum(float(Wg[r, j]) * float(x[j]) for j in range(d))
        u = math.fsum(float(Wu[r, j]) * float(x[j]) for j in range(d))
        h.append(g / (1.0 + math.exp(-g)) * u)
    return np.array([math.fsum(float(Wd[i, r]) * h[r] for r in range(f)) for i in range(Wd.shape[0])])


def test_silu_values():
    v = np.array([0.0, 30.0, -30.0, 1.0])
    s = O.silu(v)
    assert s[0] == 0.0
    assert abs(s[1] - 30.0) < 1e-9 and abs(s[2]) < 1e-9
    assert abs(s[3] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15


def test_ffn_bruteforce_small():
    cfg = get_config("tiny", d=64, f=64)
    ex = make_expert(cfg, 1, seed=2, with_w16=True)
    x = make_tokens(cfg, 3, seed=2).astype(np.float64)
    for b in (3, 5, 16):
        Wg, Wu, Wd = O.expert_weights(ex, b)
        y = O.swiglu_ffn(Wg, Wu, Wd, x)
        for t in range(3):
            np.testing.assert_allclose(y[t], _brute_ffn(Wg, Wu, Wd, x[t]), rtol=1e-11, atol=1e-14)


def test_ffn_constant_lut_closed_form():
    d, f = 128, 64
    rng = np.random.default_rng(4)
    cg, cu = rng.standard_normal(f) * 0.1, rng.standard_normal(f) * 0.1
    cd = rng.standard_normal(d) * 0.1
    cg, cu, cd = [v.astype(np.float16) for v in (cg, cu, cd)]
    ex = {"code6": [rng.integers(0, 64, (f, d), dtype=np.uint8), rng.integers(0, 64, (f, d), dtype=np.uint8),
                    rng.integers(0, 64, (d, f), dtype=np.uint8)],
          "lut": [[np.tile(c[:, None], (1, 1 << b)) for b in (3, 4, 5, 6)] for c in (cg, cu, cd)],
          "w16": None}
    x = rng.standard_normal((5, d)).astype(np.float16).astype(np.float64)
    sx = x.sum(1)
    for b in (3, 4, 5, 6):
        y = O.swiglu_ffn(*O.expert_weights(ex, b), x)
        g = cg.astype(np.float64)[None, :] * sx[:, None]
        u = cu.astype(np.float64)[None, :] * sx[:, None]
        hsum = (g / (1 + np.exp(-g)) * u).sum(1)
        np.testing.assert_allclose(y, cd.astype(np.float64)[None, :] * hsum[:, None], rtol=1e-10, atol=1e-14)


def _tiny_layer(seed=0, T=16, **kw):
    cfg = get_config("tiny", **kw)
    wr, bias = make_router(cfg, seed)
    experts = [make_expert(cfg, e, seed, with_w16=True) for e in range(cfg.E)]
    bits = bits_plan(cfg, seed)
    x = make_tokens(cfg, T, seed)
    return cfg, wr, bias, experts, bits, x


def test_layer_equals_per_token_sum():
    cfg, wr, bias, experts, bits, x = _tiny_layer(d=128, f=128)
    out = O.moe_layer(x, wr, bias, experts, bits, cfg.K, cfg.renormalize)
    xd = x.astype(np.float64)
    for t in range(x.shape[0]):
        ref = np.zeros(cfg.d)
        for k in range(cfg.K):
            e = int(out["idx"][t, k])
            ref += out["w"][t, k] * O.swiglu_ffn(*O.expert_weights(experts[e], int(bits[e])), xd[t:t + 1])[0]
        np.testing.assert_allclose(out["y"][t], ref, rtol=1e-12, atol=1e-15)
    # sampled-token entry point agrees with the full layer
    sel = [0, 7, 15]
    part = O.moe_tokens(x, wr, bias, lambda e: experts[e], bits, cfg.K, cfg.renormalize, sel)
    np.testing.assert_allclose(part["y"], out["y"][sel], rtol=1e-12, atol=1e-15)


def test_unrouted_expert_bitwidth_does_not_matter():
    cfg, wr, bias, experts, bits, x = _tiny_layer(d=128, f=128, E=8, K=1, T=3)
    out = O.moe_layer(x, wr, bias, experts, bits, cfg.K, cfg.renormalize)
    unused = [e for e in range(cfg.E) if out["offsets"][e + 1] == out["offsets"][e]]
    assert unused
    bits2 = bits.copy()
    for e in unused:
        bits2[e] = 3 if bits[e] != 3 else 6
    out2 = O.moe_layer(x, wr, bias, experts, bits2, cfg.K, cfg.renormalize)
    assert np.array_equal(out["y"], out2["y"])


def test_k1_renorm_is_plain_gather():
    cfg, wr, bias, experts, bits, x = _tiny_layer(d=128, f=128, K=1, T=10)
    out = O.moe_layer(x, wr, bias, experts, bits, 1, 1)
    assert np.allclose(out["w"], 1.0)
    np.testing.assert_array_equal(out["y"], out["y_perm"][out["inv_slot"]])


def test_shared_ffn_added_unweighted():
    cfg = get_config("qwen", d=128, f=64, E=6, K=2, shared_ffn=192)
    wr, bias = make_router(cfg)
    experts = [make_expert(cfg, e, with_w16=True) for e in range(cfg.E)]
    bits = bits_plan(cfg)
    sh = make_shared(cfg)
    x = make_tokens(cfg, 4)
    a = O.moe_layer(x, wr, bias, experts, bits, cfg.K, 0, shared=sh)
    b = O.moe_layer(x, wr, bias, experts, bits, cfg.K, 0)
    xd = x.astype(np.float64)
    for t in range(4):
        ref = _brute_ffn(*[m.astype(np.float64) for m in sh], xd[t])
        np.testing.assert_allclose(a["y"][t] - b["y"][t], ref, rtol=1e-9, atol=1e-12)


def test_greedy_plan_respects_floor_and_budget():
    cfg = get_config("qwen")
    bits = bits_plan(cfg)
    assert bits.min() >= 3
    cost = sum(16 if b == 16 else b for b in bits.tolist())
    assert cost <= 4 * cfg.E + 1e-9
    _, bias = make_router(cfg)
    assert bits[int(np.argmax(bias))] == 16
