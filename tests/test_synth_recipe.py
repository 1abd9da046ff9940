"""The synthetic workloads follow their stated recipe (no GPU): shapes, value
ranges and distributions, the per-config bitwidth plans, the Zipf router bias
and the sweep's bitwidth requests, and every draw is reproducible from its seed.
These are the inputs of both the oracle tests and the GPU tests and bench."""
import numpy as np
import pytest

from synth import (CONFIGS, bits_plan, get_config, make_expert, make_router, make_sensitivity, make_shared,
                   make_tokens, zipf_bias)
from synth.workloads import sweep_changes


def test_shapes_of_the_named_layers():
    want = {"tiny": (512, 1024, 8, 2, 0), "qwen": (2048, 1408, 60, 4, 5632), "mixtral": (4096, 14336, 8, 2, 0),
            "e128": (2816, 704, 128, 8, 0), "sweep": (4096, 14336, 8, 2, 0)}
    for name, (d, f, E, K, fs) in want.items():
        c = CONFIGS[name]
        assert (c.d, c.f, c.E, c.K, c.shared_ffn) == (d, f, E, K, fs), name
    assert CONFIGS["sweep"].n_layers == 32
    assert (CONFIGS["qwen"].renormalize, CONFIGS["mixtral"].renormalize, CONFIGS["e128"].renormalize) == (0, 1, 1)


def test_expert_values_follow_the_recipe():
    cfg = get_config("tiny", d=128, f=192)
    ex = make_expert(cfg, 3, seed=5, with_w16=True)
    shapes = [(cfg.f, cfg.d), (cfg.f, cfg.d), (cfg.d, cfg.f)]
    for m in range(3):
        c = ex["code6"][m]
        assert c.shape == shapes[m] and c.dtype == np.uint8 and c.max() <= 63
        assert len(np.unique(c)) == 64  # uniform over 0..63
        for i, b in enumerate((3, 4, 5, 6)):
            lut = ex["lut"][m][i]
            assert lut.shape == (shapes[m][0], 1 << b) and lut.dtype == np.float16
            assert (np.diff(lut.astype(np.float64), axis=1) >= 0).all()  # sorted draws per row
        w = ex["w16"][m].astype(np.float64)
        assert w.shape == shapes[m] and abs(w.std() - 0.02) < 0.002
    luts = np.concatenate([ex["lut"][m][3].astype(np.float64).ravel() for m in range(3)])
    assert abs(luts.std() - 0.02) < 0.002  # N(0, 0.02) quantiles


def test_router_tokens_and_shared_ffn():
    cfg = get_config("qwen", d=256, f=128, shared_ffn=192)
    wr, bias = make_router(cfg, 1)
    assert wr.shape == (cfg.E, cfg.d) and wr.dtype == np.float16
    assert abs(wr.astype(np.float64).std() - 0.02) < 0.002
    x = make_tokens(cfg, 64, 1).astype(np.float64)
    assert x.shape == (64, cfg.d) and abs(x.std() - 1.0) < 0.05
    sh = make_shared(cfg, 1)
    assert [m.shape for m in sh] == [(192, 256), (192, 256), (256, 192)]


def test_zipf_bias_is_minus_s_log_rank():
    cfg = get_config("qwen")
    b = zipf_bias(cfg, 0).astype(np.float64)
    rank = np.rint(np.exp(-b / cfg.zipf_s) - 1.0).astype(int)
    assert sorted(rank.tolist()) == list(range(cfg.E))  # a permutation of the ranks
    np.testing.assert_allclose(b, -cfg.zipf_s * np.log(rank + 1.0), rtol=1e-6, atol=1e-6)
    assert zipf_bias(get_config("tiny"), 0) is None


def test_bitwidth_plans():
    assert bits_plan(CONFIGS["mixtral"]).tolist() == [6, 5, 4, 3, 6, 5, 4, 3]
    e128 = bits_plan(CONFIGS["e128"])
    assert {b: int((e128 == b).sum()) for b in (3, 4, 6, 16)} == {3: 45, 4: 45, 6: 30, 16: 8}
    for l in (0, 1, 7):
        assert bits_plan(CONFIGS["sweep"], layer=l).tolist() == [(6, 5, 4, 3, 16)[(e + l) % 5] for e in range(8)]
    tiny = bits_plan(CONFIGS["tiny"])
    assert set(tiny.tolist()) <= {3, 4, 5, 6, 16}
    qwen = bits_plan(CONFIGS["qwen"])
    assert qwen.min() >= 3 and sum(qwen.tolist()) <= 4 * 60  # greedy under a 4-bit budget with a 3-bit floor


def test_sweep_requests_a_quarter_of_the_pairs_below_their_initial_bits():
    cfg = CONFIGS["sweep"]
    initial = [bits_plan(cfg, layer=l) for l in range(cfg.n_layers)]
    for step in range(5):
        req = sweep_changes(cfg, step, initial)
        assert len(req) == cfg.n_layers * cfg.E // 4
        assert len({(l, e) for l, e, _ in req}) == len(req)
        for l, e, b in req:
            assert b in (3, 4, 5, 6, 16) and b <= initial[l][e]
    assert sweep_changes(cfg, 3, initial) == sweep_changes(cfg, 3, initial)
    assert sweep_changes(cfg, 3, initial) != sweep_changes(cfg, 4, initial)


@pytest.mark.parametrize("fn", [
    lambda s: make_expert(get_config("tiny", d=64, f=64), 2, seed=s, with_w16=True)["code6"][1],
    lambda s: make_router(get_config("qwen", d=64), s)[0],
    lambda s: make_tokens(get_config("tiny"), 4, s),
    lambda s: make_sensitivity(get_config("qwen"), s),
])
def test_draws_are_reproducible_and_seed_dependent(fn):
    a, b, c = fn(0), fn(0), fn(1)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c)
