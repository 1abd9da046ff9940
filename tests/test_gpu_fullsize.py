"""Parity at full layer sizes on sampled tokens.

The oracle recomputes a few sampled tokens one by one (routing, the routed
experts at their bitwidths, the shared FFN, the combine) and the GPU output of
the whole batch is checked at those tokens: the Qwen-shaped layer exactly as
bench.py times it (decode batch of 64 tokens, and 256 tokens where the busiest
experts take the tensor-core GEMM), the Mixtral-shaped layer at decode and
prefill sizes, and the 128-expert layer at prefill size.
"""
import numpy as np
import pytest
import torch

import any_precision_expert_gb300 as pw
from oracle import pw_oracle as O
from synth import bits_plan, get_config, make_expert, make_router, make_tokens

from gpu_layers import assert_close, pool_bytes

pytestmark = pytest.mark.gpu


def _check_sampled(cfg, layer, wr, bias, experts_get, bits, x16, sample, shared=None):
    T = x16.shape[0]
    buf = pw.Buffers(layer, T)
    x = torch.from_numpy(x16).cuda()
    y = pw.moe_forward(layer, x, torch.from_numpy(wr).cuda(),
                       torch.from_numpy(bias).cuda() if bias is not None else None, buf)
    torch.cuda.synchronize()
    assert layer.check_device() == 0
    y = y.float().cpu().numpy()
    gidx = buf.idx[:T].cpu().numpy()
    ref = O.moe_tokens(x16, wr, bias, experts_get, bits, cfg.K, cfg.renormalize, sample, shared=shared)
    if not np.array_equal(gidx[sample], ref["idx"]):
        diff = (gidx[sample] != ref["idx"]).any(1)
        near = O.near_tie_tokens(ref["logits"], cfg.K)
        assert near[diff].all()
        ref = O.moe_tokens(x16, wr, bias, experts_get, bits, cfg.K, cfg.renormalize, sample, shared=shared,
                           idx_override=gidx[sample])
    assert_close(buf.w[:T].cpu().numpy()[sample], ref["w"], tol=1e-5, what="router weights")
    assert_close(y[sample], ref["y"], what="layer output")
    # whole-batch invariants: finite, permutation consistent
    assert np.isfinite(y).all()
    off = buf.offsets.cpu().numpy()
    assert off[-1] == T * cfg.K and (np.diff(off) >= 0).all()


@pytest.mark.parametrize("T", [64, 256])
def test_qwen_layer_as_benchmarked(T):
    import bench
    wl = bench.build_workload(n_copies=1, T=T)
    try:
        cfg = wl["cfg"]
        rng = np.random.default_rng(T)
        sample = sorted(rng.choice(T, size=6, replace=False).tolist())
        _check_sampled(cfg, wl["layers"][0], wl["wr"], wl["bias"], lambda e: wl["experts"][e], wl["bits"],
                       wl["xs"][0], sample, shared=wl["shared"])
    finally:
        for L in wl["layers"]:
            L.destroy()
        wl["pool"].close()


def _full_layer(name, seed=0):
    cfg = get_config(name)
    bits = bits_plan(cfg, seed)
    wr, bias = make_router(cfg, seed)
    pool = pw.Pool(pool_bytes(cfg, bits))
    layer = pw.Layer(pool, cfg.d, cfg.f, cfg.E, cfg.K, cfg.renormalize, cfg.shared_ffn)
    for e in range(cfg.E):
        ex = make_expert(cfg, e, seed)
        layer.load_expert(e, int(bits[e]), ex["code6"], ex["lut"], ex["w16"])
    return cfg, bits, wr, bias, pool, layer


@pytest.mark.parametrize("T", [64, 4096])
def test_mixtral_layer_full_size(T):
    cfg, bits, wr, bias, pool, layer = _full_layer("mixtral")
    try:
        x16 = make_tokens(cfg, T, 0)
        sample = [0, T // 3, T - 1]
        _check_sampled(cfg, layer, wr, bias, lambda e: make_expert(cfg, e, 0), bits, x16, sample)
    finally:
        layer.destroy()
        pool.close()


def test_e128_layer_prefill_full_size():
    cfg, bits, wr, bias, pool, layer = _full_layer("e128")
    try:
        T = 8192
        x16 = make_tokens(cfg, T, 0)
        sample = [1, 4000, 8191]
        _check_sampled(cfg, layer, wr, bias, lambda e: make_expert(cfg, e, 0), bits, x16, sample)
    finally:
        layer.destroy()
        pool.close()
