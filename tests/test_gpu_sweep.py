"""Multi-layer decode with bitwidth changes between steps, as in the 32-layer
sweep: layers built by device copies of one uploaded expert set
(pw_layer_copy_expert), a seeded quarter of the (layer, expert) pairs changing
bitwidth each step, one CUDA graph of all layers captured once and replayed
after every change (it reads bitwidths and page tables from device memory).
Every layer's output is checked against the oracle at the bitwidths of that
step."""
import numpy as np
import pytest
import torch

import any_precision_expert_gb300 as pw
from oracle import pw_oracle as O
from synth import get_config, make_expert, make_router, make_tokens
from synth.workloads import sweep_changes

from gpu_layers import assert_close

pytestmark = pytest.mark.gpu


def _init_bits(cfg, l):
    return np.array([(6, 5, 4, 3, 16)[(e + l) % 5] for e in range(cfg.E)], dtype=np.int32)


def _check(cfg, x16, wr, bias, experts, bits, buf, T):
    y = buf.y[:T].float().cpu().numpy()
    gidx = buf.idx[:T].cpu().numpy()
    ref = O.moe_layer(x16, wr, bias, experts, bits, cfg.K, cfg.renormalize)
    diff = (gidx != ref["idx"]).any(1)
    if diff.any():
        assert O.near_tie_tokens(ref["logits"], cfg.K)[diff].all()
        ref = O.moe_layer(x16, wr, bias, experts, bits, cfg.K, cfg.renormalize, idx_override=gidx)
    assert_close(y, ref["y"], what="layer output")


@pytest.mark.parametrize("T", [1, 24])
def test_sweep_steps_with_bitwidth_changes(T):
    cfg = get_config("tiny", n_layers=3)
    n_layers = cfg.n_layers
    init = [_init_bits(cfg, l) for l in range(n_layers)]
    experts = [make_expert(cfg, e, 0, with_w16=True) for e in range(cfg.E)]
    per = 3 * cfg.d * cfg.f
    pool = pw.Pool((n_layers + 1) * cfg.E * (per * 6 // 8 + per * 2) * 2 + (96 << 20), page_bytes=256 << 10)
    src = pw.Layer(pool, cfg.d, cfg.f, cfg.E, cfg.K, cfg.renormalize)
    for e, ex in enumerate(experts):
        src.load_expert(e, 16, ex["code6"], ex["lut"], ex["w16"])
    layers, routers, xs, bufs = [], [], [], []
    try:
        for l in range(n_layers):
            L = pw.Layer(pool, cfg.d, cfg.f, cfg.E, cfg.K, cfg.renormalize)
            for e in range(cfg.E):
                L.copy_expert(e, src, e, int(init[l][e]))
            layers.append(L)
            routers.append(make_router(cfg, 0, layer=l))
            xs.append(make_tokens(cfg, T, 0, layer=l))
            bufs.append(pw.Buffers(L, T))
        wr_d = [torch.from_numpy(w).cuda() for w, _ in routers]
        bias_d = [torch.from_numpy(b).cuda() if b is not None else None for _, b in routers]
        x_d = [torch.from_numpy(x).cuda() for x in xs]
        s = torch.cuda.Stream()

        def forward_all():
            for l in range(n_layers):
                pw.moe_forward(layers[l], x_d[l], wr_d[l], bias_d[l], bufs[l], stream=s)

        with torch.cuda.stream(s):
            forward_all()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            forward_all()
        cur = [b.copy() for b in init]
        for step in range(4):
            for l, e, b in sweep_changes(cfg, step, init):
                layers[l].set_expert_bitwidth(e, b, stream=s)
                cur[l][e] = b
            with torch.cuda.stream(s):
                g.replay()
            s.synchronize()
            for l in range(n_layers):
                assert layers[l].check_device() == 0
                _check(cfg, xs[l], routers[l][0], routers[l][1], experts, cur[l], bufs[l], T)
    finally:
        for L in layers:
            L.destroy()
        src.destroy()
        pool.close()
