"""Planner signals on the GPU (pw_route_stats) against the planner oracle, and
re-planning under growing KV-cache pressure applied to a live layer.

PagedWeight (zhichai.net/topic/178446964): section "三层感知" (routing
statistics and the prompt residual from the routing-weighted input norm);
section "安全边界与异步搬运" (floors, staged search); "动态量化优化MoE模型服务",
section 方法与技术路线 (M_w = M_total - M_kv, re-planned when the KV cache
grows).
"""
import numpy as np
import pytest
import torch

import any_precision_expert_gb300 as pw
from oracle import pw_planner as P
from synth import get_config, make_sensitivity

from gpu_layers import GpuLayer

pytestmark = pytest.mark.gpu


def _stats(gl, x16):
    T = x16.shape[0]
    L = gl.layer
    x = torch.from_numpy(x16).cuda()
    buf = pw.Buffers(L, max(T, 1))
    L.route_topk(x, gl.wr_d, gl.bias_d, T, buf.idx, buf.w)
    mass = torch.empty(gl.cfg.E, dtype=torch.float32, device="cuda")
    resid = torch.empty_like(mass)
    ws = torch.empty(max(T, 1), dtype=torch.float32, device="cuda")
    L.route_stats(x, buf.idx, buf.w, T, mass, resid, ws)
    torch.cuda.synchronize()
    return buf.idx[:T].cpu().numpy(), buf.w[:T].cpu().numpy(), mass, resid, (x, buf, ws)


@pytest.mark.parametrize("name,T,kw", [("tiny", 16, {}), ("qwen", 1, dict(E=20)), ("qwen", 200, dict(E=60)),
                                       ("e128", 300, dict(E=128, K=8)), ("tiny", 0, {})])
def test_route_stats_match_oracle(name, T, kw):
    cfg = get_config(name, **kw)
    gl = GpuLayer(cfg, seed=6, bits=[3] * cfg.E, with_w16=False)
    try:
        x16 = gl.tokens(T)
        idx, w, mass, resid, (x, buf, ws) = _stats(gl, x16)
        rm, rr = P.route_stats(x16, idx, w.astype(np.float64), cfg.E)
        m, r = mass.cpu().numpy(), resid.cpu().numpy()
        assert np.allclose(m, rm, rtol=1e-5, atol=1e-6)
        assert np.allclose(r, rr, rtol=1e-4, atol=1e-5)
        if T:
            m2, r2 = torch.empty_like(mass), torch.empty_like(resid)
            gl.layer.route_stats(x, buf.idx, buf.w, T, m2, r2, ws)
            torch.cuda.synchronize()
            assert torch.equal(m2, mass) and torch.equal(r2, resid)  # fixed summation order
    finally:
        gl.close()


def test_replan_under_kv_growth_applies_and_stays_exact():
    cfg = get_config("qwen", d=512, f=320, E=12, K=4, shared_ffn=768)
    gl = GpuLayer(cfg, seed=8, bits=[16] * cfg.E, with_w16=True)
    try:
        E = cfg.E
        x16 = gl.tokens(48)
        _, _, mass, resid, _ = _stats(gl, x16)
        mass, resid = mass.double().cpu().numpy(), resid.double().cpu().numpy()
        sens = make_sensitivity(cfg, seed=8)
        sizes = np.array([gl.layer.plan_sizes()] * E, dtype=np.uint64)
        floors = np.array([3] * E)
        floors[int(np.argmax(mass))] = 5  # the busiest expert never drops below 5 bits
        top = int(sizes[:, 0].sum())
        page = gl.pool.stats()["page_bytes"]
        prev = [16] * E
        # 2 MiB pages: an expert holds 7 pages at 16 bits and b pages at b <= 6;
        # the floors (one expert at 5, the rest at 3) need 38 of the 84 pages
        for frac in (1.0, 0.9, 0.75, 0.6, 0.5, 0.46):  # KV cache takes more of the HBM budget each time
            budget = int(top * frac)
            bits, used, ok = pw.plan_bitwidths(sens, sizes, budget, mass=mass, resid=resid, floors=floors)
            rbits, rused, rok = P.plan_bitwidths(sens.tolist(), mass.tolist(), resid.tolist(), floors.tolist(),
                                                 None, sizes.tolist(), budget)
            assert bits.tolist() == rbits and used == rused and ok == rok
            assert ok and used <= budget
            assert all(b <= a for a, b in zip(prev, bits.tolist()))  # more pressure never raises an expert
            assert gl.layer.apply_plan(bits) == []
            for e, b in enumerate(bits.tolist()):
                gl.bits[e] = b
            torch.cuda.synchronize()
            assert gl.pool.stats()["mapped_pages"] * page == used
            gl.check_forward(x16)
            prev = bits.tolist()
        assert min(prev) == 3 and prev[int(np.argmax(mass))] >= 5
    finally:
        gl.close()
