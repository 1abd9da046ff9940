"""The whole-layer call pw_moe_forward: one fused persistent kernel (router,
permutation, every expert's FFN, the shared FFN, combine) for decode-sized
batches, the separate kernels above the decode thresholds.

Checks: the same routing and output, bit for bit, as the separate calls
(pw_route_topk, pw_permute, pw_moe_ffn, pw_combine) on both sides of the
thresholds, with and without a shared FFN; the layer output against the fp64
oracle; CUDA graph replays repeat the eager result (the kernel's counters
return to zero).
"""
import numpy as np
import pytest
import torch

import any_precision_expert_gb300 as pw
from synth import get_config

from gpu_layers import GpuLayer, assert_close

pytestmark = pytest.mark.gpu


def _both(gl, T):
    x = torch.from_numpy(gl.tokens(T)).cuda()
    a = pw.Buffers(gl.layer, max(T, 1))
    b = pw.Buffers(gl.layer, max(T, 1))
    ya = pw.moe_forward(gl.layer, x, gl.wr_d, gl.bias_d, a).clone()
    yb = pw.moe_forward_fused(gl.layer, x, gl.wr_d, gl.bias_d, b).clone()
    torch.cuda.synchronize()
    assert gl.layer.check_device() == 0
    return a, b, ya, yb


@pytest.mark.parametrize("shape,bits,Ts", [
    (dict(name="qwen", d=512, f=320, E=12, K=4, shared_ffn=768),
     [3, 16, 3, 4, 3, 5, 16, 6, 3, 3, 16, 3], (1, 5, 16, 48, 64, 65, 130)),
    (dict(name="tiny", d=512, f=4096, E=5, K=2), [3, 4, 5, 6, 16], (1, 8, 32, 33, 70)),
    (dict(name="qwen", d=256, f=192, E=9, K=3, shared_ffn=4096), [16, 3, 6, 3, 4, 3, 5, 3, 3], (1, 12, 64)),
    # router sums over three (d = 2816, the last one partial) and four 1024-column slices
    (dict(name="e128", d=2816, f=256, E=128, K=8), [(3, 4, 6, 16)[e % 4] for e in range(128)], (1, 7, 16, 17)),
    (dict(name="mixtral", d=4096, f=512, E=8, K=2), [6, 5, 4, 3, 6, 5, 4, 3], (1, 2, 16)),
])
def test_fused_equals_separate(shape, bits, Ts):
    shape = dict(shape)
    cfg = get_config(shape.pop("name"), **shape)
    gl = GpuLayer(cfg, seed=12, bits=bits, with_w16=False)
    try:
        for T in Ts:
            a, b, ya, yb = _both(gl, T)
            assert torch.equal(a.idx[:T], b.idx[:T]) and torch.equal(a.w[:T], b.w[:T]), T
            assert torch.equal(ya, yb), T
    finally:
        gl.close()


def test_fused_matches_oracle_and_replays():
    cfg = get_config("qwen", E=12, shared_ffn=5632)
    gl = GpuLayer(cfg, seed=13, with_w16=False)
    try:
        for T in (1, 8, 64):
            x16 = gl.tokens(T)
            x = torch.from_numpy(x16).cuda()
            buf = pw.Buffers(gl.layer, T)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                y0 = pw.moe_forward_fused(gl.layer, x, gl.wr_d, gl.bias_d, buf, stream=s).clone()
            s.synchronize()
            ref = gl.oracle(x16, idx_override=buf.idx[:T].cpu().numpy())
            assert_close(y0.float().cpu().numpy(), ref["y"], what=f"fused layer output T={T}")
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                pw.moe_forward_fused(gl.layer, x, gl.wr_d, gl.bias_d, buf, stream=s)
            for _ in range(4):
                buf.y.zero_()
                g.replay()
                torch.cuda.synchronize()
                assert torch.equal(buf.y[:T], y0)
            assert gl.layer.check_device() == 0
    finally:
        gl.close()


def test_fused_empty_batch():
    cfg = get_config("tiny")
    gl = GpuLayer(cfg, seed=14)
    try:
        buf = pw.Buffers(gl.layer, 1)
        x = torch.empty((0, cfg.d), dtype=torch.float16, device="cuda")
        gl.layer.forward(x, gl.wr_d, gl.bias_d, 0, buf.idx, buf.w, buf.y, buf.fws)
        torch.cuda.synchronize()
        assert gl.layer.check_device() == 0
    finally:
        gl.close()
