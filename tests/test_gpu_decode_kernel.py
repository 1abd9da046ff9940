"""The persistent decode kernel behind pw_moe_ffn: it runs the routed experts
(3-bit and fp16 pages) and the shared FFN in one launch, orders down tiles
after their gate/up tiles with device counters, and leaves those counters at
zero for the next launch.

Checks: the combined call gives bit-identical results to the separate routed
and shared calls (every item is computed the same way whoever runs it), down
reductions split over several warps match the oracle at every bitwidth, CUDA
graph replays give the eager result again and again, the decode / tensor-core
threshold can be crossed by the shared FFN, and the layer output stays within
the oracle's tolerance.
"""
import numpy as np
import pytest
import torch

import any_precision_expert_gb300 as pw
from synth import get_config

from gpu_layers import GpuLayer

pytestmark = pytest.mark.gpu


def _separate(gl, x, T):
    buf = pw.Buffers(gl.layer, T)
    L = gl.layer
    L.route_topk(x, gl.wr_d, gl.bias_d, T, buf.idx, buf.w)
    L.permute(buf.idx, T, x, buf.offsets, buf.perm_src, buf.inv_slot, buf.x_perm, buf.ws)
    L.expert_ffn_bitplane(buf.x_perm, buf.offsets, T, buf.y_perm, buf.ws)
    if L.fs:
        L.shared_ffn(x, T, buf.y_shared, buf.ws)
    torch.cuda.synchronize()
    return buf


@pytest.mark.parametrize("T,fs", [(1, 768), (8, 768), (64, 768), (200, 768), (1, 4096), (12, 4096)])
def test_combined_call_equals_separate_calls(T, fs):
    # fs = 4096: the shared FFN's down reduction is split over several warps per tile
    cfg = get_config("qwen", d=512, f=320, E=12, K=4, shared_ffn=fs)
    gl = GpuLayer(cfg, seed=3, bits=[3, 16, 3, 4, 3, 5, 16, 6, 3, 3, 16, 3], with_w16=False)
    try:
        x = torch.from_numpy(gl.tokens(T)).cuda()
        ref = _separate(gl, x, T)
        buf = pw.Buffers(gl.layer, T)
        pw.moe_forward(gl.layer, x, gl.wr_d, gl.bias_d, buf)
        torch.cuda.synchronize()
        assert gl.layer.check_device() == 0
        S = T * cfg.K
        assert torch.equal(buf.offsets, ref.offsets)
        assert torch.equal(buf.y_perm[:S], ref.y_perm[:S])
        assert torch.equal(buf.y_shared[:T], ref.y_shared[:T])
    finally:
        gl.close()


def test_graph_replays_repeat_the_eager_result():
    cfg = get_config("qwen", d=512, f=320, E=12, K=4, shared_ffn=768)
    gl = GpuLayer(cfg, seed=4, bits=[3, 16, 3, 3, 3, 5, 16, 3, 3, 3, 16, 3], with_w16=False)
    try:
        T = 48
        x = torch.from_numpy(gl.tokens(T)).cuda()
        buf = pw.Buffers(gl.layer, T)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            y0 = pw.moe_forward(gl.layer, x, gl.wr_d, gl.bias_d, buf, stream=s).clone()
            for _ in range(3):  # eager repeats
                y1 = pw.moe_forward(gl.layer, x, gl.wr_d, gl.bias_d, buf, stream=s)
                assert torch.equal(y1, y0)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pw.moe_forward(gl.layer, x, gl.wr_d, gl.bias_d, buf, stream=s)
        for _ in range(5):
            buf.y.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(buf.y[:T], y0)
        assert gl.layer.check_device() == 0
    finally:
        gl.close()


# Both decode configurations (three CTAs per SM with row-pair LUT tables; two
# CTAs per SM with per-lane tables at fixed shared-memory addresses) compute
# every item; the host picks one per call, PW_DECODE_NBLK forces it.
NBLK = pytest.mark.parametrize("nblk", ["2", "3"])


@NBLK
def test_layer_output_against_oracle_mixed_bits(nblk, monkeypatch):
    monkeypatch.setenv("PW_DECODE_NBLK", nblk)
    cfg = get_config("qwen", d=512, f=320, E=12, K=4, shared_ffn=768)
    gl = GpuLayer(cfg, seed=5, bits=[3, 16, 3, 4, 3, 5, 16, 6, 3, 3, 16, 3], with_w16=False)
    try:
        for T in (1, 3, 17, 64):
            gl.check_forward(gl.tokens(T))
    finally:
        gl.close()


def test_shared_ffn_across_the_decode_threshold(monkeypatch):
    cfg = get_config("qwen", d=512, f=320, E=8, K=2, shared_ffn=512)
    gl = GpuLayer(cfg, seed=6, bits=[3, 16, 3, 3, 16, 3, 3, 3], with_w16=False)
    try:
        monkeypatch.setenv("PW_DECODE_MAX_TOK", "64")
        monkeypatch.setenv("PW_DECODE_MAX_TOK_SHARED", "64")
        for T in (64, 65):  # shared FFN on the decode kernel, then on the tensor-core GEMM
            gl.check_forward(gl.tokens(T))
    finally:
        gl.close()


def test_many_chunks_per_expert():
    # one expert takes every token (250, above the decode threshold: the
    # tensor-core GEMM with a ragged last M-tile)
    cfg = get_config("tiny", K=1)
    gl = GpuLayer(cfg, seed=7, bits=[3] * 8, with_w16=False)
    try:
        gl.bias = np.array([0, 50, 0, 0, 0, 0, 0, 0], dtype=np.float32)
        gl.bias_d = torch.from_numpy(gl.bias).cuda()
        r = gl.check_forward(gl.tokens(250))
        assert (r["buf"].idx[:250].cpu().numpy() == 1).all()
    finally:
        gl.close()


@NBLK
@pytest.mark.parametrize("f", [4096, 4160])
def test_split_down_reduction_all_bitwidths(f, nblk, monkeypatch):
    # Down reductions of 4096 or more columns for experts with at most 16
    # tokens are shared by two (9..16 tokens) or four (1..8) warps per tile;
    # f = 4160 ends in a ragged plane group.
    monkeypatch.setenv("PW_DECODE_NBLK", nblk)
    cfg = get_config("tiny", d=512, f=f, E=5, K=2)
    gl = GpuLayer(cfg, seed=5, bits=[3, 4, 5, 6, 16])
    try:
        for T in (1, 5, 12, 40):
            gl.check_forward(gl.tokens(T))
    finally:
        gl.close()


@NBLK
def test_odd_shapes_all_bitwidths(nblk, monkeypatch):
    monkeypatch.setenv("PW_DECODE_NBLK", nblk)
    # d = 192 (three 64-column chunks per down tile row block, 12 down tiles)
    # and f = 320 (five chunks: one whole plane group and a ragged one)
    cfg = get_config("qwen", d=192, f=320, E=5, K=2, shared_ffn=320)
    gl = GpuLayer(cfg, seed=9, bits=[3, 4, 5, 6, 16])
    try:
        for T in (1, 7, 40):
            gl.check_forward(gl.tokens(T))
    finally:
        gl.close()



# Experts of 33..64 tokens on the decode kernel (two items of 32 tokens per
# tile pair; the threshold a Mixtral-shaped layer takes when its batch puts
# at most 32 tokens per expert on average); PW_DECODE_MAX_TOK forces it.
def test_experts_above_32_tokens_on_the_decode_kernel_all_bitwidths(monkeypatch):
    monkeypatch.setenv("PW_DECODE_MAX_TOK", "64")
    # d = 192, f = 320: ragged plane groups in both phases; the shared FFN too
    cfg = get_config("qwen", d=192, f=320, E=5, K=2, shared_ffn=320)
    gl = GpuLayer(cfg, seed=11, bits=[3, 4, 5, 6, 16])
    try:
        for T in (33, 40, 64, 130):  # 130: experts above 64 tokens go to the GEMM
            gl.check_forward(gl.tokens(T))
    finally:
        gl.close()
    # f = 4160: 4096+ column down reductions ending in a ragged plane group
    cfg = get_config("tiny", d=512, f=4160, E=5, K=2)
    gl = GpuLayer(cfg, seed=12, bits=[3, 4, 5, 6, 16])
    try:
        for T in (36, 64, 100):
            gl.check_forward(gl.tokens(T))
    finally:
        gl.close()


@NBLK
def test_one_expert_many_items(nblk, monkeypatch):
    # every token on expert 1: 250 tokens in eight items of 32 (the last of
    # 26 tokens), all on the decode kernel
    monkeypatch.setenv("PW_DECODE_NBLK", nblk)
    monkeypatch.setenv("PW_DECODE_MAX_TOK", "256")
    cfg = get_config("tiny", K=1)
    for bits in ([3] * 8, [5] * 8):
        gl = GpuLayer(cfg, seed=13, bits=bits, with_w16=False)
        try:
            gl.bias = np.array([0, 50, 0, 0, 0, 0, 0, 0], dtype=np.float32)
            gl.bias_d = torch.from_numpy(gl.bias).cuda()
            r = gl.check_forward(gl.tokens(250))
            assert (r["buf"].idx[:250].cpu().numpy() == 1).all()
        finally:
            gl.close()
