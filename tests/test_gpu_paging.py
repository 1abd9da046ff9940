"""Raising precision by an asynchronous plane upload (pw_raise_expert_async):
planes the expert no longer holds are copied from pinned host memory on a copy
stream and the new bitwidth commits in stream order.  A forward enqueued
before the raise computes with the old bitwidth, one enqueued after it with
the new one; both are checked against the oracle."""
import numpy as np
import pytest
import torch

import any_precision_expert_gb300 as pw
from oracle import pw_oracle as O
from synth import get_config

from gpu_layers import GpuLayer, assert_close

pytestmark = pytest.mark.gpu


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def test_async_raise_commits_in_stream_order():
    cfg = get_config("tiny")
    gl = GpuLayer(cfg, seed=12, bits=[3] * 8, with_w16=False)
    try:
        T = 24
        x = gl.tokens(T)
        s = torch.cuda.Stream()
        cs = torch.cuda.Stream()
        xd = torch.from_numpy(x).cuda()
        buf_a, buf_b = pw.Buffers(gl.layer, T), pw.Buffers(gl.layer, T)
        new_bits = [5, 6, 4, 3, 6, 5, 4, 6]
        hold = []
        with torch.cuda.stream(s):
            pw.moe_forward(gl.layer, xd, gl.wr_d, gl.bias_d, buf_a, stream=s)   # before: 3 bits
            for e, b in enumerate(new_bits):
                if b == 3:
                    continue
                planes = [[_pinned(q) for q in pw.pack_planes(gl.experts[e]["code6"][m])] for m in range(3)]
                hold.append(planes)
                gl.layer.raise_expert_async(e, b, planes=planes, copy_stream=cs, stream=s)
            pw.moe_forward(gl.layer, xd, gl.wr_d, gl.bias_d, buf_b, stream=s)   # after: new bits
        torch.cuda.synchronize()
        assert gl.layer.check_device() == 0
        # routing does not depend on bitwidths: both forwards route alike
        idx = buf_a.idx[:T].cpu().numpy()
        assert np.array_equal(idx, buf_b.idx[:T].cpu().numpy())

        def ref_at(bits):
            gl.bits[:] = bits
            ref = gl.oracle(x)
            diff = (idx != ref["idx"]).any(axis=1)
            if diff.any():
                assert O.near_tie_tokens(ref["logits"], cfg.K)[diff].all()
                ref = gl.oracle(x, idx_override=idx)
            return ref

        ref_a = ref_at([3] * 8)
        ref_b = ref_at(new_bits)
        assert_close(buf_a.y[:T].float().cpu().numpy(), ref_a["y"], what="forward before the raise")
        assert_close(buf_b.y[:T].float().cpu().numpy(), ref_b["y"], what="forward after the raise")
        gl.check_forward(x)   # and a fresh forward at the committed bitwidths
        assert [gl.layer.get_expert_bitwidth(e) for e in range(8)] == new_bits
    finally:
        gl.close()


def test_async_raise_to_fp16_page():
    cfg = get_config("tiny")
    gl = GpuLayer(cfg, seed=13, bits=[3] * 8, with_w16=True)   # loads at 16, lowered to 3
    try:
        # push the fp16 pages and planes 3..5 out of the pool's reclaim queue: reload expert 2 at 3 bits
        ex = gl.experts[2]
        gl.layer.load_expert(2, 3, ex["code6"], ex["lut"], None)
        planes = [pw.pack_planes(ex["code6"][m]) for m in range(3)]
        w16 = [pw.pack_f16(m) for m in ex["w16"]]
        gl.layer.raise_expert_async(2, 16, planes=planes, w16=w16)
        torch.cuda.synchronize()
        gl.bits[2] = 16
        gl.check_forward(gl.tokens(16))
    finally:
        gl.close()
