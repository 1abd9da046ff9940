"""The expert FFN entry point that needs no caller scratch.

pw_expert_ffn_bitplane_noalloc serves callers that cannot allocate device
memory when they run the layer (an engine that has given all of HBM to its
weight pool and KV cache, or a host program that only hands in pre-allocated
inputs and outputs).  It keeps the h activations in a fixed 8 MiB array of the
library instead of a caller workspace; its result must match the workspace
entry point's.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import any_precision_expert_gb300 as pw
from any_precision_expert_gb300 import _lib
from synth import get_config

from gpu_layers import GpuLayer, assert_close

pytestmark = pytest.mark.gpu


def _noalloc(layer, x_perm, offsets, T, y_perm, stream):
    return _lib.lib.pw_expert_ffn_bitplane_noalloc(layer.handle, x_perm.data_ptr(), offsets.data_ptr(), T,
                                                   y_perm.data_ptr(), stream)


def test_noalloc_matches_workspace_entry_point():
    cfg = get_config("tiny")
    gl = GpuLayer(cfg, seed=12)  # every bitwidth 3/4/5/6/16 present
    try:
        layer = gl.layer
        stream = torch.cuda.current_stream().cuda_stream
        for T in (24, 300):  # 300 tokens: the busiest experts take the tensor-core GEMM too
            buf = pw.Buffers(layer, T)
            x = torch.from_numpy(gl.tokens(T)).cuda()
            layer.route_topk(x, gl.wr_d, gl.bias_d, T, buf.idx, buf.w)
            layer.permute(buf.idx, T, x, buf.offsets, buf.perm_src, buf.inv_slot, buf.x_perm, buf.ws)
            layer.expert_ffn_bitplane(buf.x_perm, buf.offsets, T, buf.y_perm, buf.ws)
            torch.cuda.synchronize()
            ref = buf.y_perm[:T * cfg.K].cpu().numpy()
            for _ in range(2):  # the shared array keeps the previous call's data
                y = torch.full((T * cfg.K, cfg.d), float("nan"), dtype=torch.float32, device="cuda")
                assert _noalloc(layer, buf.x_perm, buf.offsets, T, y, stream) == 0
                torch.cuda.synchronize()
                assert_close(y.cpu().numpy(), ref, what="no-alloc expert FFN")
        assert layer.check_device() == 0
    finally:
        gl.close()


def test_noalloc_rejects_batches_beyond_its_scratch():
    cfg = get_config("tiny")
    gl = GpuLayer(cfg, seed=13, with_w16=False)
    try:
        # 8 MiB / (K * ffn * 2 bytes) = 2048 tokens fit; one more does not
        T = (8 << 20) // (cfg.K * cfg.f * 2) + 1
        x_perm = torch.zeros((T * cfg.K, cfg.d), dtype=torch.float16, device="cuda")
        offsets = torch.zeros(cfg.E + 1, dtype=torch.int32, device="cuda")
        y = torch.zeros((T * cfg.K, cfg.d), dtype=torch.float32, device="cuda")
        rc = _noalloc(gl.layer, x_perm, offsets, T, y, torch.cuda.current_stream().cuda_stream)
        assert rc == 3  # PW_ERR_OOM, nothing launched
        assert _noalloc(gl.layer, x_perm, offsets, 0, y, torch.cuda.current_stream().cuda_stream) == 0
    finally:
        gl.close()
