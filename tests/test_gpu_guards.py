"""Failure detection on the GPU without a GPU fault.

* Bounded waits: the decode kernel's down items wait (polling a counter) for
  the gate/up tiles of their token chunk, and the fused step waits for every
  down item before it combines.  A testing hook makes those waits target a
  count nothing reaches, with a short poll limit: the kernel must give up,
  flag the layer's error word (PW_ERR_TIMEOUT), finish, and leave the layer
  usable -- the next call matches the oracle.
* Bad caller tables: slot offsets that are not monotone or leave [0, T*K),
  and combine slot indices out of range, are clamped in the kernels and flag
  the error word (PW_ERR_DEVICE_CHECK); nothing outside the slot rows of
  y_perm or the documented scratch is written.
"""
import numpy as np
import pytest
import torch

import any_precision_expert_gb300 as pw
from any_precision_expert_gb300 import _lib
from synth import get_config

from gpu_layers import GpuLayer

pytestmark = pytest.mark.gpu

PW_ERR_TIMEOUT = 6
PW_ERR_DEVICE_CHECK = 7


@pytest.fixture(scope="module")
def tiny():
    gl = GpuLayer(get_config("tiny"), seed=12)  # experts at 3/4/5/6/16 bits
    yield gl
    gl.close()


@pytest.mark.parametrize("T,fused", [(40, False), (8, True)])
def test_forced_wait_timeout_is_reported_and_recovered(tiny, T, fused):
    L = tiny.layer
    x = tiny.tokens(T, stream=3)
    xd = torch.from_numpy(x).cuda()
    buf = pw.Buffers(L, T)
    assert _lib.lib.pw_testing_wait_limit(L.handle, 1000, 1) == 0  # waits for a count nothing reaches
    try:
        if fused:
            pw.moe_forward_fused(L, xd, tiny.wr_d, tiny.bias_d, buf)
        else:
            pw.moe_forward(L, xd, tiny.wr_d, tiny.bias_d, buf)
        torch.cuda.synchronize()  # the kernel gave up and returned
    finally:
        assert _lib.lib.pw_testing_wait_limit(L.handle, 0, 0) == 0
    assert L.check_device() == PW_ERR_TIMEOUT
    assert L.check_device() == 0  # read and cleared
    tiny.check_forward(x)         # counters were returned to zero: a clean call matches the oracle


def _routed_inputs(gl, T):
    L = gl.layer
    buf = pw.Buffers(L, T)
    x = torch.from_numpy(gl.tokens(T, stream=4)).cuda()
    L.route_topk(x, gl.wr_d, gl.bias_d, T, buf.idx, buf.w)
    L.permute(buf.idx, T, x, buf.offsets, buf.perm_src, buf.inv_slot, buf.x_perm, buf.ws)
    return buf


# T = 16: every bucket on the decode kernel; T = 300: clamped buckets above 32
# slots take the tcgen05 GEMM
BAD_OFFSETS = {16: [-3, 10, 5, 40, 40, 20, 32, 33, 100],
               300: [-7, 50, 40, 200, 900, 650, 600, 601, 10000]}


@pytest.mark.parametrize("T", sorted(BAD_OFFSETS))
def test_bad_offsets_stay_inside_the_slot_rows(tiny, T):
    cfg, L = tiny.cfg, tiny.layer
    S = T * cfg.K
    buf = _routed_inputs(tiny, T)
    off = torch.tensor(BAD_OFFSETS[T], dtype=torch.int32, device="cuda")
    y = torch.full((S + 64, cfg.d), 7.0, dtype=torch.float32, device="cuda")
    need = L.workspace_size(T)
    ws = torch.full((need + 4096,), 0xAB, dtype=torch.uint8, device="cuda")
    L.expert_ffn_bitplane(buf.x_perm, off, T, y, ws)
    torch.cuda.synchronize()
    assert L.check_device() == PW_ERR_DEVICE_CHECK
    assert bool((y[S:] == 7.0).all()), "rows past T*K were written"
    assert bool((ws[need:] == 0xAB).all()), "scratch past the workspace size was written"
    # the no-alloc entry point clamps the same way (its h rows live in the library's array)
    y.fill_(7.0)
    stream = torch.cuda.current_stream().cuda_stream
    if T * cfg.K * cfg.f * 2 <= 8 << 20:
        rc = _lib.lib.pw_expert_ffn_bitplane_noalloc(L.handle, buf.x_perm.data_ptr(), off.data_ptr(), T,
                                                     y.data_ptr(), stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert L.check_device() == PW_ERR_DEVICE_CHECK
        assert bool((y[S:] == 7.0).all())
    # a valid table afterwards: no flag
    L.expert_ffn_bitplane(buf.x_perm, buf.offsets, T, y, ws)
    torch.cuda.synchronize()
    assert L.check_device() == 0


def test_combine_flags_slots_out_of_range(tiny):
    cfg, L = tiny.cfg, tiny.layer
    T = 16
    buf = _routed_inputs(tiny, T)
    L.expert_ffn_bitplane(buf.x_perm, buf.offsets, T, buf.y_perm, buf.ws)
    inv = buf.inv_slot.clone()
    inv[3] = T * cfg.K + 5
    inv[7] = -1
    L.combine(buf.y_perm, inv, buf.w, T, None, buf.y)
    torch.cuda.synchronize()
    assert L.check_device() == PW_ERR_DEVICE_CHECK
    L.combine(buf.y_perm, buf.inv_slot, buf.w, T, None, buf.y)
    torch.cuda.synchronize()
    assert L.check_device() == 0
    assert np.isfinite(buf.y[:T].float().cpu().numpy()).all()


@pytest.mark.parametrize("T", [8, 40])
def test_workspace_canaries(T):
    # debug bounds: canary blocks after every scratch region of the
    # whole-layer call; a clean call leaves them intact (and the output
    # unchanged), a word changed afterwards is reported by the check
    cfg = get_config("qwen", d=512, f=320, E=12, K=4, shared_ffn=768)
    gl = GpuLayer(cfg, seed=8, bits=[3, 16, 3, 4, 3, 5, 16, 6, 3, 3, 16, 3], with_w16=False)
    try:
        x = torch.from_numpy(gl.tokens(T)).cuda()
        buf = pw.Buffers(gl.layer, T)
        y0 = pw.moe_forward_fused(gl.layer, x, gl.wr_d, gl.bias_d, buf).clone()
        gl.layer.set_debug_bounds(True)
        buf = pw.Buffers(gl.layer, T)  # scratch sized with the canaries
        y1 = pw.moe_forward_fused(gl.layer, x, gl.wr_d, gl.bias_d, buf)
        # the split calls (pw_moe_ffn fills and checks its own scratch's canaries)
        y2 = pw.moe_forward(gl.layer, x, gl.wr_d, gl.bias_d, buf).clone()
        torch.cuda.synchronize()
        assert gl.layer.check_device() == 0
        assert torch.equal(y1, y0)
        assert torch.equal(y2, y0)
        ws = buf.fws.view(torch.int32)
        pat = (ws.cpu().numpy().astype(np.int64) & 0xFFFF0000) == 0xC0DE0000
        hits = np.flatnonzero(pat)
        assert hits.size >= 10 * 64  # ten canary blocks of 64 words
        gl.layer.debug_check_workspace(T, buf.fws)
        torch.cuda.synchronize()
        assert gl.layer.check_device() == 0
        ws[int(hits[len(hits) // 2])] = 0  # as a write past a region would
        gl.layer.debug_check_workspace(T, buf.fws)
        torch.cuda.synchronize()
        assert gl.layer.check_device() == 7  # PW_ERR_DEVICE_CHECK
        gl.layer.set_debug_bounds(False)
    finally:
        gl.close()
