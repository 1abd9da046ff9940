"""The virtual-memory page table (pw_pool_create_vmm) on the GPU.

The write-ups read expert weights through a "virtual page table" (second
write-up, section 方法与技术路线); the third page's PagedTensor gives every
expert stable virtual addresses through CUDA virtual memory.  Here the caller
creates the physical pages (cuMemCreate), the library maps each (expert,
plane) block into a fixed virtual range, and the kernels read the planes
through those addresses.  Checks against the fp64 oracle: a forward pass, a
CUDA graph replayed across bitwidth changes (no mapping changes, no data
moved), and an expert whose planes were handed to another layer and then
uploaded again -- into the same virtual addresses.
"""
import pytest
import torch

import any_precision_expert_gb300 as pw
from any_precision_expert_gb300.vmm import PhysicalPages
from synth import get_config

from gpu_layers import GpuLayer, assert_close

pytestmark = pytest.mark.gpu

PAGE = 2 << 20


def _fused(gl, x16, buf):
    x = torch.from_numpy(x16).cuda()
    return pw.moe_forward_fused(gl.layer, x, gl.wr_d, gl.bias_d, buf)


def test_vmm_layer_matches_oracle_across_bitwidth_changes():
    cfg = get_config("tiny")                      # 8 experts, d 512, ffn 1024: one page per plane block
    phys = PhysicalPages(72, PAGE, torch.cuda.current_device())
    pool = pw.Pool.from_vmm_handles(phys.handles, PAGE, torch.cuda.current_device())
    try:
        gl = GpuLayer(cfg, seed=12, with_w16=True, pool=pool)  # loaded at 16 bits, then the planned bits
        try:
            T = 8
            x16 = gl.tokens(T, stream=5)
            gl.check_forward(x16)
            # a CUDA graph of the fused step keeps reading through the same
            # addresses while bitwidths change between replays
            buf = pw.Buffers(gl.layer, T)
            y0 = _fused(gl, x16, buf).clone()
            torch.cuda.synchronize()
            s = torch.cuda.Stream()
            g = torch.cuda.CUDAGraph()
            xd = torch.from_numpy(x16).cuda()
            with torch.cuda.graph(g, stream=s):
                pw.moe_forward_fused(gl.layer, xd, gl.wr_d, gl.bias_d, buf, stream=s)
            maps0 = pool.vmm_counts()
            for e, b in ((0, 3), (1, 16), (2, 4), (0, 6), (3, 5)):
                gl.set_bits(e, b)
                g.replay()
                torch.cuda.synchronize()
                ref = gl.oracle(x16, idx_override=buf.idx[:T].cpu().numpy())
                assert_close(buf.y[:T].float().cpu().numpy(), ref["y"], what=f"graph replay after e{e}->{b}")
            assert pool.vmm_counts() == maps0              # bitwidth changes map and unmap nothing
            assert gl.layer.check_device() == 0
            del y0
        finally:
            gl.close()
        maps, unmaps = pool.vmm_counts()
        assert maps == unmaps
    finally:
        pool.close()
        phys.release()


def _resident_pages(cfg, dev):
    """Pages one layer of this shape keeps resident (tables, LUTs)."""
    phys = PhysicalPages(8, PAGE, dev)
    pool = pw.Pool.from_vmm_handles(phys.handles, PAGE, dev)
    try:
        layer = pw.Layer(pool, cfg.d, cfg.f, cfg.E, cfg.K, cfg.renormalize)
        n = pool.stats()["resident_bytes"] // PAGE
        layer.destroy()
        return n
    finally:
        pool.close()
        phys.release()


def test_vmm_reused_planes_come_back_at_the_same_addresses():
    cfg = get_config("tiny")
    dev = torch.cuda.current_device()
    res = _resident_pages(cfg, dev)
    bits = [6] * cfg.E                              # six one-page plane blocks per expert
    phys = PhysicalPages(res + 6 * cfg.E + 1, PAGE, dev)
    pool = pw.Pool.from_vmm_handles(phys.handles, PAGE, dev)
    try:
        gl = GpuLayer(cfg, seed=15, bits=bits, with_w16=False, pool=pool)
        try:
            assert pool.stats()["free_pages"] == 1
            x16 = gl.tokens(12, stream=7)
            gl.check_forward(x16)
            va = [gl.layer.page_address(5, p, 0) for p in range(6)]
            gl.set_bits(5, 3)                       # planes 3..5: reclaimable (3 pages)
            torch.cuda.synchronize()
            # expert 2 re-loaded at 16 bits needs 8 pages: the free one, its own
            # six, and one of expert 5's reclaimable planes -- the oldest, plane 3
            from synth import make_expert
            ex2 = make_expert(cfg, 2, 15, with_w16=True)
            gl.layer.load_expert(2, 16, ex2["code6"], ex2["lut"], ex2["w16"])
            gl.experts[2], gl.bits[2] = ex2, 16
            assert gl.layer.page_address(5, 3, 0) == 0
            assert gl.layer.try_set_expert_bitwidth(5, 6) == 4   # PW_ERR_NOT_RESIDENT
            gl.check_forward(x16)
            # expert 2 back to 3 bits frees pages; plane 3 of expert 5 is uploaded
            # again from host memory, into its old virtual range
            gl.set_bits(2, 3)
            torch.cuda.synchronize()
            ex5 = gl.experts[5]
            packed = [pw.pack_planes(ex5["code6"][m]) for m in range(3)]
            maps, unmaps = pool.vmm_counts()
            gl.layer.raise_expert_async(5, 6, planes=packed)
            gl.bits[5] = 6
            torch.cuda.synchronize()
            assert [gl.layer.page_address(5, p, 0) for p in range(6)] == va
            assert pool.vmm_counts()[0] == maps + 1      # one page mapped into expert 5's range
            gl.check_forward(x16)
            gl.check_forward(gl.tokens(40, stream=8))
        finally:
            gl.close()
        assert pool.vmm_counts()[0] == pool.vmm_counts()[1]
    finally:
        pool.close()
        phys.release()
