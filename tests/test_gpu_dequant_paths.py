"""Bit-exact dequantisation through the FFN kernels' own decode code.

Section 核心洞察 of the PagedWeight write-up fixes every weight the kernels
use: W[r, c] = LUT_b[r][code6[r, c] >> (6 - b)] at b = 3..6 bits (the top b
bit-planes through the page table), or the fp16 page at 16 bits.  The decode
kernel's K loop (cp.async ring, 3-bit byte permutes from register LUTs, 4..6-bit
shared LUT table in both of its configurations, fp16 fragments) and the tcgen05
GEMM's dequant warps (plane loads, per-lane LUT table, the same decode
routines) each dump the A fragments they produce; every value must equal the
oracle's, bit for bit.

The shapes reach every plane-group case of the stored layout: reductions of
320, 704, 1408, 4160 and 14336 columns (full groups of four 64-column chunks
plus ragged final groups of 1, 2 and 3 chunks) and 128-row tiles of the GEMM
that end early (320 and 704 rows).
"""
import numpy as np
import pytest
import torch

from oracle import pw_oracle as O
from synth import get_config

from gpu_layers import GpuLayer

pytestmark = pytest.mark.gpu

SHAPES = [dict(d=320, f=704), dict(d=1408, f=4160), dict(d=512, f=14336)]


@pytest.mark.parametrize("kernel", ["decode_row", "decode_lane", "prefill"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"d{s['d']}_f{s['f']}")
def test_kernel_dequant_bit_exact_every_bitwidth(shape, kernel):
    cfg = get_config("tiny", E=2, **shape)
    gl = GpuLayer(cfg, seed=21, bits=[16, 16], with_w16=True)
    try:
        ex = gl.experts[0]
        for b in (16, 6, 5, 4, 3, 6, 16):  # lower plane by plane, then raise from reclaimable pages
            gl.set_bits(0, b)
            for m in range(3):
                R, C = (cfg.f, cfg.d) if m < 2 else (cfg.d, cfg.f)
                out = torch.full((R, C), float("nan"), dtype=torch.float16, device="cuda")
                gl.layer.debug_dequant_kernel(0, m, kernel, out)
                torch.cuda.synchronize()
                ref = O.dequant(ex["code6"][m], ex["lut"][m], b, ex["w16"][m]).astype(np.float16)
                got = out.cpu().numpy().view(np.uint16)
                bad = got != ref.view(np.uint16)
                assert not bad.any(), (f"{kernel} b={b} m={m}: {int(bad.sum())} of {bad.size} values differ, "
                                       f"first at {np.argwhere(bad)[0].tolist()}")
        assert gl.layer.check_device() == 0
    finally:
        gl.close()
