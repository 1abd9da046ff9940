"""Helpers for GPU tests: build a device layer from a synthetic config and
compare it with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import any_precision_expert_gb300 as pw
from oracle import pw_oracle as O
from synth import bits_plan, make_expert, make_router, make_shared, make_tokens

TOL = 2e-3  # max |err| <= TOL * (1 + |ref|) for fp32-accumulated outputs


def assert_close(got, ref, tol=TOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = tol * (1.0 + np.abs(ref))
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                           f"max err {err.max():.3e}, worst ratio {(err / bound).max():.3f}")
    return float((err / bound).max()) if err.size else 0.0


def pool_bytes(cfg, bits, page=2 << 20, layers=1, slack=64 << 20):
    d, f, E = int(cfg.d), int(cfg.f), int(cfg.E)
    bits = [int(b) for b in bits]
    plane = 3 * d * f // 8
    pages = 0
    for b in bits:
        np_ = 6 if b == 16 else b
        pages += np_ * (plane // page + 3)
        if b == 16:
            pages += 3 * d * f * 2 // page + 4
    lut = E * (2 * f + d) * 240
    sh = 3 * d * cfg.shared_ffn * 2
    return layers * (pages * page + lut + sh + 2 * page) + slack


class GpuLayer:
    """A synthetic layer uploaded to the GPU plus its host copies for the oracle."""

    def __init__(self, cfg, seed=0, bits=None, with_w16=True, page=2 << 20, pool_extra=0, pool=None):
        self.cfg = cfg
        self.seed = seed
        self.bits = np.array(bits if bits is not None else bits_plan(cfg, seed), dtype=np.int32)
        self.wr, self.bias = make_router(cfg, seed)
        self.experts = [make_expert(cfg, e, seed, with_w16=with_w16 or self.bits[e] == 16)
                        for e in range(cfg.E)]
        self.shared = make_shared(cfg, seed)
        self.own_pool = pool is None
        if pool is None:
            nb = pool_bytes(cfg, [16 if with_w16 else b for b in self.bits], page) + pool_extra
            pool = pw.Pool(nb, page_bytes=page)
        self.pool = pool
        self.layer = pw.Layer(self.pool, cfg.d, cfg.f, cfg.E, cfg.K, cfg.renormalize, cfg.shared_ffn)
        for e, ex in enumerate(self.experts):
            b0 = 16 if (with_w16 and ex["w16"] is not None) else int(self.bits[e])
            self.layer.load_expert(e, b0, ex["code6"], ex["lut"], ex["w16"])
            if b0 != self.bits[e]:
                self.layer.set_expert_bitwidth(e, int(self.bits[e]))
        if self.shared is not None:
            self.layer.load_shared(self.shared)
        self.wr_d = torch.from_numpy(self.wr).cuda()
        self.bias_d = torch.from_numpy(self.bias).cuda() if self.bias is not None else None
        torch.cuda.synchronize()

    def set_bits(self, e, b):
        self.layer.set_expert_bitwidth(e, b)
        self.bits[e] = b

    def tokens(self, T, stream=0):
        return make_tokens(self.cfg, T, self.seed, stream=stream)

    def forward(self, x16, buf=None):
        T = x16.shape[0]
        buf = buf or pw.Buffers(self.layer, max(T, 1))
        x = torch.from_numpy(x16).cuda()
        y = pw.moe_forward(self.layer, x, self.wr_d, self.bias_d, buf)
        torch.cuda.synchronize()
        return y.float().cpu().numpy(), buf

    def oracle(self, x16, idx_override=None):
        return O.moe_layer(x16, self.wr, self.bias, self.experts, self.bits, self.cfg.K,
                           self.cfg.renormalize, shared=self.shared, idx_override=idx_override)

    def check_forward(self, x16, buf=None, tol=TOL):
        """Run the layer, compare routing (near ties allowed) and the output."""
        y, buf = self.forward(x16, buf)
        assert self.layer.check_device() == 0, "device error word set (timeout or bounds check)"
        T = x16.shape[0]
        ref = self.oracle(x16)
        gidx = buf.idx[:T].cpu().numpy()
        diff = (gidx != ref["idx"]).any(axis=1)
        if diff.any():
            near = O.near_tie_tokens(ref["logits"], self.cfg.K)
            assert near[diff].all(), f"routing differs on non-near-tie tokens {np.nonzero(diff & ~near)[0]}"
            ref = self.oracle(x16, idx_override=gidx)
        assert_close(buf.w[:T].cpu().numpy(), ref["w"], tol=1e-5, what="router weights")
        ratio = assert_close(y, ref["y"], tol=tol, what="layer output")
        return {"y": y, "ref": ref, "buf": buf, "ratio": ratio, "near_ties": int(diff.sum())}

    def close(self):
        self.layer.destroy()
        if self.own_pool:
            self.pool.close()
