"""Thin Python binding over the C ABI in include/pw.h.

Only argument marshalling happens here: torch tensors are turned into device
pointers and streams; every step of the layer runs in libpw.so's kernels.
PyTorch provides device memory (the page pool buffer, activations, scratch)
and streams.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from ._lib import (LUTP, U8P3, U16P3, U32P6, LayerDesc, PoolStats, check, lib)

BITS_ALLOWED = (3, 4, 5, 6, 16)


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _host(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        a = a.astype(dtype)
    return a


def pack_planes(code6: np.ndarray):
    """Library packer: six uint32 plane arrays for a uint8 code matrix [R, C]."""
    code6 = _host(code6, np.uint8)
    R, Cc = code6.shape
    outs = [np.zeros(R * Cc // 32, dtype=np.uint32) for _ in range(6)]
    arr = U32P6(*[o.ctypes.data for o in outs])
    check(lib.pw_pack_planes(code6.ctypes.data, R, Cc, C.byref(arr)), "pw_pack_planes")
    return outs


def pack_f16(w16: np.ndarray) -> np.ndarray:
    w = _host(w16, np.float16)
    R, Cc = w.shape
    out = np.zeros(R * Cc, dtype=np.uint16)
    check(lib.pw_pack_f16(w.ctypes.data, R, Cc, out.ctypes.data), "pw_pack_f16")
    return out


def _host_blocks(planes, w16):
    """C arrays of host pointers (numpy arrays or torch tensors; None allowed)."""
    def hp(a):
        if a is None:
            return None
        return a.data_ptr() if hasattr(a, "data_ptr") else a.ctypes.data
    arr = None
    if planes is not None:
        arr = (U32P6 * 3)(*[U32P6(*[hp(planes[m][q]) for q in range(6)]) for m in range(3)])
    w = U16P3(*[hp(w16[m]) for m in range(3)]) if w16 is not None else None
    return arr, w


LEVELS = (16, 6, 5, 4, 3)  # planner levels, least aggressive first


def plan_bitwidths(sens, sizes, budget: int, mass=None, resid=None, floors=None, ceils=None):
    """Staged greedy bitwidth plan (pw_plan_bitwidths): sens [E][4] damage at
    3..6 bits, sizes [E][5] bytes at 16, 6, 5, 4, 3 bits, budget in bytes;
    mass / resid [E] from Layer.route_stats (None switches a signal off).
    Returns (bits int32 [E], bytes used, feasible)."""
    sens = _host(np.asarray(sens, dtype=np.float64), np.float64)
    E = sens.shape[0]
    sizes = _host(np.asarray(sizes, dtype=np.uint64), np.uint64)
    if sens.shape != (E, 4) or sizes.shape != (E, 5):
        raise ValueError("sens must be [E][4] and sizes [E][5]")

    def opt(a, dtype):
        return None if a is None else _host(np.asarray(a, dtype=dtype).reshape(E), dtype)
    mass, resid = opt(mass, np.float64), opt(resid, np.float64)
    floors, ceils = opt(floors, np.int32), opt(ceils, np.int32)
    bits = np.zeros(E, dtype=np.int32)
    used = C.c_uint64(0)

    def ptr(a):
        return None if a is None else a.ctypes.data
    st = lib.pw_plan_bitwidths(E, ptr(sens), ptr(mass), ptr(resid), ptr(floors), ptr(ceils), ptr(sizes),
                               int(budget), bits.ctypes.data, C.byref(used))
    if st not in (0, 3):  # PW_OK, PW_ERR_OOM (infeasible: the floors)
        check(st, "pw_plan_bitwidths")
    return bits, int(used.value), st == 0


def decode_plan(d: int, ffn: int, n_experts: int, top_k: int, T: int, shared_ffn: int = 0) -> dict:
    """pw_decode_plan: the token thresholds between the decode kernel and the
    tensor-core GEMM for a batch of T tokens, and whether pw_moe_forward
    takes its one-launch fused step (host only)."""
    desc = LayerDesc(d, ffn, n_experts, top_k, 1, shared_ffn)
    r, s, f = C.c_int32(0), C.c_int32(0), C.c_int32(0)
    check(lib.pw_decode_plan(C.byref(desc), int(T), C.byref(r), C.byref(s), C.byref(f)), "pw_decode_plan")
    return {"routed_max": r.value, "shared_max": s.value, "fused": bool(f.value)}


class Pool:
    """Page pool over one device buffer (a torch uint8 tensor)."""

    def __init__(self, nbytes: int, page_bytes: int = 2 << 20, device=None, buffer=None):
        if buffer is None:
            dev = device if device is not None else ("cuda" if torch.cuda.is_available() else "cpu")
            buffer = torch.empty(nbytes + 256, dtype=torch.uint8, device=dev)
        self.buffer = buffer
        base = buffer.data_ptr()
        pad = (-base) % 256
        self.handle = C.c_void_p()
        check(lib.pw_pool_create(base + pad, buffer.numel() - pad, page_bytes, C.byref(self.handle)),
              "pw_pool_create")

    @classmethod
    def from_vmm_handles(cls, handles, page_bytes: int = 2 << 20, device: int = 0):
        """Pool over caller-created physical pages (pw_pool_create_vmm): handles
        are CUmemGenericAllocationHandle values of page_bytes each; the caller
        keeps them alive until close() and releases them afterwards."""
        self = cls.__new__(cls)
        self.buffer = None
        arr = (C.c_ulonglong * len(handles))(*[int(h) for h in handles])
        self.handle = C.c_void_p()
        check(lib.pw_pool_create_vmm(arr, len(handles), page_bytes, device, C.byref(self.handle)),
              "pw_pool_create_vmm")
        return self

    def vmm_counts(self):
        """(pages mapped, pages unmapped) so far by a virtual-memory pool."""
        a, b = C.c_uint64(0), C.c_uint64(0)
        check(lib.pw_testing_vmm_counts(self.handle, C.byref(a), C.byref(b)), "pw_testing_vmm_counts")
        return a.value, b.value

    def stats(self) -> dict:
        s = PoolStats()
        check(lib.pw_pool_get_stats(self.handle, C.byref(s)), "pw_pool_get_stats")
        return {f: getattr(s, f) for f, _ in PoolStats._fields_}

    def close(self):
        if self.handle:
            check(lib.pw_pool_destroy(self.handle), "pw_pool_destroy")
            self.handle = C.c_void_p()


class Layer:
    """One MoE layer: page-table handle plus the hot-path calls."""

    def __init__(self, pool: Pool, d: int, ffn: int, n_experts: int, top_k: int,
                 renormalize: int, shared_ffn: int = 0):
        self.pool = pool
        self.desc = LayerDesc(d, ffn, n_experts, top_k, renormalize, shared_ffn)
        self.handle = C.c_void_p()
        check(lib.pw_layer_create(pool.handle, C.byref(self.desc), C.byref(self.handle)), "pw_layer_create")
        self.d, self.ffn, self.E, self.K = d, ffn, n_experts, top_k
        self.renormalize, self.fs = renormalize, shared_ffn

    # -- setup ---------------------------------------------------------------
    def load_expert(self, e: int, bits: int, code6, luts, w16=None, stream=None):
        """code6: 3 uint8 [R,C]; luts: 3 x [LUT_3..LUT_6] fp16; w16: 3 fp16 [R,C] or None."""
        c = [_host(m, np.uint8) for m in code6]
        lt = [[_host(t, np.float16) for t in row] for row in luts]
        ws = [_host(m, np.float16) for m in w16] if w16 is not None else None
        a_code = U8P3(*[m.ctypes.data for m in c])
        a_lut = LUTP(*[(C.c_void_p * 4)(*[t.ctypes.data for t in row]) for row in lt])
        a_w16 = U16P3(*[m.ctypes.data for m in ws]) if ws is not None else U16P3(None, None, None)
        check(lib.pw_layer_load_expert(self.handle, e, bits, C.byref(a_code), C.byref(a_lut),
                                       C.byref(a_w16), _s(stream)), f"pw_layer_load_expert(e={e})")

    def copy_expert(self, e: int, src: "Layer", e_src: int, bits: int, stream=None):
        """Device-to-device copy of src's expert e_src (at `bits`) into expert e."""
        check(lib.pw_layer_copy_expert(self.handle, e, src.handle, e_src, bits, _s(stream)),
              f"pw_layer_copy_expert(e={e})")

    def load_shared(self, w16, stream=None):
        ws = [_host(m, np.float16) for m in w16]
        arr = U16P3(*[m.ctypes.data for m in ws])
        check(lib.pw_layer_load_shared(self.handle, C.byref(arr), _s(stream)), "pw_layer_load_shared")

    def destroy(self):
        if self.handle:
            check(lib.pw_layer_destroy(self.handle), "pw_layer_destroy")
            self.handle = C.c_void_p()

    # -- precision -------------------------------------------------------------
    def set_expert_bitwidth(self, e: int, bits: int, stream=None):
        check(lib.pw_set_expert_bitwidth(self.handle, e, bits, _s(stream)), "pw_set_expert_bitwidth")

    def raise_expert_async(self, e: int, bits: int, planes=None, w16=None, copy_stream=None, stream=None):
        """Raise expert e to `bits`, uploading missing planes from host memory on
        copy_stream and committing on stream (pw_raise_expert_async).

        planes: 3 lists (gate, up, down) of 6 packed plane arrays (pack_planes
        output; entries may be None for planes still resident); w16: 3 packed
        fp16 pages (pack_f16 output) when raising to 16.  numpy arrays or
        (preferably pinned) torch tensors; the caller keeps them alive until
        `stream` has passed this call.
        """
        arr, w = _host_blocks(planes, w16)
        check(lib.pw_raise_expert_async(self.handle, e, bits, arr, w, _s(copy_stream), _s(stream)),
              f"pw_raise_expert_async(e={e}, bits={bits})")

    def prefetch_expert(self, e: int, bits: int, planes=None, w16=None, copy_stream=None):
        """Upload the blocks expert e needs at `bits` on copy_stream without
        raising it (pw_prefetch_expert); a later set_expert_bitwidth commits."""
        arr, w = _host_blocks(planes, w16)
        check(lib.pw_prefetch_expert(self.handle, e, bits, arr, w, _s(copy_stream)),
              f"pw_prefetch_expert(e={e}, bits={bits})")

    def try_set_expert_bitwidth(self, e: int, bits: int, stream=None) -> int:
        return lib.pw_set_expert_bitwidth(self.handle, e, bits, _s(stream))

    def get_expert_bitwidth(self, e: int) -> int:
        b = C.c_int32(0)
        check(lib.pw_get_expert_bitwidth(self.handle, e, C.byref(b)), "pw_get_expert_bitwidth")
        return b.value

    def expert_resident_bytes(self, bits: int) -> int:
        n = C.c_uint64(0)
        check(lib.pw_expert_resident_bytes(self.handle, bits, C.byref(n)), "pw_expert_resident_bytes")
        return n.value

    def plan_sizes(self):
        """Bytes one expert holds at 16, 6, 5, 4, 3 bits (the planner's size row)."""
        return [self.expert_resident_bytes(b) for b in LEVELS]

    def apply_plan(self, bits, stream=None):
        """Set every expert to its planned bitwidth in stream order (lowering
        unmaps planes; raising re-maps planes still held).  Returns the experts
        whose planes are gone and need pw_raise_expert_async with host data."""
        missing = []
        for e, b in enumerate(np.asarray(bits).tolist()):
            if self.get_expert_bitwidth(e) == b:
                continue
            st = self.try_set_expert_bitwidth(e, int(b), stream)
            if st == 4:  # PW_ERR_NOT_RESIDENT
                missing.append(e)
            else:
                check(st, f"pw_set_expert_bitwidth(e={e}, bits={b})")
        return missing

    def forward_workspace_size(self, T: int) -> int:
        n = C.c_size_t(0)
        check(lib.pw_moe_forward_workspace_size(self.handle, T, C.byref(n)), "pw_moe_forward_workspace_size")
        return n.value

    def workspace_size(self, T: int) -> int:
        n = C.c_size_t(0)
        check(lib.pw_workspace_size(self.handle, T, C.byref(n)), "pw_workspace_size")
        return n.value

    def check_device(self, stream=None) -> int:
        return lib.pw_layer_check_device(self.handle, _s(stream))

    def set_debug_bounds(self, on: bool):
        """Workspace canaries around every scratch region (size workspaces after changing it)."""
        check(lib.pw_layer_set_debug_bounds(self.handle, 1 if on else 0), "pw_layer_set_debug_bounds")

    def debug_check_workspace(self, T: int, ws, stream=None):
        """Check a whole-layer workspace's canaries; the result lands in the device error word."""
        check(lib.pw_debug_check_workspace(self.handle, T, _p(ws), ws.numel() * ws.element_size(), _s(stream)),
              "pw_debug_check_workspace")

    # -- hot path ----------------------------------------------------------------
    def route_topk(self, x, wr, bias, T, idx, w, counts=None, stream=None):
        check(lib.pw_route_topk(self.handle, _p(x), _p(wr), _p(bias), T, _p(idx), _p(w), _p(counts),
                                _s(stream)), "pw_route_topk")

    def route_stats(self, x, idx, w, T, mass, resid, ws, stream=None):
        check(lib.pw_route_stats(self.handle, _p(x), _p(idx), _p(w), T, _p(mass), _p(resid), _p(ws),
                                 ws.numel() * ws.element_size(), _s(stream)), "pw_route_stats")

    def permute(self, idx, T, x, offsets, perm_src, inv_slot, x_perm, ws, stream=None):
        check(lib.pw_permute(self.handle, _p(idx), T, _p(x), _p(offsets), _p(perm_src), _p(inv_slot),
                             _p(x_perm), _p(ws), ws.numel() * ws.element_size(), _s(stream)), "pw_permute")

    def expert_ffn_bitplane(self, x_perm, offsets, T, y_perm, ws, stream=None):
        check(lib.pw_expert_ffn_bitplane(self.handle, _p(x_perm), _p(offsets), T, _p(y_perm), _p(ws),
                                         ws.numel() * ws.element_size(), _s(stream)), "pw_expert_ffn_bitplane")

    def shared_ffn(self, x, T, y_shared, ws, stream=None):
        check(lib.pw_shared_ffn(self.handle, _p(x), T, _p(y_shared), _p(ws), ws.numel() * ws.element_size(),
                                _s(stream)), "pw_shared_ffn")

    def moe_ffn(self, x, x_perm, offsets, T, y_perm, y_shared, ws, stream=None):
        check(lib.pw_moe_ffn(self.handle, _p(x), _p(x_perm), _p(offsets), T, _p(y_perm), _p(y_shared), _p(ws),
                             ws.numel() * ws.element_size(), _s(stream)), "pw_moe_ffn")

    def forward(self, x, wr, bias, T, idx, w, y, ws, stream=None):
        """The whole layer (pw_moe_forward): routing into idx / w, output y."""
        check(lib.pw_moe_forward(self.handle, _p(x), _p(wr), _p(bias), T, _p(idx), _p(w), _p(y), _p(ws),
                                 ws.numel() * ws.element_size(), _s(stream)), "pw_moe_forward")

    def combine(self, y_perm, inv_slot, w, T, y_shared, y, stream=None):
        check(lib.pw_combine(self.handle, _p(y_perm), _p(inv_slot), _p(w), T, _p(y_shared), _p(y), _s(stream)),
              "pw_combine")

    def debug_dequant(self, e: int, m: int, out, stream=None):
        check(lib.pw_debug_dequant(self.handle, e, m, _p(out), _s(stream)), "pw_debug_dequant")

    def debug_dequant_kernel(self, e: int, m: int, kernel: str, out, stream=None):
        """Dump through the decode kernel's ('decode': the layer's configuration; 'decode_row' /
        'decode_lane': a given LUT-table configuration) or the tcgen05 GEMM's ('prefill') own decode path."""
        which = {"decode": 0, "prefill": 1, "decode_row": 2, "decode_lane": 3}[kernel]
        check(lib.pw_debug_dequant_kernel(self.handle, e, m, which, _p(out), _s(stream)), "pw_debug_dequant_kernel")

    def page_address(self, e: int, p: int, vpage: int) -> int:
        a = C.c_uint64(0)
        check(lib.pw_debug_page_address(self.handle, e, p, vpage, C.byref(a)), "pw_debug_page_address")
        return a.value


class Buffers:
    """Device buffers for one layer call at up to T_max tokens (reused every step)."""

    def __init__(self, layer: Layer, T_max: int, device="cuda"):
        d, K, E = layer.d, layer.K, layer.E
        S = T_max * K
        self.T_max = T_max
        self.idx = torch.empty((T_max, K), dtype=torch.int32, device=device)
        self.w = torch.empty((T_max, K), dtype=torch.float32, device=device)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, device=device)
        self.perm_src = torch.empty(S, dtype=torch.int32, device=device)
        self.inv_slot = torch.empty(S, dtype=torch.int32, device=device)
        self.x_perm = torch.empty((S, d), dtype=torch.float16, device=device)
        self.y_perm = torch.empty((S, d), dtype=torch.float32, device=device)
        self.y_shared = (torch.empty((T_max, d), dtype=torch.float32, device=device)
                         if layer.fs else None)
        self.y = torch.empty((T_max, d), dtype=torch.float16, device=device)
        self.ws = torch.empty(max(layer.workspace_size(T_max), 256), dtype=torch.uint8, device=device)
        self._layer, self._device, self._fws = layer, device, None

    @property
    def fws(self):
        """Scratch of the whole-layer call (pw_moe_forward), allocated on first use."""
        if self._fws is None:
            n = max(self._layer.forward_workspace_size(self.T_max), 256)
            self._fws = torch.empty(n, dtype=torch.uint8, device=self._device)
        return self._fws


def moe_forward_fused(layer: Layer, x, wr, bias, buf: Buffers, stream=None):
    """The whole hot path for x [T, d] in one library call (pw_moe_forward); returns buf.y[:T]."""
    T = x.shape[0]
    layer.forward(x, wr, bias, T, buf.idx, buf.w, buf.y, buf.fws, stream)
    return buf.y[:T]


def moe_forward(layer: Layer, x, wr, bias, buf: Buffers, stream=None):
    """The whole hot path for x [T, d] (device fp16); returns buf.y[:T]."""
    T = x.shape[0]
    layer.route_topk(x, wr, bias, T, buf.idx, buf.w, None, stream)
    layer.permute(buf.idx, T, x, buf.offsets, buf.perm_src, buf.inv_slot, buf.x_perm, buf.ws, stream)
    ysh = buf.y_shared if layer.fs else None
    layer.moe_ffn(x, buf.x_perm, buf.offsets, T, buf.y_perm, ysh, buf.ws, stream)
    layer.combine(buf.y_perm, buf.inv_slot, buf.w, T, ysh, buf.y, stream)
    return buf.y[:T]
