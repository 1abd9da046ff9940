"""Caller-side physical pages for a virtual-memory pool (pw_pool_create_vmm).

The library maps pages but never allocates them: the caller creates one
physical allocation per page with the CUDA driver (cuMemCreate: pinned device
memory, no export handle) and releases them after the pool is closed.  This
module does exactly that through ctypes on the driver library, so Python users
and the tests need nothing beyond the driver.
"""
from __future__ import annotations

import ctypes as C

_CU_MEM_ALLOCATION_TYPE_PINNED = 1
_CU_MEM_LOCATION_TYPE_DEVICE = 1
_CU_MEM_HANDLE_TYPE_NONE = 0


class _Location(C.Structure):
    _fields_ = [("type", C.c_int), ("id", C.c_int)]


class _AllocFlags(C.Structure):
    _fields_ = [("compressionType", C.c_ubyte), ("gpuDirectRDMACapable", C.c_ubyte),
                ("usage", C.c_ushort), ("reserved", C.c_ubyte * 4)]


class _AllocProp(C.Structure):  # CUmemAllocationProp
    _fields_ = [("type", C.c_int), ("requestedHandleTypes", C.c_int), ("location", _Location),
                ("win32HandleMetaData", C.c_void_p), ("allocFlags", _AllocFlags)]


def _driver():
    lib = C.CDLL("libcuda.so.1")
    lib.cuMemCreate.argtypes = [C.POINTER(C.c_ulonglong), C.c_size_t, C.POINTER(_AllocProp), C.c_ulonglong]
    lib.cuMemCreate.restype = C.c_int
    lib.cuMemRelease.argtypes = [C.c_ulonglong]
    lib.cuMemRelease.restype = C.c_int
    return lib


class PhysicalPages:
    """n physical allocations of page_bytes each on `device` (cuMemCreate);
    release() frees them (after every pool that maps them is closed)."""

    def __init__(self, n: int, page_bytes: int = 2 << 20, device: int = 0):
        import torch
        torch.cuda.init()
        torch.zeros(1, device=f"cuda:{device}")  # the device's primary context exists and is current
        self._lib = _driver()
        prop = _AllocProp()
        prop.type = _CU_MEM_ALLOCATION_TYPE_PINNED
        prop.requestedHandleTypes = _CU_MEM_HANDLE_TYPE_NONE
        prop.location.type = _CU_MEM_LOCATION_TYPE_DEVICE
        prop.location.id = device
        self.page_bytes, self.device = page_bytes, device
        self.handles = []
        try:
            for _ in range(n):
                h = C.c_ulonglong(0)
                rc = self._lib.cuMemCreate(C.byref(h), page_bytes, C.byref(prop), 0)
                if rc != 0:
                    raise RuntimeError(f"cuMemCreate failed: CUresult {rc}")
                self.handles.append(h.value)
        except Exception:
            self.release()
            raise

    def release(self):
        for h in self.handles:
            self._lib.cuMemRelease(h)
        self.handles = []
