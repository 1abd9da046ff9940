"""ctypes loader for libpw.so: argument types of every exported C function.

There is no fallback: importing this module fails loudly if the library has
not been built (run ``python -m any_precision_expert_gb300.build`` or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpw.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                      "(python -c 'import __graft_entry__ as g; g.build()')")

lib = C.CDLL(LIB_PATH)

vp = C.c_void_p
i32 = C.c_int
sz = C.c_size_t
P_i32 = C.POINTER(C.c_int32)


class LayerDesc(C.Structure):
    _fields_ = [("d", i32), ("ffn", i32), ("n_experts", i32), ("top_k", i32),
                ("renormalize", i32), ("shared_ffn", i32)]


class PoolStats(C.Structure):
    _fields_ = [("total_pages", sz), ("free_pages", sz), ("mapped_pages", sz),
                ("reclaimable_pages", sz), ("resident_bytes", sz), ("page_bytes", sz)]


U8P3 = C.c_void_p * 3          # const uint8_t* const [3]
U16P3 = C.c_void_p * 3         # const uint16_t* const [3]
LUTP = (C.c_void_p * 4) * 3    # const uint16_t* const [3][4]
U32P6 = C.c_void_p * 6

_SIGS = {
    "pw_status_str": (C.c_char_p, [i32]),
    "pw_last_cuda_error": (i32, [P_i32]),
    "pw_pool_create": (i32, [vp, sz, sz, C.POINTER(vp)]),
    "pw_pool_destroy": (i32, [vp]),
    "pw_pool_create_vmm": (i32, [vp, sz, sz, i32, C.POINTER(vp)]),
    "pw_pool_get_stats": (i32, [vp, C.POINTER(PoolStats)]),
    "pw_layer_create": (i32, [vp, C.POINTER(LayerDesc), C.POINTER(vp)]),
    "pw_layer_destroy": (i32, [vp]),
    "pw_layer_load_expert": (i32, [vp, i32, i32, C.POINTER(U8P3), C.POINTER(LUTP), C.POINTER(U16P3), vp]),
    "pw_layer_load_shared": (i32, [vp, C.POINTER(U16P3), vp]),
    "pw_layer_copy_expert": (i32, [vp, i32, vp, i32, i32, vp]),
    "pw_route_topk": (i32, [vp, vp, vp, vp, i32, vp, vp, vp, vp]),
    "pw_permute": (i32, [vp, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
    "pw_expert_ffn_bitplane": (i32, [vp, vp, vp, i32, vp, vp, sz, vp]),
    "pw_expert_ffn_bitplane_noalloc": (i32, [vp, vp, vp, i32, vp, vp]),
    "pw_shared_ffn": (i32, [vp, vp, i32, vp, vp, sz, vp]),
    "pw_moe_ffn": (i32, [vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]),
    "pw_combine": (i32, [vp, vp, vp, vp, i32, vp, vp, vp]),
    "pw_moe_forward": (i32, [vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp]),
    "pw_moe_forward_workspace_size": (i32, [vp, i32, C.POINTER(sz)]),
    "pw_set_expert_bitwidth": (i32, [vp, i32, i32, vp]),
    "pw_raise_expert_async": (i32, [vp, i32, i32, C.POINTER(U32P6 * 3), C.POINTER(U16P3), vp, vp]),
    "pw_prefetch_expert": (i32, [vp, i32, i32, C.POINTER(U32P6 * 3), C.POINTER(U16P3), vp]),
    "pw_get_expert_bitwidth": (i32, [vp, i32, P_i32]),
    "pw_route_stats": (i32, [vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]),
    "pw_expert_resident_bytes": (i32, [vp, i32, C.POINTER(C.c_uint64)]),
    "pw_plan_bitwidths": (i32, [i32, vp, vp, vp, vp, vp, vp, C.c_uint64, vp, C.POINTER(C.c_uint64)]),
    "pw_workspace_size": (i32, [vp, i32, C.POINTER(sz)]),
    "pw_decode_plan": (i32, [C.POINTER(LayerDesc), i32, P_i32, P_i32, P_i32]),
    "pw_layer_check_device": (i32, [vp, vp]),
    "pw_layer_set_debug_bounds": (i32, [vp, i32]),
    "pw_debug_check_workspace": (i32, [vp, i32, vp, C.c_size_t, vp]),
    "pw_pack_planes": (i32, [vp, i32, i32, C.POINTER(U32P6)]),
    "pw_pack_f16": (i32, [vp, i32, i32, vp]),
    "pw_debug_dequant": (i32, [vp, i32, i32, vp, vp]),
    "pw_debug_dequant_kernel": (i32, [vp, i32, i32, i32, vp, vp]),
    "pw_debug_page_address": (i32, [vp, i32, i32, i32, C.POINTER(C.c_uint64)]),
    "pw_testing_host_sim": (i32, [i32]),
    "pw_testing_complete_events": (i32, []),
    "pw_testing_wait_limit": (i32, [vp, C.c_longlong, i32]),
    "pw_testing_vmm_counts": (i32, [vp, C.POINTER(C.c_uint64), C.POINTER(C.c_uint64)]),
}

for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)

STATUS = {0: "PW_OK", 1: "PW_ERR_INVALID_ARG", 2: "PW_ERR_UNSUPPORTED", 3: "PW_ERR_OOM",
          4: "PW_ERR_NOT_RESIDENT", 5: "PW_ERR_CUDA", 6: "PW_ERR_TIMEOUT", 7: "PW_ERR_DEVICE_CHECK"}


class PwError(RuntimeError):
    def __init__(self, status: int, where: str):
        detail = ""
        if status == 5:
            ce = C.c_int32(0)
            lib.pw_last_cuda_error(C.byref(ce))
            detail = f" (cudaError {ce.value})"
        super().__init__(f"{where}: {STATUS.get(status, status)}{detail}")
        self.status = status


def check(status: int, where: str = "pw"):
    if status != 0:
        raise PwError(status, where)
    return status
