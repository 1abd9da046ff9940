"""GB300 (sm_103a) routed any-precision MoE expert layer.

The CUDA library ``libpw.so`` (C ABI in include/pw.h) does all the work; this
package only loads it and marshals torch tensors into its calls.  Importing
fails if the library has not been built: there is no CPU fallback.
"""
from ._lib import EXPORTED, LIB_PATH, PwError, check, lib  # noqa: F401
from .api import (BITS_ALLOWED, LEVELS, Buffers, Layer, Pool, moe_forward, moe_forward_fused,  # noqa: F401
                  decode_plan, pack_f16, pack_planes, plan_bitwidths)
