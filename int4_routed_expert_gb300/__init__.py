"""int4 routed-expert MoE layer for one NVIDIA GB300 (sm_103a).

The layer lives in the C-ABI library ``libmoe.so`` (include/moe.h); this
package holds its CUDA sources (``csrc/``), the in-tree build
(``build.py``) and the ctypes binding (``moe.py``).
"""
from .moe import (  # noqa: F401
    EXPORTED,
    ExpertTier,
    SlotCache,
    MOE_BF16,
    MOE_F32,
    MoeError,
    MoELayer,
    Plan,
    load,
    moe_destroy,
    moe_device_status,
    moe_forward,
    moe_last_error,
    moe_layer_create,
    moe_route,
    moe_selftest_bounded_wait,
    moe_selftest_desync,
    moe_route_noalloc,
    moe_trace_enable,
    moe_trace_phase_name,
    moe_trace_read,
    moe_workspace_bytes,
)
