"""GB300-native MoE token re-routing (MoeReRoutingV2): rank-major -> expert-major.

The op lives in the CUDA library ``lib/libmrr_v2.so`` (C ABI: include/mrr_v2.h);
``moe_expert_token_gb300.mrr_v2`` is its ctypes binding and ``moe_re_routing`` the torch-level
call.  Build the library with ``python -m moe_expert_token_gb300.build``.
"""
from .mrr_v2 import (  # noqa: F401
    MrrError,
    load_library,
    moe_re_routing,
    moe_re_routing_inverse,
    moe_re_routing_multi,
    moe_re_routing_v1,
    moe_gating_top_k,
    mrr_gating_topk_run,
    mrr_v1_run,
    mrr_status_str,
    mrr_v2_plan,
    mrr_v2_read_status,
    mrr_v2_run,
    mrr_v2_run_multi,
    mrr_v2_run_plan,
    mrr_v2_run_plan_multi,
    mrr_v2_unroute,
    mrr_v2_unroute_plan,
)
