"""GB300-native (sm_103a) sparse Mixture-of-Experts feed-forward layer.

The computation is the MoE FFN of the "Qwen3.6-35B-A3B -- Architecture Overview" page
(MoE FFN: 256 Experts): an fp32-scored router, softmax, top-K with renormalised weights,
SwiGLU experts over a merged gate_up tensor, and a sigmoid-gated shared expert, summed into
the residual. Every step runs in the hand-written CUDA kernels of ``libmoe_gb300.so``
behind the C ABI of ``include/moe.h``; this package only marshals torch tensors into that
ABI. There is no CPU path: a call fails loudly when the library or a GPU is missing.
"""
from .binding import (  # noqa: F401
    FLAG_BF16_SCORES,
    TEST_SUPPRESS_SCORE,
    TEST_SUPPRESS_STAGE,
    ForwardHostIO,
    MoEError,
    Weights,
    library_path,
    load_library,
    moe_expert_shadow_size,
    moe_forward,
    moe_forward_host_experts,
    moe_forward_host_io,
    moe_last_device_error,
    moe_launch_count,
    moe_set_trace,
    moe_test_set_wait,
    moe_rmsnorm,
    moe_route,
    moe_route_noalloc,
    moe_router_stats,
    moe_workspace_init,
    moe_workspace_size,
    moe_workspace_tap,
    new_workspace,
)
