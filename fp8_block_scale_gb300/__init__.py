"""GB300-native block-scaled FP8 MoE expert library (sm_103a).

The compute path lives in ``libmoe_fp8.so`` (CUDA kernels behind the C ABI of
``include/moe_fp8.h`` and, for E2M1-K32 weights, ``include/moe_w4a8.h``);
``_lib`` is its ctypes binding and ``problem`` assembles device buffers for a
workload using only the library's kernels.  The seeded synthetic inputs come
from the top-level ``workloads`` module, which the CPU oracle imports too.
"""

from ._lib import (  # noqa: F401
    MoeError,
    MoeFwdArgs,
    MoeW4A8Args,
    load,
    make_fwd_args,
    make_w4a8_args,
    moe_forward_workspace_size,
    moe_fp8_block_scale_forward,
    moe_plan,
    moe_plan_capacity,
    moe_plan_workspace_size,
    moe_prep_weights,
    moe_quantize_act_1x128,
    moe_quantize_act_1x128_ue8m0,
    moe_quantize_act_per_row,
    moe_quantize_weight_128x128,
    moe_quantize_weight_k32,
    moe_route_plan,
    moe_route_topk,
    moe_requant_scales_ue8m0,
    moe_status_string,
    moe_w4a8_forward,
    moe_w4a8_workspace_size,
    moe_workspace_init,
)
