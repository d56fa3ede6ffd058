"""Quantized MoE decode step (softmax router, affine 4-bit experts) for GB300.

Python binding of the C ABI declared in include/moe_decode.h. The functions
keep the C names (moe_plan_create, moe_decode_forward, moe_get_routing,
moe_plan_free, ...). Every step of the decode path runs in the CUDA library
libmoe_decode.so, built by build.build(). PyTorch supplies device memory and
streams only.
"""
from ._abi import (  # noqa: F401
    EXPORTED,
    LIB_PATH,
    MOE_ACT_GEGLU,
    MOE_ACT_GEGLU_TANH,
    MOE_ACT_SWIGLU,
    MOE_ACT_SWIGLU_CLAMPED,
    MOE_DTYPE_BF16,
    MOE_DTYPE_F32,
    MOE_ERR_CUDA,
    MOE_ERR_INVALID_ARG,
    MOE_ERR_OOM,
    MOE_ERR_RANGE,
    MOE_ERR_TIMEOUT,
    MOE_ERR_UNSUPPORTED,
    MOE_FLAG_F32_DEBUG,
    MOE_FLAG_GROUPED_COHORTS,
    MOE_FLAG_PHASE_TIMES,
    MOE_FLAG_TEST_STALL,
    MOE_FLAG_TRACE,
    MOE_OK,
    PLANE_FIELDS,
    PHASES,
    MoeError,
    lib,
    make_config,
    make_planes,
    moe_abi_version,
    moe_config,
    moe_decode_forward,
    moe_decode_forward_host,
    moe_decode_forward_layers,
    moe_decode_forward_noalloc,
    moe_expert_planes,
    moe_get_phase_times,
    moe_get_routing,
    moe_layer_io,
    moe_plan_check,
    moe_plan_create,
    moe_plan_free,
    moe_plan_launch_count,
    moe_plan_workspace_bytes,
    moe_status_str,
)
from .layer import DeviceLayer, MoeDecodeLayer  # noqa: F401
