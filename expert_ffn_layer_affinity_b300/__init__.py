"""DeepSeekMoE layer forward with auxiliary-loss-free load balancing on one
B300 (sm_103a): C-ABI library libmoe_b300.so (include/moe.h) plus a thin
ctypes binding with the same function names."""
from ._lib import (  # noqa: F401
    LIB_PATH, MoEError, lib, moe_abi_version, moe_bias_update, moe_combine,
    moe_grouped_swiglu, moe_grouped_swiglu_tiled, moe_tile_expert_weights, moe_permute, moe_permute_static, moe_router_prepare, moe_router_topk, moe_replica_plan, moe_replica_remap,
    moe_seq_balance_loss, moe_quantize_fp8, moe_quantize_weights_fp8, moe_permute_fp8,
    moe_grouped_swiglu_fp8, moe_grouped_swiglu_save, moe_wait_selftest, moe_router_splits, moe_combine_backward, moe_swiglu_backward, moe_grouped_gemm,
    moe_grouped_gemm_wgrad, moe_grouped_gemm_kn, moe_router_backward,
    moe_combine_dx,
    moe_workspace_bytes, MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE,
    MOE_ERR_CUDA, MOE_ERR_WORKSPACE, MOE_ERR_SCRATCH_LIMIT, MOE_DEV_TIMEOUT, MOE_DEV_NONFINITE, MOE_DEV_BAD_INDEX,
)
from .synth import CONFIGS, LayerConfig  # noqa: F401
