"""B300-native (sm_103a) routed Mixture-of-Experts layer forward pass.

The compute lives in libmoe.so (hand-written CUDA: tcgen05 tensor-core grouped GEMMs fed by
TMA, warp-level router top-k, deterministic permutation and combine). This package is the
thin Python binding of its C ABI (include/moe.h). Torch supplies device memory and streams.
"""
from ._binding import (  # noqa: F401
    Fp8Weights,
    MoeError,
    Nvfp4Weights,
    SIGNATURES,
    get_device_status,
    latent_moe,
    latent_moe_shared,
    latent_moe_workspace_size,
    lib,
    moe_combine,
    moe_forward,
    moe_forward_fp8,
    moe_forward_fp8_workspace_size,
    moe_forward_nvfp4,
    moe_forward_nvfp4_workspace_size,
    moe_forward_shared,
    moe_forward_workspace_size,
    moe_forward_fused_combine_workspace_size,
    moe_grouped_ffn,
    moe_grouped_ffn_fp8,
    moe_grouped_ffn_nvfp4,
    moe_linear,
    moe_permute,
    moe_quantize_fp8_weights,
    moe_quantize_nvfp4_weights,
    moe_route,
    moe_route_dispatch,
    quant_view,
    status_string,
)
