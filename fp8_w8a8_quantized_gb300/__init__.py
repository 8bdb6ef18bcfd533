"""GB300-native (sm_103a) FP8_DYNAMIC W8A8 linear layer.

The layer runs in a CUDA library with a C ABI (include/fp8w8a8.h): dynamic
per-token E4M3 activation quantization, a tcgen05 FP8 x FP8 GEMM with fp32
accumulation in tensor memory, and a fused per-token x per-channel dequant
epilogue that writes bf16.  This package is its thin Python binding.
"""
from ._binding import (  # noqa: F401
    FP8_OK,
    LIBRARY_PATH,
    Fp8Error,
    QuantizedLinear,
    fp8_device_status,
    fp8_kv_cache_quant,
    fp8_kv_cache_quant_kv,
    fp8_linear,
    fp8_linear_blockwise,
    fp8_linear_blockwise_workspace_size,
    fp8_linear_rmsnorm,
    fp8_linear_workspace_size,
    fp8_quant_per_channel_weights,
    fp8_quant_per_tensor,
    fp8_quant_per_token,
    fp8_quant_per_token_group,
    fp8_quant_weight_blocks,
    fp8_rmsnorm_quant,
    fp8_quant_static,
    fp8_scaled_gemm,
    fp8_scaled_gemm_blockwise,
    fp8_status_string,
    lib,
)
