"""GB300 (sm_103a) MoE grouped matmul with blockwise FP8 quantization.

The computation lives in the CUDA library ``libgmm_gb300.so`` (C ABI in
``include/gmm.h``); this package holds its Python binding, its build script,
the seeded synthetic workloads and the FP8 tile autotuner (``tune``:
``python -m fp8_blockwise_quantized_gb300.tune`` tunes the production layer).
"""
from .binding import (EXPORTED, GmmError, LIB_PATH, STATUS_NAMES, Workspace, bf16_fwd, dgrad, fp8_fwd,
                      gmm_bf16_dgrad, gmm_selftest_wait_timeout, gmm_fp8_fwd_swiglu_quant, fp8_fwd_swiglu_quant,
                      gmm_bf16_fwd, gmm_fp8_fwd, gmm_fp8_fwd_noalloc, gmm_fp8_fwd_tiled,
                      gmm_fp8_fwd_swiglu_quant_tiled, gmm_get_device_status,
                      gmm_group_metadata, TileConfig,
                      gmm_quantize_lhs, gmm_quantize_rhs, gmm_tiles_offset, gmm_workspace_bytes,
                      group_metadata, load, quantize_lhs, quantize_rhs, tgmm, tgmm_bf16,
                      gmm_quantize_rhs_w4, gmm_fp8_w4_fwd, gmm_fp8_w4_fwd_swiglu_quant, quantize_rhs_w4,
                      fp8_w4_fwd, fp8_w4_fwd_swiglu_quant, tgmm_bf16_tiled, TgmmConfig)

__all__ = ["EXPORTED", "GmmError", "LIB_PATH", "STATUS_NAMES", "Workspace", "bf16_fwd", "dgrad", "fp8_fwd",
           "gmm_bf16_dgrad", "gmm_selftest_wait_timeout", "gmm_fp8_fwd_swiglu_quant", "fp8_fwd_swiglu_quant",
           "gmm_bf16_fwd", "gmm_fp8_fwd", "gmm_fp8_fwd_noalloc", "gmm_fp8_fwd_tiled",
           "gmm_fp8_fwd_swiglu_quant_tiled", "gmm_get_device_status",
           "gmm_group_metadata", "TileConfig",
           "gmm_quantize_lhs", "gmm_quantize_rhs", "gmm_tiles_offset", "gmm_workspace_bytes",
           "group_metadata", "load", "quantize_lhs", "quantize_rhs", "tgmm", "tgmm_bf16",
           "gmm_quantize_rhs_w4", "gmm_fp8_w4_fwd", "gmm_fp8_w4_fwd_swiglu_quant", "quantize_rhs_w4",
           "fp8_w4_fwd", "fp8_w4_fwd_swiglu_quant", "tgmm_bf16_tiled", "TgmmConfig"]
