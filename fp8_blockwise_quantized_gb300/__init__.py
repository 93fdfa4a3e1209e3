"""GB300 (sm_103a) MoE grouped matmul with blockwise FP8 quantization."""
