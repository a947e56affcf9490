"""libforge: a GB300-native fused weight-gradient GEMM with AdamW in the epilogue.

``forge_wgrad_adamw`` computes dW = dY^T X with a tcgen05 bf16 GEMM whose fp32
accumulator lives in tensor memory, applies AdamW to each accumulator tile and
writes back only the new weight and moments.  ``forge_wgrad`` and
``forge_adamw`` are the unfused pair.  The CUDA library is loaded on first use
of :mod:`weight_gradient_gemm_gb300.forge`.
"""
__all__ = ["forge", "inputs"]
