"""Uno draft+verify hot path on B300 (sm_103a): gated-LoRA projection, block
verifier and draft sampler as hand-written CUDA kernels behind a C ABI
(include/uno.h, libuno.so).  This package is the thin Python binding.

    from lossless_draft_verify_gated_b300 import uno_gated_lora_linear, uno_verify_block
"""
from .binding import (  # noqa: F401
    UNO_BF16, UNO_F32, UNO_OK, UNO_SEQ_BAD_DRAFT, UNO_SEQ_NONFINITE, UNO_SEQ_OK, UnoError, lib,
    status_string, uno_device_error, uno_draft_sample, uno_gated_lora_linear,
    uno_tree_verify, uno_tree_verify_workspace, uno_lm_head_verify, uno_lm_head_verify_workspace,
    uno_gated_lora_linear_batched, uno_gated_lora_linear_batched_workspace,
    uno_gated_lora_linear_workspace, uno_verify_block, uno_verify_block_ex,
    uno_verify_block_workspace, uno_version)

__all__ = ["uno_gated_lora_linear", "uno_gated_lora_linear_workspace", "uno_gated_lora_linear_batched",
           "uno_gated_lora_linear_batched_workspace", "uno_verify_block",
           "uno_verify_block_workspace", "uno_verify_block_ex", "uno_tree_verify", "uno_tree_verify_workspace",
           "uno_lm_head_verify", "uno_lm_head_verify_workspace",
           "uno_draft_sample", "uno_device_error", "uno_version",
           "status_string", "UnoError", "lib"]
