"""Layer-streamed NF4 LoRA fine-tuning on one B300 (sm_103a).

The compute path is libls.so (hand-written CUDA kernels behind a C ABI, declared in
include/ls.h and include/ls_kernels.h); this package is its thin Python binding
plus host-side helpers that lay out pinned host buffers.  Importing the package
does not require a GPU; calling a compute entry point without the built library
or without a CUDA device raises.
"""
from ._binding import (LSError, LS_OK, LS_ERR_ARG, LS_ERR_CAP, LS_ERR_CUDA, LS_ERR_TIMEOUT, LS_ERR_STATE,
                       LS_ERR_DEVICE, ls_config, ls_layer_host, ls_nf4_host, ls_profile_t, ls_stats_t, ls_vocab_host, lib, call,
                       check, last_error, header_functions, LIB_PATH, lsk_gemm_plan)
from .runtime import (Stack, make_config, plan_bytes, quantize_host, layer_layout, gemm_plan)

__all__ = ["LSError", "ls_config", "ls_layer_host", "ls_nf4_host", "ls_profile_t", "ls_stats_t", "ls_vocab_host", "lib", "call",
           "check", "last_error", "header_functions", "Stack", "make_config", "plan_bytes", "quantize_host",
           "layer_layout", "LIB_PATH", "LS_OK", "LS_ERR_ARG", "LS_ERR_CAP", "LS_ERR_CUDA", "LS_ERR_TIMEOUT",
           "LS_ERR_STATE", "LS_ERR_DEVICE", "lsk_gemm_plan", "gemm_plan"]
