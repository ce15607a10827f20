"""KVarN 2-bit KV cache for GB300 (sm_103a): quantise-on-append and decode
attention as hand-written CUDA behind a C ABI (include/kvarn.h).

This package is the thin Python face of that library: ``build`` compiles it
in-tree, and the functions re-exported from ``_abi`` marshal torch tensors to
the C entry points of the same names.
"""
from ._abi import (BF16, FP32, KIND_K, KIND_V, DEVERR_BLOCK_ID, DEVERR_NONFINITE,  # noqa: F401
                   FLAG_NO_CHANNEL_PASS, FLAG_NO_ROTATION, FLAG_NO_TOKEN_PASS, FLAG_TEST_WAIT_TIMEOUT,
                   DEVERR_POSITION, DEVERR_WAIT_TIMEOUT, Config, KVarNError, alloc_pool,
                   alloc_staging, alloc_workspace, append, block_bytes, clear_error, decode_attn, prefill_attn, prefill_workspace_bytes, alloc_prefill_workspace,
                   decode_attn_bf16, decode_attn_noalloc, dequantize, error_decomposition, head_block_bytes, header_symbols, lib, make_config,
                   quantize_block, read_error, staging_bytes, status_string, version,
                   workspace_bytes)
from .build import build  # noqa: F401
