"""Cached denoising step of a masked diffusion LM on one GB300 (sm_103a).

The compute path is libdllmkv.so (hand-written CUDA kernels behind a C ABI,
declared in include/dllm_kv.h); this package holds its ctypes binding
(``_lib``), the step-loop driver (``loop``) and the build script (``build``).
"""
from . import _lib
from ._lib import (DllmError, dllm_cache_init, dllm_cache_free, dllm_cache_reset, dllm_cache_check,
                   dllm_state_copy, refresh_all, kv_refresh, block_attn, block_attn_rows, attn_out,
                   ffn_gelu, lmhead_conf, stab_update, make_cfg)

__all__ = ["DllmError", "dllm_cache_init", "dllm_cache_free", "dllm_cache_reset", "dllm_cache_check",
           "dllm_state_copy", "refresh_all", "kv_refresh", "block_attn", "block_attn_rows", "attn_out",
           "ffn_gelu", "lmhead_conf", "stab_update", "make_cfg"]
