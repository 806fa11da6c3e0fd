"""GB300-native (sm_103a) exact IO-aware attention.

The compute lives in libattn_gb300.so (C ABI in include/attn.h): tcgen05 tensor-core kernels
for fp16/bf16 and CUDA-core kernels for fp32.  This package is the thin PyTorch binding.
"""
from .attention import (bwd, bwd_cross, bwd_varlen, flash_attention, flash_attn_varlen_qkvpacked_func, fwd, fwd_kvcache,
                        fwd_varlen, get_device_status, kvcache_workspace_bytes)
from ._lib import AttnError

__all__ = ["flash_attention", "flash_attn_varlen_qkvpacked_func", "fwd", "bwd", "fwd_varlen", "bwd_varlen",
           "fwd_kvcache", "kvcache_workspace_bytes", "bwd_cross", "get_device_status", "AttnError"]
