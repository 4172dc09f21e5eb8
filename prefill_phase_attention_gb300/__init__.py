"""GB300 (sm_103a) causal varlen prefill attention with the KV-cache write.

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/prefill_attn.h``); ``binding`` marshals PyTorch tensors into it.
"""
from .binding import (PrefillAttnError, load, prefill_attn_device_status, prefill_attn_last_launch_count,
                      prefill_attn_release, prefill_attn_varlen, prefill_attn_varlen_ex, prefill_attn_varlen_noalloc,
                      prefill_attn_varlen_validate)

__all__ = ["PrefillAttnError", "load", "prefill_attn_varlen", "prefill_attn_varlen_ex", "prefill_attn_varlen_noalloc",
           "prefill_attn_varlen_validate",
           "prefill_attn_device_status", "prefill_attn_release", "prefill_attn_last_launch_count"]
