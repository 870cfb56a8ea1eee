"""GB300-native dense bidirectional long-sequence attention for DiT denoising.

The compute path is libditattn.so (hand-written sm_103a CUDA behind a C ABI,
``include/dit_attn.h``); ``binding`` is a thin ctypes layer over it.  Importing
the package does not load the library; the first use of an operation does, and
fails loudly if the library has not been built.
"""
__all__ = ["attn_fwd", "attn_fwd_ws", "attn_fwd_workspace_bytes", "attn_fwd_masked", "attn_fwd_masked_noalloc", "masked_workspace_bytes", "masked_split_workspace_bytes", "attn_fwd_accumulate", "lse_merge", "qkv_to_head_major", "qkv_norm_rope_to_head_major",
           "qkv_cast_fp8", "attn_fwd_fp8", "attn_fwd_fp8_ws",
           "split_stacked_fp8", "check_watchdog", "watchdog_selftest", "DitError", "library_path"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
