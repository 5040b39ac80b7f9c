"""Fused exact-attention forward (bf16 and FP8 e4m3) for GB300 (sm_103a).

The compute lives in a C-ABI shared library (``libattn_sm103.so``) of
hand-written CUDA kernels; this package is a thin ctypes binding over it.
"""
__all__ = ["attn_fwd", "attn_fwd_fp8", "attn_fp8_prep", "synth"]


def __getattr__(name):
    if name in ("attn_fwd", "attn_fwd_fp8", "attn_fp8_prep", "attn_fwd_host",
                "fp8_prepare_qkv", "library", "AttnError", "MODE_BLOCK",
                "MODE_BLOCK_HADAMARD", "MODE_PER_TENSOR", "device_status"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
