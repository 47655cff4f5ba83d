"""LongStraw branch replay on GB300: a C-ABI CUDA library and its thin Python binding.

The binding is imported lazily so that the workload generators can be used without a
built library; every compute call goes through the CUDA library and fails loudly when
it is missing.
"""
__version__ = "0.1.0"

_BINDING = ("Prefix", "grpo_loss", "grpo_loss_workspace_bytes", "device_status",
            "LongStrawError", "library_path", "STATUS_NAMES", "timing_enable", "timing_read", "token_logp",
            "KERNEL_NAMES", "attn_merge", "sum_bf16", "bf16_to_f32", "f32_to_bf16")


def __getattr__(name):
    if name in _BINDING:
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)
