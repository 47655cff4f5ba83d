"""LongStraw branch replay on GB300: a C-ABI CUDA library and its thin Python binding.

The binding is imported lazily so that the workload generators can be used without a
built library; every compute call goes through the CUDA library and fails loudly when
it is missing.
"""
__version__ = "0.1.0"


def __getattr__(name):
    if name in ("Prefix", "grpo_loss", "lib", "LongStrawError", "library_path"):
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)
