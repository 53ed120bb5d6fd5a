"""GB300 (sm_103a) sparse KV-cache refresh for bidirectional diffusion-LLM layers.

The compute lives in libdllm.so (C ABI, include/dllm.h).  `binding` wraps it for
torch tensors with the same function names; `synth` draws the seeded inputs.
Importing this package loads nothing; the first binding call loads the library
and fails loudly when it has not been built (see `build()`).
"""
from __future__ import annotations

__all__ = ["build", "binding", "synth"]


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile the CUDA library in-tree for sm_103a; returns the .so path."""
    from . import _build
    return _build.build(verbose=verbose, force=force)


def __getattr__(name):
    if name in ("binding", "synth"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
