"""GB300-native fused causal flash-attention (forward + backward).

The compute path is the C-ABI library ``libxfa.so`` built from ``csrc/`` for
sm_103a; ``binding`` marshals torch tensors into it and ``tape`` exposes the
operator as one node of a small define-by-run autograd tape.  Submodules load
lazily so that ``inputs`` (the seeded generator) can be imported without the
CUDA library.
"""
import importlib

__all__ = ["binding", "tape", "inputs", "build", "flash_attention", "Var"]


def __getattr__(name):
    if name in ("binding", "tape", "inputs", "build"):
        return importlib.import_module(f"{__name__}.{name}")
    if name in ("flash_attention", "Var"):
        return getattr(importlib.import_module(f"{__name__}.tape"), name)
    raise AttributeError(name)
