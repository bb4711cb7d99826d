"""Prox sparse SwiGLU FFN decode on B300 (sm_103a).

The compute lives in ``libprox.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/prox.h``).  ``free_swiglu_ffn_prox_b300.prox`` is the
thin Python binding with the same entry-point names; ``synth`` draws seeded
synthetic layers and hidden states.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "prox"]


def __getattr__(name):
    if name == "prox":
        from . import prox as _prox

        return _prox
    raise AttributeError(name)
