"""Prox sparse SwiGLU FFN decode on B300 (sm_103a).

The compute lives in ``libprox.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/prox.h``).  ``free_swiglu_ffn_prox_b300.prox`` is the
thin Python binding with the same entry-point names (import it explicitly);
``synth`` draws seeded synthetic layers and hidden states.
"""
