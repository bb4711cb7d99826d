"""Seeded synthetic inputs for one SwiGLU FFN layer at batch-1 decode.

This module only draws random numbers; it holds none of the method's
arithmetic and is shared by the tests, the benchmark and the CPU oracle's
callers.  No checkpoint or dataset is used: the pages evaluate on trained
models, which stand in here as i.i.d. Gaussian bf16 weights and a
heavy-tailed (Laplace) hidden state with a few outlier dimensions, the shape
of a decoder's residual stream.

Recipe (all draws in fp32, then rounded to bf16 with ties to even):
  * weights, one ``torch.Generator`` seeded with ``seed``, drawn in the order
    W_gate [F][d], W_up [F][d], W_down [d][F], each ``randn * sigma``;
  * x: a second generator seeded with ``x_seed``: ``rand(d)`` -> Laplace(0,1)
    by inverse CDF, then ``randperm(d)``; the first ``n_outlier`` dims of the
    permutation are multiplied by ``outlier_scale``.
Draws on a CUDA generator differ from draws on a CPU generator with the same
seed; every consumer states the device it drew on.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class LayerShape:
    name: str
    d_model: int
    d_ff: int
    sigma: float
    n_outlier: int
    outlier_scale: float = 20.0
    keep_fractions: tuple = (0.5, 0.3, 0.1)
    layers: int = 1


# Llama-shaped FFN layers at batch 1 (d_model, d_ff); outlier dims = 1% of d,
# except the tiny case, which has four.
TINY = LayerShape("tiny_d256_f688", 256, 688, 0.02, 4, keep_fractions=(0.5,))
LLAMA2_7B = LayerShape("llama2_7b_ffn_d4096_f11008", 4096, 11008, 0.02, 41)
LLAMA3_8B = LayerShape("llama3_8b_ffn_d4096_f14336", 4096, 14336, 0.02, 41)
LLAMA3_70B = LayerShape("llama3_70b_ffn_d8192_f28672", 8192, 28672, 0.015, 82)
STACK32 = dataclasses.replace(LLAMA3_8B, name="stack32_llama3_8b_ffn", layers=32,
                              keep_fractions=(0.3,))

SHAPES = {s.name: s for s in (TINY, LLAMA2_7B, LLAMA3_8B, LLAMA3_70B, STACK32)}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def make_weights(d_model: int, d_ff: int, sigma: float, seed: int, device="cpu"):
    """(W_gate [F][d], W_up [F][d], W_down [d][F]) as bf16 on ``device``."""
    g = _gen(seed, device)
    kw = dict(generator=g, device=device, dtype=torch.float32)
    w_gate = (torch.randn(d_ff, d_model, **kw) * sigma).to(torch.bfloat16)
    w_up = (torch.randn(d_ff, d_model, **kw) * sigma).to(torch.bfloat16)
    w_down = (torch.randn(d_model, d_ff, **kw) * sigma).to(torch.bfloat16)
    return w_gate, w_up, w_down


def make_x(d_model: int, n_outlier: int, outlier_scale: float, seed: int, device="cpu"):
    """Hidden state x [d] as bf16: Laplace(0,1) with ``n_outlier`` scaled dims."""
    g = _gen(seed, device)
    u = torch.rand(d_model, generator=g, device=device, dtype=torch.float64) - 0.5
    # inverse CDF of Laplace(0, 1); keep |u| < 1/2 so the log stays finite
    a = u.abs().clamp(max=0.5 - 2.0 ** -40)
    x = -torch.sign(u) * torch.log1p(-2.0 * a)
    perm = torch.randperm(d_model, generator=g, device=device)
    x[perm[:n_outlier]] *= outlier_scale
    return x.to(torch.float32).to(torch.bfloat16)


def layer(shape: LayerShape, seed: int = 0, device="cpu"):
    return make_weights(shape.d_model, shape.d_ff, shape.sigma, seed, device)


def hidden(shape: LayerShape, seed: int = 0, device="cpu"):
    return make_x(shape.d_model, shape.n_outlier, shape.outlier_scale, seed, device)


def bits(t: torch.Tensor):
    """Raw 16-bit patterns of a bf16 tensor as a numpy uint16 array (host)."""
    import numpy as np

    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
