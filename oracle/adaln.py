"""adaLN modulation, fp64.

Source: "Nemotron-Labs-TwoTower" wiki, "Motivation: one network, two roles" - the
denoiser is conditioned on the diffusion timestep through adaptive layer
normalization in the DiT / PixArt-alpha style; "Ablations" - adaLN time conditioning
adds about 1.5M parameters.  The pages give no formula.  Reading used here: a
LayerNorm with no learned affine and biased variance,

    y = (x - mean(x)) / sqrt(var(x) + eps) * (1 + scale(t)) + shift(t),

over the hidden dimension, where shift(t), scale(t) are the per-timestep modulation
vectors (the timestep MLP and modulation tables themselves need trained weights and
are inputs here).
"""
import numpy as np

from ._bf16 import bf16_to_f64


def adaln_modulate(x_bf16, shift, scale, eps: float = 1e-5) -> np.ndarray:
    """x bf16 bits [..., H]; shift, scale broadcastable to [..., H] (fp32 or fp64).

    Returns float64 [..., H] (unrounded).
    """
    x = bf16_to_f64(x_bf16)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    xhat = (x - mu) / np.sqrt(var + eps)
    return xhat * (1.0 + np.asarray(scale, dtype=np.float64)) + np.asarray(shift, dtype=np.float64)
