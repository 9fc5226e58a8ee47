"""The denoiser's query/key/value projection of the adaLN output, fp64.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source: "Nemotron-Labs-TwoTower" wiki, sections "Motivation: one network, two roles"
(the denoiser is conditioned on the timestep through adaptive layer normalisation)
and "Architecture" (the block's queries, and its own keys/values, are the denoiser's
projections of its hidden states; the block attends over the context tower's cache
followed by those keys/values).  So at every step Q, K_blk and V_blk are linear
images of the t-modulated hidden rows.

Readings where the pages are silent:
* one fused projection without bias, W_qkv stored [(Hq + 2 Hkv) D][H]: output column
  c < Hq D is query head c // D, lane c % D; the next Hkv D columns are the keys (kv
  head, lane), the last Hkv D the values - the layout [B][S][heads][D] of q, k_blk,
  v_blk row by row;
* the hidden rows are the adaLN output (bf16), W_qkv is bf16, the product is exact
  here and rounded to bf16 once on the GPU (RNE) when stored.
"""
import numpy as np

from ._bf16 import bf16_to_f64


def qkv_projection(y_bits, W_bits, Hq: int, Hkv: int, D: int):
    """y bf16 bits [B][S][H], W bf16 bits [(Hq + 2 Hkv) D][H] -> fp64 (q [B][S][Hq][D],
    k [B][S][Hkv][D], v [B][S][Hkv][D]), unrounded."""
    y = bf16_to_f64(y_bits)
    W = bf16_to_f64(W_bits)
    B, S, H = y.shape
    assert W.shape == ((Hq + 2 * Hkv) * D, H)
    out = y.reshape(B * S, H) @ W.T
    q = out[:, :Hq * D].reshape(B, S, Hq, D)
    k = out[:, Hq * D:(Hq + Hkv) * D].reshape(B, S, Hkv, D)
    v = out[:, (Hq + Hkv) * D:].reshape(B, S, Hkv, D)
    return q, k, v
