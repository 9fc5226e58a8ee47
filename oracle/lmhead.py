"""LM head feeding the confidence-unmasking step, fp64.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source: "Nemotron-Labs-TwoTower" wiki, section "Block-wise generation": at every step
the denoiser predicts all masked positions of the block, i.e. its LM head turns the
hidden row of each masked position into logits over the vocabulary, and the
confidence-unmasking step (oracle/unmask.py, oracle/samplers.py) reads those logits.

Readings where the pages are silent:
* the head is a linear map without bias: logit[j] = sum_k h[k] * W[j][k], W stored as
  [V][H] (one row per token id, the layout of a linear layer's weight);
* the hidden rows are bf16 and so is W; the product is taken exactly (fp64);
* only masked positions need logits; the rows of decoded positions are not formed.
"""
import numpy as np

from ._bf16 import bf16_to_f64
from .samplers import sampler_step


def lm_head_logits(h_bits, W_bits) -> np.ndarray:
    """fp64 logits [n][V] of n hidden rows (bf16 bits [n][H]) through W (bf16 bits [V][H])."""
    h = bf16_to_f64(h_bits)
    W = bf16_to_f64(W_bits)
    return h @ W.T


def lm_head_step(h_bits, W_bits, ids, steps: int, mask_id: int, T: int, kind: int = 0,
                 gamma: float = 0.8, temperature: float = 1.0, commit_step=None) -> dict:
    """One sampler step of one sequence whose logits come from the LM head.

    h_bits: bf16 bits [S][H] (rows of decoded positions are not used); the other
    arguments and the result are those of oracle.sampler_step.
    """
    h = np.asarray(h_bits)

    def rows(positions):
        return lm_head_logits(h[list(positions)], W_bits)

    return sampler_step(rows, ids, steps, mask_id, T, kind, gamma, temperature, commit_step)
