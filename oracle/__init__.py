"""CPU oracle for one TwoTower denoise step: plain numpy, fp64 arithmetic.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this package: only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import, call or execute anything under ``oracle/``.  It shares no
code with the CUDA path; its inputs come from the seeded generators in
``block_wise_mask_tt_b300.synth`` (which hold none of the method's arithmetic) or
from the tests themselves.

Sources ("Nemotron-Labs-TwoTower" wiki page unless stated otherwise):
* adaLN time conditioning - sections "Motivation: one network, two roles" and
  "Ablations" (adaptive layer normalization on the diffusion timestep);
* denoise attention - section "Architecture" (block queries attend over the context
  tower's layer-i cache followed by the block's own keys, bidirectional in the block);
* confidence unmasking and the timestep rule - section "Block-wise generation";
* sampler variants (temperature, mock-AR, predict-and-noise) - sections
  "Block-wise generation" and "Release history and artifacts" and the opening summary;
* the outer loop (block append, stopping) - section "Block-wise generation" and the
  MLX README's "Configuration (diffusion)";
* the LM head that feeds the unmask step - section "Block-wise generation";
* the query/key/value projection of the adaLN output - sections "Motivation: one
  network, two roles" and "Architecture".

Every function computes the plain definition: no blocking, no fusion, no reordering
beyond what the definition states.  Readings where the pages are silent are listed
in each module's docstring.
"""
from .adaln import adaln_modulate
from .attention import denoise_attention, denoise_attention_rows, context_kv
from .unmask import row_confidence, unmask_step
from .loop import denoise_block, denoise_block_batch
from .samplers import sampler_step, sampler_block, row_confidence_t
from .outer import append_block, generate
from .lmhead import lm_head_logits, lm_head_step
from .qkv import qkv_projection

__all__ = [
    "adaln_modulate",
    "denoise_attention",
    "denoise_attention_rows",
    "context_kv",
    "row_confidence",
    "unmask_step",
    "denoise_block",
    "denoise_block_batch",
    "sampler_step",
    "sampler_block",
    "row_confidence_t",
    "append_block",
    "generate",
    "lm_head_logits",
    "lm_head_step",
    "qkv_projection",
]
