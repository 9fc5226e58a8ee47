"""One block denoised to completion (the single-block sampler), fp64.

Source: "Nemotron-Labs-TwoTower" wiki, section "Block-wise generation": a new block
of S positions starts as all [MASK] tokens and is refined over up to T steps; the
timestep fed to the denoiser at each step is the fraction of the block still masked;
each step runs confidence unmasking (``oracle.unmask.unmask_step``).  The MLX port's
README ("Configuration (diffusion)") gives the same knobs: block size 16, 16 steps per
block, mask token id 3.

The denoiser itself needs trained weights, so the per-step logits are supplied by the
caller (a function of the step index and the masked positions).  The timestep of each
step is recorded; it selects the adaLN modulation row n_masked (t = n_masked / S).
"""
import numpy as np

from .unmask import unmask_step


def denoise_block(S: int, T: int, mask_id: int, gamma: float, logits_fn, ids=None,
                  steps: int = 0, commit_step=None) -> dict:
    """logits_fn(step, positions) -> fp32 [len(positions)][V].

    Returns dict(ids, steps, commit_step, n_masked, trace) where trace is a list of
    per-step dicts (t, n_masked_before, committed positions, conf, tok, k_min).
    """
    ids = np.full(S, mask_id, dtype=np.int64) if ids is None else np.array(ids, np.int64)
    cs = np.zeros(S, np.uint8) if commit_step is None else np.array(commit_step, np.uint8)
    trace = []
    while np.any(ids == mask_id) and steps < T:
        m = int(np.sum(ids == mask_id))
        step_index = steps
        r = unmask_step(lambda pos: logits_fn(step_index, pos), ids, steps, mask_id, gamma, T, cs)
        trace.append(dict(t=m / S, n_masked_before=m, committed=np.flatnonzero(r["commit"]),
                          conf=r["conf"], tok=r["tok"], k_min=r["k_min"], ids_before=ids))
        ids, steps, cs = r["ids"], r["steps"], r["commit_step"]
    return dict(ids=ids, steps=steps, commit_step=cs, n_masked=int(np.sum(ids == mask_id)),
                trace=trace)


def denoise_block_batch(B: int, S: int, T: int, mask_id: int, gamma: float, logits_fn_b) -> list:
    """Independent sequences: logits_fn_b(b, step, positions).  Returns one dict per b."""
    return [denoise_block(S, T, mask_id, gamma,
                          lambda step, pos, b=b: logits_fn_b(b, step, pos)) for b in range(B)]
