"""Confidence unmasking, one denoising step of one sequence, fp64.

Source: "Nemotron-Labs-TwoTower" wiki, section "Block-wise generation" (the paper's
single-block sampler, "confidence unmasking"): every step predicts all masked
positions in parallel; predictions whose confidence clears a threshold gamma are
committed and the rest stay masked; a floor guarantees the block completes within T
steps; the mask token is never emitted and already-decoded positions stay fixed.
The wispaper summary ("Adaptive Step-wise Generation") states the threshold is met
(confidence >= gamma, gamma = 0.8 by default).

Readings where the pages are silent or loose:
* confidence of a position = the largest softmax probability over the vocabulary,
  with the mask id removed from the distribution (its logit treated as -inf: it can
  neither win the argmax nor add to the normaliser);
* the predicted token is the argmax, ties going to the lowest token id;
* committed when confidence >= gamma;
* floor: with m positions still masked and T - steps steps left, at least
  k_min = ceil(m / (T - steps)) positions are committed; when fewer than k_min clear
  gamma, the k_min most confident are committed instead, equal confidences ordered by
  lower position.  With T = S this is "at least the single most confident one";
* positions committed earlier are neither read nor changed; their confidence is
  reported as 0.
"""
import math

import numpy as np


def row_confidence(logits_row, mask_id: int):
    """(token, confidence) for one masked position from its fp32 logits [V]."""
    a = np.asarray(logits_row, dtype=np.float64).copy()
    if 0 <= mask_id < a.size:
        a[mask_id] = -np.inf
    tok = int(np.argmax(a))  # first index of the maximum: the lowest id on ties
    conf = 1.0 / float(np.sum(np.exp(a - a[tok])))
    return tok, conf


def floor_count(m: int, steps: int, T: int) -> int:
    """Fewest commits this step that still lets the block finish within T steps."""
    if m == 0:
        return 0
    left = T - steps
    if left <= 0:
        return m
    return int(math.ceil(m / left))


def unmask_step(logits, ids, steps: int, mask_id: int, gamma: float, T: int,
                commit_step=None) -> dict:
    """One step of one sequence.

    logits: fp32 [S][V] (rows of committed positions are ignored) or a callable
    ``rows(positions) -> [len][V]``; ids int [S]; steps = steps taken so far.

    Returns dict with ids, commit (uint8 [S]), conf (float64 [S]), tok (int [S], -1
    where not masked), n_masked, steps, commit_step (uint8 [S], 1-based step of
    commitment, 0 while masked), k_min.
    """
    ids = np.array(ids, dtype=np.int64)
    S = ids.size
    masked = [i for i in range(S) if ids[i] == mask_id]
    m = len(masked)
    cs = np.zeros(S, np.uint8) if commit_step is None else np.array(commit_step, np.uint8)
    conf = np.zeros(S)
    tok = np.full(S, -1, dtype=np.int64)
    commit = np.zeros(S, np.uint8)
    if m == 0:
        return dict(ids=ids, commit=commit, conf=conf, tok=tok, n_masked=0, steps=steps,
                    commit_step=cs, k_min=0)
    rows = logits(masked) if callable(logits) else np.asarray(logits)[masked]
    for j, i in enumerate(masked):
        tok[i], conf[i] = row_confidence(rows[j], mask_id)
    k_min = floor_count(m, steps, T)
    chosen = [i for i in masked if conf[i] >= gamma]
    if len(chosen) < k_min:
        chosen = sorted(masked, key=lambda i: (-conf[i], i))[:k_min]
    steps += 1
    for i in chosen:
        ids[i] = tok[i]
        commit[i] = 1
        cs[i] = steps
    return dict(ids=ids, commit=commit, conf=conf, tok=tok, n_masked=m - len(chosen),
                steps=steps, commit_step=cs, k_min=k_min)
