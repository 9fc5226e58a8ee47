"""Sampler variants of one denoising step (one sequence), fp64.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Sources ("Nemotron-Labs-TwoTower" wiki page):
* "Block-wise generation": the main sampler is confidence unmasking (oracle/unmask.py);
  the paper also names the standard predict-and-noise sampler of the block-diffusion
  literature, which predicts a clean block and re-masks the low-confidence positions
  according to the noise schedule;
* the model-card example in "Release history and artifacts" passes a sampling
  temperature;
* the opening summary describes a "mock-AR" two-tower mode that predicts one token per
  step.

Readings where the pages are silent:
* temperature tau > 0 divides the logits before the softmax: the confidence of a
  masked position is max_j softmax(l / tau)_j with the mask id removed; the predicted
  token (the argmax, lowest id on ties) does not depend on tau;
* mock-AR commits exactly one position per step, the leftmost still-masked one (the
  order an autoregressive decoder would take);
* predict-and-noise follows the linear schedule of masked diffusion: after the step
  taken with `steps` steps already done, floor(S * (T - steps - 1) / T) positions stay
  masked (0 at the last step); the positions committed are the most confident ones
  (equal confidences by lower position), at least one per step while any is masked;
* in every mode the mask token is never emitted and decoded positions stay fixed.
"""
import math

import numpy as np

CONFIDENCE, MOCK_AR, PREDICT_NOISE = 0, 1, 2


def row_confidence_t(logits_row, mask_id: int, temperature: float):
    """(token, confidence) of one masked position at temperature tau."""
    a = np.asarray(logits_row, dtype=np.float64).copy()
    if 0 <= mask_id < a.size:
        a[mask_id] = -np.inf
    tok = int(np.argmax(a))
    conf = 1.0 / float(np.sum(np.exp((a - a[tok]) / float(temperature))))
    return tok, conf


def schedule_keep(S: int, steps: int, T: int) -> int:
    """Positions the linear noise schedule leaves masked after the step (steps done before it)."""
    left = T - steps - 1
    if left <= 0:
        return 0
    return (S * left) // T


def sampler_step(logits, ids, steps: int, mask_id: int, T: int, kind: int = CONFIDENCE,
                 gamma: float = 0.8, temperature: float = 1.0, commit_step=None) -> dict:
    """One step of one sequence under the given sampler.

    logits: fp32 [S][V] (rows of decoded positions ignored) or ``rows(positions) ->
    [len][V]``; ids int [S]; steps = steps taken so far.  Returns the same fields as
    oracle.unmask_step (k_min is the number of commits the rule asks for at least).
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
        tok[i], conf[i] = row_confidence_t(rows[j], mask_id, temperature)
    by_conf = sorted(masked, key=lambda i: (-conf[i], i))
    if kind == CONFIDENCE:
        left = T - steps
        k_min = m if left <= 0 else int(math.ceil(m / left))
        chosen = [i for i in masked if conf[i] >= gamma]
        if len(chosen) < k_min:
            chosen = by_conf[:k_min]
    elif kind == MOCK_AR:
        k_min = 1
        chosen = [masked[0]]
    elif kind == PREDICT_NOISE:
        k_min = min(m, max(1, m - schedule_keep(S, steps, T)))
        chosen = by_conf[:k_min]
    else:
        raise ValueError(f"unknown sampler kind {kind}")
    steps += 1
    for i in chosen:
        ids[i] = tok[i]
        commit[i] = 1
        cs[i] = steps
    return dict(ids=ids, commit=commit, conf=conf, tok=tok, n_masked=m - len(chosen),
                steps=steps, commit_step=cs, k_min=k_min)


def sampler_block(S: int, T: int, mask_id: int, logits_fn, kind: int = CONFIDENCE,
                  gamma: float = 0.8, temperature: float = 1.0) -> dict:
    """Decodes one block from fully masked: logits_fn(step, positions) -> [len][V]."""
    ids = np.full(S, mask_id, np.int64)
    cs = np.zeros(S, np.uint8)
    steps = 0
    trace = []
    while np.any(ids == mask_id) and steps < 255:
        r = sampler_step(lambda pos: logits_fn(steps, pos), ids, steps, mask_id, T, kind, gamma,
                         temperature, cs)
        trace.append(dict(ids_before=ids.copy(), conf=r["conf"], commit=r["commit"]))
        ids, cs, steps = r["ids"], r["commit_step"], r["steps"]
    return dict(ids=ids, steps=steps, commit_step=cs, trace=trace)
