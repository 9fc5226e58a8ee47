"""tt_confidence_unmask against the oracle's unmask step (bit-exact decisions)."""
import numpy as np
import pytest

import oracle
from block_wise_mask_tt_b300 import synth
from gpu_util import compare_unmask, oracle_unmask_batch, record_excluded, run_unmask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tt():
    from block_wise_mask_tt_b300 import tt as _tt
    return _tt


def _logits(B, S, V, mask, seed, kind=synth.LOGITS_UNIFORM, lo=0.0, hi=20.0, step=0):
    return np.stack([synth.logits_rows(seed, b, 0, step, np.arange(S), V, mask, kind, lo, hi)
                     for b in range(B)])


def _state(B, S, mask, seed, frac_committed=0.0, max_step=0):
    rng = np.random.default_rng(seed)
    ids = np.full((B, S), mask, np.int32)
    cs = np.zeros((B, S), np.uint8)
    steps = rng.integers(0, max_step + 1, size=B).astype(np.int32) if max_step else np.zeros(B, np.int32)
    for b in range(B):
        done = rng.random(S) < frac_committed
        ids[b, done] = rng.integers(4, 1000, size=done.sum())
        cs[b, done] = 1
    return ids, steps, cs


CASES = [
    # B, S, V, gamma, T, frac_committed, kind, lo, hi
    (1, 16, 1024, 0.8, 16, 0.0, synth.LOGITS_UNIFORM, 0.0, 12.0),
    (4, 16, 1024, 0.8, 16, 0.4, synth.LOGITS_UNIFORM, 0.0, 12.0),
    (2, 16, 131072, 0.8, 16, 0.0, synth.LOGITS_UNIFORM, 0.0, 20.0),
    (3, 32, 16384, 0.8, 32, 0.3, synth.LOGITS_BIMODAL, 0.0, 0.0),
    (5, 7, 4096, 0.5, 7, 0.2, synth.LOGITS_UNIFORM, 0.0, 14.0),
    (2, 16, 2048, 0.0, 16, 0.0, synth.LOGITS_UNIFORM, 0.0, 12.0),
    (2, 16, 2048, 1.01, 16, 0.5, synth.LOGITS_UNIFORM, 0.0, 12.0),
    (3, 16, 2052, 0.95, 4, 0.0, synth.LOGITS_UNIFORM, 0.0, 12.0),
    (1, 1, 1024, 0.8, 16, 0.0, synth.LOGITS_UNIFORM, 0.0, 12.0),
    (64, 32, 1024, 0.8, 32, 0.5, synth.LOGITS_BIMODAL, 0.0, 0.0),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}S{c[1]}V{c[2]}g{c[3]}T{c[4]}" for c in CASES])
def test_unmask_matches_oracle(tt, case):
    B, S, V, gamma, T, frac, kind, lo, hi = case
    mask = 3
    for seed in (0, 1):
        logits = _logits(B, S, V, mask, seed, kind, lo, hi)
        ids0, steps0, cs0 = _state(B, S, mask, seed, frac, max_step=max(0, min(T - 1, 3)))
        gpu = run_unmask(tt, logits, ids0, steps0, cs0, mask, gamma, T)
        ora = oracle_unmask_batch(logits, ids0, steps0, cs0, mask, gamma, T)
        n = compare_unmask(gpu, ora, ids0, steps0, mask, gamma, what=f"seed {seed}")
        record_excluded(f"unmask B{B} S{S} V{V} gamma={gamma}", n, B)


def test_ties_and_mask_id(tt):
    """Exact ties go to the lowest id; the mask id never wins even with the largest logit."""
    B, S, V, mask = 1, 4, 4096, 3
    logits = np.zeros((B, S, V), np.float32)
    logits[0, 0, [9, 5, 4000]] = 9.0          # tie -> id 5
    logits[0, 1, mask] = 50.0                  # mask id largest -> next best (id 7)
    logits[0, 1, 7] = 8.0
    logits[0, 2, [1028, 1027]] = 12.0          # tie across a vector boundary -> 1027
    logits[0, 3, [V - 1, 2048]] = 11.0         # tie across CTA chunks -> 2048
    ids0 = np.full((B, S), mask, np.int32)
    steps0 = np.zeros(B, np.int32)
    cs0 = np.zeros((B, S), np.uint8)
    gpu = run_unmask(tt, logits, ids0, steps0, cs0, mask, 0.0, 16)
    assert gpu["ids"][0].tolist() == [5, 7, 1027, 2048]
    ora = oracle_unmask_batch(logits, ids0, steps0, cs0, mask, 0.0, 16)
    compare_unmask(gpu, ora, ids0, steps0, mask, 0.0)


def test_done_sequences_untouched(tt):
    B, S, V, mask = 3, 16, 1024, 3
    logits = _logits(B, S, V, mask, 4)
    ids0 = np.full((B, S), mask, np.int32)
    ids0[1] = np.arange(100, 100 + S)
    steps0 = np.array([0, 5, 2], np.int32)
    cs0 = np.zeros((B, S), np.uint8)
    cs0[1] = 3
    gpu = run_unmask(tt, logits, ids0, steps0, cs0, mask, 0.8, 16)
    assert np.array_equal(gpu["ids"][1], ids0[1])
    assert gpu["steps"][1] == 5 and gpu["n_masked"][1] == 0
    assert np.all(gpu["commit"][1] == 0) and np.all(gpu["conf"][1] == 0)
    assert np.all(gpu["commit_step"][1] == 3)


def test_repeated_calls_reuse_workspace(tt):
    """The tickets in the workspace are left zeroed: back-to-back calls on one workspace agree."""
    import torch
    from gpu_util import dev, host
    B, S, V, mask = 4, 16, 8192, 3
    ws = tt.workspace(tt.tt_confidence_unmask_workspace(B, S, V))
    ids = dev(np.full((B, S), mask, np.int32))
    steps = dev(np.zeros(B, np.int32))
    cs = torch.zeros((B, S), dtype=torch.uint8, device="cuda")
    ids_h = np.full((B, S), mask, np.int32)
    steps_h = np.zeros(B, np.int32)
    cs_h = np.zeros((B, S), np.uint8)
    for k in range(S + 2):
        logits = np.stack([synth.logits_rows(9, b, 0, int(steps_h[b]), np.arange(S), V, mask, 0,
                                             0.0, 14.0) for b in range(B)])
        tt.tt_confidence_unmask(dev(logits), ids, steps, B, S, V, mask, 0.8, S, commit_step=cs, ws=ws)
        ora = oracle_unmask_batch(logits, ids_h, steps_h, cs_h, mask, 0.8, S)
        torch.cuda.synchronize()
        got_ids, got_steps = host(ids), host(steps)
        for b in range(B):
            if not np.any(ids_h[b] == mask):
                assert np.array_equal(got_ids[b], ids_h[b])
                continue
            if np.any(np.abs(ora[b]["conf"][ids_h[b] == mask] - 0.8) <= 1e-5):
                pytest.skip("gamma-band position; teacher forcing covered elsewhere")
            assert np.array_equal(got_ids[b], ora[b]["ids"])
            assert got_steps[b] == ora[b]["steps"]
        ids_h, steps_h = got_ids.copy(), got_steps.copy()
        cs_h = host(cs).copy()
    assert np.all(ids_h != mask) and np.all(steps_h <= S)
