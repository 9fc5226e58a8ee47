"""The LM-head oracle against its pins, and planted mistakes that the pins reject."""
import numpy as np
import pytest

import oracle
from gpu_util import bf16_to_f64
import pins
from oracle.samplers import sampler_step


@pytest.mark.parametrize("check", pins.LMHEAD_LOGIT_CHECKS, ids=lambda c: c.__name__)
def test_lm_head_logits(check):
    check(oracle.lm_head_logits)


@pytest.mark.parametrize("check", pins.LMHEAD_STEP_CHECKS, ids=lambda c: c.__name__)
def test_lm_head_step(check):
    check(oracle.lm_head_step)


# planted mistakes in copies of the LM head
def _f64(bits):
    return bf16_to_f64(bits)


def _logits_mut(h, W, *, transposed=False, half_k=False, bias=False):
    hf, Wf = _f64(h), _f64(W)
    if half_k:
        k = hf.shape[1] // 2
        return hf[:, :k] @ Wf[:, :k].T
    out = hf @ Wf if transposed else hf @ Wf.T
    return out + 1.0 if bias else out


def _step_mut(h, W, ids, steps, mask_id, T, kind=0, gamma=0.8, temperature=1.0, commit_step=None,
              *, shift_rows=False, **kw):
    h = np.asarray(h)

    def rows(positions):
        pos = [(p + 1) % h.shape[0] for p in positions] if shift_rows else list(positions)
        return _logits_mut(h[pos], W, **kw)

    return sampler_step(rows, ids, steps, mask_id, T, kind, gamma, temperature, commit_step)


def _rejected(checks, fn):
    for check in checks:
        try:
            check(fn)
        except (AssertionError, ValueError, IndexError):
            return True
    return False


def test_sanity_copies_pass():
    assert not _rejected(pins.LMHEAD_LOGIT_CHECKS, lambda *a: _logits_mut(*a))
    assert not _rejected(pins.LMHEAD_STEP_CHECKS, lambda *a: _step_mut(*a))


@pytest.mark.parametrize("kw", [dict(transposed=True), dict(half_k=True), dict(bias=True)],
                         ids=lambda k: next(iter(k)))
def test_logit_mutant_rejected(kw):
    assert _rejected(pins.LMHEAD_LOGIT_CHECKS, lambda *a: _logits_mut(*a, **kw))


@pytest.mark.parametrize("kw", [dict(transposed=True), dict(half_k=True), dict(shift_rows=True)],
                         ids=lambda k: next(iter(k)))
def test_step_mutant_rejected(kw):
    assert _rejected(pins.LMHEAD_STEP_CHECKS, lambda *a: _step_mut(*a, **kw))
