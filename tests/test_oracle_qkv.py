"""The QKV-projection oracle against its pins, and planted mistakes the pins reject."""
import numpy as np
import pytest

import oracle
from gpu_util import bf16_to_f64
import pins


@pytest.mark.parametrize("check", pins.QKV_CHECKS, ids=lambda c: c.__name__)
def test_qkv(check):
    check(oracle.qkv_projection)


def _mut(y, W, Hq, Hkv, D, *, kv_swapped=False, k_from_q=False, transposed_heads=False):
    yf = bf16_to_f64(y)
    Wf = bf16_to_f64(W)
    B, S, H = yf.shape
    out = yf.reshape(B * S, H) @ Wf.T
    q = out[:, :Hq * D]
    k = out[:, Hq * D:(Hq + Hkv) * D]
    v = out[:, (Hq + Hkv) * D:]
    if kv_swapped:
        k, v = v, k
    if k_from_q:
        k = q[:, :Hkv * D]
    q = q.reshape(B, S, Hq, D)
    if transposed_heads:
        q = q.reshape(B, S, D, Hq).transpose(0, 1, 3, 2)
    return q, k.reshape(B, S, Hkv, D), v.reshape(B, S, Hkv, D)


def _rejected(fn):
    for check in pins.QKV_CHECKS:
        try:
            check(fn)
        except (AssertionError, ValueError, IndexError):
            return True
    return False


def test_sanity_copy_passes():
    assert not _rejected(lambda *a: _mut(*a))


@pytest.mark.parametrize("kw", [dict(kv_swapped=True), dict(k_from_q=True), dict(transposed_heads=True)],
                         ids=lambda k: next(iter(k)))
def test_mutant_rejected(kw):
    assert _rejected(lambda *a: _mut(*a, **kw))
