"""The CUDA logits stand-in reproduces the seeded generator bit for bit."""
import numpy as np
import pytest
import torch

from block_wise_mask_tt_b300 import synth
from gpu_util import dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tt():
    from block_wise_mask_tt_b300 import tt as _tt
    return _tt


@pytest.mark.parametrize("B,S,V,kind,lo,hi,seed,block", [
    (1, 16, 1024, synth.LOGITS_UNIFORM, 0.0, 12.0, 0, 0),
    (2, 16, 131072, synth.LOGITS_UNIFORM, 0.0, 20.0, 7, 3),
    (3, 32, 8192, synth.LOGITS_BIMODAL, 0.0, 0.0, 123456789, 63),
    (1, 5, 1028, synth.LOGITS_UNIFORM, 1.5, 2.5, 2 ** 32 - 1, 1),
])
def test_logits_bit_exact(tt, B, S, V, kind, lo, hi, seed, block):
    mask = 3
    steps = np.array([(5 * b) % 16 for b in range(B)], np.int32)
    out = torch.full((B, S, V), float("nan"), dtype=torch.float32, device="cuda")
    spec = tt.tt_logits_spec(seed & 0xFFFFFFFF, block, kind, lo, hi)
    tt.tt_synthetic_logits(spec, out, B, S, V, mask, steps=dev(steps))
    torch.cuda.synchronize()
    got = host(out)
    rows = [(b, s) for b in range(B) for s in range(S)]
    if len(rows) > 24:
        rows = rows[:8] + rows[-8:] + rows[len(rows) // 2: len(rows) // 2 + 8]
    for b, s in rows:
        ref = synth.logits_rows(seed, b, block, int(steps[b]), [s], V, mask, kind, lo, hi)[0]
        assert np.array_equal(got[b, s].view(np.uint32), ref.view(np.uint32)), (b, s)


def test_only_masked_rows_written(tt):
    B, S, V, mask = 2, 8, 1024, 3
    ids = np.full((B, S), mask, np.int32)
    ids[0, 2] = 17
    ids[1, 7] = 4
    out = torch.full((B, S, V), -123.0, dtype=torch.float32, device="cuda")
    spec = tt.tt_logits_spec(1, 0, 0, 0.0, 12.0)
    tt.tt_synthetic_logits(spec, out, B, S, V, mask, ids=dev(ids))
    torch.cuda.synchronize()
    got = host(out)
    assert np.all(got[0, 2] == -123.0) and np.all(got[1, 7] == -123.0)
    ref = synth.logits_rows(1, 1, 0, 0, [3], V, mask, 0, 0.0, 12.0)[0]
    assert np.array_equal(got[1, 3], ref)
