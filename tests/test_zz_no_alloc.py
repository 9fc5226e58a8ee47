"""tt_confidence_unmask_noalloc: the unmask step for callers that cannot allocate.

Some callers cannot give the library a workspace: all of their device memory is held
by another allocator, or their hot path may not call cudaMalloc (it can synchronise
the device and has no latency bound).  The no-allocation entry point keeps its
scratch in a fixed array inside the library instead.  These tests call it through
the C ABI and compare it with tt_confidence_unmask (which takes a workspace) on the
same inputs, using the parity rules of the other unmask tests: token ids, commit
masks, step counts and commit steps bit-exact, confidences within 1e-5 relative.
Two calls in a row are checked.  The first (12 sequences at V = 131072) fills the
front of the scratch with its per-chunk partial results; the second (5 sequences at
V = 8192) is smaller, so its completion counters fall on words the first call left
non-zero: the second call decides correctly only if the entry point clears them.
Both calls are also compared directly with the oracle's unmask step.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from block_wise_mask_tt_b300 import synth
from gpu_util import CONF_REL, compare_unmask, dev, host


@pytest.fixture(scope="module")
def tt():
    from block_wise_mask_tt_b300 import tt as _tt
    return _tt


def _logits(w, B, steps0, ids0, seed, block):
    """Synthetic logits for the masked rows (zeros elsewhere), as the step would make them."""
    lg = np.zeros((B, w.S, w.V), np.float32)
    for b in range(B):
        pos = np.flatnonzero(ids0[b] == w.mask_id)
        if pos.size:
            lg[b, pos] = synth.logits_rows(seed, b, block, int(steps0[b]), pos, w.V, w.mask_id,
                                           w.logits_kind, w.boost_lo, w.boost_hi)
    return lg


def _run(tt, fn, logits, ids0, steps0, w):
    B = ids0.shape[0]
    ids = dev(ids0.astype(np.int32))
    steps = dev(steps0.astype(np.int32))
    n_masked = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    conf = torch.full((B, w.S), -1.0, dtype=torch.float32, device="cuda")
    commit = torch.full((B, w.S), 7, dtype=torch.uint8, device="cuda")
    cs = torch.zeros((B, w.S), dtype=torch.uint8, device="cuda")
    fn(logits, ids, steps, B, w.S, w.V, w.mask_id, w.gamma, w.steps_max, n_masked=n_masked,
       conf=conf, commit=commit, commit_step=cs)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    return dict(ids=host(ids), steps=host(steps), n_masked=host(n_masked), conf=host(conf),
                commit=host(commit), commit_step=host(cs))


def _same(a, b, what):
    for k in ("ids", "steps", "n_masked", "commit", "commit_step"):
        assert np.array_equal(a[k], b[k]), f"{what}: {k} differs"
    m = b["conf"] > 0
    rel = np.abs(a["conf"][m] - b["conf"][m]) / b["conf"][m]
    assert rel.size == 0 or rel.max() <= CONF_REL, f"{what}: conf rel err {rel.max()}"
    assert np.array_equal(a["conf"][~m], b["conf"][~m]), f"{what}: conf of decoded positions"


def _oracle(w, lg, ids0, steps0, got, what):
    """The oracle's unmask step of every sequence from the same state and the same
    host-generated logits."""
    ora = [oracle.unmask_step(lg[b], ids0[b], int(steps0[b]), w.mask_id, w.gamma, w.steps_max,
                              np.zeros(w.S, np.uint8)) for b in range(ids0.shape[0])]
    compare_unmask(got, ora, ids0, steps0, w.mask_id, w.gamma, what=what)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(tt):
    w = synth.BATCHED.replace(B=12)
    rng = np.random.default_rng(7)
    # call 1: 12 sequences at V = 131072, some positions already decoded
    ids0 = np.full((w.B, w.S), w.mask_id, np.int64)
    # some positions of the first four sequences already decoded; the later rows stay
    # masked, so their chunk partials (scratch bytes 8192 .. 24575) are all written
    ids0[:4][rng.random((4, w.S)) < 0.3] = 11
    steps0 = rng.integers(0, 4, w.B)
    lg_h = _logits(w, w.B, steps0, ids0, seed=1, block=0)
    lg = dev(lg_h)
    ref = _run(tt, tt.tt_confidence_unmask, lg, ids0, steps0, w)
    got = _run(tt, tt.tt_confidence_unmask_noalloc, lg, ids0, steps0, w)
    _same(got, ref, "call 1")
    _oracle(w, lg_h, ids0, steps0, got, "call 1")
    # call 2, straight after: fewer sequences and a smaller vocabulary, from the state
    # call 1 produced; its counters (scratch bytes 11520 .. 11859) sit where call 1
    # left partial results
    w2 = w.replace(B=5, V=8192)
    ids1, steps1 = ref["ids"][:5].astype(np.int64), ref["steps"][:5]
    lg2_h = _logits(w2, w2.B, steps1, ids1, seed=2, block=0)
    lg2 = dev(lg2_h)
    ref2 = _run(tt, tt.tt_confidence_unmask, lg2, ids1, steps1, w2)
    got2 = _run(tt, tt.tt_confidence_unmask_noalloc, lg2, ids1, steps1, w2)
    _same(got2, ref2, "call 2")
    _oracle(w2, lg2_h, ids1, steps1, got2, "call 2")
    assert ref2["commit"].sum() > 0


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch(tt):
    # 4096 rows x 128 vocabulary chunks of 16 bytes exceed the fixed 8 MiB; the call is
    # rejected on the host before anything touches the device (the pointers are never
    # dereferenced, so this runs without a GPU as well).
    fake = 256
    st = tt.lib.tt_confidence_unmask_noalloc(fake, fake, None, fake, None, None, None, 128, 32,
                                             131072, 3, 0.8, 16, None)
    assert st == tt.TT_ERR_UNSUPPORTED
    assert "fixed scratch" in tt.lib.tt_last_error().decode()
