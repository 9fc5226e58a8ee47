"""The outer loop (Algorithm 1) of the oracle against its pins."""
import numpy as np
import pytest

import pins
from oracle.outer import append_block, generate
from oracle.loop import denoise_block


@pytest.mark.parametrize("check", pins.OUTER_CHECKS, ids=lambda f: f.__name__)
def test_outer(check):
    check(append_block)


def test_generate_blocks_are_single_block_decodes_and_stop():
    """Block k of every sequence is the single-block decode with block index k; a
    sequence stops after max_new tokens (here two blocks) and is padded afterwards."""
    from block_wise_mask_tt_b300 import synth
    B, S, T, V, mask = 3, 4, 4, 64, 3

    def fn(b, blk, step, pos):
        return synth.logits_rows(5, b, blk, step, pos, V, mask, 0, 0.0, 12.0)
    r = generate(B, S, T, mask, 0.8, 3, fn, eos_id=-1, pad_id=0, max_new=2 * S)
    assert r["done"].tolist() == [1, 1, 1] and r["generated"].tolist() == [8, 8, 8]
    for b in range(B):
        for k in range(2):
            d = denoise_block(S, T, mask, 0.8, lambda st, pos: fn(b, k, st, pos))
            assert np.array_equal(r["tokens"][b, k * S:(k + 1) * S], d["ids"])
        assert np.all(r["tokens"][b, 2 * S:] == 0)
    # an EOS id that block 0 of sequence 1 commits stops that sequence only
    eos = int(r["tokens"][1, 1])
    r2 = generate(B, S, T, mask, 0.8, 3, fn, eos_id=eos, pad_id=0, max_new=100)
    for b in range(B):
        stop = next((k for k in range(3) if eos in r2["tokens"][b, k * S:(k + 1) * S]), None)
        if stop is not None:
            assert np.all(r2["tokens"][b, (stop + 1) * S:] == 0)
    assert r2["done"][1] == 1


# planted mistakes in a copy of append_block: each must be rejected by some pin
def _append_mut(cache, k_blk, v_blk, ctx_len, ids, eos_id, max_new, generated, done, *,
                off_by_one=False, append_done=False, no_eos=False, strict_len=False):
    out = {k: np.array(v, copy=True) for k, v in cache.items()}
    ctx_len = np.array(ctx_len, np.int64, copy=True)
    generated = np.array(generated, np.int64, copy=True)
    done = np.array(done, np.uint8, copy=True)
    B, S = np.asarray(ids).shape
    for b in range(B):
        if done[b] and not append_done:
            continue
        for s in range(S):
            pos = int(ctx_len[b]) + s - (1 if off_by_one and ctx_len[b] > 0 else 0)
            if "page_table" in out:
                pg = int(out["page_table"][b, pos // 64])
                out["k_pages"][pg, pos % 64] = k_blk[b, s]
                out["v_pages"][pg, pos % 64] = v_blk[b, s]
            else:
                out["k_ctx"][b, pos] = k_blk[b, s]
                out["v_ctx"][b, pos] = v_blk[b, s]
        ctx_len[b] += S
        generated[b] += S
        hit = (not no_eos) and np.any(np.asarray(ids)[b] == eos_id)
        if hit or (generated[b] > max_new if strict_len else generated[b] >= max_new):
            done[b] = 1
    out.update(ctx_len=ctx_len, generated=generated, done=done)
    return out


def _rejected(fn):
    for check in pins.OUTER_CHECKS:
        try:
            check(fn)
        except (AssertionError, IndexError, ValueError):
            return True
    return False


def test_outer_sanity_copy_passes():
    assert not _rejected(lambda *a: _append_mut(*a))


@pytest.mark.parametrize("kw", [dict(off_by_one=True), dict(append_done=True), dict(no_eos=True),
                                dict(strict_len=True)], ids=lambda k: next(iter(k)))
def test_outer_mutant_rejected(kw):
    assert _rejected(lambda *a: _append_mut(*a, **kw))
