"""Plant a plausible mistake in a copy of the oracle; some pin must reject every copy.

This shows the pins constrain the oracle: a dropped term, a wrong sign or index, a
transposed operand or a flipped comparison anywhere in it fails at least one check.
Mistakes are planted only in these CPU copies, never in the real oracle.
"""
import math

import numpy as np
import pytest

import oracle
import pins
from oracle._bf16 import bf16_to_f64
from oracle import unmask as U


# ----------------------------------------------------------------------------------
# attention mutants
# ----------------------------------------------------------------------------------

def _attn_generic(inp, scale, *, drop_block=False, causal_block=False, gqa_mod=False,
                  no_scale=False, pv_keys=False, ctx_off_by_one=False):
    q = bf16_to_f64(inp["q"])
    kb, vb = bf16_to_f64(inp["k_blk"]), bf16_to_f64(inp["v_blk"])
    B, S, Hq, D = q.shape
    Hkv = kb.shape[2]
    G = Hq // Hkv
    O = np.zeros((B, S, Hq, D))
    lse = np.zeros((B, S, Hq))
    for b in range(B):
        kc, vc = oracle.context_kv(inp, b)
        if ctx_off_by_one and len(kc):
            kc, vc = kc[:-1], vc[:-1]
        for h in range(Hq):
            g = (h % Hkv) if gqa_mod else (h // G)
            keys = kc[:, g] if drop_block else np.concatenate([kc[:, g], kb[b, :, g]])
            vals = vc[:, g] if drop_block else np.concatenate([vc[:, g], vb[b, :, g]])
            if keys.shape[0] == 0:
                continue
            a = (1.0 if no_scale else scale) * (q[b, :, h] @ keys.T)
            if causal_block and not drop_block:
                n = kc.shape[0]
                for s in range(S):
                    a[s, n + s + 1:] = -np.inf
            m = a.max(axis=1, keepdims=True)
            e = np.exp(a - m)
            p = e / e.sum(axis=1, keepdims=True)
            O[b, :, h] = p @ (keys if pv_keys else vals)
            lse[b, :, h] = (m + np.log(e.sum(axis=1, keepdims=True)))[:, 0]
    return O, lse


ATTN_MUTANTS = {
    "drop_block_keys": dict(drop_block=True),
    "causal_inside_block": dict(causal_block=True),
    "wrong_gqa_mapping": dict(gqa_mod=True),
    "missing_softmax_scale": dict(no_scale=True),
    "pv_uses_keys": dict(pv_keys=True),
    "context_off_by_one": dict(ctx_off_by_one=True),
}


def _rejected(checks, fn):
    for check in checks:
        try:
            check(fn)
        except (AssertionError, ValueError, IndexError, ZeroDivisionError):
            return True
    return False


def test_sanity_generic_attention_passes():
    assert not _rejected(pins.ATTENTION_CHECKS, lambda i, s: _attn_generic(i, s))


@pytest.mark.parametrize("name", sorted(ATTN_MUTANTS))
def test_attention_mutant_rejected(name):
    kw = ATTN_MUTANTS[name]
    assert _rejected(pins.ATTENTION_CHECKS, lambda i, s: _attn_generic(i, s, **kw))


# ----------------------------------------------------------------------------------
# adaLN mutants
# ----------------------------------------------------------------------------------

def _adaln_generic(x_bf16, shift, scale, eps=1e-5, *, ddof=0, no_eps=False, plain_scale=False,
                   minus_shift=False):
    x = bf16_to_f64(x_bf16)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - ddof)
    xh = (x - mu) / np.sqrt(var + (0.0 if no_eps else eps))
    sc = np.asarray(scale, np.float64)
    sh = np.asarray(shift, np.float64)
    y = xh * (sc if plain_scale else 1.0 + sc)
    return y - sh if minus_shift else y + sh


ADALN_MUTANTS = {
    "unbiased_variance": dict(ddof=1),
    "missing_eps": dict(no_eps=True),
    "scale_without_one": dict(plain_scale=True),
    "shift_sign": dict(minus_shift=True),
}


def test_sanity_generic_adaln_passes():
    assert not _rejected(pins.ADALN_CHECKS, lambda *a: _adaln_generic(*a))


@pytest.mark.parametrize("name", sorted(ADALN_MUTANTS))
def test_adaln_mutant_rejected(name):
    kw = ADALN_MUTANTS[name]
    with np.errstate(all="ignore"):
        assert _rejected(pins.ADALN_CHECKS, lambda *a: _adaln_generic(*a, **kw))


# ----------------------------------------------------------------------------------
# unmask mutants
# ----------------------------------------------------------------------------------

def _row_generic(row, mask_id, *, keep_mask=False, ties_high=False, mask_in_sum=False):
    a = np.asarray(row, np.float64).copy()
    full = a.copy()
    if not keep_mask:
        a[mask_id] = -np.inf
    tok = int(a.size - 1 - np.argmax(a[::-1])) if ties_high else int(np.argmax(a))
    base = full if mask_in_sum else a
    conf = 1.0 / float(np.sum(np.exp(base - a[tok])))
    return tok, conf


ROW_MUTANTS = {
    "mask_id_not_excluded": dict(keep_mask=True),
    "ties_to_highest_id": dict(ties_high=True),
    "mask_logit_in_normaliser": dict(mask_in_sum=True),
}


def test_sanity_generic_row_passes():
    assert not _rejected(pins.UNMASK_ROW_CHECKS, lambda r, m: _row_generic(r, m))


@pytest.mark.parametrize("name", sorted(ROW_MUTANTS))
def test_row_mutant_rejected(name):
    kw = ROW_MUTANTS[name]
    assert _rejected(pins.UNMASK_ROW_CHECKS, lambda r, m: _row_generic(r, m, **kw))


def _step_generic(logits, ids, steps, mask_id, gamma, T, commit_step=None, *, strict=False,
                  no_floor=False, floor_high_pos=False, floor_least=False, floor_plain_one=False,
                  step_off=False, refresh_committed=False):
    ids = np.array(ids, np.int64)
    S = ids.size
    masked = [i for i in range(S) if ids[i] == mask_id]
    if refresh_committed:
        masked_rows = list(range(S))
    else:
        masked_rows = masked
    cs = np.zeros(S, np.uint8) if commit_step is None else np.array(commit_step, np.uint8)
    conf = np.zeros(S)
    tok = np.full(S, -1, np.int64)
    commit = np.zeros(S, np.uint8)
    m = len(masked)
    if m == 0:
        return dict(ids=ids, commit=commit, conf=conf, tok=tok, n_masked=0, steps=steps,
                    commit_step=cs, k_min=0)
    rows = logits(masked_rows) if callable(logits) else np.asarray(logits)[masked_rows]
    for j, i in enumerate(masked_rows):
        tok[i], conf[i] = U.row_confidence(rows[j], mask_id)
    k_min = 0 if no_floor else (1 if floor_plain_one else U.floor_count(m, steps, T))
    chosen = [i for i in masked if (conf[i] > gamma if strict else conf[i] >= gamma)]
    if refresh_committed:
        chosen = [i for i in range(S) if conf[i] >= gamma and (i in masked or True)]
    if len(chosen) < k_min:
        if floor_least:
            key = lambda i: (conf[i], i)
        elif floor_high_pos:
            key = lambda i: (-conf[i], -i)
        else:
            key = lambda i: (-conf[i], i)
        chosen = sorted(masked, key=key)[:k_min]
    steps += 1
    for i in chosen:
        ids[i] = tok[i]
        commit[i] = 1
        cs[i] = steps + (1 if step_off else 0)
    return dict(ids=ids, commit=commit, conf=conf, tok=tok,
                n_masked=int(np.sum(ids == mask_id)), steps=steps, commit_step=cs, k_min=k_min)


def _block_with(step_kw):
    def block(S, T, mask_id, gamma, logits_fn, ids=None, steps=0, commit_step=None):
        ids = np.full(S, mask_id, np.int64)
        cs = np.zeros(S, np.uint8)
        trace = []
        while np.any(ids == mask_id) and steps < T:
            m = int(np.sum(ids == mask_id))
            k = steps
            r = _step_generic(lambda pos: logits_fn(k, pos), ids, steps, mask_id, gamma, T, cs,
                              **step_kw)
            trace.append(dict(t=m / S, n_masked_before=m, committed=np.flatnonzero(r["commit"]),
                              conf=r["conf"], tok=r["tok"], k_min=r["k_min"], ids_before=ids))
            ids, steps, cs = r["ids"], r["steps"], r["commit_step"]
        return dict(ids=ids, steps=steps, commit_step=cs, n_masked=int(np.sum(ids == mask_id)),
                    trace=trace)
    return block


STEP_MUTANTS = {
    "strict_threshold": dict(strict=True),
    "no_floor": dict(no_floor=True),
    "floor_ties_high_position": dict(floor_high_pos=True),
    "floor_least_confident": dict(floor_least=True),
    "floor_ignores_steps_left": dict(floor_plain_one=True),
    "commit_step_off_by_one": dict(step_off=True),
    "committed_positions_recommitted": dict(refresh_committed=True),
}


def test_sanity_generic_block_passes():
    assert not _rejected(pins.BLOCK_CHECKS, _block_with({}))
    assert not _rejected(pins.UNMASK_STEP_CHECKS, lambda *a, **k: _step_generic(*a, **k))


@pytest.mark.parametrize("name", sorted(STEP_MUTANTS))
def test_step_mutant_rejected(name):
    kw = STEP_MUTANTS[name]
    checks = pins.BLOCK_CHECKS
    block_ok = not _rejected(checks, _block_with(kw))
    step_ok = not _rejected(pins.UNMASK_STEP_CHECKS, lambda *a, **k: _step_generic(*a, **k, **kw))
    assert not (block_ok and step_ok)


# ----------------------------------------------------------------------------------
# sampler variants
# ----------------------------------------------------------------------------------
def _sampler_generic(logits, ids, steps, mask_id, T, kind=0, gamma=0.8, temperature=1.0,
                     commit_step=None, *, temp_multiplies=False, ar_rightmost=False,
                     ar_most_confident=False, schedule_off_by_one=False, pn_least=False):
    import math
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
        a = np.asarray(rows[j], np.float64).copy()
        a[mask_id] = -np.inf
        tok[i] = int(np.argmax(a))
        z = (a - a[tok[i]]) * temperature if temp_multiplies else (a - a[tok[i]]) / temperature
        conf[i] = 1.0 / float(np.sum(np.exp(z)))
    by_conf = sorted(masked, key=lambda i: (-conf[i], i))
    if kind == 0:
        left = T - steps
        k_min = m if left <= 0 else int(math.ceil(m / left))
        chosen = [i for i in masked if conf[i] >= gamma]
        if len(chosen) < k_min:
            chosen = by_conf[:k_min]
    elif kind == 1:
        k_min = 1
        chosen = [masked[-1]] if ar_rightmost else [by_conf[0]] if ar_most_confident else [masked[0]]
    else:
        left = T - steps - (0 if schedule_off_by_one else 1)
        keep = 0 if left <= 0 else (S * left) // T
        k_min = min(m, max(1, m - keep))
        chosen = (by_conf[::-1] if pn_least else by_conf)[:k_min]
    steps += 1
    for i in chosen:
        ids[i] = tok[i]
        commit[i] = 1
        cs[i] = steps
    return dict(ids=ids, commit=commit, conf=conf, tok=tok, n_masked=m - len(chosen),
                steps=steps, commit_step=cs, k_min=k_min)


SAMPLER_MUTANTS = {
    "temperature_multiplies": dict(temp_multiplies=True),
    "mock_ar_rightmost": dict(ar_rightmost=True),
    "mock_ar_most_confident": dict(ar_most_confident=True),
    "schedule_off_by_one": dict(schedule_off_by_one=True),
    "predict_noise_least_confident": dict(pn_least=True),
}


def test_sanity_generic_sampler_passes():
    assert not _rejected(pins.SAMPLER_CHECKS, lambda *a: _sampler_generic(*a))


@pytest.mark.parametrize("name", sorted(SAMPLER_MUTANTS))
def test_sampler_mutant_rejected(name):
    kw = SAMPLER_MUTANTS[name]
    assert _rejected(pins.SAMPLER_CHECKS, lambda *a: _sampler_generic(*a, **kw))
