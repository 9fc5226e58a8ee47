"""Sampler variants of the unmask step (temperature, mock-AR, predict-and-noise)
against the oracle's sampler_step, and the block loop driven by each of them.

Parity rules as for the main sampler: token ids, commit masks, step counts and
commit steps bit-exact, except sequences where the rule decides between confidences
within 1e-5 of each other (or of gamma), which are checked for validity only;
confidences within 1e-5 relative."""
import numpy as np
import pytest
import torch

from block_wise_mask_tt_b300 import synth
from gpu_util import CONF_REL, GAMMA_BAND, check_decision_validity, dev, host
from oracle.samplers import sampler_block, sampler_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tt():
    from block_wise_mask_tt_b300 import tt as _tt
    return _tt


def _ambiguous(r, ids0_b, mask_id, kind, gamma):
    masked = np.flatnonzero(ids0_b == mask_id)
    if masked.size == 0 or kind == 1:
        return False
    conf = r["conf"][masked]
    k = r["k_min"]
    if kind == 0 and np.any(np.abs(conf - gamma) <= GAMMA_BAND):
        return True
    srt = np.sort(conf)[::-1]
    if 0 < k < masked.size and abs(srt[k - 1] - srt[k]) <= GAMMA_BAND * srt[k - 1]:
        return kind == 2 or int(np.sum(conf >= gamma)) < k
    return False


@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("tau", [0.5, 1.0, 2.0])
def test_sampler_unmask_matches_oracle(tt, kind, tau):
    B, S, V, mask, T, gamma = 6, 16, 8192, 3, 8, 0.8
    rng = np.random.default_rng(100 * kind + int(10 * tau))
    ids0 = np.full((B, S), mask, np.int64)
    ids0[rng.random((B, S)) < 0.3] = 17
    steps0 = rng.integers(0, T - 1, B)
    logits = np.zeros((B, S, V), np.float32)
    for b in range(B):
        pos = np.flatnonzero(ids0[b] == mask)
        logits[b, pos] = synth.logits_rows(9, b, 0, int(steps0[b]), pos, V, mask, 0, 0.0, 12.0)
    ids = dev(ids0.astype(np.int32))
    steps = dev(steps0.astype(np.int32))
    n_masked = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    conf = torch.full((B, S), -1.0, dtype=torch.float32, device="cuda")
    commit = torch.full((B, S), 7, dtype=torch.uint8, device="cuda")
    cs = torch.zeros((B, S), dtype=torch.uint8, device="cuda")
    sm = tt.tt_sampler(kind, gamma, tau, T)
    tt.tt_sampler_unmask(dev(logits), ids, steps, B, S, V, mask, sm, n_masked=n_masked, conf=conf,
                         commit=commit, commit_step=cs)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    g = dict(ids=host(ids), steps=host(steps), n_masked=host(n_masked), conf=host(conf),
             commit=host(commit), commit_step=host(cs))
    excluded = 0
    for b in range(B):
        r = sampler_step(logits[b], ids0[b], int(steps0[b]), mask, T, kind, gamma, tau)
        msk = ids0[b] == mask
        rel = np.abs(g["conf"][b][msk] - r["conf"][msk]) / r["conf"][msk]
        assert rel.size == 0 or rel.max() <= CONF_REL
        assert np.all(g["conf"][b][~msk] == 0)
        # every sequence: the decision is one the sampler's rule allows, given the
        # confidence tolerance
        assert g["steps"][b] == r["steps"]
        check_decision_validity(g["ids"][b], g["commit"][b], ids0[b], r["tok"], r["conf"], mask, kind,
                                gamma, r["k_min"], CONF_REL * r["conf"], what=f"b={b}")
        assert g["n_masked"][b] == int(msk.sum()) - int(g["commit"][b].sum())
        if _ambiguous(r, ids0[b], mask, kind, gamma):
            excluded += 1
            continue
        assert np.array_equal(g["ids"][b], r["ids"]), b
        assert np.array_equal(g["commit"][b], r["commit"]), b
        assert np.array_equal(g["commit_step"][b], r["commit_step"]), b
        assert g["steps"][b] == r["steps"] and g["n_masked"][b] == r["n_masked"]
    assert excluded <= B // 2


@pytest.mark.parametrize("kind,T,tau", [(1, 16, 1.0), (2, 4, 1.0), (2, 5, 0.7), (0, 16, 0.5)])
def test_block_loop_with_sampler_matches_oracle(tt, kind, T, tau):
    w = synth.TINY.replace(T=T)
    B, S = w.B, w.S
    inp = synth.make_attention_inputs(w, 4)
    ad = synth.make_adaln_inputs(w, 4)
    dims = tt.attn_dims(B, S, w.Hq, w.Hkv, w.D, inp["k_ctx"].shape[1], 0, 0, 0, w.softmax_scale, 0)
    desc = tt.step_desc(dims, w.H, w.V, w.mask_id, w.gamma, T, w.ln_eps, 4, 1, w.logits_kind,
                        w.boost_lo, w.boost_hi, sampler=kind, temperature=tau)
    t = dict(x=dev(ad["x"]), shift_table=dev(ad["shift_table"]), scale_table=dev(ad["scale_table"]),
             q=dev(inp["q"]), k_blk=dev(inp["k_blk"]), v_blk=dev(inp["v_blk"]), k_ctx=dev(inp["k_ctx"]),
             v_ctx=dev(inp["v_ctx"]), ctx_len=dev(inp["ctx_len"]),
             ids=torch.full((B, S), w.mask_id, dtype=torch.int32, device="cuda"),
             n_masked=torch.zeros(B, dtype=torch.int32, device="cuda"),
             steps=torch.zeros(B, dtype=torch.int32, device="cuda"),
             commit_step=torch.zeros((B, S), dtype=torch.uint8, device="cuda"),
             y=torch.zeros((B, S, w.H), dtype=torch.int16, device="cuda"),
             attn_out=torch.zeros((B, S, w.Hq, w.D), dtype=torch.int16, device="cuda"),
             logits=torch.zeros((B, S, w.V), dtype=torch.float32, device="cuda"))
    ws = tt.workspace(tt.tt_denoise_workspace(desc))
    tt.tt_denoise_block_loop(desc, tt.step_tensors(**t), ws)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    ids, steps, cs = host(t["ids"])[0], int(host(t["steps"])[0]), host(t["commit_step"])[0]
    r = sampler_block(S, T, w.mask_id, lambda step, pos: synth.logits_rows(
        4, 0, 1, step, pos, w.V, w.mask_id, w.logits_kind, w.boost_lo, w.boost_hi), kind, w.gamma, tau)
    if kind == 1:
        assert cs.tolist() == list(range(1, S + 1)) and steps == S
    if kind == 2:
        # the schedule fixes how many commit at each step, whatever the tie-breaking
        assert np.array_equal(np.bincount(cs, minlength=T + 1), np.bincount(r["commit_step"], minlength=T + 1))
    amb = any(_ambiguous(dict(conf=tr["conf"], k_min=int(tr["commit"].sum())), tr["ids_before"],
                         w.mask_id, kind, w.gamma)
              for tr in r["trace"])
    if not amb:
        assert np.array_equal(ids, r["ids"]) and steps == r["steps"]
        assert np.array_equal(cs, r["commit_step"])
    assert np.all(ids != w.mask_id)
