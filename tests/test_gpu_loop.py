"""The whole denoise step and the device-driven block loop against the oracle.

tt_denoise_step is run one step at a time and every step is compared with the
oracle evaluated from the GPU's own pre-step state (teacher forcing), so a position
excluded for lying within 1e-5 of gamma cannot cascade into later steps.  Then
tt_denoise_block_loop (one CUDA-graph launch with a device-side WHILE loop) must
reproduce the step-by-step final state bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_wise_mask_tt_b300 import synth
from gpu_util import (adaln_tol, bf16_to_f64, check_attention, compare_unmask, dev, host,
                      record_excluded)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tt():
    from block_wise_mask_tt_b300 import tt as _tt
    return _tt


LOOP_CASES = {
    "c0": synth.TINY,
    "c1_B2_L512": synth.SINGLE.replace(B=2, L=512),
    "c4_B3_paged": synth.RAGGED_PAGED.replace(B=3, L=700, L_min=64, V=16384),
    "c3_gamma05_B2": synth.LONG_CONTEXT.replace(B=2, L=256, V=8192, gamma=0.5),
    "T_lt_S": synth.TINY.replace(T=5, gamma=0.97),
}


class Loop:
    def __init__(self, tt, w, seed, block):
        self.tt, self.w, self.seed, self.block = tt, w, seed, block
        self.inp = synth.make_attention_inputs(w, seed)
        self.ad = synth.make_adaln_inputs(w, seed)
        B, S = w.B, w.S
        if w.paged:
            kp = self.inp["k_pages"]
            dims = tt.attn_dims(B, S, w.Hq, w.Hkv, w.D, 0, w.page_size,
                                self.inp["page_table"].shape[1], kp.shape[0], w.softmax_scale, 0)
            self.k_ctx, self.v_ctx = dev(kp), dev(self.inp["v_pages"])
            self.page_table = dev(self.inp["page_table"])
        else:
            dims = tt.attn_dims(B, S, w.Hq, w.Hkv, w.D, self.inp["k_ctx"].shape[1], 0, 0, 0,
                                w.softmax_scale, 0)
            self.k_ctx, self.v_ctx = dev(self.inp["k_ctx"]), dev(self.inp["v_ctx"])
            self.page_table = None
        self.desc = tt.step_desc(dims, w.H, w.V, w.mask_id, w.gamma, w.steps_max, w.ln_eps, seed,
                                 block, w.logits_kind, w.boost_lo, w.boost_hi)
        self.t = dict(
            x=dev(self.ad["x"]), shift_table=dev(self.ad["shift_table"]),
            scale_table=dev(self.ad["scale_table"]), q=dev(self.inp["q"]),
            k_blk=dev(self.inp["k_blk"]), v_blk=dev(self.inp["v_blk"]), k_ctx=self.k_ctx,
            v_ctx=self.v_ctx, page_table=self.page_table, ctx_len=dev(self.inp["ctx_len"]),
            ids=torch.full((B, S), w.mask_id, dtype=torch.int32, device="cuda"),
            n_masked=torch.full((B,), S, dtype=torch.int32, device="cuda"),
            steps=torch.zeros(B, dtype=torch.int32, device="cuda"),
            commit_step=torch.zeros((B, S), dtype=torch.uint8, device="cuda"),
            y=torch.zeros((B, S, w.H), dtype=torch.int16, device="cuda"),
            attn_out=torch.zeros((B, S, w.Hq, w.D), dtype=torch.int16, device="cuda"),
            logits=torch.zeros((B, S, w.V), dtype=torch.float32, device="cuda"),
            conf=torch.zeros((B, S), dtype=torch.float32, device="cuda"),
            commit=torch.zeros((B, S), dtype=torch.uint8, device="cuda"))
        self.ts = tt.step_tensors(**self.t)
        self.ws = tt.workspace(tt.tt_denoise_workspace(self.desc))

    def reset(self):
        self.t["ids"].fill_(self.w.mask_id)
        self.t["n_masked"].fill_(self.w.S)
        self.t["steps"].zero_()
        self.t["commit_step"].zero_()

    def logits_fn(self, b, step, positions):
        w = self.w
        return synth.logits_rows(self.seed, b, self.block, step, positions, w.V, w.mask_id,
                                 w.logits_kind, w.boost_lo, w.boost_hi)


@pytest.mark.parametrize("name", sorted(LOOP_CASES))
def test_step_by_step_teacher_forced_then_graph_loop(tt, name):
    w = LOOP_CASES[name]
    lp = Loop(tt, w, seed=3, block=2)
    B, S, T, mask = w.B, w.S, w.steps_max, w.mask_id
    O_ref, _ = oracle.denoise_attention(lp.inp, w.softmax_scale)
    excluded = 0
    decisions = 0
    n_steps = 0
    for k in range(T + 1):
        ids0 = host(lp.t["ids"]).copy()
        steps0 = host(lp.t["steps"]).copy()
        cs0 = host(lp.t["commit_step"]).copy()
        nm0 = (ids0 == mask).sum(axis=1)
        if not np.any(nm0 > 0):
            break
        tt.tt_denoise_step(lp.desc, lp.ts, lp.ws)
        torch.cuda.synchronize()
        assert tt.tt_device_status(True) == 0
        n_steps += 1
        active = nm0 > 0
        # logits of the masked rows are the generator's, bit for bit
        lg = host(lp.t["logits"])
        logits = np.zeros((B, S, w.V), np.float32)
        for b in np.flatnonzero(active):
            pos = np.flatnonzero(ids0[b] == mask)
            logits[b, pos] = lp.logits_fn(b, int(steps0[b]), pos)
            assert np.array_equal(lg[b, pos].view(np.uint32), logits[b, pos].view(np.uint32))
        # unmask decisions, teacher-forced from the GPU's pre-step state
        ora = [oracle.unmask_step(logits[b], ids0[b], int(steps0[b]), mask, w.gamma, T, cs0[b])
               for b in range(B)]
        gpu = dict(ids=host(lp.t["ids"]), steps=host(lp.t["steps"]), n_masked=host(lp.t["n_masked"]),
                   conf=host(lp.t["conf"]), commit=host(lp.t["commit"]),
                   commit_step=host(lp.t["commit_step"]))
        for b in np.flatnonzero(~active):  # finished sequences are left alone by the step
            gpu["conf"][b] = 0.0
            gpu["commit"][b] = 0
        excluded += compare_unmask(gpu, ora, ids0, steps0, mask, w.gamma, what=f"{name} step {k}")
        decisions += int(active.sum())
        # adaLN of the active sequences uses table row n_masked (t = n_masked / S)
        y = bf16_to_f64(host(lp.t["y"]))
        for b in np.flatnonzero(active):
            ref = oracle.adaln_modulate(lp.ad["x"][b], lp.ad["shift_table"][nm0[b]],
                                        lp.ad["scale_table"][nm0[b]], w.ln_eps)
            sh = np.broadcast_to(lp.ad["shift_table"][nm0[b]], ref.shape)
            assert np.all(np.abs(y[b] - ref) <= adaln_tol(ref, sh))
        O = bf16_to_f64(host(lp.t["attn_out"]))
        check_attention(O[active], O_ref[active], what=f"{name} step {k}")
    record_excluded(f"reduced loop {name}", excluded, decisions)
    final = (host(lp.t["ids"]).copy(), host(lp.t["steps"]).copy(), host(lp.t["commit_step"]).copy())
    assert np.all(final[0] != mask)
    assert np.all(final[1] <= T) and n_steps <= T
    assert np.all((final[2] >= 1) & (final[2] <= final[1][:, None]))

    # the graph loop from a fresh block reproduces the step-by-step run exactly
    for rep in range(2):
        lp.reset()
        tt.tt_denoise_block_loop(lp.desc, lp.ts, lp.ws)
        torch.cuda.synchronize()
        assert tt.tt_device_status(True) == 0
        assert np.array_equal(host(lp.t["ids"]), final[0])
        assert np.array_equal(host(lp.t["steps"]), final[1])
        assert np.array_equal(host(lp.t["commit_step"]), final[2])
        assert np.all(host(lp.t["n_masked"]) == 0)


def test_graph_loop_changes_block_index_without_rebuild(tt):
    """Block index / seed enter through the workspace: successive blocks differ as the oracle says."""
    w = synth.TINY
    lp = Loop(tt, w, seed=5, block=0)
    outs = []
    for block in (0, 1, 0):
        lp.desc.logits.block_index = block
        lp.block = block
        lp.reset()
        tt.tt_denoise_block_loop(lp.desc, lp.ts, lp.ws)
        torch.cuda.synchronize()
        ids = host(lp.t["ids"]).copy()
        outs.append(ids)
        r = oracle.denoise_block(w.S, w.steps_max, w.mask_id, w.gamma,
                                 lambda step, pos: lp.logits_fn(0, step, pos))
        amb = any(np.any(np.abs(tr["conf"][tr["ids_before"] == w.mask_id] - w.gamma) <= 1e-5)
                  for tr in r["trace"])
        if not amb:
            assert np.array_equal(ids[0], r["ids"])
            assert host(lp.t["steps"])[0] == r["steps"]
    assert np.array_equal(outs[0], outs[2])
    assert not np.array_equal(outs[0], outs[1])
