"""tt_qkv_project and the step with the projection on (qkv_proj = 1) against the oracle.

The kernel accumulates each output in fp32 over H products (added into the
accumulator in 16-wide slices) and rounds it to bf16 once, so it may differ from the
exact fp64 value by one bf16 ulp of that value (the rounding, and a rounding boundary
crossed by the accumulation error) plus delta = (H/16 + 16) 2^-24 sum_k |y_k W_ck|.

In the step, every tt_denoise_step is checked against the oracle from the GPU's own
inputs (teacher forcing): the adaLN output y; q, k_blk, v_blk against the projection
of that y; the attention output against the oracle attention over the GPU's q, k_blk,
v_blk and the context cache; the unmask decision against the oracle on the stand-in
logits.  Then the block graph must reproduce the step-by-step result bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from block_wise_mask_tt_b300 import synth
from gpu_util import (adaln_tol, bf16_to_f64, bf16_ulp, check_attention, compare_unmask, dev, host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tt():
    from block_wise_mask_tt_b300 import tt as _tt
    return _tt


def _abs_bound(y_bits, W_bits):
    ya = np.abs(bf16_to_f64(y_bits)).reshape(-1, y_bits.shape[-1])
    Wa = np.abs(bf16_to_f64(W_bits))
    return ya @ Wa.T


def check_qkv(y, W, q, k, v, Hq, Hkv, D, what=""):
    B, S, H = y.shape
    rq, rk, rv = oracle.qkv_projection(y, W, Hq, Hkv, D)
    bound = ((H / 16 + 16) * 2.0 ** -24) * _abs_bound(y, W)
    got = np.concatenate([bf16_to_f64(q).reshape(B * S, -1), bf16_to_f64(k).reshape(B * S, -1),
                          bf16_to_f64(v).reshape(B * S, -1)], axis=1)
    ref = np.concatenate([rq.reshape(B * S, -1), rk.reshape(B * S, -1), rv.reshape(B * S, -1)], axis=1)
    err = np.abs(got - ref)
    tol = bf16_ulp(ref) + bound
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} entries off, worst excess {(err - tol).max()}"


CASES = [
    # (B, S, H, Hq, Hkv, D): one and several 128-row tiles, a partial 64-slice of H,
    # column segments of 64 and 128 lanes, and 74 / 75 single-unit work items (half the
    # SMs of the part and one more)
    (1, 16, 2688, 32, 2, 128),
    (3, 16, 256, 4, 1, 64),
    (20, 16, 200, 8, 2, 64),
    (1, 8, 512, 72, 1, 64),
    (1, 8, 512, 73, 1, 64),
    (9, 32, 512, 16, 4, 128),
    (1, 1, 64, 1, 1, 64),
]


@pytest.mark.parametrize("B,S,H,Hq,Hkv,D", CASES)
def test_qkv_project_matches_oracle(tt, B, S, H, Hq, Hkv, D):
    w = synth.Workload("qkv", B=B, L=0, S=S, Hq=Hq, Hkv=Hkv, D=D, H=H, V=64)
    y = synth.make_hidden(w, B + H)
    W = synth.make_qkv_weights(w, D + S)
    q = torch.full((B, S, Hq, D), -1, dtype=torch.int16, device="cuda")
    k = torch.full((B, S, Hkv, D), -1, dtype=torch.int16, device="cuda")
    v = torch.full((B, S, Hkv, D), -1, dtype=torch.int16, device="cuda")
    tt.tt_qkv_project(dev(y), dev(W), q, k, v, B, S, H, Hq, Hkv, D)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    check_qkv(y, W, host(q), host(k), host(v), Hq, Hkv, D, what=str((B, S, H, Hq, Hkv, D)))


def test_qkv_rejects_bad_arguments(tt):
    def z(*shape):
        return torch.zeros(shape, dtype=torch.int16, device="cuda")
    y = z(1, 4, 64)
    with pytest.raises(tt.TTError):  # D = 32
        tt.tt_qkv_project(y, z(3 * 32, 64), z(1, 4, 1, 32), z(1, 4, 1, 32), z(1, 4, 1, 32), 1, 4, 64, 1, 1, 32)
    with pytest.raises(tt.TTError):  # Hkv does not divide Hq
        tt.tt_qkv_project(y, z(7 * 64, 64), z(1, 4, 3, 64), z(1, 4, 2, 64), z(1, 4, 2, 64), 1, 4, 64, 3, 2, 64)
    with pytest.raises(tt.TTError):  # H below 64
        tt.tt_qkv_project(z(1, 4, 32), z(3 * 64, 32), z(1, 4, 1, 64), z(1, 4, 1, 64), z(1, 4, 1, 64), 1, 4, 32, 1, 1, 64)


STEP_CASES = {
    "tiny_B2": synth.TINY.replace(B=2),
    "single_B2_L512": synth.SINGLE.replace(B=2, L=512, V=8192, softmax_scale=1.0 / 128 ** 0.5,
                                               q_prescale=1.0),
}


@pytest.mark.parametrize("name", sorted(STEP_CASES))
def test_step_and_loop_with_projection(tt, name):
    w = STEP_CASES[name]
    seed, block = 4, 1
    B, S, T, mask = w.B, w.S, w.steps_max, w.mask_id
    inp = synth.make_attention_inputs(w, seed)
    ad = synth.make_adaln_inputs(w, seed)
    W = synth.make_qkv_weights(w, seed)
    dims = tt.attn_dims(B, S, w.Hq, w.Hkv, w.D, inp["k_ctx"].shape[1], 0, 0, 0, w.softmax_scale, 0)
    desc = tt.step_desc(dims, w.H, w.V, mask, w.gamma, T, w.ln_eps, seed, block, w.logits_kind, w.boost_lo,
                        w.boost_hi, qkv_proj=True)
    t = dict(x=dev(ad["x"]), shift_table=dev(ad["shift_table"]), scale_table=dev(ad["scale_table"]),
             q=torch.zeros((B, S, w.Hq, w.D), dtype=torch.int16, device="cuda"),
             k_blk=torch.zeros((B, S, w.Hkv, w.D), dtype=torch.int16, device="cuda"),
             v_blk=torch.zeros((B, S, w.Hkv, w.D), dtype=torch.int16, device="cuda"),
             k_ctx=dev(inp["k_ctx"]), v_ctx=dev(inp["v_ctx"]), ctx_len=dev(inp["ctx_len"]),
             ids=torch.full((B, S), mask, dtype=torch.int32, device="cuda"),
             n_masked=torch.full((B,), S, dtype=torch.int32, device="cuda"),
             steps=torch.zeros(B, dtype=torch.int32, device="cuda"),
             commit_step=torch.zeros((B, S), dtype=torch.uint8, device="cuda"),
             y=torch.zeros((B, S, w.H), dtype=torch.int16, device="cuda"),
             attn_out=torch.zeros((B, S, w.Hq, w.D), dtype=torch.int16, device="cuda"),
             logits=torch.zeros((B, S, w.V), dtype=torch.float32, device="cuda"),
             conf=torch.zeros((B, S), dtype=torch.float32, device="cuda"),
             commit=torch.zeros((B, S), dtype=torch.uint8, device="cuda"),
             w_qkv=dev(W))
    ts = tt.step_tensors(**t)
    ws = tt.workspace(tt.tt_denoise_workspace(desc))

    def logits_fn(b, step, pos):
        return synth.logits_rows(seed, b, block, step, pos, w.V, mask, w.logits_kind, w.boost_lo, w.boost_hi)

    excluded = 0
    for kstep in range(T + 1):
        ids0, steps0, cs0 = host(t["ids"]).copy(), host(t["steps"]).copy(), host(t["commit_step"]).copy()
        nm0 = (ids0 == mask).sum(axis=1)
        if not np.any(nm0 > 0):
            break
        tt.tt_denoise_step(desc, ts, ws)
        torch.cuda.synchronize()
        assert tt.tt_device_status(True) == 0
        active = nm0 > 0
        y = host(t["y"])
        for b in np.flatnonzero(active):
            ref = oracle.adaln_modulate(ad["x"][b], ad["shift_table"][nm0[b]], ad["scale_table"][nm0[b]], w.ln_eps)
            sh = np.broadcast_to(ad["shift_table"][nm0[b]], ref.shape)
            assert np.all(np.abs(bf16_to_f64(y[b]) - ref) <= adaln_tol(ref, sh))
        q, kb, vb = host(t["q"]), host(t["k_blk"]), host(t["v_blk"])
        act = np.flatnonzero(active)
        check_qkv(y[act], W, q[act], kb[act], vb[act], w.Hq, w.Hkv, w.D, what=f"{name} step {kstep}")
        cur = dict(q=q[act], k_blk=kb[act], v_blk=vb[act], ctx_len=inp["ctx_len"][act],
                   k_ctx=inp["k_ctx"][act], v_ctx=inp["v_ctx"][act])
        O_ref, _ = oracle.denoise_attention(cur, w.softmax_scale)
        check_attention(bf16_to_f64(host(t["attn_out"]))[act], O_ref, what=f"{name} step {kstep}")
        logits = np.zeros((B, S, w.V), np.float32)
        for b in act:
            pos = np.flatnonzero(ids0[b] == mask)
            logits[b, pos] = logits_fn(b, int(steps0[b]), pos)
        ora = [oracle.unmask_step(logits[b], ids0[b], int(steps0[b]), mask, w.gamma, T, cs0[b]) for b in range(B)]
        gpu = dict(ids=host(t["ids"]), steps=host(t["steps"]), n_masked=host(t["n_masked"]),
                   conf=host(t["conf"]), commit=host(t["commit"]), commit_step=host(t["commit_step"]))
        for b in np.flatnonzero(~active):  # finished sequences are left alone by the step
            gpu["conf"][b] = 0.0
            gpu["commit"][b] = 0
        excluded += compare_unmask(gpu, ora, ids0, steps0, mask, w.gamma, what=f"{name} step {kstep}")
    final = (host(t["ids"]).copy(), host(t["steps"]).copy(), host(t["commit_step"]).copy())
    assert np.all(final[0] != mask)
    t["ids"].fill_(mask)
    t["n_masked"].fill_(S)
    t["steps"].zero_()
    t["commit_step"].zero_()
    tt.tt_denoise_block_loop(desc, ts, ws)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    assert np.array_equal(host(t["ids"]), final[0])
    assert np.array_equal(host(t["steps"]), final[1])
    assert np.array_equal(host(t["commit_step"]), final[2])
