"""tt_denoise_attn against the fp64 oracle: contiguous and paged caches, GQA packing,
ragged tails, several row tiles and KV tiles, split invariance, empty contexts."""
import math

import numpy as np
import pytest
import torch

import oracle
from block_wise_mask_tt_b300 import synth
from gpu_util import bf16_to_f64, check_attention, check_guards, dev, guarded, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tt():
    from block_wise_mask_tt_b300 import tt as _tt
    return _tt


def run_attn(tt, w, inp, num_splits=0):
    B, S, Hq, Hkv, D = w.B, w.S, w.Hq, w.Hkv, w.D
    if w.paged:
        kp, vp = inp["k_pages"], inp["v_pages"]
        dims = tt.attn_dims(B, S, Hq, Hkv, D, 0, w.page_size, inp["page_table"].shape[1], kp.shape[0],
                            w.softmax_scale, num_splits)
        kc, vc, pt = dev(kp), dev(vp), dev(inp["page_table"])
    else:
        L = inp["k_ctx"].shape[1]
        dims = tt.attn_dims(B, S, Hq, Hkv, D, L, 0, 0, 0, w.softmax_scale, num_splits)
        kc = dev(inp["k_ctx"]) if L else None
        vc = dev(inp["v_ctx"]) if L else None
        pt = None
    # outputs between canaries (bf16 NaN pattern / NaN) that must come back untouched
    g_out, out = guarded(B * S * Hq * D, torch.int16, 0x7FC0)
    g_lse, lse = guarded(B * S * Hq, torch.float32, float("nan"))
    tt.tt_denoise_attn(dims, dev(inp["q"]), dev(inp["k_blk"]), dev(inp["v_blk"]), kc, vc, pt,
                       dev(inp["ctx_len"]), out, lse)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    check_guards(g_out, 0x7FC0, "out")
    check_guards(g_lse, float("nan"), "lse")
    return (bf16_to_f64(host(out)).reshape(B, S, Hq, D),
            host(lse).astype(np.float64).reshape(B, S, Hq))


def W(**kw):
    base = dict(name="t", B=1, L=256, S=16, Hq=4, Hkv=1, D=64, H=256, V=1024)
    base.update(kw)
    return synth.Workload(**base)


CASES = {
    "c0_shape": W(softmax_scale=1 / 8.0, qkv_fp32_source=True),
    "g16_d128_L300": W(B=2, L=300, Hq=32, Hkv=2, D=128, q_prescale=1 / math.sqrt(128)),
    "g16_d128_s32_ragged": W(B=3, L=200, L_min=1, S=32, Hq=32, Hkv=2, D=128, q_prescale=1 / math.sqrt(128)),
    "g4_d64_L1000": W(B=2, L=1000, S=16, Hq=8, Hkv=2, D=64, softmax_scale=0.125),
    "g12_d128_s13": W(B=2, L=130, S=13, Hq=24, Hkv=2, D=128, softmax_scale=0.09),
    "g1_d64_s1": W(B=3, L=70, S=1, Hq=2, Hkv=2, D=64, softmax_scale=0.125),
    "g32_d64_s16": W(B=1, L=513, S=16, Hq=32, Hkv=1, D=64, softmax_scale=0.125),
    "paged_g16_s32": W(B=4, L=700, L_min=1, S=32, Hq=32, Hkv=2, D=128, paged=True,
                       q_prescale=1 / math.sqrt(128)),
    "paged_g4_d64": W(B=3, L=300, L_min=1, S=16, Hq=8, Hkv=2, D=64, paged=True, softmax_scale=0.125),
    "empty_ctx": W(B=2, L=0, S=16, Hq=32, Hkv=2, D=128, q_prescale=1 / math.sqrt(128)),
    "large_logits": W(B=1, L=640, S=16, Hq=16, Hkv=1, D=128, softmax_scale=1.0, qkv_std=2.5),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_attention_matches_oracle(tt, name):
    w = CASES[name]
    inp = synth.make_attention_inputs(w, seed=len(name))
    O, lse = run_attn(tt, w, inp)
    Or, lr = oracle.denoise_attention(inp, w.softmax_scale)
    check_attention(O, Or, lse, lr, what=name, out_rounding=w.qkv_std > 1.0)


def test_context_length_zero_for_some_sequences(tt):
    w = W(B=3, L=256, S=16, Hq=32, Hkv=2, D=128, q_prescale=1 / math.sqrt(128))
    inp = synth.make_attention_inputs(w, seed=3, ctx_len=np.array([0, 256, 65], np.int32))
    O, lse = run_attn(tt, w, inp)
    Or, lr = oracle.denoise_attention(inp, w.softmax_scale)
    check_attention(O, Or, lse, lr)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 0])
def test_split_invariance(tt, splits):
    w = W(B=2, L=1024, S=16, Hq=32, Hkv=2, D=128, q_prescale=1 / math.sqrt(128))
    inp = synth.make_attention_inputs(w, seed=11)
    O, lse = run_attn(tt, w, inp, num_splits=splits)
    Or, lr = oracle.denoise_attention(inp, w.softmax_scale)
    check_attention(O, Or, lse, lr, what=f"splits={splits}")


@pytest.mark.parametrize("splits", [0, 3, 7])
def test_ragged_paged_longest_first(tt, splits):
    """A ragged paged batch of more work units than SMs: the units are dispatched
    longest first from a device-side sort (empty splits of short sequences left out);
    with 7 splits the combine pass merges them, with 3 the split CTAs' partials too."""
    w = W(B=40, L=700, L_min=1, S=16, Hq=8, Hkv=2, D=64, paged=True, softmax_scale=0.125)
    inp = synth.make_attention_inputs(w, seed=15)
    O, lse = run_attn(tt, w, inp, num_splits=splits)
    Or, lr = oracle.denoise_attention(inp, w.softmax_scale)
    check_attention(O, Or, lse, lr, what=f"splits={splits}")


@pytest.mark.parametrize("n_long", [0, 4])
def test_ragged_paged_split_chosen_per_call(tt, n_long):
    """More row groups than SMs in a ragged paged batch: the prep kernel chooses the
    split length from the sequences' actual lengths.  All short: every row group in one
    split, written directly.  Four long ones among 76 short: the long ones are cut into
    64-tile units and merged by the combine pass, the short ones still written directly."""
    w = W(B=80, L=16384, L_min=1, S=16, Hq=4, Hkv=2, D=64, paged=True, softmax_scale=0.125)
    rng = np.random.default_rng(21 + n_long)
    ctx = rng.integers(200, 700, size=w.B).astype(np.int32)
    ctx[rng.choice(w.B, size=n_long, replace=False)] = rng.integers(14000, 16385, size=n_long)
    inp = synth.make_attention_inputs(w, seed=16, ctx_len=ctx)
    O, lse = run_attn(tt, w, inp)
    Or, lr = oracle.denoise_attention(inp, w.softmax_scale)
    check_attention(O, Or, lse, lr, what=f"{n_long} long sequences")


def test_small_ragged_batch_in_128_row_groups(tt):
    """Short contexts over many sequences: a few tile-rounds per SM in all, so each CTA
    serves one 128-row tile (here R = 256 rows per kv head, two groups), and with more
    row groups than SMs the prep kernel orders them and picks the split length."""
    w = W(B=100, L=512, L_min=64, S=16, Hq=32, Hkv=2, D=64, paged=True, softmax_scale=0.125)
    inp = synth.make_attention_inputs(w, seed=17)
    O, lse = run_attn(tt, w, inp)
    Or, lr = oracle.denoise_attention(inp, w.softmax_scale)
    check_attention(O, Or, lse, lr, what="128-row groups")


def test_ragged_batch_beyond_the_order_kernels_tile_cache(tt):
    """More row-group items (4100 sequences x 1 kv head x 1 group) than the prep kernel
    keeps tile counts for in shared memory (4096): its two passes over the units then
    read ctx_len from global memory.  One-tile contexts of 1..128 tokens, S = 1."""
    w = W(B=4100, L=128, L_min=1, S=1, Hq=1, Hkv=1, D=64, paged=True, softmax_scale=0.125)
    inp = synth.make_attention_inputs(w, seed=23)
    O, lse = run_attn(tt, w, inp)
    Or, lr = oracle.denoise_attention(inp, w.softmax_scale)
    check_attention(O, Or, lse, lr, what="4100 one-tile sequences")


@pytest.mark.parametrize("splits", [2, 5, 16])
def test_fused_combine_option(tt, splits, monkeypatch):
    """With TT_ATTN_FUSED_COMBINE=1 the split CTAs of a contiguous call that fits one
    wave merge their row groups themselves (counters in the workspace, left at zero):
    three calls on one workspace, a ragged batch with some sequences shorter than one
    split, each against the oracle."""
    monkeypatch.setenv("TT_ATTN_FUSED_COMBINE", "1")
    w = W(B=3, L=2600, L_min=100, S=16, Hq=32, Hkv=2, D=128, q_prescale=1 / math.sqrt(128))
    inp = synth.make_attention_inputs(w, seed=18)
    L = inp["k_ctx"].shape[1]
    dims = tt.attn_dims(w.B, w.S, w.Hq, w.Hkv, w.D, L, 0, 0, 0, w.softmax_scale, splits)
    ws = tt.workspace(tt.tt_denoise_attn_workspace(dims))
    Or, lr = oracle.denoise_attention(inp, w.softmax_scale)
    args = [dev(inp[k]) for k in ("q", "k_blk", "v_blk", "k_ctx", "v_ctx")]
    cl = dev(inp["ctx_len"])
    for call in range(3):
        g_out, out = guarded(w.B * w.S * w.Hq * w.D, torch.int16, 0x7FC0)
        g_lse, lse = guarded(w.B * w.S * w.Hq, torch.float32, float("nan"))
        tt.tt_denoise_attn(dims, *args, None, cl, out, lse, ws=ws)
        torch.cuda.synchronize()
        assert tt.tt_device_status(True) == 0
        check_guards(g_out, 0x7FC0, "out")
        check_guards(g_lse, float("nan"), "lse")
        O = bf16_to_f64(host(out)).reshape(w.B, w.S, w.Hq, w.D)
        check_attention(O, Or, host(lse).astype(np.float64).reshape(w.B, w.S, w.Hq), lr,
                        what=f"fused combine, {splits} splits, call {call}")


def test_paged_equals_contiguous(tt):
    w = W(B=3, L=500, L_min=1, S=16, Hq=32, Hkv=2, D=128, paged=True, q_prescale=1 / math.sqrt(128))
    inp = synth.make_attention_inputs(w, seed=12)
    Op, lp = run_attn(tt, w, inp, num_splits=2)
    L = 512
    kc = np.zeros((w.B, L, w.Hkv, w.D), np.uint16)
    vc = np.zeros((w.B, L, w.Hkv, w.D), np.uint16)
    for b in range(w.B):
        n = int(inp["ctx_len"][b])
        t = np.arange(n)
        kc[b, :n] = inp["k_pages"][inp["page_table"][b, t // 64], t % 64]
        vc[b, :n] = inp["v_pages"][inp["page_table"][b, t // 64], t % 64]
    inp_c = dict(q=inp["q"], k_blk=inp["k_blk"], v_blk=inp["v_blk"], ctx_len=inp["ctx_len"], k_ctx=kc,
                 v_ctx=vc)
    Oc, lc = run_attn(tt, w.replace(paged=False), inp_c, num_splits=2)
    np.testing.assert_array_equal(Op, Oc)
    np.testing.assert_array_equal(lp, lc)


def test_block_permutation_equivariance(tt):
    w = W(B=1, L=256, S=16, Hq=32, Hkv=2, D=128, q_prescale=1 / math.sqrt(128))
    inp = synth.make_attention_inputs(w, seed=13)
    O, _ = run_attn(tt, w, inp)
    perm = np.random.default_rng(0).permutation(16)
    inp2 = dict(inp)
    for k in ("q", "k_blk", "v_blk"):
        inp2[k] = np.ascontiguousarray(inp[k][:, perm])
    O2, _ = run_attn(tt, w, inp2)
    np.testing.assert_allclose(O2, O[:, perm], atol=2e-2, rtol=0)


@pytest.mark.parametrize("splits", [0, 2, 6])
def test_bad_page_id_is_reported(tt, splits):
    """A page id outside the pool sets the error word and skips that sequence's
    context, whether the CTA writes the output itself, merges the splits itself (2) or
    leaves them to the combine pass (6); the other sequence is unaffected."""
    w = W(B=2, L=700, L_min=1, S=16, Hq=8, Hkv=2, D=64, paged=True, softmax_scale=0.125)
    inp = synth.make_attention_inputs(w, seed=14, ctx_len=np.array([650, 700], np.int32))
    inp["page_table"][1, 0] = 10 ** 6
    kp = inp["k_pages"]
    dims = tt.attn_dims(w.B, w.S, w.Hq, w.Hkv, w.D, 0, 64, inp["page_table"].shape[1], kp.shape[0],
                        w.softmax_scale, splits)
    out = torch.zeros((w.B, w.S, w.Hq, w.D), dtype=torch.int16, device="cuda")
    assert tt.tt_device_status(True) == 0
    tt.tt_denoise_attn(dims, dev(inp["q"]), dev(inp["k_blk"]), dev(inp["v_blk"]), dev(kp),
                       dev(inp["v_pages"]), dev(inp["page_table"]), dev(inp["ctx_len"]), out)
    assert tt.tt_device_status(True) == tt.TT_ERR_DEVICE
    # sequence 0 is unaffected
    Or, _ = oracle.denoise_attention({k: (v[:1] if k in ("q", "k_blk", "v_blk", "ctx_len", "page_table")
                                          else v) for k, v in inp.items()}, w.softmax_scale)
    check_attention(bf16_to_f64(host(out))[:1], Or)
