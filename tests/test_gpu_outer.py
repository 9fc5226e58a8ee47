"""Algorithm 1's outer loop on the GPU against the oracle: the block append into a
contiguous or paged cache with its stop rules, and tt_generate over several blocks
(tokens, cache lengths, stops, and the attention of the last block over the grown
cache)."""

import numpy as np
import pytest
import torch

import oracle
import pins
from block_wise_mask_tt_b300 import synth
from gpu_util import bf16_to_f64, check_attention, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tt():
    from block_wise_mask_tt_b300 import tt as _tt
    return _tt


@pytest.mark.parametrize("paged", [False, True])
def test_append_block_matches_oracle(tt, paged):
    cache, base, lens, cap = pins._append_case(21 + paged, paged, D=64)
    B, S, Hkv, D = base["k_blk"].shape
    ids = np.array([[1, 2, 3], [4, 99, 6], [7, 8, 9]], np.int32)
    gen0 = np.array([0, 0, 3], np.int32)
    done0 = np.array([0, 0, 0], np.uint8)
    want = oracle.append_block(cache, base["k_blk"], base["v_blk"], lens, ids, 99, 6, gen0, done0)
    if paged:
        pt = cache["page_table"]
        dims = tt.attn_dims(B, S, 4, Hkv, D, 0, 64, pt.shape[1], cache["k_pages"].shape[0], 1.0, 0)
        kc, vc, ptd = dev(cache["k_pages"]), dev(cache["v_pages"]), dev(pt.astype(np.int32))
    else:
        dims = tt.attn_dims(B, S, 4, Hkv, D, cap, 0, 0, 0, 1.0, 0)
        kc, vc, ptd = dev(cache["k_ctx"]), dev(cache["v_ctx"]), None
    ctx = dev(lens.astype(np.int32))
    gen = dev(gen0)
    done = dev(done0)
    out = torch.full((B, 8), -7, dtype=torch.int32, device="cuda")
    stop = tt.tt_stop_spec(99, 0, 6)
    tt.tt_append_block(dims, dev(base["k_blk"]), dev(base["v_blk"]), kc, vc, ptd, ctx, dev(ids), stop,
                       gen, done, out, 8, 2)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    assert host(ctx).tolist() == want["ctx_len"].tolist()
    assert host(gen).tolist() == want["generated"].tolist()
    assert host(done).tolist() == want["done"].tolist()
    o = host(out)
    assert np.array_equal(o[:, 2:5], ids) and np.all(o[:, :2] == -7) and np.all(o[:, 5:] == -7)
    if paged:
        assert np.array_equal(host(kc), want["k_pages"]) and np.array_equal(host(vc), want["v_pages"])
    else:
        assert np.array_equal(host(kc), want["k_ctx"]) and np.array_equal(host(vc), want["v_ctx"])
    # a second call leaves the finished sequences alone and pads their tokens
    want2 = oracle.append_block({k: want[k] for k in cache}, base["k_blk"], base["v_blk"], want["ctx_len"],
                                ids, 99, 100, want["generated"], want["done"])
    tt.tt_append_block(dims, dev(base["k_blk"]), dev(base["v_blk"]), kc, vc, ptd, ctx, dev(ids),
                       tt.tt_stop_spec(99, 5, 100), gen, done, out, 8, 5)
    torch.cuda.synchronize()
    assert host(ctx).tolist() == want2["ctx_len"].tolist()
    assert host(out)[1, 5:8].tolist() == [5, 5, 5] and host(out)[2, 5:8].tolist() == [5, 5, 5]
    key = "k_pages" if paged else "k_ctx"
    assert np.array_equal(host(kc), want2[key])


def test_append_block_rejects_rows_that_do_not_fit(tt):
    cache, base, lens, cap = pins._append_case(5, False, D=64)
    B, S, Hkv, D = base["k_blk"].shape
    dims = tt.attn_dims(B, S, 4, Hkv, D, cap, 0, 0, 0, 1.0, 0)
    ctx = dev(np.array([cap - 1, 0, 0], np.int32))  # sequence 0 has one free row
    kc = dev(cache["k_ctx"])
    before = host(kc).copy()
    gen, done = dev(np.zeros(B, np.int32)), dev(np.zeros(B, np.uint8))
    assert tt.tt_device_status(True) == 0
    tt.tt_append_block(dims, dev(base["k_blk"]), dev(base["v_blk"]), kc, dev(cache["v_ctx"]), None, ctx,
                       dev(np.ones((B, S), np.int32)), tt.tt_stop_spec(-1, 0, 100), gen, done)
    assert tt.tt_device_status(True) == tt.TT_ERR_DEVICE
    after = host(kc)
    assert np.array_equal(after[0], before[0])          # nothing written for sequence 0
    assert host(ctx).tolist() == [cap - 1, S, S]        # the others were appended


def test_generate_matches_oracle(tt):
    B, S, Hq, Hkv, D, V, mask, T = 3, 16, 8, 2, 64, 1024, 3, 16
    n_blocks, lens = 3, np.array([200, 64, 130], np.int32)
    cap = int(lens.max()) + n_blocks * S
    w = synth.Workload("gen", B=B, L=int(lens.max()), S=S, Hq=Hq, Hkv=Hkv, D=D, H=64, V=V, T=T,
                       softmax_scale=0.125, boost_lo=0.0, boost_hi=12.0)
    inp = synth.make_attention_inputs(w, 8, ctx_len=lens)
    ad = synth.make_adaln_inputs(w, 8)
    kc = np.zeros((B, cap, Hkv, D), np.uint16)
    vc = np.zeros((B, cap, Hkv, D), np.uint16)
    kc[:, :inp["k_ctx"].shape[1]] = inp["k_ctx"]
    vc[:, :inp["v_ctx"].shape[1]] = inp["v_ctx"]

    def fn(b, blk, step, pos):
        return synth.logits_rows(8, b, blk, step, pos, V, mask, w.logits_kind, w.boost_lo, w.boost_hi)
    # an EOS id that sequence 2 commits in its first block; everyone stops after 2 blocks
    first = oracle.generate(B, S, T, mask, w.gamma, 1, fn, eos_id=-1, pad_id=0, max_new=10**6)
    eos = int(first["tokens"][2, 5])
    want = oracle.generate(B, S, T, mask, w.gamma, n_blocks, fn, eos_id=eos, pad_id=0, max_new=2 * S)

    dims = tt.attn_dims(B, S, Hq, Hkv, D, cap, 0, 0, 0, w.softmax_scale, 0)
    desc = tt.step_desc(dims, w.H, V, mask, w.gamma, T, w.ln_eps, 8, 0, w.logits_kind, w.boost_lo, w.boost_hi)
    t = dict(x=dev(ad["x"]), shift_table=dev(ad["shift_table"]), scale_table=dev(ad["scale_table"]),
             q=dev(inp["q"]), k_blk=dev(inp["k_blk"]), v_blk=dev(inp["v_blk"]), k_ctx=dev(kc), v_ctx=dev(vc),
             ctx_len=dev(lens), ids=torch.zeros((B, S), dtype=torch.int32, device="cuda"),
             n_masked=torch.zeros(B, dtype=torch.int32, device="cuda"),
             steps=torch.zeros(B, dtype=torch.int32, device="cuda"),
             commit_step=torch.zeros((B, S), dtype=torch.uint8, device="cuda"),
             y=torch.zeros((B, S, w.H), dtype=torch.int16, device="cuda"),
             attn_out=torch.zeros((B, S, Hq, D), dtype=torch.int16, device="cuda"),
             logits=torch.zeros((B, S, V), dtype=torch.float32, device="cuda"))
    ws = tt.workspace(tt.tt_denoise_workspace(desc))
    gen = torch.zeros(B, dtype=torch.int32, device="cuda")
    done = torch.zeros(B, dtype=torch.uint8, device="cuda")
    out = torch.full((B, n_blocks * S), -1, dtype=torch.int32, device="cuda")
    tt.tt_generate(desc, tt.step_tensors(**t), n_blocks, tt.tt_stop_spec(eos, 0, 2 * S), gen, done, out, ws)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    excluded = [b for b in range(B) if any(
        np.any(np.abs(tr["conf"][tr["ids_before"] == mask] - w.gamma) <= 1e-5)
        for k in range(n_blocks)
        for tr in oracle.denoise_block(S, T, mask, w.gamma, lambda st, pos: fn(b, k, st, pos))["trace"])]
    for b in range(B):
        if b not in excluded:
            assert np.array_equal(host(out)[b], want["tokens"][b]), b
    assert host(gen).tolist() == want["generated"].tolist()
    assert host(done).tolist() == want["done"].tolist()
    blocks_run = (want["generated"] // S).astype(np.int32)
    assert host(t["ctx_len"]).tolist() == (lens + S * blocks_run).tolist()
    # the last block a sequence decoded attended over its cache grown by the blocks before it
    for b in range(B):
        k_last = int(blocks_run[b]) - 1
        cur = dict(q=inp["q"][b:b + 1], k_blk=inp["k_blk"][b:b + 1], v_blk=inp["v_blk"][b:b + 1],
                   ctx_len=np.array([lens[b] + S * k_last], np.int32),
                   k_ctx=np.concatenate([kc[b:b + 1, :lens[b]]] + [inp["k_blk"][b:b + 1]] * k_last, 1),
                   v_ctx=np.concatenate([vc[b:b + 1, :lens[b]]] + [inp["v_blk"][b:b + 1]] * k_last, 1))
        ref, _ = oracle.denoise_attention(cur, w.softmax_scale)
        # later blocks skip a finished sequence, so its output is from its own last block
        check_attention(bf16_to_f64(host(t["attn_out"]))[b:b + 1], ref, what=f"seq {b}")


def test_generate_paged_matches_oracle(tt):
    """Outer loop over a paged cache: the blocks are appended into pages the table
    already names (shuffled, with spare pages for the growth)."""
    B, S, Hq, Hkv, D, V, mask, T = 3, 16, 8, 2, 64, 1024, 3, 16
    n_blocks, lens = 3, np.array([100, 64, 150], np.int32)
    cap = int(lens.max()) + n_blocks * S
    w = synth.Workload("genp", B=B, L=int(lens.max()), S=S, Hq=Hq, Hkv=Hkv, D=D, H=64, V=V, T=T,
                       softmax_scale=0.125, boost_lo=0.0, boost_hi=12.0)
    inp = synth.make_attention_inputs(w, 9, ctx_len=lens)
    ad = synth.make_adaln_inputs(w, 9)
    per_seq = (cap + 63) // 64
    n_pages = B * per_seq + 2  # two pages nobody uses
    perm = np.random.default_rng(4).permutation(n_pages)[:B * per_seq].reshape(B, per_seq).astype(np.int32)
    kp = np.zeros((n_pages, 64, Hkv, D), np.uint16)
    vp = np.zeros((n_pages, 64, Hkv, D), np.uint16)
    for b in range(B):
        for t_ in range(int(lens[b])):
            kp[perm[b, t_ // 64], t_ % 64] = inp["k_ctx"][b, t_]
            vp[perm[b, t_ // 64], t_ % 64] = inp["v_ctx"][b, t_]

    def fn(b, blk, step, pos):
        return synth.logits_rows(9, b, blk, step, pos, V, mask, w.logits_kind, w.boost_lo, w.boost_hi)
    want = oracle.generate(B, S, T, mask, w.gamma, n_blocks, fn, eos_id=-1, pad_id=0, max_new=n_blocks * S)

    dims = tt.attn_dims(B, S, Hq, Hkv, D, 0, 64, per_seq, n_pages, w.softmax_scale, 0)
    desc = tt.step_desc(dims, w.H, V, mask, w.gamma, T, w.ln_eps, 9, 0, w.logits_kind, w.boost_lo, w.boost_hi)
    t = dict(x=dev(ad["x"]), shift_table=dev(ad["shift_table"]), scale_table=dev(ad["scale_table"]),
             q=dev(inp["q"]), k_blk=dev(inp["k_blk"]), v_blk=dev(inp["v_blk"]), k_ctx=dev(kp), v_ctx=dev(vp),
             page_table=dev(perm), ctx_len=dev(lens),
             ids=torch.zeros((B, S), dtype=torch.int32, device="cuda"),
             n_masked=torch.zeros(B, dtype=torch.int32, device="cuda"),
             steps=torch.zeros(B, dtype=torch.int32, device="cuda"),
             commit_step=torch.zeros((B, S), dtype=torch.uint8, device="cuda"),
             y=torch.zeros((B, S, w.H), dtype=torch.int16, device="cuda"),
             attn_out=torch.zeros((B, S, Hq, D), dtype=torch.int16, device="cuda"),
             logits=torch.zeros((B, S, V), dtype=torch.float32, device="cuda"))
    ws = tt.workspace(tt.tt_denoise_workspace(desc))
    gen = torch.zeros(B, dtype=torch.int32, device="cuda")
    done = torch.zeros(B, dtype=torch.uint8, device="cuda")
    out = torch.full((B, n_blocks * S), -1, dtype=torch.int32, device="cuda")
    tt.tt_generate(desc, tt.step_tensors(**t), n_blocks, tt.tt_stop_spec(-1, 0, n_blocks * S), gen, done, out, ws)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    excluded = [b for b in range(B) if any(
        np.any(np.abs(tr["conf"][tr["ids_before"] == mask] - w.gamma) <= 1e-5)
        for k in range(n_blocks)
        for tr in oracle.denoise_block(S, T, mask, w.gamma, lambda st, pos: fn(b, k, st, pos))["trace"])]
    for b in range(B):
        if b not in excluded:
            assert np.array_equal(host(out)[b], want["tokens"][b]), b
    assert host(t["ctx_len"]).tolist() == (lens + n_blocks * S).tolist()
    assert host(gen).tolist() == want["generated"].tolist() == [n_blocks * S] * B
    assert host(done).tolist() == want["done"].tolist()  # the length limit was reached
    # the appended rows sit in the named pages; the spare pages are untouched
    kph = host(t["k_ctx"])
    for b in range(B):
        for k in range(n_blocks):
            for s in range(S):
                pos = int(lens[b]) + k * S + s
                assert np.array_equal(kph[perm[b, pos // 64], pos % 64], inp["k_blk"][b, s])
    spare = sorted(set(range(n_pages)) - set(perm.reshape(-1).tolist()))
    assert np.all(kph[spare] == 0)
    # the last block attended over the paged cache grown by the blocks before it
    last = n_blocks - 1
    for b in range(B):
        kc = np.concatenate([inp["k_ctx"][b:b + 1, :lens[b]]] + [inp["k_blk"][b:b + 1]] * last, 1)
        vc = np.concatenate([inp["v_ctx"][b:b + 1, :lens[b]]] + [inp["v_blk"][b:b + 1]] * last, 1)
        ref, _ = oracle.denoise_attention(dict(q=inp["q"][b:b + 1], k_blk=inp["k_blk"][b:b + 1],
                                               v_blk=inp["v_blk"][b:b + 1],
                                               ctx_len=np.array([lens[b] + S * last], np.int32),
                                               k_ctx=kc, v_ctx=vc), w.softmax_scale)
        check_attention(bf16_to_f64(host(t["attn_out"]))[b:b + 1], ref, what=f"paged seq {b}")


def test_generate_with_projection_and_lm_head_equals_manual_loop(tt):
    """tt_generate with the projection and the LM head in the step equals the same
    blocks driven one call at a time (block start by hand, tt_denoise_block_loop,
    tt_append_block): the orchestration adds nothing and drops nothing."""
    B, S, Hq, Hkv, D, V, H, mask, T = 2, 16, 8, 2, 64, 2048, 256, 3, 16
    n_blocks, lens = 3, np.array([90, 40], np.int32)
    cap = int(lens.max()) + n_blocks * S
    w = synth.Workload("genlm", B=B, L=int(lens.max()), S=S, Hq=Hq, Hkv=Hkv, D=D, H=H, V=V, T=T,
                       softmax_scale=0.125)
    inp = synth.make_attention_inputs(w, 2, ctx_len=lens)
    ad = synth.make_adaln_inputs(w, 2)
    Wv, Wq = synth.make_lmhead_weights(w, 2), synth.make_qkv_weights(w, 2)
    kc0 = np.zeros((B, cap, Hkv, D), np.uint16)
    vc0 = np.zeros((B, cap, Hkv, D), np.uint16)
    kc0[:, :inp["k_ctx"].shape[1]] = inp["k_ctx"]
    vc0[:, :inp["v_ctx"].shape[1]] = inp["v_ctx"]
    dims = tt.attn_dims(B, S, Hq, Hkv, D, cap, 0, 0, 0, w.softmax_scale, 0)
    desc = tt.step_desc(dims, H, V, mask, w.gamma, T, w.ln_eps, 2, 0, tt.LOGITS_LM_HEAD, 0.0, 0.0, qkv_proj=True)

    def fresh():
        return dict(x=dev(ad["x"]), shift_table=dev(ad["shift_table"]), scale_table=dev(ad["scale_table"]),
                    q=dev(inp["q"]), k_blk=dev(inp["k_blk"]), v_blk=dev(inp["v_blk"]), k_ctx=dev(kc0),
                    v_ctx=dev(vc0), ctx_len=dev(lens),
                    ids=torch.zeros((B, S), dtype=torch.int32, device="cuda"),
                    n_masked=torch.zeros(B, dtype=torch.int32, device="cuda"),
                    steps=torch.zeros(B, dtype=torch.int32, device="cuda"),
                    commit_step=torch.zeros((B, S), dtype=torch.uint8, device="cuda"),
                    y=torch.zeros((B, S, H), dtype=torch.int16, device="cuda"),
                    attn_out=torch.zeros((B, S, Hq, D), dtype=torch.int16, device="cuda"),
                    w_vocab=dev(Wv), w_qkv=dev(Wq))
    stop = tt.tt_stop_spec(-1, 0, n_blocks * S)
    a = fresh()
    ws = tt.workspace(tt.tt_denoise_workspace(desc))
    gen_a = torch.zeros(B, dtype=torch.int32, device="cuda")
    done_a = torch.zeros(B, dtype=torch.uint8, device="cuda")
    out_a = torch.full((B, n_blocks * S), -1, dtype=torch.int32, device="cuda")
    tt.tt_generate(desc, tt.step_tensors(**a), n_blocks, stop, gen_a, done_a, out_a, ws)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    b_ = fresh()
    ws_b = tt.workspace(tt.tt_denoise_workspace(desc))
    gen_b = torch.zeros(B, dtype=torch.int32, device="cuda")
    done_b = torch.zeros(B, dtype=torch.uint8, device="cuda")
    out_b = torch.full((B, n_blocks * S), -1, dtype=torch.int32, device="cuda")
    ts_b = tt.step_tensors(**b_)
    for k in range(n_blocks):
        b_["ids"].fill_(mask)
        b_["steps"].zero_()
        b_["commit_step"].zero_()
        desc.logits.block_index = k
        tt.tt_denoise_block_loop(desc, ts_b, ws_b)
        tt.tt_append_block(dims, b_["k_blk"], b_["v_blk"], b_["k_ctx"], b_["v_ctx"], None, b_["ctx_len"],
                           b_["ids"], stop, gen_b, done_b, out_b, n_blocks * S, k * S)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    assert np.array_equal(host(out_a), host(out_b))
    assert np.all(host(out_a) != mask) and np.all(host(out_a) >= 0)
    assert host(a["ctx_len"]).tolist() == host(b_["ctx_len"]).tolist() == (lens + n_blocks * S).tolist()
    assert np.array_equal(host(a["k_ctx"]), host(b_["k_ctx"]))
    assert np.array_equal(host(a["attn_out"]), host(b_["attn_out"]))
