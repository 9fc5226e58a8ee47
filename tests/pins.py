"""Checks that pin the oracle to something other than itself.

Each ``check_*`` takes the oracle function(s) under test as arguments, so that the
same checks run against the real oracle (tests/test_oracle_*.py) and against copies
with a planted mistake (tests/test_oracle_mutations.py), which they must reject.
The pins are library routines other than the ones the oracle calls (torch SDPA and
layer_norm, scipy softmax), closed forms, invariants and special cases.
"""
import math

import numpy as np
import torch
import torch.nn.functional as F

from block_wise_mask_tt_b300 import synth


# ----------------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------------

def tiny_attention_inputs(seed, B, S, Hq, Hkv, D, lens, paged=False, page_size=4):
    w = synth.Workload("tiny", B=B, L=max(lens) if len(lens) else 0, S=S, Hq=Hq, Hkv=Hkv, D=D,
                       H=8, V=16, paged=paged, page_size=page_size,
                       L_min=1 if paged else 0)
    return synth.make_attention_inputs(w, seed, ctx_len=np.asarray(lens, np.int32))


def _bf(x):
    return torch.from_numpy(synth.bf16_bits_to_f32(x).astype(np.float64))


def torch_reference(inp, scale):
    """torch SDPA (fp64, CPU) over [context ++ block] keys per sequence; lse by logsumexp."""
    q = _bf(inp["q"])  # B S Hq D
    kb, vb = _bf(inp["k_blk"]), _bf(inp["v_blk"])
    B, S, Hq, D = q.shape
    Hkv = kb.shape[2]
    G = Hq // Hkv
    outs, lses = [], []
    for b in range(B):
        n = int(inp["ctx_len"][b])
        if "page_table" in inp:
            ps = inp["k_pages"].shape[1]
            kc = torch.stack([_bf(inp["k_pages"][inp["page_table"][b, t // ps], t % ps])
                              for t in range(n)]) if n else torch.zeros(0, Hkv, D, dtype=torch.float64)
            vc = torch.stack([_bf(inp["v_pages"][inp["page_table"][b, t // ps], t % ps])
                              for t in range(n)]) if n else torch.zeros(0, Hkv, D, dtype=torch.float64)
        else:
            kc, vc = _bf(inp["k_ctx"][b, :n]), _bf(inp["v_ctx"][b, :n])
        k = torch.cat([kc, kb[b]], 0).permute(1, 0, 2).repeat_interleave(G, 0)  # Hq, L+S, D
        v = torch.cat([vc, vb[b]], 0).permute(1, 0, 2).repeat_interleave(G, 0)
        qq = q[b].permute(1, 0, 2)  # Hq S D
        o = F.scaled_dot_product_attention(qq[None], k[None], v[None], scale=scale)[0]
        outs.append(o.permute(1, 0, 2))
        lses.append(torch.logsumexp(scale * qq @ k.transpose(1, 2), dim=-1).permute(1, 0))
    return torch.stack(outs).numpy(), torch.stack(lses).numpy()


def check_attention_vs_torch(attn_fn):
    cases = [
        dict(B=2, S=3, Hq=4, Hkv=2, D=8, lens=[5, 0]),
        dict(B=1, S=16, Hq=4, Hkv=1, D=16, lens=[37]),
        dict(B=3, S=1, Hq=6, Hkv=3, D=8, lens=[1, 9, 4]),
        dict(B=2, S=5, Hq=2, Hkv=2, D=4, lens=[13, 2]),
    ]
    for i, c in enumerate(cases):
        for paged in (False, True):
            inp = tiny_attention_inputs(100 + i, paged=paged, **c)
            scale = 1.0 / math.sqrt(c["D"])
            O, lse = attn_fn(inp, scale)
            Ot, lset = torch_reference(inp, scale)
            np.testing.assert_allclose(O, Ot, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse, lset, rtol=1e-12, atol=1e-12)


def check_identical_keys_mean(attn_fn):
    """Every key equal => uniform weights => output is the mean of all value rows."""
    B, S, Hq, Hkv, D, L = 2, 4, 4, 2, 8, 6
    inp = tiny_attention_inputs(7, B, S, Hq, Hkv, D, [L, L])
    key = synth.f32_to_bf16_bits(np.linspace(-1, 1, D).astype(np.float32))
    inp["k_ctx"][:] = key
    inp["k_blk"][:] = key
    O, _ = attn_fn(inp, 0.7)
    vc = synth.bf16_bits_to_f32(inp["v_ctx"]).astype(np.float64)
    vb = synth.bf16_bits_to_f32(inp["v_blk"]).astype(np.float64)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            g = h // G
            mean = np.concatenate([vc[b, :L, g], vb[b, :, g]]).mean(axis=0)
            for s in range(S):
                np.testing.assert_allclose(O[b, s, h], mean, rtol=1e-12, atol=1e-12)


def check_block_permutation(attn_fn):
    """Bidirectional block: permuting block tokens (q, k_blk, v_blk together) permutes O."""
    inp = tiny_attention_inputs(8, 2, 6, 4, 2, 8, [5, 3])
    O, lse = attn_fn(inp, 0.35)
    perm = np.array([3, 0, 5, 1, 4, 2])
    inp2 = dict(inp)
    for k in ("q", "k_blk", "v_blk"):
        inp2[k] = inp[k][:, perm]
    O2, lse2 = attn_fn(inp2, 0.35)
    np.testing.assert_allclose(O2, O[:, perm], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse2, lse[:, perm], rtol=1e-12, atol=1e-12)


def check_single_key(attn_fn):
    """No context and a one-token block: the only key gets weight 1, O = v, lse = scale*q.k."""
    inp = tiny_attention_inputs(9, 1, 1, 2, 1, 8, [0])
    O, lse = attn_fn(inp, 0.5)
    v = synth.bf16_bits_to_f32(inp["v_blk"][0, 0, 0]).astype(np.float64)
    q = synth.bf16_bits_to_f32(inp["q"][0, 0]).astype(np.float64)
    k = synth.bf16_bits_to_f32(inp["k_blk"][0, 0, 0]).astype(np.float64)
    for h in range(2):
        np.testing.assert_allclose(O[0, 0, h], v, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[0, 0, h], 0.5 * q[h] @ k, rtol=1e-12, atol=1e-12)


def check_dominant_key(attn_fn):
    """One context key aligned with q and much larger than the rest selects its value row."""
    B, S, Hq, Hkv, D, L = 1, 2, 2, 1, 8, 7
    inp = tiny_attention_inputs(10, B, S, Hq, Hkv, D, [L])
    q = np.zeros((B, S, Hq, D), np.float32)
    q[..., 0] = 1.0
    inp["q"] = synth.f32_to_bf16_bits(q)
    k = synth.bf16_bits_to_f32(inp["k_ctx"]).copy()
    k[..., 0] = 0.0
    k[0, 4, 0, 0] = 64.0  # exp(64*1) dominates every other weight (others are exp(0))
    inp["k_ctx"] = synth.f32_to_bf16_bits(k)
    kb = synth.bf16_bits_to_f32(inp["k_blk"]).copy()
    kb[..., 0] = 0.0
    inp["k_blk"] = synth.f32_to_bf16_bits(kb)
    O, _ = attn_fn(inp, 1.0)
    v = synth.bf16_bits_to_f32(inp["v_ctx"][0, 4, 0]).astype(np.float64)
    for s in range(S):
        for h in range(Hq):
            np.testing.assert_allclose(O[0, s, h], v, rtol=1e-12, atol=1e-12)


ATTENTION_CHECKS = (check_attention_vs_torch, check_identical_keys_mean, check_block_permutation,
                    check_single_key, check_dominant_key)


# ----------------------------------------------------------------------------------
# adaLN
# ----------------------------------------------------------------------------------

def check_adaln_vs_torch(adaln_fn):
    rng = np.random.default_rng(3)
    for H in (1, 7, 256, 2688):
        x = synth.f32_to_bf16_bits(rng.standard_normal((3, H)).astype(np.float32) * 2 + 0.5)
        shift = rng.standard_normal((3, H)).astype(np.float32) * 0.1
        scale = rng.standard_normal((3, H)).astype(np.float32) * 0.1
        y = adaln_fn(x, shift, scale, 1e-5)
        xt = _bf(x)
        for r in range(3):
            ref = F.layer_norm(xt[r], (H,), weight=1 + torch.from_numpy(scale[r]).double(),
                               bias=torch.from_numpy(shift[r]).double(), eps=1e-5).numpy()
            np.testing.assert_allclose(y[r], ref, rtol=1e-12, atol=1e-12)
        y0 = adaln_fn(x, np.zeros(H, np.float32), np.zeros(H, np.float32), 1e-3)
        ref0 = F.layer_norm(xt, (H,), eps=1e-3).numpy()
        np.testing.assert_allclose(y0, ref0, rtol=1e-12, atol=1e-12)


def check_adaln_constant_row(adaln_fn):
    """x constant => x - mean = 0 => y = shift exactly, whatever scale is."""
    H = 64
    x = np.full((2, H), synth.f32_to_bf16_bits(np.float32(1.75)), np.uint16)
    shift = np.linspace(-1, 1, H).astype(np.float32)
    scale = np.linspace(2, -3, H).astype(np.float32)
    y = adaln_fn(x, shift, scale, 1e-5)
    np.testing.assert_array_equal(y, np.broadcast_to(shift.astype(np.float64), (2, H)))


def check_adaln_moments(adaln_fn):
    """With shift = scale = 0 the row has mean 0 and biased variance var/(var+eps)."""
    rng = np.random.default_rng(4)
    H, eps = 512, 0.25
    xf = rng.standard_normal(H).astype(np.float32)
    x = synth.f32_to_bf16_bits(xf)
    y = adaln_fn(x, np.zeros(H, np.float32), np.zeros(H, np.float32), eps)
    xd = synth.bf16_bits_to_f32(x).astype(np.float64)
    var = np.var(xd)
    assert abs(y.mean()) < 1e-12
    np.testing.assert_allclose(np.mean(y ** 2), var / (var + eps), rtol=1e-12)


ADALN_CHECKS = (check_adaln_vs_torch, check_adaln_constant_row, check_adaln_moments)


# ----------------------------------------------------------------------------------
# unmask
# ----------------------------------------------------------------------------------

def check_conf_two_valued(row_conf_fn):
    """Logit a at one id, b elsewhere (mask id included at b): conf = e^a/(e^a+(V-2)e^b)."""
    for V, a, bval, j, mask in ((16, 3.0, 1.0, 9, 3), (1024, 0.5, -2.0, 0, 3), (50, 10.0, 9.0, 49, 0)):
        row = np.full(V, bval, np.float32)
        row[j] = a
        tok, conf = row_conf_fn(row, mask)
        exp = math.exp(a) / (math.exp(a) + (V - 2) * math.exp(bval))
        assert tok == j
        assert abs(conf - exp) <= 1e-14 * exp


def check_conf_vs_scipy(row_conf_fn):
    import scipy.special
    rng = np.random.default_rng(5)
    for V in (8, 1000, 131072):
        for mask in (3, 0, V - 1):
            row = (rng.standard_normal(V) * 3).astype(np.float32)
            tok, conf = row_conf_fn(row, mask)
            keep = np.delete(np.arange(V), mask)
            p = scipy.special.softmax(row[keep].astype(np.float64))
            assert tok == keep[int(np.argmax(p))]
            assert abs(conf - p.max()) <= 1e-12 * p.max()


def check_mask_never_emitted(row_conf_fn):
    """The mask id holds the largest logit by far: it is neither emitted nor counted."""
    V, mask = 64, 3
    row = np.linspace(-1, 1, V).astype(np.float32)
    row[mask] = 50.0
    tok, conf = row_conf_fn(row, mask)
    assert tok == V - 1
    keep = np.delete(row.astype(np.float64), mask)
    assert abs(conf - 1.0 / np.sum(np.exp(keep - keep.max()))) < 1e-14


def check_ties_lowest_id(row_conf_fn):
    V, mask = 32, 3
    row = np.zeros(V, np.float32)
    for ids in ((5, 6), (30, 7, 19), (0, 31), (2, 4)):
        r = row.copy()
        r[list(ids)] = 2.5
        tok, conf = row_conf_fn(r, mask)
        assert tok == min(ids)
        assert abs(conf - math.exp(2.5) / (len(ids) * math.exp(2.5) + (V - 1 - len(ids)))) < 1e-14


def check_threshold_inclusive(step_fn):
    """Two equal live logits => conf = 1/2 exactly; gamma = 0.5 commits it (>=)."""
    V, mask, S = 3, 2, 2
    logits = np.zeros((S, V), np.float32)
    logits[:, mask] = 5.0
    r = step_fn(logits, np.full(S, mask), 0, mask, 0.5, 8)
    assert r["conf"][0] == 0.5 and r["conf"][1] == 0.5
    assert r["commit"].tolist() == [1, 1]
    assert r["ids"].tolist() == [0, 0]  # tie between ids 0 and 1 -> 0


def _random_logits_fn(seed, V, mask, boost=(0.0, 12.0)):
    def fn(step, positions):
        return synth.logits_rows(seed, 0, 0, step, positions, V, mask, synth.LOGITS_UNIFORM, *boost)
    return fn


def check_gamma_zero_one_step(block_fn):
    for seed in range(3):
        r = block_fn(16, 16, 3, 0.0, _random_logits_fn(seed, 256, 3))
        assert r["steps"] == 1
        assert np.all(r["ids"] != 3)
        assert np.all(r["commit_step"] == 1)


def check_gamma_above_one_takes_s_steps(block_fn):
    """gamma > 1 => only the floor commits: exactly one per step, most confident first."""
    for S in (1, 5, 16):
        r = block_fn(S, S, 3, 1.01, _random_logits_fn(11 + S, 256, 3))
        assert r["steps"] == S
        assert sorted(r["commit_step"].tolist()) == list(range(1, S + 1))
        for tr in r["trace"]:
            assert len(tr["committed"]) == 1
            i = tr["committed"][0]
            live = [p for p in range(S) if tr["ids_before"][p] == 3]
            assert all(tr["conf"][i] > tr["conf"][p] or (tr["conf"][i] == tr["conf"][p] and i <= p)
                       for p in live)


def check_floor_ceil_rule(block_fn):
    """T < S with gamma > 1: each step commits ceil(m / steps_left) positions."""
    for S, T in ((16, 4), (16, 5), (7, 3), (32, 16)):
        r = block_fn(S, T, 3, 2.0, _random_logits_fn(S * T, 128, 3))
        assert r["steps"] == T
        m = S
        for k, tr in enumerate(r["trace"]):
            want = math.ceil(m / (T - k))
            assert len(tr["committed"]) == want
            m -= want
        assert m == 0


def check_frozen_and_bounded(block_fn):
    """Committed ids never change, the mask id is never emitted, steps <= T, t = m/S."""
    for seed, gamma in ((1, 0.8), (2, 0.5), (3, 0.95), (4, 0.3)):
        S, T = 16, 16
        r = block_fn(S, T, 3, gamma, _random_logits_fn(seed, 512, 3, (0.0, 14.0)))
        assert 1 <= r["steps"] <= T
        assert np.all(r["ids"] != 3)
        prev = None
        for tr in r["trace"]:
            ids_b = tr["ids_before"]
            assert tr["t"] == np.sum(ids_b == 3) / S
            if prev is not None:
                done = prev != 3
                assert np.array_equal(ids_b[done], prev[done])
            prev = ids_b
        assert r["trace"][0]["t"] == 1.0
        # a position's final id is the token predicted at its commit step
        for tr in r["trace"]:
            for i in tr["committed"]:
                assert r["ids"][i] == tr["tok"][i]
        # commits above gamma are exactly the positions at or above gamma (when any exist)
        for tr in r["trace"]:
            live = np.flatnonzero(tr["ids_before"] == 3)
            above = [i for i in live if tr["conf"][i] >= gamma]
            if len(above) >= tr["k_min"]:
                assert sorted(above) == sorted(tr["committed"].tolist())


def check_floor_ties_lower_position(block_fn):
    """Equal confidence everywhere and gamma > 1: the floor commits positions in order."""
    S = 6

    def fn(step, positions):
        return np.zeros((len(positions), 16), np.float32)
    r = block_fn(S, S, 3, 1.5, fn)
    assert [int(tr["committed"][0]) for tr in r["trace"]] == list(range(S))


UNMASK_ROW_CHECKS = (check_conf_two_valued, check_conf_vs_scipy, check_mask_never_emitted,
                     check_ties_lowest_id)
UNMASK_STEP_CHECKS = (check_threshold_inclusive,)
BLOCK_CHECKS = (check_gamma_zero_one_step, check_gamma_above_one_takes_s_steps,
                check_floor_ceil_rule, check_frozen_and_bounded, check_floor_ties_lower_position)


# ----------------------------------------------------------------------------------
# sampler variants (temperature, mock-AR, predict-and-noise)
# ----------------------------------------------------------------------------------
# Each check takes sampler_step(logits, ids, steps, mask_id, T, kind, gamma,
# temperature, commit_step) from oracle.samplers (or a mutated copy).
SAMPLER_CONFIDENCE, SAMPLER_MOCK_AR, SAMPLER_PREDICT_NOISE = 0, 1, 2


def _run_block(step_fn, S, T, mask_id, logits_fn, kind, gamma=0.8, temperature=1.0):
    ids = np.full(S, mask_id, np.int64)
    cs = np.zeros(S, np.uint8)
    steps = 0
    per_step = []
    while np.any(ids == mask_id) and steps < 64:
        k = steps
        r = step_fn(lambda pos: logits_fn(k, pos), ids, steps, mask_id, T, kind, gamma, temperature, cs)
        per_step.append(r)
        ids, cs, steps = r["ids"], r["commit_step"], r["steps"]
    return ids, cs, steps, per_step


def check_temperature_closed_form(step_fn):
    """Two-valued row (a at one id, b at the other V-2, the mask id excluded):
    conf = 1 / (1 + (V-2) exp((b-a)/tau)); the token is the argmax for every tau."""
    V, mask = 40, 5
    for tau in (0.1, 0.5, 1.0, 3.0):
        a, b = 2.0, 0.5
        row = np.full(V, b, np.float32)
        row[17] = a
        row[mask] = 50.0  # largest, but excluded
        logits = np.tile(row, (3, 1))
        ids = np.array([mask, 9, mask])
        r = step_fn(logits, ids, 0, mask, 16, SAMPLER_CONFIDENCE, 2.0, tau, None)
        want = 1.0 / (1.0 + (V - 2) * math.exp((b - a) / tau))
        assert abs(r["conf"][0] - want) <= 1e-12 * want
        assert r["tok"][0] == 17 and r["tok"][2] == 17 and r["conf"][1] == 0.0


def check_temperature_vs_scipy(step_fn):
    from scipy.special import softmax
    rng = np.random.default_rng(3)
    V, mask, S = 300, 3, 6
    logits = rng.standard_normal((S, V)).astype(np.float32) * 2
    for tau in (0.25, 1.0, 2.5):
        r = step_fn(logits, np.full(S, mask), 0, mask, S, SAMPLER_CONFIDENCE, 2.0, tau, None)
        for i in range(S):
            l = logits[i].astype(np.float64).copy()
            l[mask] = -np.inf
            p = softmax(l / tau)
            assert abs(r["conf"][i] - p.max()) <= 1e-12
            assert r["tok"][i] == int(np.argmax(l))


def check_temperature_one_is_plain_confidence(step_fn):
    """tau = 1 with gamma = 0 commits the whole block in one step; gamma > 1 one per step."""
    ids, cs, steps, _ = _run_block(step_fn, 8, 8, 3, _random_logits_fn(5, 256, 3), SAMPLER_CONFIDENCE, 0.0)
    assert steps == 1 and np.all(cs == 1)
    ids, cs, steps, _ = _run_block(step_fn, 8, 8, 3, _random_logits_fn(6, 256, 3), SAMPLER_CONFIDENCE, 1.01)
    assert steps == 8 and sorted(cs.tolist()) == list(range(1, 9))


def check_mock_ar_left_to_right(step_fn):
    """One token per step, in position order: commit_step[i] = i + 1, S steps."""
    for S in (1, 7, 16):
        ids, cs, steps, per = _run_block(step_fn, S, S, 3, _random_logits_fn(40 + S, 256, 3), SAMPLER_MOCK_AR)
        assert steps == S
        assert cs.tolist() == list(range(1, S + 1))
        assert np.all(ids != 3)
        assert all(int(r["commit"].sum()) == 1 for r in per)


def check_mock_ar_skips_decoded_positions(step_fn):
    mask = 3
    logits = np.zeros((5, 16), np.float32)
    ids = np.array([7, mask, 9, mask, mask])
    r = step_fn(logits, ids, 0, mask, 5, SAMPLER_MOCK_AR, 0.8, 1.0, None)
    assert r["commit"].tolist() == [0, 1, 0, 0, 0]
    assert r["ids"][0] == 7 and r["ids"][2] == 9


def check_predict_noise_schedule(step_fn):
    """Linear schedule: floor(S (T - k - 1) / T) stay masked after step k (at least one
    commit per step); the committed positions are the most confident (by scipy)."""
    from scipy.special import softmax
    for S, T, counts in ((16, 4, [4, 4, 4, 4]), (16, 16, [1] * 16), (16, 5, [4, 3, 3, 3, 3]),
                         (8, 3, [3, 3, 2])):
        fn = _random_logits_fn(60 + T, 256, 3)
        ids, cs, steps, per = _run_block(step_fn, S, T, 3, fn, SAMPLER_PREDICT_NOISE)
        assert [int(r["commit"].sum()) for r in per] == counts
        assert steps == T and np.all(ids != 3)
        # first step: the committed set is the top-k by confidence
        lg = fn(0, np.arange(S)).astype(np.float64)
        lg[:, 3] = -np.inf
        conf = np.array([softmax(row).max() for row in lg])
        top = sorted(range(S), key=lambda i: (-conf[i], i))[:counts[0]]
        assert sorted(np.flatnonzero(per[0]["commit"]).tolist()) == sorted(top)


SAMPLER_CHECKS = [check_temperature_closed_form, check_temperature_vs_scipy,
                  check_temperature_one_is_plain_confidence, check_mock_ar_left_to_right,
                  check_mock_ar_skips_decoded_positions, check_predict_noise_schedule]


# ----------------------------------------------------------------------------------
# outer loop (Algorithm 1): cache append and stopping
# ----------------------------------------------------------------------------------
def _append_case(seed, paged, D=8):
    """A small batch: context lengths 5 / 0 / 9 with room for two more blocks of S=3."""
    rng = np.random.default_rng(seed)
    B, S, Hkv, Hq = 3, 3, 2, 4
    lens = np.array([5, 0, 9])
    w = synth.Workload("tiny", B=B, L=int(lens.max()), S=S, Hq=Hq, Hkv=Hkv, D=D, H=8, V=16,
                       paged=False)
    base = synth.make_attention_inputs(w, seed, ctx_len=lens.astype(np.int32))
    cap = int(lens.max()) + 2 * S
    kc = np.zeros((B, cap, Hkv, D), np.uint16)
    vc = np.zeros((B, cap, Hkv, D), np.uint16)
    for b in range(B):
        kc[b, :lens[b]] = base["k_ctx"][b, :lens[b]]
        vc[b, :lens[b]] = base["v_ctx"][b, :lens[b]]
    if not paged:
        return dict(k_ctx=kc, v_ctx=vc), base, lens, cap
    # the same logical rows in shuffled 64-row pages
    n_pages = B * ((cap + 63) // 64)
    perm = rng.permutation(n_pages)
    pt = perm.reshape(B, -1).astype(np.int64)
    kp = np.zeros((n_pages, 64, Hkv, D), np.uint16)
    vp = np.zeros((n_pages, 64, Hkv, D), np.uint16)
    for b in range(B):
        for t in range(cap):
            kp[pt[b, t // 64], t % 64] = kc[b, t]
            vp[pt[b, t // 64], t % 64] = vc[b, t]
    return dict(k_pages=kp, v_pages=vp, page_table=pt), base, lens, cap


def check_append_then_attend_equals_concatenation(append_fn):
    """Two blocks appended, then a third block attends: torch SDPA over the explicitly
    concatenated keys [context ; block 0 ; block 1 ; own block] must agree."""
    for paged in (False, True):
        cache, base, lens, cap = _append_case(7 + paged, paged)
        B, S, Hkv, D = base["k_blk"].shape
        rng = np.random.default_rng(3)
        blks = [synth.f32_to_bf16_bits(rng.standard_normal((2, B, S, Hkv, D)).astype(np.float32))
                for _ in range(2)]
        ctx, gen, done = lens.copy(), np.zeros(B, np.int64), np.zeros(B, np.uint8)
        for kb_vb in blks:
            ids = np.full((B, S), 11)
            r = append_fn(cache, kb_vb[0], kb_vb[1], ctx, ids, 99, 1000, gen, done)
            cache = {k: r[k] for k in cache}
            ctx, gen, done = r["ctx_len"], r["generated"], r["done"]
        assert ctx.tolist() == (lens + 2 * S).tolist()
        # attention of the current block over the appended cache
        inp = dict(q=base["q"], k_blk=base["k_blk"], v_blk=base["v_blk"], ctx_len=ctx.astype(np.int32))
        if paged:
            inp.update(k_pages=cache["k_pages"], v_pages=cache["v_pages"], page_table=cache["page_table"])
        else:
            inp.update(k_ctx=cache["k_ctx"], v_ctx=cache["v_ctx"])
        # explicit concatenation, contiguous
        L = int(ctx.max())
        kc = np.zeros((B, L, Hkv, D), np.uint16)
        vc = np.zeros((B, L, Hkv, D), np.uint16)
        for b in range(B):
            n = int(lens[b])
            kc[b, :n] = base["k_ctx"][b, :n]
            vc[b, :n] = base["v_ctx"][b, :n]
            for i, kb_vb in enumerate(blks):
                kc[b, n + i * S:n + (i + 1) * S] = kb_vb[0][b]
                vc[b, n + i * S:n + (i + 1) * S] = kb_vb[1][b]
        ref = dict(q=base["q"], k_blk=base["k_blk"], v_blk=base["v_blk"], ctx_len=ctx.astype(np.int32),
                   k_ctx=kc, v_ctx=vc)
        want, _ = torch_reference(ref, 0.35)
        import oracle
        got, _ = oracle.denoise_attention(inp, 0.35)
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def check_append_stops(append_fn):
    cache, base, lens, cap = _append_case(11, False)
    B, S = base["k_blk"].shape[:2]
    ids = np.array([[1, 2, 3], [4, 99, 6], [7, 8, 9]])  # sequence 1 commits the EOS id 99
    gen0 = np.array([0, 0, 3])  # sequence 2 reaches max_new = 6 exactly
    done0 = np.array([0, 0, 0], np.uint8)
    r = append_fn(cache, base["k_blk"], base["v_blk"], lens, ids, 99, 6, gen0, done0)
    assert r["done"].tolist() == [0, 1, 1]          # EOS; 3 + 3 reaches 6
    assert r["generated"].tolist() == [3, 3, 6]
    assert r["ctx_len"].tolist() == (lens + S).tolist()
    # a done sequence is left alone: no rows written, ctx_len and generated unchanged
    r2 = append_fn({k: r[k] for k in cache}, base["k_blk"], base["v_blk"], r["ctx_len"], ids, 99, 100,
                   r["generated"], r["done"])
    assert r2["ctx_len"].tolist() == [lens[0] + 2 * S, lens[1] + S, lens[2] + S]
    assert np.array_equal(r2["k_ctx"][1], r["k_ctx"][1]) and np.array_equal(r2["k_ctx"][2], r["k_ctx"][2])
    assert r2["generated"].tolist() == [6, 3, 6]


OUTER_CHECKS = [check_append_then_attend_equals_concatenation, check_append_stops]


# ----------------------------------------------------------------------------------
# LM head feeding the unmask step
# ----------------------------------------------------------------------------------
BF16_ONE = 0x3F80


def _rand_bf16(seed, shape, std=1.0):
    rng = np.random.default_rng(seed)
    return synth.f32_to_bf16_bits((rng.standard_normal(shape) * std).astype(np.float32))


def check_lm_head_one_hot_rows(logits_fn):
    """W[j] = e_{pi(j)} (exact ones): logit[r][j] is the hidden component pi(j), exactly."""
    V, H = 40, 24
    pi = np.random.default_rng(1).integers(0, H, V)
    W = np.zeros((V, H), np.uint16)
    W[np.arange(V), pi] = BF16_ONE
    h = _rand_bf16(2, (5, H))
    got = logits_fn(h, W)
    assert got.shape == (5, V)
    want = synth.bf16_bits_to_f32(h).astype(np.float64)[:, pi]
    assert np.array_equal(got, want)


def check_lm_head_vs_torch_linear(logits_fn):
    h = _rand_bf16(3, (5, 96))
    W = _rand_bf16(4, (70, 96), 0.3)
    want = F.linear(_bf(h), _bf(W)).numpy()
    np.testing.assert_allclose(logits_fn(h, W), want, rtol=1e-12, atol=1e-12)


def check_lm_head_scaled_basis_rows(step_fn):
    """h[s] = a_s e_{k_s}: logit[j] = a_s W[j][k_s]; token and confidence follow from
    column k_s of W alone (closed form written out with loops)."""
    V = H = 48
    mask = 5
    W = _rand_bf16(6, (V, H))
    Wf = synth.bf16_bits_to_f32(W).astype(np.float64)
    S = 6
    ks = [0, 7, 7, 19, 33, 47]
    amps = [0.5, 1.0, 2.0, 3.0, 1.5, 4.0]
    h = np.zeros((S, H), np.uint16)
    for s in range(S):
        h[s, ks[s]] = synth.f32_to_bf16_bits(np.array([amps[s]], np.float32))[0]
    r = step_fn(h, W, np.full(S, mask), 0, mask, 16, 0, 2.0, 1.0, None)
    for s in range(S):
        best, tok = -math.inf, -1
        for j in range(V):
            if j != mask and amps[s] * Wf[j, ks[s]] > best:
                best, tok = amps[s] * Wf[j, ks[s]], j
        den = 0.0
        for j in range(V):
            if j != mask:
                den += math.exp(amps[s] * Wf[j, ks[s]] - best)
        assert r["tok"][s] == tok
        assert abs(r["conf"][s] - 1.0 / den) <= 1e-12


def check_lm_head_mask_row_never_emitted(step_fn):
    """The mask id's row of W is aligned with every hidden row (largest logit): it is
    neither emitted nor counted in the confidence."""
    V, H, mask, S = 32, 16, 3, 4
    W = _rand_bf16(8, (V, H), 0.1)
    h = _rand_bf16(9, (S, H))
    W[mask] = synth.f32_to_bf16_bits(np.sign(synth.bf16_bits_to_f32(h).sum(0)).astype(np.float32) * 8)
    r = step_fn(h, W, np.full(S, mask), 0, mask, S, 0, 0.0, 1.0, None)
    assert np.all(r["ids"] != mask)
    lg = synth.bf16_bits_to_f32(h).astype(np.float64) @ synth.bf16_bits_to_f32(W).astype(np.float64).T
    lg[:, mask] = -np.inf
    from scipy.special import softmax
    for s in range(S):
        assert abs(r["conf"][s] - softmax(lg[s]).max()) <= 1e-12


def check_lm_head_decoded_rows_unused(step_fn):
    """Hidden rows of decoded positions are never read: NaN there changes nothing."""
    V, H, mask, S = 64, 32, 3, 6
    W = _rand_bf16(10, (V, H), 0.4)
    h = _rand_bf16(11, (S, H))
    ids = np.array([mask, 17, mask, mask, 40, mask])
    a = step_fn(h, W, ids, 1, mask, S, 0, 0.8, 1.0, None)
    h2 = h.copy()
    h2[[1, 4]] = 0x7FC0  # bf16 NaN
    b = step_fn(h2, W, ids, 1, mask, S, 0, 0.8, 1.0, None)
    assert np.array_equal(a["ids"], b["ids"]) and np.array_equal(a["conf"], b["conf"])
    assert np.all(np.isfinite(b["conf"]))


LMHEAD_LOGIT_CHECKS = [check_lm_head_one_hot_rows, check_lm_head_vs_torch_linear]
LMHEAD_STEP_CHECKS = [check_lm_head_scaled_basis_rows, check_lm_head_mask_row_never_emitted,
                      check_lm_head_decoded_rows_unused]


# ----------------------------------------------------------------------------------
# query/key/value projection of the adaLN output
# ----------------------------------------------------------------------------------

def check_qkv_one_hot_rows(proj_fn):
    """Row r of W_qkv = e_{pi(r)} (exact ones): every output entry is one hidden component,
    placed by the (q heads, k heads, v heads) x D column order."""
    B, S, H, Hq, Hkv, D = 2, 3, 16, 4, 2, 8
    n = (Hq + 2 * Hkv) * D
    pi = np.random.default_rng(12).integers(0, H, n)
    W = np.zeros((n, H), np.uint16)
    W[np.arange(n), pi] = BF16_ONE
    y = _rand_bf16(13, (B, S, H))
    q, k, v = proj_fn(y, W, Hq, Hkv, D)
    yf = synth.bf16_bits_to_f32(y).astype(np.float64)
    for h in range(Hq):
        for d in range(D):
            assert np.array_equal(q[:, :, h, d], yf[:, :, pi[h * D + d]])
    for h in range(Hkv):
        for d in range(D):
            assert np.array_equal(k[:, :, h, d], yf[:, :, pi[(Hq + h) * D + d]])
            assert np.array_equal(v[:, :, h, d], yf[:, :, pi[(Hq + Hkv + h) * D + d]])


def check_qkv_vs_torch_linear(proj_fn):
    B, S, H, Hq, Hkv, D = 3, 5, 40, 4, 1, 16
    y = _rand_bf16(14, (B, S, H))
    W = _rand_bf16(15, ((Hq + 2 * Hkv) * D, H), 0.2)
    q, k, v = proj_fn(y, W, Hq, Hkv, D)
    full = F.linear(_bf(y), _bf(W)).numpy()
    got = np.concatenate([q.reshape(B, S, -1), k.reshape(B, S, -1), v.reshape(B, S, -1)], axis=-1)
    np.testing.assert_allclose(got, full, rtol=1e-12, atol=1e-12)


QKV_CHECKS = [check_qkv_one_hot_rows, check_qkv_vs_torch_linear]
