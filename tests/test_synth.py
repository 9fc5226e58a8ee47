"""The seeded input generators: pinned to library routines and to their own contracts."""
import numpy as np
import pytest
import torch

from block_wise_mask_tt_b300 import synth


def test_murmur3_matches_sklearn():
    murmurhash3_32 = pytest.importorskip("sklearn.utils").murmurhash3_32
    rng = np.random.default_rng(0)
    keys = rng.integers(0, 2 ** 32, size=4096, dtype=np.uint64)
    seeds = rng.integers(0, 2 ** 32, size=64, dtype=np.uint64)
    for s in seeds:
        ours = synth.murmur3_32(keys, int(s))
        ref = murmurhash3_32(keys.astype(np.uint32).view(np.int32), seed=int(s), positive=True)
        np.testing.assert_array_equal(ours, np.asarray(ref, np.uint32))
    for k in (0, 1, 0xFFFFFFFF, 0xFFFFFFFE, 0xFFFFFFFD):
        assert synth.murmur3_32(k, 7)[0] == murmurhash3_32(np.array([k], np.uint32).view(np.int32),
                                                           seed=7, positive=True)[0]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 7,
                        # exact ties: low 16 bits 0x8000
                        (np.arange(1000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)])
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = synth.bf16_bits_to_f32(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_logits_noise_moments_and_plant():
    V, mask = 131072, 3
    rows = synth.logits_rows(0, 0, 0, 0, np.arange(4), V, mask, synth.LOGITS_UNIFORM, 0.0, 20.0)
    h = synth.row_seed(0, 0, 0, 0, np.arange(4))
    pid = synth.planted_token(h, V, mask)
    boost = synth.planted_boost(h, synth.LOGITS_UNIFORM, 0.0, 20.0)
    for i in range(4):
        r = np.delete(rows[i], pid[i]).astype(np.float64)
        assert abs(r.mean()) < 0.02 and abs(r.var() - 1.0) < 0.02
        assert 0.0 <= boost[i] < 20.0
        assert pid[i] != mask
    # the planted logit is noise + boost with one fp32 add
    r = synth.row_seed(0, 0, 0, 0, 2)
    noise = synth.logits_rows(0, 0, 0, 0, [2], V, mask, synth.LOGITS_UNIFORM, 0.0, 0.0)[0]
    assert rows[2][pid[2]] == np.float32(noise[pid[2]] + boost[2])


def test_planted_never_mask_id():
    V = 7
    h = synth.row_seed(5, 0, 0, 0, np.arange(20000))
    for mask in range(V):
        assert not np.any(synth.planted_token(h, V, mask) == mask)


def test_bimodal_boost_ranges():
    h = synth.row_seed(3, 1, 2, 3, np.arange(20000))
    b = synth.planted_boost(h, synth.LOGITS_BIMODAL, 0, 0)
    lo = (b >= 0) & (b < 4)
    hi = (b >= 10) & (b < 20)
    assert np.all(lo | hi)
    assert 0.45 < lo.mean() < 0.55


def test_paged_layout_is_a_permutation():
    w = synth.RAGGED_PAGED.replace(B=5, L=700, L_min=1, D=8, Hq=4, Hkv=2)
    inp = synth.make_attention_inputs(w, 3)
    n = (inp["ctx_len"] + 63) // 64
    used = np.concatenate([inp["page_table"][b, : n[b]] for b in range(w.B)])
    assert sorted(used.tolist()) == list(range(inp["k_pages"].shape[0]))
    for b in range(w.B):
        assert np.all(inp["page_table"][b, n[b]:] == -1)


@pytest.mark.parametrize("w", synth.WORKLOADS, ids=lambda w: w.name)
def test_configs_well_formed(w):
    assert w.Hq % w.Hkv == 0
    assert w.S <= 32 and w.D in (64, 128)
    assert w.G * w.S <= 512


def test_lm_head_weights_follow_the_recipe():
    """W [V][H] ~ N(0, (lm_logit_std / sqrt(H))^2): unit-RMS hidden rows then give logits
    of standard deviation lm_logit_std; the draw is seeded and independent of block size."""
    w = synth.SINGLE.replace(V=4096, H=512)
    W = synth.make_lmhead_weights(w, 5)
    assert W.shape == (4096, 512) and W.dtype == np.uint16
    Wf = synth.bf16_bits_to_f32(W).astype(np.float64)
    assert abs(Wf.std() - w.lm_logit_std / np.sqrt(w.H)) < 0.01 * w.lm_logit_std / np.sqrt(w.H)
    assert abs(Wf.mean()) < 3 * Wf.std() / np.sqrt(Wf.size)
    h = synth.bf16_bits_to_f32(synth.make_hidden(w.replace(B=2), 6)).astype(np.float64).reshape(-1, w.H)
    logit_std = (h @ Wf.T).std()
    assert abs(logit_std - w.lm_logit_std) < 0.05 * w.lm_logit_std
    assert np.array_equal(W, synth.make_lmhead_weights(w, 5, rows=4096))  # same stream, one block
    assert not np.array_equal(W, synth.make_lmhead_weights(w, 6))


def test_qkv_weights_follow_the_recipe():
    """W_qkv [(Hq + 2 Hkv) D][H] ~ N(0, 1/H): unit-RMS hidden rows give unit-variance q/k/v."""
    w = synth.TINY
    W = synth.make_qkv_weights(w, 2)
    assert W.shape == ((w.Hq + 2 * w.Hkv) * w.D, w.H) and W.dtype == np.uint16
    Wf = synth.bf16_bits_to_f32(W).astype(np.float64)
    assert abs(Wf.std() * np.sqrt(w.H) - 1.0) < 0.02
    assert np.array_equal(W, synth.make_qkv_weights(w, 2))
