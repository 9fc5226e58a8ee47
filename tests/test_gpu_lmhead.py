"""tt_lmhead_unmask (LM head fused with the sampler step) against the oracle.

The oracle forms the logits exactly (fp64 products of the bf16 operands); the kernel
accumulates in fp32 on the tensor cores.  Tolerances follow from that accumulation:
with K = H products per logit added in 16-wide slices, each logit's error is at most
delta = (K/16 + 16) * 2^-24 * sum_k |h_k W_jk|, so
* tokens must equal the oracle's where its top two logits differ by more than
  2 delta, and otherwise be within 2 delta of the top (a near-tie);
* confidences must agree within exp(2 delta / tau) - 1 relative, plus the 1e-5 of
  the fp32 softmax sums;
* commits, ids, steps and commit_step must be bit-exact, except in sequences where
  the decision compares values closer than that (a confidence near gamma, a floor or
  schedule ranking between near-equal confidences, or a token near-tie): those are
  checked for validity only and counted.
"""
import numpy as np
import pytest
import torch

import oracle
from block_wise_mask_tt_b300 import synth
from gpu_util import compare_lmhead as compare, dev, host

pytestmark = pytest.mark.gpu

CONFIDENCE, MOCK_AR, PREDICT_NOISE = 0, 1, 2


@pytest.fixture(scope="module")
def tt():
    from block_wise_mask_tt_b300 import tt as _tt
    return _tt


def _weights(seed, V, H, logit_std=10.0):
    w = synth.Workload("lm", B=1, L=0, S=1, Hq=1, Hkv=1, D=64, H=H, V=V, lm_logit_std=logit_std)
    return synth.make_lmhead_weights(w, seed, rows=4096)


def _hidden(seed, B, S, H):
    w = synth.Workload("lm", B=B, L=0, S=S, Hq=1, Hkv=1, D=64, H=H, V=64)
    return synth.make_hidden(w, seed)


def _state(seed, B, S, mask, frac_masked, V):
    rng = np.random.default_rng(seed)
    ids = np.full((B, S), mask, np.int64)
    dec = rng.random((B, S)) >= frac_masked
    ids[dec] = rng.integers(0, V, int(dec.sum()))
    ids[dec & (ids == mask)] = (mask + 1) % V
    steps = rng.integers(0, 3, B).astype(np.int32) * (dec.any(1))
    cs = np.where(dec, rng.integers(1, 3, (B, S)), 0).astype(np.uint8)
    return ids.astype(np.int32), steps.astype(np.int32), cs


def run_gpu(tt, h, W, ids0, steps0, cs0, mask, kind, gamma, T, tau):
    B, S, H = h.shape
    V = W.shape[0]
    ids, steps, cs = dev(ids0), dev(steps0), dev(cs0)
    n_masked = torch.full((B,), -5, dtype=torch.int32, device="cuda")
    conf = torch.full((B, S), -1.0, dtype=torch.float32, device="cuda")
    commit = torch.full((B, S), 7, dtype=torch.uint8, device="cuda")
    tt.tt_lmhead_unmask(dev(h), dev(W), ids, steps, B, S, H, V, mask, tt.tt_sampler(kind, gamma, tau, T),
                        n_masked=n_masked, conf=conf, commit=commit, commit_step=cs)
    torch.cuda.synchronize()
    assert tt.tt_device_status(True) == 0
    return dict(ids=host(ids), steps=host(steps), n_masked=host(n_masked), conf=host(conf),
                commit=host(commit), commit_step=host(cs))


CASES = [
    # (B, S, H, V, mask, frac_masked): one and several 128-row tiles, ragged vocabulary
    # tails (units of 64 ids and 256-id tiles), H with and without a partial 64-slice
    (1, 16, 256, 1024, 3, 1.0),
    (3, 16, 192, 3000, 3, 0.7),
    (20, 16, 256, 5000, 4999, 0.9),
    (9, 32, 200, 777, 0, 0.6),
    (40, 8, 128, 2048, 100, 0.5),
    (2, 5, 64, 64, 63, 1.0),
    (128, 32, 128, 1024, 5, 0.9),  # the largest batch: B*S = 4096 rows, 32 row tiles
]


@pytest.mark.parametrize("B,S,H,V,mask,frac", CASES)
def test_lmhead_confidence_matches_oracle(tt, B, S, H, V, mask, frac):
    h = _hidden(B * 7 + V, B, S, H)
    W = _weights(V + H, V, H)
    ids0, steps0, cs0 = _state(B + S, B, S, mask, frac, V)
    T = S
    gpu = run_gpu(tt, h, W, ids0, steps0, cs0, mask, CONFIDENCE, 0.8, T, 1.0)
    excl = compare(gpu, h, W, ids0, steps0, cs0, mask, CONFIDENCE, 0.8, T, 1.0)
    assert excl <= max(1, B // 3)


@pytest.mark.parametrize("kind,tau", [(CONFIDENCE, 0.5), (CONFIDENCE, 2.0), (MOCK_AR, 1.0),
                                      (PREDICT_NOISE, 1.0)])
def test_lmhead_samplers(tt, kind, tau):
    B, S, H, V, mask = 12, 16, 320, 4096, 7
    h = _hidden(5, B, S, H)
    W = _weights(6, V, H)
    ids0, steps0, cs0 = _state(9, B, S, mask, 0.8, V)
    gpu = run_gpu(tt, h, W, ids0, steps0, cs0, mask, kind, 0.8, S, tau)
    compare(gpu, h, W, ids0, steps0, cs0, mask, kind, 0.8, S, tau)


def test_lmhead_equal_rows_tie_to_lowest_id(tt):
    """Two identical rows of W produce bit-identical logits; the lower id must win."""
    B, S, H, V, mask = 2, 8, 128, 1000, 3
    h = _hidden(21, B, S, H)
    h[:, :, 5] = synth.f32_to_bf16_bits(np.array([4.0], np.float32))[0]
    W = _weights(22, V, H, 1.0)
    strong = np.zeros(H, np.uint16)
    strong[5] = synth.f32_to_bf16_bits(np.array([2.0], np.float32))[0]  # logit exactly 8
    W[611] = strong
    W[37] = strong
    W[998] = strong
    ids0 = np.full((B, S), mask, np.int32)
    gpu = run_gpu(tt, h, W, ids0, np.zeros(B, np.int32), np.zeros((B, S), np.uint8), mask, CONFIDENCE,
                  0.0, S, 1.0)
    lg = synth.bf16_bits_to_f32(h).astype(np.float64).reshape(-1, H) @ synth.bf16_bits_to_f32(W).astype(np.float64).T
    top = np.argmax(np.where(np.arange(V) == mask, -np.inf, lg), axis=1)
    assert np.all(top == 37)
    assert np.all(gpu["ids"] == 37)


def test_lmhead_nothing_masked(tt):
    B, S, H, V, mask = 3, 4, 64, 256, 5
    h = _hidden(1, B, S, H)
    W = _weights(2, V, H)
    ids0 = np.arange(B * S, dtype=np.int32).reshape(B, S) + 10
    steps0 = np.array([2, 0, 4], np.int32)
    gpu = run_gpu(tt, h, W, ids0, steps0, np.ones((B, S), np.uint8), mask, CONFIDENCE, 0.8, S, 1.0)
    assert np.array_equal(gpu["ids"], ids0) and np.array_equal(gpu["steps"], steps0)
    assert np.all(gpu["n_masked"] == 0) and not gpu["commit"].any() and np.all(gpu["conf"] == 0)


def test_lmhead_rejects_bad_arguments(tt):
    h = torch.zeros((1, 4, 64), dtype=torch.int16, device="cuda")
    W = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    ids = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    steps = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = tt.tt_sampler(0, 0.8, 1.0, 4)
    with pytest.raises(tt.TTError):
        tt.tt_lmhead_unmask(h, W, ids, steps, 1, 4, 64, 64, 64, s)  # mask id outside V
    with pytest.raises(tt.TTError):
        tt.tt_lmhead_unmask(h, W[:32], ids, steps, 1, 4, 64, 32, 3, s)  # V < 64
    with pytest.raises(tt.TTError):
        tt.tt_lmhead_unmask(h, W, ids, steps, 1, 4, 64, 64, 3, tt.tt_sampler(0, 0.8, 0.0, 4))


@pytest.mark.parametrize("B", [1, 32])
def test_lmhead_full_vocabulary(tt, B):
    """H = 2688, V = 131072 as in the single-sequence and batched workloads, all rows
    masked (the first step of a block); the oracle checks sampled sequences."""
    S, H, V, mask = 16, 2688, 131072, 3
    w = synth.SINGLE.replace(B=B)
    h = synth.make_hidden(w, 3)
    W = synth.make_lmhead_weights(w, 4)
    ids0 = np.full((B, S), mask, np.int32)
    gpu = run_gpu(tt, h, W, ids0, np.zeros(B, np.int32), np.zeros((B, S), np.uint8), mask, CONFIDENCE,
                  0.8, S, 1.0)
    seqs = [0] if B == 1 else [0, 13, 31]
    excl = compare(gpu, h, W, ids0, np.zeros(B, np.int32), np.zeros((B, S), np.uint8), mask, CONFIDENCE,
                   0.8, S, 1.0, seqs=seqs)
    # every sampled sequence was checked for validity in full; at least one of the
    # batched ones also bit for bit
    assert B == 1 or excl < len(seqs)
    # every sequence took one step and committed at least one position
    assert np.all(gpu["steps"] == 1) and np.all(gpu["commit"].sum(1) >= 1)
