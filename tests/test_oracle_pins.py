"""The oracle against its pins (library routines, closed forms, invariants)."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("check", pins.ATTENTION_CHECKS, ids=lambda f: f.__name__)
def test_attention(check):
    check(oracle.denoise_attention)


def test_attention_rows_match_full():
    import numpy as np
    inp = pins.tiny_attention_inputs(21, 2, 5, 4, 2, 8, [7, 3], paged=True, page_size=4)
    O, lse = oracle.denoise_attention(inp, 0.4)
    rows = [(0, 0, 0), (1, 4, 3), (1, 2, 1), (0, 3, 2)]
    Or, lr = oracle.denoise_attention_rows(inp, 0.4, rows)
    for i, (b, s, h) in enumerate(rows):
        np.testing.assert_allclose(Or[i], O[b, s, h], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lr[i], lse[b, s, h], rtol=1e-13, atol=1e-13)


def test_paged_equals_contiguous():
    import numpy as np
    a = pins.tiny_attention_inputs(22, 3, 4, 4, 2, 8, [9, 1, 16], paged=True, page_size=4)
    c = {k: a[k] for k in ("q", "k_blk", "v_blk", "ctx_len")}
    L = 16
    B, Hkv, D = 3, 2, 8
    kc = np.zeros((B, L, Hkv, D), np.uint16)
    vc = np.zeros((B, L, Hkv, D), np.uint16)
    for b in range(B):
        for t in range(int(a["ctx_len"][b])):
            kc[b, t] = a["k_pages"][a["page_table"][b, t // 4], t % 4]
            vc[b, t] = a["v_pages"][a["page_table"][b, t // 4], t % 4]
    c["k_ctx"], c["v_ctx"] = kc, vc
    Oa, la = oracle.denoise_attention(a, 0.3)
    Oc, lc = oracle.denoise_attention(c, 0.3)
    np.testing.assert_array_equal(Oa, Oc)
    np.testing.assert_array_equal(la, lc)


@pytest.mark.parametrize("check", pins.ADALN_CHECKS, ids=lambda f: f.__name__)
def test_adaln(check):
    check(oracle.adaln_modulate)


@pytest.mark.parametrize("check", pins.UNMASK_ROW_CHECKS, ids=lambda f: f.__name__)
def test_unmask_row(check):
    check(oracle.row_confidence)


@pytest.mark.parametrize("check", pins.UNMASK_STEP_CHECKS, ids=lambda f: f.__name__)
def test_unmask_step(check):
    check(oracle.unmask_step)


@pytest.mark.parametrize("check", pins.BLOCK_CHECKS, ids=lambda f: f.__name__)
def test_block(check):
    check(oracle.denoise_block)


def test_operating_point_golden():
    """The workloads use the pages' operating point (tests/golden/operating_point.json)."""
    import json
    import os
    from block_wise_mask_tt_b300 import synth
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "operating_point.json")))
    for w in synth.WORKLOADS[:4]:
        assert w.gamma == g["confidence_threshold"]["value"]
        assert w.S == g["block_size"]["value"]
        assert w.steps_max == g["steps_per_block"]["value"]
        assert w.mask_id == g["mask_token_id"]["value"]
    r = oracle.denoise_block(16, 16, 3, 0.8, pins._random_logits_fn(0, 64, 3))
    assert r["trace"][0]["t"] == g["first_timestep"]["value"]


@pytest.mark.parametrize("check", pins.SAMPLER_CHECKS, ids=lambda f: f.__name__)
def test_samplers(check):
    from oracle.samplers import sampler_step
    check(sampler_step)


def test_sampler_confidence_equals_unmask_step():
    """The confidence sampler at tau = 1 is the main oracle's step."""
    import numpy as np
    from oracle.samplers import sampler_step
    fn = pins._random_logits_fn(9, 512, 3)
    ids = np.full(16, 3)
    ids[[1, 4]] = [10, 11]
    lg = fn(2, np.arange(16))
    a = oracle.unmask_step(lg, ids, 2, 3, 0.8, 16)
    b = sampler_step(lg, ids, 2, 3, 16, 0, 0.8, 1.0)
    for k in ("ids", "commit", "commit_step", "n_masked", "steps", "k_min"):
        assert np.array_equal(a[k], b[k]), k
    assert np.allclose(a["conf"], b["conf"], rtol=1e-15, atol=0)
