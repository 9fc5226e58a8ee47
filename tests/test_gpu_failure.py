"""The device-side failure path, exercised without any fault: a bounded wait that
runs out reports TT_ERR_TIMEOUT through the device error word, the kernel returns,
and the context stays usable for the next call."""
import math

import numpy as np
import pytest
import torch

import oracle
from block_wise_mask_tt_b300 import synth
from gpu_util import bf16_to_f64, check_attention, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tt():
    from block_wise_mask_tt_b300 import tt as _tt
    return _tt


def test_wait_that_runs_out_reports_timeout_and_context_survives(tt):
    assert tt.tt_device_status(True) == tt.TT_OK
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    tt.tt_selftest_wait_timeout(2000)  # 2 ms on an mbarrier nothing arrives on
    t1.record()
    t1.synchronize()
    assert t0.elapsed_time(t1) >= 1.9  # the wait really waited for its limit
    assert tt.tt_device_status(False) == tt.TT_ERR_TIMEOUT
    assert "ran out" in tt.lib.tt_last_error().decode()
    assert tt.tt_device_status(True) == tt.TT_ERR_TIMEOUT  # read and cleared
    assert tt.tt_device_status(True) == tt.TT_OK

    # the context is usable: an attention call right after agrees with the oracle
    w = synth.Workload("t", B=2, L=300, S=16, Hq=32, Hkv=2, D=128, H=256, V=1024,
                       q_prescale=1 / math.sqrt(128))
    inp = synth.make_attention_inputs(w, seed=8)
    dims = tt.attn_dims(w.B, w.S, w.Hq, w.Hkv, w.D, inp["k_ctx"].shape[1], 0, 0, 0, w.softmax_scale, 0)
    out = torch.zeros((w.B, w.S, w.Hq, w.D), dtype=torch.int16, device="cuda")
    tt.tt_denoise_attn(dims, dev(inp["q"]), dev(inp["k_blk"]), dev(inp["v_blk"]), dev(inp["k_ctx"]),
                       dev(inp["v_ctx"]), None, dev(inp["ctx_len"]), out)
    assert tt.tt_device_status(True) == tt.TT_OK
    Or, _ = oracle.denoise_attention(inp, w.softmax_scale)
    check_attention(bf16_to_f64(host(out)), Or)


def test_first_error_wins_and_timeout_repeats(tt):
    """Two runs in a row on one stream: the word keeps the first code until reset."""
    tt.tt_selftest_wait_timeout(500)
    tt.tt_selftest_wait_timeout(500)
    assert tt.tt_device_status(True) == tt.TT_ERR_TIMEOUT
    assert tt.tt_device_status(True) == tt.TT_OK
