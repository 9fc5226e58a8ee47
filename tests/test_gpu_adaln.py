"""tt_adaln_modulate against the fp64 oracle (one bf16 ulp plus the fp32 statistics error)."""
import numpy as np
import pytest
import torch

import oracle
from block_wise_mask_tt_b300 import synth
from gpu_util import adaln_tol, bf16_to_f64, bf16_ulp, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tt():
    from block_wise_mask_tt_b300 import tt as _tt
    return _tt


def _check(y_bits, ref, shift):
    got = bf16_to_f64(y_bits)
    err = np.abs(got - ref)
    tol = adaln_tol(ref, np.broadcast_to(shift, ref.shape))
    assert np.all(err <= tol), float((err / tol).max())


@pytest.mark.parametrize("B,S,H", [(1, 16, 256), (1, 16, 2688), (4, 32, 2688), (3, 5, 8), (2, 3, 8192)])
def test_adaln_per_sequence(tt, B, S, H):
    w = synth.SINGLE.replace(B=B, S=S, H=H)
    a = synth.make_adaln_inputs(w, seed=B * 100 + S)
    y = torch.empty((B, S, H), dtype=torch.int16, device="cuda")
    tt.tt_adaln_modulate(dev(a["x"]), dev(a["shift"]), dev(a["scale"]), y, eps=1e-5)
    torch.cuda.synchronize()
    ref = oracle.adaln_modulate(a["x"], a["shift"][:, None, :], a["scale"][:, None, :], 1e-5)
    _check(host(y), ref, a["shift"][:, None, :])


def test_adaln_table_rows(tt):
    B, S, H = 6, 16, 2688
    w = synth.SINGLE.replace(B=B, S=S, H=H)
    a = synth.make_adaln_inputs(w, seed=5)
    rows = np.array([16, 0, 7, 16, 1, 9], np.int32)
    y = torch.empty((B, S, H), dtype=torch.int16, device="cuda")
    tt.tt_adaln_modulate(dev(a["x"]), dev(a["shift_table"]), dev(a["scale_table"]), y, eps=1e-5,
                         row_index=dev(rows), table_rows=S + 1)
    torch.cuda.synchronize()
    ref = oracle.adaln_modulate(a["x"], a["shift_table"][rows][:, None, :],
                                a["scale_table"][rows][:, None, :], 1e-5)
    _check(host(y), ref, a["shift_table"][rows][:, None, :])


def test_adaln_constant_row_and_scale(tt):
    B, S, H = 1, 4, 512
    x = np.full((B, S, H), synth.f32_to_bf16_bits(np.float32(-2.5)), np.uint16)
    x[0, 1] = synth.f32_to_bf16_bits(np.linspace(-3, 3, H).astype(np.float32))
    shift = (np.arange(H, dtype=np.float32) / H)[None]
    scale = np.full((1, H), 0.5, np.float32)
    y = torch.empty((B, S, H), dtype=torch.int16, device="cuda")
    tt.tt_adaln_modulate(dev(x), dev(shift), dev(scale), y, eps=1e-5)
    torch.cuda.synchronize()
    got = bf16_to_f64(host(y))
    # constant rows give exactly shift (rounded to bf16)
    np.testing.assert_array_equal(got[0, 0], bf16_to_f64(synth.f32_to_bf16_bits(shift[0])))
    _check(host(y), oracle.adaln_modulate(x, shift[:, None, :], scale[:, None, :], 1e-5),
           shift[:, None, :])


def test_adaln_bad_table_row_is_reported(tt):
    B, S, H = 2, 4, 64
    x = dev(synth.f32_to_bf16_bits(np.ones((B, S, H), np.float32)))
    tab = dev(np.zeros((S + 1, H), np.float32))
    rows = dev(np.array([1, S + 1], np.int32))
    y = torch.zeros((B, S, H), dtype=torch.int16, device="cuda")
    assert tt.tt_device_status(True) == 0
    tt.tt_adaln_modulate(x, tab, tab, y, row_index=rows, table_rows=S + 1)
    assert tt.tt_device_status(True) == tt.TT_ERR_DEVICE
    assert np.all(host(y)[1] == 0)  # the bad sequence was skipped
    assert tt.tt_device_status(True) == 0
