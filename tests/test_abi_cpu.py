"""The C ABI on a machine without a GPU: loading, exports, struct layout, host validation.

Every call below fails host-side validation before anything touches CUDA, so it
runs without a device.
"""
import ctypes
import os
import re
import subprocess

import pytest

from block_wise_mask_tt_b300 import build as tt_build

tt_build.build(quiet=True)
from block_wise_mask_tt_b300 import tt  # noqa: E402


def test_exports_every_header_symbol():
    declared = tt.header_symbols()
    assert len(declared) >= 13
    out = subprocess.run(["nm", "-D", "--defined-only", tt.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (tt_\w+)$", out, flags=re.M))
    assert set(declared) <= exported, set(declared) - exported
    assert exported <= set(declared), exported - set(declared)
    for name in declared:
        assert hasattr(tt.lib, name)


def test_abi_version_and_status_strings():
    assert tt.tt_abi_version() == 4
    names = [tt.lib.tt_status_string(i).decode() for i in range(7)]
    assert names == ["TT_OK", "TT_ERR_INVALID_ARG", "TT_ERR_UNSUPPORTED", "TT_ERR_CUDA",
                     "TT_ERR_DEVICE", "TT_ERR_TIMEOUT", "TT_ERR_WORKSPACE"]


def _c_sizeof(type_name: str) -> int:
    src = ('#include "tt.h"\n#include <stdio.h>\nint main(void){printf("%%zu\\n", sizeof(%s));return 0;}\n'
           % type_name)
    import tempfile
    d = tempfile.mkdtemp(prefix="tt_sizeof_")
    c = os.path.join(d, "s.c")
    exe = os.path.join(d, "s")
    open(c, "w").write(src)
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(tt.HEADER_PATH), c, "-o", exe], check=True)
    return int(subprocess.run([exe], capture_output=True, text=True, check=True).stdout)


@pytest.mark.parametrize("name,cls", [("tt_attn_dims", tt.tt_attn_dims),
                                      ("tt_logits_spec", tt.tt_logits_spec),
                                      ("tt_step_desc", tt.tt_step_desc),
                                      ("tt_step_tensors", tt.tt_step_tensors)])
def test_struct_layout_matches_header(name, cls):
    assert ctypes.sizeof(cls) == _c_sizeof(name)


def _dims(**kw):
    base = dict(B=2, S=16, Hq=32, Hkv=2, D=128, max_ctx=256, page_size=0, max_pages=0, num_pages=0,
                softmax_scale=1.0, num_splits=0)
    base.update(kw)
    return tt.attn_dims(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), tt.TT_ERR_UNSUPPORTED),
    (dict(S=33), tt.TT_ERR_UNSUPPORTED),
    (dict(Hq=31), tt.TT_ERR_INVALID_ARG),
    (dict(B=0), tt.TT_ERR_INVALID_ARG),
    (dict(max_ctx=-1), tt.TT_ERR_INVALID_ARG),
    (dict(page_size=32, max_pages=4, num_pages=4), tt.TT_ERR_UNSUPPORTED),
    (dict(softmax_scale=0.0), tt.TT_ERR_INVALID_ARG),
    (dict(Hq=256, Hkv=1), tt.TT_ERR_UNSUPPORTED),
])
def test_attention_dims_rejected(kw, status):
    d = _dims(**kw)
    assert tt.tt_denoise_attn_workspace(d) == 0
    r = tt.lib.tt_denoise_attn(ctypes.byref(d), None, None, None, None, None, None, None, None, None,
                               None, 0, None)
    assert r == status, tt.lib.tt_last_error()


def test_attention_null_and_misaligned_pointers():
    d = _dims()
    assert tt.tt_denoise_attn_workspace(d) > 0
    r = tt.lib.tt_denoise_attn(ctypes.byref(d), None, 16, 16, 16, 16, None, None, 16, None, 16,
                               1 << 30, None)
    assert r == tt.TT_ERR_INVALID_ARG and b"q is null" in tt.lib.tt_last_error()
    r = tt.lib.tt_denoise_attn(ctypes.byref(d), 24, 16, 16, 16, 16, None, None, 16, None, 16,
                               1 << 30, None)
    assert r == tt.TT_ERR_INVALID_ARG and b"aligned" in tt.lib.tt_last_error()
    # paged cache needs a page table and lengths
    dp = _dims(page_size=64, max_pages=4, num_pages=8)
    r = tt.lib.tt_denoise_attn(ctypes.byref(dp), 16, 16, 16, 16, 16, None, None, 16, None, 16,
                               1 << 30, None)
    assert r == tt.TT_ERR_INVALID_ARG and b"page_table" in tt.lib.tt_last_error()
    # contiguous cache must not get one
    r = tt.lib.tt_denoise_attn(ctypes.byref(d), 16, 16, 16, 16, 16, 16, None, 16, None, 16,
                               1 << 30, None)
    assert r == tt.TT_ERR_INVALID_ARG


def test_unmask_validation():
    assert tt.tt_confidence_unmask_workspace(2, 16, 1024) > 0
    assert tt.tt_confidence_unmask_workspace(2, 33, 1024) == 0
    assert tt.tt_confidence_unmask_workspace(2, 16, 1022) == 0
    f = tt.lib.tt_confidence_unmask
    # mask id outside the vocabulary
    assert f(16, 16, None, 16, None, None, None, 2, 16, 1024, 1024, 0.8, 16, 16, 1 << 20, None) == \
        tt.TT_ERR_INVALID_ARG
    # max_steps range
    assert f(16, 16, None, 16, None, None, None, 2, 16, 1024, 3, 0.8, 0, 16, 1 << 20, None) == \
        tt.TT_ERR_INVALID_ARG
    # NaN gamma
    assert f(16, 16, None, 16, None, None, None, 2, 16, 1024, 3, float("nan"), 16, 16, 1 << 20,
             None) == tt.TT_ERR_INVALID_ARG
    # workspace too small / null
    need = tt.tt_confidence_unmask_workspace(2, 16, 1024)
    assert f(16, 16, None, 16, None, None, None, 2, 16, 1024, 3, 0.8, 16, 16, need - 16, None) == \
        tt.TT_ERR_WORKSPACE
    assert f(16, 16, None, 16, None, None, None, 2, 16, 1024, 3, 0.8, 16, None, need, None) == \
        tt.TT_ERR_WORKSPACE
    # misaligned logits
    assert f(20, 16, None, 16, None, None, None, 2, 16, 1024, 3, 0.8, 16, 16, need, None) == \
        tt.TT_ERR_INVALID_ARG


def test_adaln_validation():
    f = tt.lib.tt_adaln_modulate
    assert f(16, 16, 16, None, 0, 32, 2, 16, 100, 1e-5, None) == tt.TT_ERR_UNSUPPORTED  # H % 8
    assert f(16, 16, 16, None, 0, 32, 2, 16, 16384, 1e-5, None) == tt.TT_ERR_UNSUPPORTED
    assert f(16, 16, 16, None, 0, 16, 2, 16, 256, 1e-5, None) == tt.TT_ERR_INVALID_ARG  # alias
    assert f(None, 16, 16, None, 0, 32, 2, 16, 256, 1e-5, None) == tt.TT_ERR_INVALID_ARG
    assert f(16, 16, 16, 16, 0, 32, 2, 16, 256, 1e-5, None) == tt.TT_ERR_INVALID_ARG  # rows
    assert f(16, 16, 16, None, 0, 32, 2, 16, 256, -1.0, None) == tt.TT_ERR_INVALID_ARG


def test_step_validation():
    d = tt.step_desc(_dims(), 2688, 131072, 3, 0.8, 16, 1e-5, 0, 0, 0, 0.0, 20.0)
    assert tt.tt_denoise_workspace(d) > 0
    bad = tt.step_desc(_dims(), 2688, 131072, 3, 0.8, 0, 1e-5, 0, 0, 0, 0.0, 20.0)
    assert tt.tt_denoise_workspace(bad) == 0
    bad = tt.step_desc(_dims(), 2688, 131072, 131072, 0.8, 16, 1e-5, 0, 0, 0, 0.0, 20.0)
    assert tt.tt_denoise_workspace(bad) == 0
    bad = tt.step_desc(_dims(), 2688, 131072, 3, 0.8, 16, 1e-5, 0, 0, 2, 0.0, 20.0)
    assert tt.tt_denoise_workspace(bad) == 0
    t = tt.tt_step_tensors()
    r = tt.lib.tt_denoise_step(ctypes.byref(d), ctypes.byref(t), 16, 1 << 40, None)
    assert r == tt.TT_ERR_INVALID_ARG and b"x is null" in tt.lib.tt_last_error()


def test_split_count_and_workspace_scale():
    small = tt.tt_denoise_attn_workspace(_dims(max_ctx=256, num_splits=1))
    many = tt.tt_denoise_attn_workspace(_dims(max_ctx=256, num_splits=4))
    assert many > 3 * small // 2


def test_lmhead_validation():
    f = tt.lib.tt_lmhead_unmask
    ok_sampler = tt.tt_sampler(0, 0.8, 1.0, 16)

    def call(B=2, S=16, H=256, V=1024, mask=3, sampler=ok_sampler, hidden=16, w=16, ids=16, steps=16):
        return f(hidden, w, ids, None, steps, None, None, None, B, S, H, V, mask, ctypes.byref(sampler),
                 16, 1 << 20, None)
    assert call(B=0) == tt.TT_ERR_INVALID_ARG
    assert call(S=33) == tt.TT_ERR_UNSUPPORTED
    assert call(B=200, S=32) == tt.TT_ERR_UNSUPPORTED  # B*S above 4096
    assert call(H=100) == tt.TT_ERR_UNSUPPORTED        # H % 8
    assert call(H=32) == tt.TT_ERR_UNSUPPORTED         # H below one 64-wide slice
    assert call(V=32) == tt.TT_ERR_UNSUPPORTED         # V below one 64-row box
    assert call(mask=1024) == tt.TT_ERR_INVALID_ARG
    assert call(sampler=tt.tt_sampler(3, 0.8, 1.0, 16)) == tt.TT_ERR_INVALID_ARG
    assert call(sampler=tt.tt_sampler(0, 0.8, 0.0, 16)) == tt.TT_ERR_INVALID_ARG
    assert call(sampler=tt.tt_sampler(0, 0.8, 1.0, 0)) == tt.TT_ERR_INVALID_ARG
    assert call(hidden=None) == tt.TT_ERR_INVALID_ARG
    assert call(hidden=24) == tt.TT_ERR_INVALID_ARG and b"aligned" in tt.lib.tt_last_error()
    assert call(w=None) == tt.TT_ERR_INVALID_ARG
    assert call(steps=None) == tt.TT_ERR_INVALID_ARG
    assert tt.tt_lmhead_unmask_workspace(2, 33, 256) == 0


def test_qkv_validation():
    f = tt.lib.tt_qkv_project

    def call(B=2, S=16, H=256, Hq=4, Hkv=1, D=64, y=16, w=16, q=16, k=16, v=16):
        return f(y, w, q, k, v, B, S, H, Hq, Hkv, D, None)
    assert call(D=96) == tt.TT_ERR_UNSUPPORTED
    assert call(Hq=3, Hkv=2) == tt.TT_ERR_INVALID_ARG
    assert call(B=0) == tt.TT_ERR_INVALID_ARG
    assert call(H=32) == tt.TT_ERR_UNSUPPORTED
    assert call(H=100) == tt.TT_ERR_UNSUPPORTED
    assert call(y=None) == tt.TT_ERR_INVALID_ARG
    assert call(w=None) == tt.TT_ERR_INVALID_ARG
    assert call(q=24) == tt.TT_ERR_INVALID_ARG and b"aligned" in tt.lib.tt_last_error()
    assert call(v=None) == tt.TT_ERR_INVALID_ARG


def test_step_kind_and_projection_flags_validated():
    d = tt.step_desc(_dims(), 2688, 131072, 3, 0.8, 16, 1e-5, 0, 0, 5, 0.0, 20.0)
    assert tt.tt_denoise_workspace(d) == 0  # logits.kind outside 0, 1, TT_LOGITS_LM_HEAD
    d = tt.step_desc(_dims(), 2688, 131072, 3, 0.8, 16, 1e-5, 0, 0, 0, 0.0, 20.0)
    d.qkv_proj = 2
    assert tt.tt_denoise_workspace(d) == 0
    d.qkv_proj = 1
    assert tt.tt_denoise_workspace(d) > 0   # the projection needs no workspace of its own
    d = tt.step_desc(_dims(D=96), 2688, 131072, 3, 0.8, 16, 1e-5, 0, 0, 0, 0.0, 20.0, qkv_proj=True)
    assert tt.tt_denoise_workspace(d) == 0


def test_sampler_unmask_validation():
    f = tt.lib.tt_sampler_unmask
    need = tt.tt_confidence_unmask_workspace(2, 16, 1024)

    def call(sampler, mask=3, V=1024):
        s = None if sampler is None else ctypes.byref(sampler)
        return f(16, 16, None, 16, None, None, None, 2, 16, V, mask, s, 16, need, None)
    assert call(None) == tt.TT_ERR_INVALID_ARG
    assert call(tt.tt_sampler(3, 0.8, 1.0, 16)) == tt.TT_ERR_INVALID_ARG      # unknown kind
    assert call(tt.tt_sampler(0, 0.8, 1.0, 256)) == tt.TT_ERR_INVALID_ARG     # max_steps
    assert call(tt.tt_sampler(0, float("nan"), 1.0, 16)) == tt.TT_ERR_INVALID_ARG
    assert call(tt.tt_sampler(0, 0.8, -1.0, 16)) == tt.TT_ERR_INVALID_ARG     # temperature
    assert call(tt.tt_sampler(0, 0.8, float("inf"), 16)) == tt.TT_ERR_INVALID_ARG
    assert call(tt.tt_sampler(1, 0.8, 1.0, 16), mask=1024) == tt.TT_ERR_INVALID_ARG
    assert call(tt.tt_sampler(2, 0.8, 1.0, 16), V=1022) == tt.TT_ERR_UNSUPPORTED


@pytest.mark.parametrize("limit_us", [0, 1000001])
def test_selftest_wait_limit_rejected(limit_us):
    assert tt.lib.tt_selftest_wait_timeout(limit_us, None) == tt.TT_ERR_INVALID_ARG
    assert "limit_us" in tt.lib.tt_last_error().decode()
