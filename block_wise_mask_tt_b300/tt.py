"""ctypes binding of libtt (include/tt.h).

Argument marshalling only: every function here checks tensor placement/dtype/shape
against the C signature, passes raw device pointers and the current torch stream,
and raises ``TTError`` on a non-OK status.  All computation happens in the CUDA
kernels of ``libtt.so``; if the library is missing, importing this module fails.
PyTorch is used only to hold device memory and to name the stream.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtt.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "tt.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libtt.so not found at {LIB_PATH}: build it with `python -m block_wise_mask_tt_b300.build`"
        " (there is no CPU fallback)")
lib = ctypes.CDLL(LIB_PATH)

TT_OK, TT_ERR_INVALID_ARG, TT_ERR_UNSUPPORTED, TT_ERR_CUDA, TT_ERR_DEVICE, TT_ERR_TIMEOUT, \
    TT_ERR_WORKSPACE = range(7)


class TTError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        name = lib.tt_status_string(status).decode()
        super().__init__(f"{name}: {message}")


class tt_attn_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("S", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("D", ctypes.c_int), ("max_ctx", ctypes.c_int),
                ("page_size", ctypes.c_int), ("max_pages", ctypes.c_int),
                ("num_pages", ctypes.c_int), ("softmax_scale", ctypes.c_float),
                ("num_splits", ctypes.c_int)]


class tt_logits_spec(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint32), ("block_index", ctypes.c_int), ("kind", ctypes.c_int),
                ("boost_lo", ctypes.c_float), ("boost_hi", ctypes.c_float)]


class tt_step_desc(ctypes.Structure):
    _fields_ = [("attn", tt_attn_dims), ("H", ctypes.c_int), ("V", ctypes.c_int),
                ("mask_id", ctypes.c_int32), ("gamma", ctypes.c_float),
                ("max_steps", ctypes.c_int), ("ln_eps", ctypes.c_float),
                ("logits", tt_logits_spec), ("sampler", ctypes.c_int),
                ("temperature", ctypes.c_float), ("qkv_proj", ctypes.c_int)]


SAMPLER_CONFIDENCE, SAMPLER_MOCK_AR, SAMPLER_PREDICT_NOISE = 0, 1, 2
LOGITS_LM_HEAD = 2  # tt_logits_spec.kind of a step whose logits come from the LM head


class tt_stop_spec(ctypes.Structure):
    _fields_ = [("eos_id", ctypes.c_int32), ("pad_id", ctypes.c_int32), ("max_new_tokens", ctypes.c_int)]


class tt_sampler(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("gamma", ctypes.c_float), ("temperature", ctypes.c_float),
                ("max_steps", ctypes.c_int)]


_STEP_TENSOR_FIELDS = ("x", "shift_table", "scale_table", "q", "k_blk", "v_blk", "k_ctx", "v_ctx",
                       "page_table", "ctx_len", "ids", "n_masked", "steps", "commit_step", "y",
                       "attn_out", "logits", "conf", "commit", "w_vocab", "w_qkv")


class tt_step_tensors(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _STEP_TENSOR_FIELDS]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "tt_abi_version": (_I, []),
    "tt_status_string": (ctypes.c_char_p, [_I]),
    "tt_last_error": (ctypes.c_char_p, []),
    "tt_device_status": (_I, [_I]),
    "tt_adaln_modulate": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, ctypes.c_float, _P]),
    "tt_denoise_attn_workspace": (ctypes.c_size_t, [ctypes.POINTER(tt_attn_dims)]),
    "tt_denoise_attn": (_I, [ctypes.POINTER(tt_attn_dims), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                             ctypes.c_size_t, _P]),
    "tt_synthetic_logits": (_I, [ctypes.POINTER(tt_logits_spec), _P, _P, _P, _I, _I, _I,
                                 ctypes.c_int32, _P]),
    "tt_confidence_unmask_workspace": (ctypes.c_size_t, [_I, _I, _I]),
    "tt_confidence_unmask": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, ctypes.c_int32,
                                  ctypes.c_float, _I, _P, ctypes.c_size_t, _P]),
    "tt_sampler_unmask": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, ctypes.c_int32,
                               ctypes.POINTER(tt_sampler), _P, ctypes.c_size_t, _P]),
    "tt_confidence_unmask_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, ctypes.c_int32,
                                          ctypes.c_float, _I, _P]),
    "tt_lmhead_unmask_workspace": (ctypes.c_size_t, [_I, _I, _I]),
    "tt_lmhead_unmask": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_int32,
                              ctypes.POINTER(tt_sampler), _P, ctypes.c_size_t, _P]),
    "tt_qkv_project": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "tt_selftest_wait_timeout": (_I, [ctypes.c_uint32, _P]),
    "tt_denoise_workspace": (ctypes.c_size_t, [ctypes.POINTER(tt_step_desc)]),
    "tt_append_block": (_I, [ctypes.POINTER(tt_attn_dims), _P, _P, _P, _P, _P, _P, _P,
                             ctypes.POINTER(tt_stop_spec), _P, _P, _P, _I, _I, _P]),
    "tt_generate": (_I, [ctypes.POINTER(tt_step_desc), ctypes.POINTER(tt_step_tensors), _I,
                         ctypes.POINTER(tt_stop_spec), _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "tt_denoise_step": (_I, [ctypes.POINTER(tt_step_desc), ctypes.POINTER(tt_step_tensors), _P,
                             ctypes.c_size_t, _P]),
    "tt_denoise_block_loop": (_I, [ctypes.POINTER(tt_step_desc), ctypes.POINTER(tt_step_tensors),
                                   _P, ctypes.c_size_t, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def header_symbols() -> list[str]:
    """Names of the functions include/tt.h declares (parsed from the header text)."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^TT_API\s+[\w\s\*]+?\b(tt_\w+)\s*\(", text, flags=re.M)))


def _check(status: int) -> None:
    if status != TT_OK:
        raise TTError(status, lib.tt_last_error().decode())


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor], name: str, dtypes=None, numel: Optional[int] = None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
    return t.data_ptr()


_BF16 = (torch.bfloat16, torch.int16, torch.uint16)
_F32 = (torch.float32,)
_I32 = (torch.int32,)
_U8 = (torch.uint8,)


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """Zero-filled device scratch of at least nbytes (the caller owns it)."""
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device or "cuda")


# ------------------------------------------------------------------------- calls
def tt_abi_version() -> int:
    return lib.tt_abi_version()


def tt_device_status(reset: bool = True) -> int:
    return lib.tt_device_status(1 if reset else 0)


def tt_adaln_modulate(x, shift, scale, y, eps: float = 1e-5, row_index=None, table_rows: int = 0,
                      stream=None) -> None:
    B, S, H = x.shape
    nvec = (B if row_index is None else table_rows) * H
    _check(lib.tt_adaln_modulate(
        _ptr(x, "x", _BF16), _ptr(shift, "shift", _F32, nvec), _ptr(scale, "scale", _F32, nvec),
        _ptr(row_index, "row_index", _I32, B), int(table_rows), _ptr(y, "y", _BF16, B * S * H),
        B, S, H, float(eps), _stream(stream)))


def attn_dims(B, S, Hq, Hkv, D, max_ctx=0, page_size=0, max_pages=0, num_pages=0,
              softmax_scale=1.0, num_splits=0) -> tt_attn_dims:
    return tt_attn_dims(B, S, Hq, Hkv, D, max_ctx, page_size, max_pages, num_pages,
                        float(softmax_scale), num_splits)


def tt_denoise_attn_workspace(dims: tt_attn_dims) -> int:
    return int(lib.tt_denoise_attn_workspace(ctypes.byref(dims)))


def tt_denoise_attn(dims: tt_attn_dims, q, k_blk, v_blk, k_ctx, v_ctx, page_table, ctx_len, out,
                    lse=None, ws=None, stream=None) -> None:
    if ws is None:
        ws = workspace(tt_denoise_attn_workspace(dims), q.device)
    _check(lib.tt_denoise_attn(
        ctypes.byref(dims), _ptr(q, "q", _BF16), _ptr(k_blk, "k_blk", _BF16),
        _ptr(v_blk, "v_blk", _BF16), _ptr(k_ctx, "k_ctx", _BF16), _ptr(v_ctx, "v_ctx", _BF16),
        _ptr(page_table, "page_table", _I32), _ptr(ctx_len, "ctx_len", _I32, dims.B),
        _ptr(out, "out", _BF16, dims.B * dims.S * dims.Hq * dims.D),
        _ptr(lse, "lse", _F32, dims.B * dims.S * dims.Hq), ws.data_ptr(), ws.numel(),
        _stream(stream)))


def tt_synthetic_logits(spec: tt_logits_spec, logits, B, S, V, mask_id, ids=None, steps=None,
                        stream=None) -> None:
    _check(lib.tt_synthetic_logits(
        ctypes.byref(spec), _ptr(ids, "ids", _I32, B * S), _ptr(steps, "steps", _I32, B),
        _ptr(logits, "logits", _F32, B * S * V), B, S, V, int(mask_id), _stream(stream)))


def tt_confidence_unmask_workspace(B, S, V) -> int:
    return int(lib.tt_confidence_unmask_workspace(B, S, V))


def tt_confidence_unmask(logits, ids, steps, B, S, V, mask_id, gamma, max_steps, n_masked=None,
                         conf=None, commit=None, commit_step=None, ws=None, stream=None) -> None:
    if ws is None:
        ws = workspace(tt_confidence_unmask_workspace(B, S, V), logits.device)
    _check(lib.tt_confidence_unmask(
        _ptr(logits, "logits", _F32, B * S * V), _ptr(ids, "ids", _I32, B * S),
        _ptr(n_masked, "n_masked", _I32, B), _ptr(steps, "steps", _I32, B),
        _ptr(conf, "conf", _F32, B * S), _ptr(commit, "commit", _U8, B * S),
        _ptr(commit_step, "commit_step", _U8, B * S), B, S, V, int(mask_id), float(gamma),
        int(max_steps), ws.data_ptr(), ws.numel(), _stream(stream)))


def tt_sampler_unmask(logits, ids, steps, B, S, V, mask_id, sampler: tt_sampler, n_masked=None,
                      conf=None, commit=None, commit_step=None, ws=None, stream=None) -> None:
    if ws is None:
        ws = workspace(tt_confidence_unmask_workspace(B, S, V), logits.device)
    _check(lib.tt_sampler_unmask(
        _ptr(logits, "logits", _F32, B * S * V), _ptr(ids, "ids", _I32, B * S),
        _ptr(n_masked, "n_masked", _I32, B), _ptr(steps, "steps", _I32, B),
        _ptr(conf, "conf", _F32, B * S), _ptr(commit, "commit", _U8, B * S),
        _ptr(commit_step, "commit_step", _U8, B * S), B, S, V, int(mask_id),
        ctypes.byref(sampler), ws.data_ptr(), ws.numel(), _stream(stream)))


def tt_qkv_project(y, w_qkv, q, k_blk, v_blk, B, S, H, Hq, Hkv, D, stream=None) -> None:
    _check(lib.tt_qkv_project(
        _ptr(y, "y", _BF16, B * S * H), _ptr(w_qkv, "w_qkv", _BF16, (Hq + 2 * Hkv) * D * H),
        _ptr(q, "q", _BF16, B * S * Hq * D), _ptr(k_blk, "k_blk", _BF16, B * S * Hkv * D),
        _ptr(v_blk, "v_blk", _BF16, B * S * Hkv * D), B, S, H, Hq, Hkv, D, _stream(stream)))


def tt_lmhead_unmask_workspace(B, S, H) -> int:
    return int(lib.tt_lmhead_unmask_workspace(B, S, H))


def tt_lmhead_unmask(hidden, w_vocab, ids, steps, B, S, H, V, mask_id, sampler: tt_sampler,
                     n_masked=None, conf=None, commit=None, commit_step=None, ws=None,
                     stream=None) -> None:
    if ws is None:
        ws = workspace(tt_lmhead_unmask_workspace(B, S, H), hidden.device)
    _check(lib.tt_lmhead_unmask(
        _ptr(hidden, "hidden", _BF16, B * S * H), _ptr(w_vocab, "w_vocab", _BF16, V * H),
        _ptr(ids, "ids", _I32, B * S), _ptr(n_masked, "n_masked", _I32, B),
        _ptr(steps, "steps", _I32, B), _ptr(conf, "conf", _F32, B * S),
        _ptr(commit, "commit", _U8, B * S), _ptr(commit_step, "commit_step", _U8, B * S),
        B, S, H, V, int(mask_id), ctypes.byref(sampler), ws.data_ptr(), ws.numel(),
        _stream(stream)))


def tt_confidence_unmask_noalloc(logits, ids, steps, B, S, V, mask_id, gamma, max_steps,
                                 n_masked=None, conf=None, commit=None, commit_step=None,
                                 stream=None) -> None:
    """tt_confidence_unmask without a workspace: the library's fixed device scratch is
    used instead (for callers that cannot allocate; calls must not overlap)."""
    _check(lib.tt_confidence_unmask_noalloc(
        _ptr(logits, "logits", _F32, B * S * V), _ptr(ids, "ids", _I32, B * S),
        _ptr(n_masked, "n_masked", _I32, B), _ptr(steps, "steps", _I32, B),
        _ptr(conf, "conf", _F32, B * S), _ptr(commit, "commit", _U8, B * S),
        _ptr(commit_step, "commit_step", _U8, B * S), B, S, V, int(mask_id), float(gamma),
        int(max_steps), _stream(stream)))


def tt_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launches a wait that is meant to run out after limit_us microseconds (the
    library's failure path); tt_device_status() then reports TT_ERR_TIMEOUT."""
    _check(lib.tt_selftest_wait_timeout(int(limit_us), _stream(stream)))


def step_desc(attn: tt_attn_dims, H, V, mask_id, gamma, max_steps, ln_eps, seed, block_index,
              kind, boost_lo, boost_hi, sampler: int = SAMPLER_CONFIDENCE,
              temperature: float = 1.0, qkv_proj: bool = False) -> tt_step_desc:
    return tt_step_desc(attn, H, V, mask_id, float(gamma), max_steps, float(ln_eps),
                        tt_logits_spec(seed & 0xFFFFFFFF, block_index, kind, float(boost_lo),
                                       float(boost_hi)), int(sampler), float(temperature),
                        1 if qkv_proj else 0)


def step_tensors(**tensors) -> tt_step_tensors:
    t = tt_step_tensors()
    for name in _STEP_TENSOR_FIELDS:
        v = tensors.pop(name, None)
        if v is not None:
            setattr(t, name, _ptr(v, name))
    if tensors:
        raise TypeError(f"unknown step tensors {sorted(tensors)}")
    return t


def tt_denoise_workspace(desc: tt_step_desc) -> int:
    return int(lib.tt_denoise_workspace(ctypes.byref(desc)))


def tt_denoise_step(desc: tt_step_desc, tensors: tt_step_tensors, ws, stream=None) -> None:
    _check(lib.tt_denoise_step(ctypes.byref(desc), ctypes.byref(tensors), ws.data_ptr(),
                               ws.numel(), _stream(stream)))


def tt_denoise_block_loop(desc: tt_step_desc, tensors: tt_step_tensors, ws, stream=None) -> None:
    _check(lib.tt_denoise_block_loop(ctypes.byref(desc), ctypes.byref(tensors), ws.data_ptr(),
                                     ws.numel(), _stream(stream)))


def tt_append_block(dims: tt_attn_dims, k_blk, v_blk, k_ctx, v_ctx, page_table, ctx_len, ids,
                    stop: tt_stop_spec, generated, done, out_tokens=None, out_stride=0, out_offset=0,
                    stream=None) -> None:
    _check(lib.tt_append_block(
        ctypes.byref(dims), _ptr(k_blk, "k_blk", _BF16), _ptr(v_blk, "v_blk", _BF16),
        _ptr(k_ctx, "k_ctx", _BF16), _ptr(v_ctx, "v_ctx", _BF16), _ptr(page_table, "page_table", _I32),
        _ptr(ctx_len, "ctx_len", _I32, dims.B), _ptr(ids, "ids", _I32, dims.B * dims.S),
        ctypes.byref(stop), _ptr(generated, "generated", _I32, dims.B), _ptr(done, "done", _U8, dims.B),
        _ptr(out_tokens, "out_tokens", _I32), int(out_stride), int(out_offset), _stream(stream)))


def tt_generate(desc: tt_step_desc, tensors: tt_step_tensors, n_blocks: int, stop: tt_stop_spec,
                generated, done, out_tokens, ws, stream=None) -> None:
    B, S = desc.attn.B, desc.attn.S
    _check(lib.tt_generate(ctypes.byref(desc), ctypes.byref(tensors), int(n_blocks), ctypes.byref(stop),
                           _ptr(generated, "generated", _I32, B), _ptr(done, "done", _U8, B),
                           _ptr(out_tokens, "out_tokens", _I32, B * n_blocks * S), ws.data_ptr(),
                           ws.numel(), _stream(stream)))
