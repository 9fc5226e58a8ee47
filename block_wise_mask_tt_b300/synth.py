"""Seeded synthetic inputs for one TwoTower denoise step.

This module only manufactures inputs: bf16 tensors for attention and adaLN, context
lengths and shuffled page tables, and the per-step logits that stand in for the
denoiser's LM head. It contains none of the method's arithmetic (no LayerNorm, no
attention, no softmax, no unmask decision), so both the CUDA path and the CPU oracle
can be fed from it without sharing any part of the computation they are compared on.

Logits stand-in ("Nemotron-Labs-TwoTower" wiki, Block-wise generation: every denoising
step predicts all masked positions in parallel).  The real LM head needs trained
weights, so each step's logits are regenerated from a counter-based hash of
(seed, sequence, block, step, position, vocabulary id):

* the hash is MurmurHash3_x86_32 of one 4-byte little-endian key with a 32-bit seed,
  implemented here from its published definition (Austin Appleby, public domain);
* noise for id v is an Irwin-Hall(4) sum of the four bytes of hash(v, h_row),
  centred and scaled to unit variance with one fp32 multiply (an approximately
  N(0,1) value; the integer sum and its conversion to fp32 are exact);
* one planted id per row gets a boost lo + u*(hi-lo), u a 24-bit uniform, added
  with single fp32 operations.

The CUDA logits kernel implements the same hash independently; the two are compared
bit for bit on the GPU, and this implementation is pinned to scikit-learn's
``murmurhash3_32`` on the CPU.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

# ----------------------------------------------------------------------------------
# bf16 storage helpers (round-to-nearest-even from fp32)
# ----------------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------------
# MurmurHash3_x86_32 over one 4-byte key
# ----------------------------------------------------------------------------------

_M3_C1 = np.uint32(0xCC9E2D51)
_M3_C2 = np.uint32(0x1B873593)
_M3_ADD = np.uint32(0xE6546B64)
_M3_F1 = np.uint32(0x85EBCA6B)
_M3_F2 = np.uint32(0xC2B2AE35)


def _rotl32(x: np.ndarray, r: int) -> np.ndarray:
    return (x << np.uint32(r)) | (x >> np.uint32(32 - r))


def murmur3_32(key, seed) -> np.ndarray:
    """MurmurHash3_x86_32 of the 4 little-endian bytes of ``key`` (uint32) under ``seed``.

    Vectorised over numpy broadcasting; always returns a uint32 ndarray.
    """
    k = np.atleast_1d(np.asarray(key, dtype=np.int64).astype(np.uint32))
    h = np.atleast_1d(np.asarray(seed, dtype=np.int64).astype(np.uint32))
    k = k * _M3_C1
    k = _rotl32(k, 15)
    k = k * _M3_C2
    h = h ^ k
    h = _rotl32(h, 13)
    h = h * np.uint32(5) + _M3_ADD
    h = h ^ np.uint32(4)  # total key length in bytes
    h = h ^ (h >> np.uint32(16))
    h = h * _M3_F1
    h = h ^ (h >> np.uint32(13))
    h = h * _M3_F2
    h = h ^ (h >> np.uint32(16))
    return h


# ----------------------------------------------------------------------------------
# Logits stand-in
# ----------------------------------------------------------------------------------

LOGITS_UNIFORM = 0  # boost ~ U(boost_lo, boost_hi)
LOGITS_BIMODAL = 1  # boost ~ U(0, 4) or U(10, 20), one hash bit picks which
BIMODAL_RANGES = ((0.0, 4.0), (10.0, 20.0))

KEY_PLANTED = 0xFFFFFFFF  # hash keys >= 2**31 are never vocabulary ids
KEY_BOOST = 0xFFFFFFFE
KEY_MODE = 0xFFFFFFFD

# Irwin-Hall(4) of bytes: sum of four U{0..255} has mean 510 and variance 4*(256^2-1)/12.
NOISE_CENTER = 510
NOISE_SCALE = np.float32(1.0 / math.sqrt(4.0 * (256.0 * 256.0 - 1.0) / 12.0))
U24_SCALE = np.float32(2.0 ** -24)


def row_seed(seed: int, b: int, block: int, step: int, pos) -> np.ndarray:
    """Per-(sequence, block, step, position) hash seed: a chain of murmur3 calls."""
    h = murmur3_32(b, seed)
    h = murmur3_32(block, h)
    h = murmur3_32(step, h)
    return murmur3_32(np.asarray(pos), h)


def planted_token(h_row: np.ndarray, V: int, mask_id: int) -> np.ndarray:
    pid = (murmur3_32(KEY_PLANTED, h_row) % np.uint32(V)).astype(np.int64)
    return np.where(pid == mask_id, (pid + 1) % V, pid)


def planted_boost(h_row: np.ndarray, kind: int, boost_lo: float, boost_hi: float) -> np.ndarray:
    u = (murmur3_32(KEY_BOOST, h_row) >> np.uint32(8)).astype(np.float32) * U24_SCALE
    if kind == LOGITS_UNIFORM:
        lo = np.full(h_row.shape, boost_lo, np.float32)
        hi = np.full(h_row.shape, boost_hi, np.float32)
    elif kind == LOGITS_BIMODAL:
        sel = (murmur3_32(KEY_MODE, h_row) & np.uint32(1)).astype(bool)
        lo = np.where(sel, np.float32(BIMODAL_RANGES[1][0]), np.float32(BIMODAL_RANGES[0][0]))
        hi = np.where(sel, np.float32(BIMODAL_RANGES[1][1]), np.float32(BIMODAL_RANGES[0][1]))
    else:
        raise ValueError(f"unknown logits kind {kind}")
    width = (hi - lo).astype(np.float32)
    return (lo + (u * width).astype(np.float32)).astype(np.float32)


def logits_rows(seed: int, b: int, block: int, step: int, positions, V: int, mask_id: int,
                kind: int, boost_lo: float, boost_hi: float) -> np.ndarray:
    """fp32 logits [len(positions)][V] of sequence b at (block, step)."""
    positions = np.atleast_1d(np.asarray(positions, dtype=np.int64))
    out = np.empty((positions.size, V), dtype=np.float32)
    ids = np.arange(V, dtype=np.uint32)
    for i, pos in enumerate(positions):
        h = row_seed(seed, b, block, step, int(pos))
        r = murmur3_32(ids, h)
        s = ((r & np.uint32(0xFF)) + ((r >> np.uint32(8)) & np.uint32(0xFF))
             + ((r >> np.uint32(16)) & np.uint32(0xFF)) + (r >> np.uint32(24))).astype(np.int32)
        row = (s - NOISE_CENTER).astype(np.float32) * NOISE_SCALE
        pid = int(planted_token(h, V, mask_id)[0])
        boost = planted_boost(h, kind, boost_lo, boost_hi)[0]
        row[pid] = np.float32(row[pid] + boost)
        out[i] = row
    return out


# ----------------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int                      # context length (max length when ragged)
    S: int
    Hq: int
    Hkv: int
    D: int
    H: int
    V: int
    gamma: float = 0.8
    gammas: tuple = (0.8,)
    T: int = 0                  # max denoise steps per block; 0 means S
    mask_id: int = 3
    softmax_scale: float = 1.0
    q_prescale: float = 1.0
    qkv_fp32_source: bool = False
    paged: bool = False
    L_min: int = 0              # ragged lengths drawn uniformly from [L_min, L]
    page_size: int = 64
    logits_kind: int = LOGITS_UNIFORM
    boost_lo: float = 0.0
    boost_hi: float = 20.0
    ln_eps: float = 1e-5
    blocks: int = 1
    qkv_std: float = 1.0
    mod_std: float = 0.1
    lm_logit_std: float = 10.0  # spread of the LM head's logits for unit-RMS hidden rows

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def steps_max(self) -> int:
        return self.T if self.T > 0 else self.S

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the tiny / single-sequence / batched / long-context / ragged-paged
# denoise step.  The tiny one names no hidden size; 256 is used for its adaLN.
WORKLOADS = (
    Workload("c0_tiny_B1_L256_S16_G4_D64", B=1, L=256, S=16, Hq=4, Hkv=1, D=64, H=256, V=1024,
             softmax_scale=1.0 / 8.0, qkv_fp32_source=True, boost_lo=0.0, boost_hi=12.0),
    Workload("c1_single_B1_L4096_S16_32q2kv_D128", B=1, L=4096, S=16, Hq=32, Hkv=2, D=128,
             H=2688, V=131072, q_prescale=1.0 / math.sqrt(128.0)),
    Workload("c2_batched_B32_L8192_S16_32q2kv_D128", B=32, L=8192, S=16, Hq=32, Hkv=2, D=128,
             H=2688, V=131072, q_prescale=1.0 / math.sqrt(128.0), blocks=64),
    Workload("c3_longctx_B4_L65536_S16_32q2kv_D128", B=4, L=65536, S=16, Hq=32, Hkv=2, D=128,
             H=2688, V=131072, q_prescale=1.0 / math.sqrt(128.0), gammas=(0.5, 0.8, 0.95)),
    Workload("c4_paged_B64_L512-32768_S32_32q2kv_D128", B=64, L=32768, L_min=512, S=32, Hq=32,
             Hkv=2, D=128, H=2688, V=131072, q_prescale=1.0 / math.sqrt(128.0), paged=True,
             logits_kind=LOGITS_BIMODAL),
)
TINY, SINGLE, BATCHED, LONG_CONTEXT, RAGGED_PAGED = WORKLOADS


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[seed & 0xFFFFFFFFFFFFFFFF, stream]))


def _normal_bf16(rng: np.random.Generator, shape, std: float, prescale: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    f = np.float32(std * prescale)
    if f != np.float32(1.0):
        x *= f
    return f32_to_bf16_bits(x)


def context_lengths(w: Workload, seed: int) -> np.ndarray:
    """int32 [B] context lengths: L for every sequence, or uniform on [L_min, L] if ragged."""
    if w.L_min > 0:
        return _rng(seed, 11).integers(w.L_min, w.L + 1, size=w.B).astype(np.int32)
    return np.full(w.B, w.L, dtype=np.int32)


def make_attention_inputs(w: Workload, seed: int = 0, ctx_len: Optional[np.ndarray] = None) -> dict:
    """bf16 (uint16 bit patterns) Q, block K/V and context K/V for one denoise step.

    Layouts: q [B][S][Hq][D]; k_blk, v_blk [B][S][Hkv][D]; contiguous context
    k_ctx, v_ctx [B][L][Hkv][D]; or, when ``w.paged``, a page pool
    k_pages, v_pages [P][page_size][Hkv][D] with an int32 page_table [B][max_pages]
    (unused entries are -1) whose physical pages are a seeded shuffle.
    """
    B, S, Hq, Hkv, D = w.B, w.S, w.Hq, w.Hkv, w.D
    if ctx_len is None:
        ctx_len = context_lengths(w, seed)
    ctx_len = np.asarray(ctx_len, dtype=np.int32)
    out = {"ctx_len": ctx_len}
    out["q"] = _normal_bf16(_rng(seed, 1), (B, S, Hq, D), w.qkv_std, w.q_prescale)
    out["k_blk"] = _normal_bf16(_rng(seed, 2), (B, S, Hkv, D), w.qkv_std, 1.0)
    out["v_blk"] = _normal_bf16(_rng(seed, 3), (B, S, Hkv, D), w.qkv_std, 1.0)
    if not w.paged:
        L = int(ctx_len.max()) if ctx_len.size else 0
        L = max(L, w.L)
        out["k_ctx"] = _normal_bf16(_rng(seed, 4), (B, L, Hkv, D), w.qkv_std, 1.0)
        out["v_ctx"] = _normal_bf16(_rng(seed, 5), (B, L, Hkv, D), w.qkv_std, 1.0)
    else:
        P_sz = w.page_size
        n_pages = (ctx_len.astype(np.int64) + P_sz - 1) // P_sz
        total = int(n_pages.sum())
        max_pages = max(1, (w.L + P_sz - 1) // P_sz)
        perm = _rng(seed, 6).permutation(total).astype(np.int32)
        table = np.full((B, max_pages), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            table[b, : n_pages[b]] = perm[off: off + n_pages[b]]
            off += int(n_pages[b])
        out["page_table"] = table
        rk, rv = _rng(seed, 4), _rng(seed, 5)
        kp = np.empty((total, P_sz, Hkv, D), dtype=np.uint16)
        vp = np.empty((total, P_sz, Hkv, D), dtype=np.uint16)
        chunk = 4096
        for p0 in range(0, total, chunk):
            p1 = min(total, p0 + chunk)
            kp[p0:p1] = _normal_bf16(rk, (p1 - p0, P_sz, Hkv, D), w.qkv_std, 1.0)
            vp[p0:p1] = _normal_bf16(rv, (p1 - p0, P_sz, Hkv, D), w.qkv_std, 1.0)
        out["k_pages"] = kp
        out["v_pages"] = vp
    return out


def make_adaln_inputs(w: Workload, seed: int = 0) -> dict:
    """x bf16 [B][S][H]; per-sequence shift/scale fp32 [B][H]; per-timestep tables fp32 [S+1][H].

    Row n of a table is the modulation for timestep t = n/S.  The standalone call's
    per-sequence vectors stand for one timestep t ~ U(0,1) each, recorded in ``t``.
    """
    B, S, H = w.B, w.S, w.H
    r = _rng(seed, 20)
    return {
        "x": _normal_bf16(r, (B, S, H), 1.0, 1.0),
        "t": _rng(seed, 21).random(B).astype(np.float32),
        "shift": (_rng(seed, 22).standard_normal((B, H), dtype=np.float32) * np.float32(w.mod_std)),
        "scale": (_rng(seed, 23).standard_normal((B, H), dtype=np.float32) * np.float32(w.mod_std)),
        "shift_table": (_rng(seed, 24).standard_normal((S + 1, H), dtype=np.float32)
                        * np.float32(w.mod_std)),
        "scale_table": (_rng(seed, 25).standard_normal((S + 1, H), dtype=np.float32)
                        * np.float32(w.mod_std)),
    }


def make_hidden(w: Workload, seed: int = 0) -> np.ndarray:
    """bf16 hidden rows [B][S][H], N(0, 1): the input of the LM head in standalone calls."""
    return _normal_bf16(_rng(seed, 30), (w.B, w.S, w.H), 1.0, 1.0)


def make_lmhead_weights(w: Workload, seed: int = 0, rows: int = 8192) -> np.ndarray:
    """bf16 vocabulary projection [V][H] (one row per token id), N(0, sigma^2) with
    sigma = lm_logit_std / sqrt(H), so unit-RMS hidden rows give logits of standard
    deviation lm_logit_std.  Drawn in blocks of rows to bound host memory."""
    V, H = w.V, w.H
    out = np.empty((V, H), dtype=np.uint16)
    r = _rng(seed, 31)
    sigma = w.lm_logit_std / math.sqrt(H)
    for v0 in range(0, V, rows):
        v1 = min(V, v0 + rows)
        out[v0:v1] = _normal_bf16(r, (v1 - v0, H), sigma, 1.0)
    return out


def make_qkv_weights(w: Workload, seed: int = 0) -> np.ndarray:
    """bf16 fused projection [(Hq + 2 Hkv) D][H]: rows 0 .. Hq D - 1 make the queries
    (head-major), then the keys, then the values.  N(0, 1/H), so unit-RMS hidden rows
    give unit-variance q/k/v entries like the directly drawn workloads."""
    n = (w.Hq + 2 * w.Hkv) * w.D
    return _normal_bf16(_rng(seed, 32), (n, w.H), 1.0 / math.sqrt(w.H), 1.0)
