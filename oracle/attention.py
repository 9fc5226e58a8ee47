"""Denoise attention, fp64.

Source: "Nemotron-Labs-TwoTower" wiki, section "Architecture": queries from the noisy
block b attend over one concatenated key/value sequence made of the context tower's
layer-i cache for blocks 0..b-1 followed by the denoiser's own layer-i keys and values
for block b; attention inside the block is bidirectional and adds no parameters.

Definition computed for every (sequence b, query head h, block position s):

    keys   = [K_ctx[b, 0..ctx_len_b), kv(h)] ++ [K_blk[b, 0..S), kv(h)]
    values = [V_ctx[b, 0..ctx_len_b), kv(h)] ++ [V_blk[b, 0..S), kv(h)]
    a_j    = softmax_scale * <q[b, s, h], keys_j>
    O[b, s, h] = sum_j softmax(a)_j * values_j,   lse[b, s, h] = log sum_j exp(a_j)

with no causal mask anywhere (the whole context precedes the block; the block is
bidirectional).  Readings where the pages are silent: layout [B][len][heads][D];
grouped-query mapping kv(h) = h // (Hq / Hkv); the paged cache maps logical token t
of sequence b to physical page page_table[b, t // page_size], row t % page_size.
"""
import numpy as np

from ._bf16 import bf16_to_f64


def context_kv(inp: dict, b: int):
    """Context K, V of sequence b as float64 [ctx_len_b][Hkv][D] (contiguous or paged)."""
    n = int(inp["ctx_len"][b])
    if "page_table" in inp:
        kp, vp = inp["k_pages"], inp["v_pages"]
        page_size = kp.shape[1]
        t = np.arange(n)
        phys = inp["page_table"][b, t // page_size]
        if n and (phys.min() < 0 or phys.max() >= kp.shape[0]):
            raise ValueError("page table entry out of range")
        return bf16_to_f64(kp[phys, t % page_size]), bf16_to_f64(vp[phys, t % page_size])
    return bf16_to_f64(inp["k_ctx"][b, :n]), bf16_to_f64(inp["v_ctx"][b, :n])


def _head_attention(qs, keys, vals, softmax_scale):
    """qs [n][D], keys/vals [m][D] -> (O [n][D], lse [n]) by the plain softmax definition."""
    a = softmax_scale * (qs @ keys.T)
    amax = a.max(axis=1, keepdims=True)
    e = np.exp(a - amax)
    denom = e.sum(axis=1, keepdims=True)
    p = e / denom
    return p @ vals, (amax + np.log(denom))[:, 0]


def denoise_attention(inp: dict, softmax_scale: float):
    """All outputs.  Returns (O float64 [B][S][Hq][D], lse float64 [B][S][Hq])."""
    q = bf16_to_f64(inp["q"])
    kb, vb = bf16_to_f64(inp["k_blk"]), bf16_to_f64(inp["v_blk"])
    B, S, Hq, D = q.shape
    Hkv = kb.shape[2]
    G = Hq // Hkv
    O = np.zeros((B, S, Hq, D))
    lse = np.zeros((B, S, Hq))
    for b in range(B):
        kc, vc = context_kv(inp, b)
        for h in range(Hq):
            g = h // G
            keys = np.concatenate([kc[:, g, :], kb[b, :, g, :]], axis=0)
            vals = np.concatenate([vc[:, g, :], vb[b, :, g, :]], axis=0)
            O[b, :, h, :], lse[b, :, h] = _head_attention(q[b, :, h, :], keys, vals, softmax_scale)
    return O, lse


def denoise_attention_rows(inp: dict, softmax_scale: float, rows):
    """Selected outputs only: rows is an iterable of (b, s, h).

    Returns (O float64 [n][D], lse float64 [n]) in the order given.
    """
    rows = [tuple(int(v) for v in r) for r in rows]
    Hq = inp["q"].shape[2]
    Hkv = inp["k_blk"].shape[2]
    G = Hq // Hkv
    D = inp["q"].shape[3]
    O = np.zeros((len(rows), D))
    lse = np.zeros(len(rows))
    by_b = {}
    for i, (b, s, h) in enumerate(rows):
        by_b.setdefault(b, []).append((i, s, h))
    for b, items in by_b.items():
        kc, vc = context_kv(inp, b)
        kb = bf16_to_f64(inp["k_blk"][b])
        vb = bf16_to_f64(inp["v_blk"][b])
        by_g = {}
        for i, s, h in items:
            by_g.setdefault(h // G, []).append((i, s, h))
        for g, rows_g in by_g.items():
            # the concatenated keys/values of kv head g, built once for all its rows
            keys = np.concatenate([kc[:, g, :], kb[:, g, :]], axis=0)
            vals = np.concatenate([vc[:, g, :], vb[:, g, :]], axis=0)
            for i, s, h in rows_g:
                qs = bf16_to_f64(inp["q"][b, s, h])[None, :]
                o, l = _head_attention(qs, keys, vals, softmax_scale)
                O[i], lse[i] = o[0], l[0]
    return O, lse
