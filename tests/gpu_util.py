"""Helpers shared by the GPU parity tests: device transfer and the comparison rules.

Comparison rules (tolerances of the parity contract):
* attention output: max |gpu - oracle| <= 1e-2 and ||gpu - oracle||_2 / ||oracle||_2 <= 5e-3
  against the fp64 oracle on the same bf16 inputs; lse within 4e-3 (natural log) -
  the kernel normalises with the bf16-rounded probabilities it multiplies V with, whose
  relative rounding error is at most 2^-9 per term;
* adaLN: within one bf16 ulp of the unrounded fp64 value plus 2^-16 of the magnitude
  of the two terms that are added, |LN(x)*(1+scale)| + |shift|: the kernel's fp32
  statistics carry a relative error of order sqrt(H) * 2^-24, and where the two terms
  nearly cancel that absolute error survives in a result far smaller than either;
* unmask: token ids, commit masks, step counts bit-exact, except sequences in which a
  masked position's oracle confidence lies within 1e-5 of gamma, or in which the floor
  decides between confidences within 1e-5 (relative) of each other - those are counted
  and checked for validity only; confidences within 1e-5 relative;
* fused LM head + sampler step: the kernel accumulates the logits in fp32, so each
  logit may differ from the exact value by delta = (H/16 + 16) 2^-24 sum_k |h_k W_jk|
  (H/16 accumulator additions of 16-product slices); tokens equal the oracle's where
  its top two logits are more than 2 delta apart and lie within 2 delta of the top
  otherwise; confidences agree within exp(2 delta / tau) - 1 + 1e-5 relative; the
  decision is bit-exact except in sequences that compare values closer than that
  (counted, validity only).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

ATTN_MAX_ABS = 1e-2
ATTN_REL_L2 = 5e-3
LSE_ABS = 4e-3
CONF_REL = 1e-5
GAMMA_BAND = 1e-5


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    a = t.detach().cpu().contiguous()
    if a.dtype in (torch.int16, torch.bfloat16):
        return a.view(torch.int16).numpy().view(np.uint16)
    return a.numpy()


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def check_attention(O_gpu: np.ndarray, O_ref: np.ndarray, lse_gpu=None, lse_ref=None, what="",
                    out_rounding=False):
    """out_rounding: also allow half a bf16 ulp of the reference per element.  The
    output is stored in bf16, so where |O| >= 4 (inputs with std > 1) rounding alone
    can exceed the flat max-abs bound; the N(0,1) workloads never need it."""
    err = np.abs(O_gpu - O_ref)
    max_abs = float(err.max()) if err.size else 0.0
    rel = float(np.linalg.norm(O_gpu - O_ref) / max(np.linalg.norm(O_ref), 1e-30))
    if out_rounding:
        excess = err - 0.5 * bf16_ulp(O_ref)
        assert float(excess.max()) <= ATTN_MAX_ABS, f"{what}: max abs err beyond rounding {excess.max()}"
    else:
        assert max_abs <= ATTN_MAX_ABS, f"{what}: max abs err {max_abs}"
    assert rel <= ATTN_REL_L2, f"{what}: rel L2 err {rel}"
    if lse_gpu is not None:
        lerr = float(np.abs(lse_gpu - lse_ref).max())
        assert lerr <= LSE_ABS, f"{what}: lse err {lerr}"
    return max_abs, rel


def adaln_tol(ref: np.ndarray, shift: np.ndarray) -> np.ndarray:
    """Allowed |gpu - oracle| for adaLN outputs (see the module docstring)."""
    terms = np.abs(ref - shift) + np.abs(shift)
    return bf16_ulp(ref) + 2.0 ** -16 * terms + 1e-30


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def oracle_unmask_batch(logits, ids0, steps0, cs0, mask_id, gamma, T):
    B = ids0.shape[0]
    out = []
    for b in range(B):
        out.append(oracle.unmask_step(logits[b], ids0[b], int(steps0[b]), mask_id, gamma, T, cs0[b]))
    return out


def ambiguous(r: dict, ids0_b: np.ndarray, mask_id: int, gamma: float) -> bool:
    masked = np.flatnonzero(ids0_b == mask_id)
    if masked.size == 0:
        return False
    conf = r["conf"][masked]
    if np.any(np.abs(conf - gamma) <= GAMMA_BAND):
        return True
    n_above = int(np.sum(conf >= gamma))
    k = r["k_min"]
    if n_above < k < masked.size:
        srt = np.sort(conf)[::-1]
        if abs(srt[k - 1] - srt[k]) <= GAMMA_BAND * srt[k - 1]:
            return True
    return False


def compare_unmask(gpu: dict, ora: list, ids0, steps0, mask_id, gamma, what="") -> int:
    """Asserts parity of one unmask call for a batch; returns the number of excluded sequences."""
    excluded = 0
    B = ids0.shape[0]
    for b in range(B):
        r = ora[b]
        masked = ids0[b] == mask_id
        cg = gpu["conf"][b]
        co = r["conf"]
        assert np.all(cg[~masked] == 0.0), f"{what} b={b}: conf of unmasked position not 0"
        if masked.any():
            rel = np.abs(cg[masked] - co[masked]) / np.maximum(co[masked], 1e-300)
            assert rel.max() <= CONF_REL, f"{what} b={b}: conf rel err {rel.max()}"
        if ambiguous(r, ids0[b], mask_id, gamma):
            excluded += 1
            # validity only: committed tokens are the oracle's argmax, decoded positions
            # unchanged, one step taken, counts consistent
            com = gpu["commit"][b].astype(bool)
            assert np.all(~com | masked)
            assert np.array_equal(gpu["ids"][b][com], r["tok"][com])
            assert np.array_equal(gpu["ids"][b][~masked], ids0[b][~masked])
            assert np.all(gpu["ids"][b][masked & ~com] == mask_id)
            assert gpu["steps"][b] == r["steps"]
            assert com.sum() >= r["k_min"]
            continue
        assert np.array_equal(gpu["ids"][b], r["ids"]), f"{what} b={b}: ids differ"
        assert np.array_equal(gpu["commit"][b], r["commit"]), f"{what} b={b}: commit differs"
        assert gpu["steps"][b] == r["steps"], f"{what} b={b}: steps differ"
        assert gpu["n_masked"][b] == r["n_masked"], f"{what} b={b}: n_masked differs"
        assert np.array_equal(gpu["commit_step"][b], r["commit_step"]), f"{what} b={b}: commit_step"
    return excluded


def run_unmask(tt, logits: np.ndarray, ids0, steps0, cs0, mask_id, gamma, T):
    B, S, V = logits.shape
    d_logits = dev(logits.astype(np.float32))
    ids = dev(ids0.astype(np.int32))
    steps = dev(steps0.astype(np.int32))
    cs = dev(cs0.astype(np.uint8))
    n_masked = torch.zeros(B, dtype=torch.int32, device="cuda")
    conf = torch.full((B, S), -1.0, dtype=torch.float32, device="cuda")
    commit = torch.full((B, S), 7, dtype=torch.uint8, device="cuda")
    tt.tt_confidence_unmask(d_logits, ids, steps, B, S, V, mask_id, gamma, T, n_masked=n_masked,
                            conf=conf, commit=commit, commit_step=cs)
    torch.cuda.synchronize()
    return dict(ids=host(ids), steps=host(steps), n_masked=host(n_masked), conf=host(conf),
                commit=host(commit), commit_step=host(cs))


def _abs_bound(hr, W, rows=16384):
    """max_j sum_k |h_rk W_jk| for every row of hr (bf16 bits), W in blocks of rows."""
    ha = np.abs(bf16_to_f64(hr))
    out = np.zeros(hr.shape[0])
    for v0 in range(0, W.shape[0], rows):
        Wa = np.abs(bf16_to_f64(W[v0:v0 + rows]))
        out = np.maximum(out, (ha @ Wa.T).max(axis=1))
    return out


def compare_lmhead(gpu, h, W, ids0, steps0, cs0, mask, kind, gamma, T, tau, seqs=None):
    """Parity of one fused LM-head sampler step (see the lmhead rules in the module
    docstring); returns the number of sequences checked for validity only."""
    B, S, H = h.shape
    seqs = list(range(B)) if seqs is None else list(seqs)
    rows = [(b, p) for b in seqs for p in np.flatnonzero(ids0[b] == mask)]
    if rows:
        hr = np.stack([h[b][p] for b, p in rows])
        lg_all = oracle.lm_head_logits(hr, W)  # the oracle's exact logits of every sampled row
        bound_all = _abs_bound(hr, W)
    excluded = 0
    at = 0
    for b in seqs:
        masked = ids0[b] == mask
        pos = np.flatnonzero(masked)
        lg = lg_all[at:at + pos.size].copy() if pos.size else None
        delta = (H / 16 + 16) * 2.0 ** -24 * bound_all[at:at + pos.size] if pos.size else None
        at += pos.size

        def rows_of(positions, lg=lg, pos=pos):
            assert list(positions) == pos.tolist()
            return lg
        r = oracle.sampler_step(rows_of, ids0[b], int(steps0[b]), mask, T, kind, gamma, tau, cs0[b])
        assert np.all(gpu["conf"][b][~masked] == 0.0), f"b={b}: conf of a decoded position"
        if not masked.any():
            assert np.array_equal(gpu["ids"][b], ids0[b]) and gpu["steps"][b] == steps0[b]
            assert gpu["n_masked"][b] == 0 and not gpu["commit"][b].any()
            continue
        lg[:, mask] = -np.inf
        srt = np.sort(lg, axis=1)
        gap = srt[:, -1] - srt[:, -2]
        near_tie = gap <= 2 * delta
        tol = np.expm1(2 * delta / tau) + 1e-5
        cg, co = gpu["conf"][b][pos], r["conf"][pos]
        rel = np.abs(cg - co) / co
        assert np.all(rel <= tol), f"b={b}: conf rel err {rel.max()} > {tol[np.argmax(rel - tol)]}"
        ambiguous = bool(near_tie.any())
        if kind == 0 and np.any(np.abs(co - gamma) <= tol * co):
            ambiguous = True
        if kind in (0, 2):
            k = r["k_min"]
            n_above = int(np.sum(co >= gamma)) if kind == 0 else 0
            if n_above < k < pos.size:
                c_sorted = np.sort(co)[::-1]
                if c_sorted[k - 1] - c_sorted[k] <= 2 * tol.max() * c_sorted[k - 1]:
                    ambiguous = True
        com = gpu["commit"][b].astype(bool)
        # validity (every sequence): commits only at masked positions, decoded ones kept,
        # each committed token within 2 delta of the top logit, the rest still masked
        assert np.all(~com | masked)
        assert np.array_equal(gpu["ids"][b][~masked], ids0[b][~masked])
        assert np.all(gpu["ids"][b][masked & ~com] == mask)
        for j, p_ in enumerate(pos):
            if com[p_]:
                t = gpu["ids"][b][p_]
                assert t != mask and lg[j, t] >= srt[j, -1] - 2 * delta[j], f"b={b} pos={p_}: token {t}"
        assert gpu["steps"][b] == r["steps"]
        if kind == 1:
            assert com.sum() == 1
        elif kind == 2:
            assert com.sum() == r["k_min"]
        else:
            assert com.sum() >= r["k_min"]
        if ambiguous:
            excluded += 1
            continue
        assert np.array_equal(gpu["ids"][b], r["ids"]), f"b={b}: ids differ"
        assert np.array_equal(gpu["commit"][b], r["commit"]), f"b={b}: commit differs"
        assert gpu["n_masked"][b] == r["n_masked"], f"b={b}: n_masked"
        assert np.array_equal(gpu["commit_step"][b], r["commit_step"]), f"b={b}: commit_step"
    return excluded
