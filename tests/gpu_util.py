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


# gamma-band exclusions per workload, reported at the end of the run (conftest.py):
# key -> [sequences excluded, sequence decisions compared]
EXCLUDED = {}


def record_excluded(key: str, excluded: int, decisions: int) -> None:
    e = EXCLUDED.setdefault(key, [0, 0])
    e[0] += int(excluded)
    e[1] += int(decisions)


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


def check_decision_validity(ids_g, com, ids0_b, tok, conf, mask_id, kind, gamma, k_min, band,
                            what=""):
    """The sampler decision of one sequence is one that the rule could have taken.

    ``conf`` holds the oracle's confidences (0 at decoded positions) and ``band`` the
    largest difference allowed between the kernel's confidence and the oracle's
    (scalar or per position), so the kernel's value of position i lies in
    [conf_i - band_i, conf_i + band_i].  The commit set C must then satisfy:
    * confidence rule (kind 0): either C is the threshold set - every position whose
      confidence is certainly >= gamma is in C and none that is certainly < gamma -
      and |C| >= k_min; or fewer than k_min are certainly >= gamma and C is a
      possible top-k_min (the floor);
    * predict-and-noise (kind 2): C is a possible top-k_min;
    * mock-AR (kind 1): C is the leftmost masked position;
    where a "possible top-k" has k elements and no position left out certainly
    beats one taken.  Committed tokens are the oracle's argmax, the other masked
    positions keep the mask id, decoded positions are unchanged."""
    masked = ids0_b == mask_id
    com = np.asarray(com).astype(bool)
    band = np.broadcast_to(np.asarray(band, dtype=np.float64), conf.shape)
    assert np.all(~com | masked), f"{what}: commit at a decoded position"
    assert np.array_equal(ids_g[~masked], ids0_b[~masked]), f"{what}: decoded position changed"
    assert np.array_equal(ids_g[com], tok[com]), f"{what}: committed token is not the oracle's argmax"
    assert np.all(ids_g[masked & ~com] == mask_id), f"{what}: uncommitted position not remasked"
    n = int(com.sum())
    lo, hi = conf - band, conf + band

    def possible_topk(k):
        if n != k:
            return False
        taken, left = masked & com, masked & ~com
        return not (taken.any() and left.any() and lo[left].max() > hi[taken].min())

    if kind == 1:
        pos = np.flatnonzero(masked)
        ok = pos.size == 0 or (n == 1 and com[pos[0]])
    elif kind == 2:
        ok = possible_topk(k_min)
    else:
        sure = masked & (lo >= gamma)
        maybe = masked & (hi >= gamma)
        threshold_set = bool(np.all(com[sure]) and np.all(~com | maybe) and n >= k_min)
        ok = threshold_set or (int(sure.sum()) < k_min and possible_topk(k_min))
    assert ok, (f"{what}: commit set {np.flatnonzero(com).tolist()} is not one the rule allows "
                f"(k_min {k_min}, confidences {np.round(conf[masked], 7).tolist()})")


def compare_unmask(gpu: dict, ora: list, ids0, steps0, mask_id, gamma, what="", kind=0) -> int:
    """Asserts parity of one unmask call for a batch; returns the number of excluded sequences.

    Every sequence is checked for validity (check_decision_validity, with the
    confidence tolerance as the band); sequences that are not ambiguous must then
    match the oracle bit for bit."""
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
        assert gpu["steps"][b] == r["steps"], f"{what} b={b}: steps differ"
        check_decision_validity(gpu["ids"][b], gpu["commit"][b], ids0[b], r["tok"], co, mask_id, kind,
                                gamma, r["k_min"], CONF_REL * co, what=f"{what} b={b}")
        com = gpu["commit"][b].astype(bool)
        assert gpu["n_masked"][b] == int(masked.sum()) - int(com.sum()), f"{what} b={b}: n_masked"
        # commit_step: the new step count where the kernel committed; elsewhere the value
        # from before the step (the oracle's, with its own commits of this step undone:
        # positions masked before the step hold 0)
        before = np.where(r["commit"].astype(bool), 0, r["commit_step"])
        exp_cs = np.where(com, r["steps"], before).astype(np.uint8)
        assert np.array_equal(gpu["commit_step"][b], exp_cs), f"{what} b={b}: commit_step"
        if ambiguous(r, ids0[b], mask_id, gamma):
            excluded += 1
            continue
        assert np.array_equal(gpu["ids"][b], r["ids"]), f"{what} b={b}: ids differ"
        assert np.array_equal(gpu["commit"][b], r["commit"]), f"{what} b={b}: commit differs"
        assert gpu["n_masked"][b] == r["n_masked"], f"{what} b={b}: n_masked differs"
        assert np.array_equal(gpu["commit_step"][b], r["commit_step"]), f"{what} b={b}: commit_step"
    return excluded


GUARD = 4096  # canary elements on each side of a guarded output buffer


def guarded(n, dtype, fill):
    """A flat device buffer with GUARD canary elements of `fill` on both sides;
    returns (whole buffer, the n-element view handed to the kernel)."""
    full = torch.full((n + 2 * GUARD,), fill, dtype=dtype, device="cuda")
    return full, full[GUARD:GUARD + n]


def guarded_copy(a: np.ndarray, canary):
    """The host array a on the device inside canaries: (whole buffer, view of a's shape)."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    full, view = guarded(t.numel(), t.dtype, canary)
    view.copy_(t.reshape(-1).cuda())
    return full, view.view(t.shape)


def check_guards(full, fill, what=""):
    """The canaries around a guarded buffer are untouched (NaN canaries stay NaN)."""
    g = torch.cat([full[:GUARD], full[-GUARD:]])
    if isinstance(fill, float) and math.isnan(fill):
        ok = bool(torch.isnan(g).all())
    else:
        ok = bool((g == fill).all())
    assert ok, f"{what}: the kernel wrote outside its buffer"


def run_unmask(tt, logits: np.ndarray, ids0, steps0, cs0, mask_id, gamma, T):
    """One tt_confidence_unmask call on host inputs; every buffer it writes sits between
    canaries that must come back untouched."""
    B, S, V = logits.shape
    d_logits = dev(logits.astype(np.float32))
    g_ids, ids = guarded_copy(ids0.astype(np.int32), -77)
    g_steps, steps = guarded_copy(steps0.astype(np.int32), -77)
    g_cs, cs = guarded_copy(cs0.astype(np.uint8), 0xA5)
    g_nm, n_masked = guarded(B, torch.int32, -77)
    g_conf, conf = guarded(B * S, torch.float32, float("nan"))
    g_com, commit = guarded(B * S, torch.uint8, 0xA5)
    conf.fill_(-1.0)
    commit.fill_(7)
    tt.tt_confidence_unmask(d_logits, ids, steps, B, S, V, mask_id, gamma, T, n_masked=n_masked,
                            conf=conf, commit=commit, commit_step=cs)
    torch.cuda.synchronize()
    for full, fill, name in ((g_ids, -77, "ids"), (g_steps, -77, "steps"), (g_cs, 0xA5, "commit_step"),
                             (g_nm, -77, "n_masked"), (g_conf, float("nan"), "conf"),
                             (g_com, 0xA5, "commit")):
        check_guards(full, fill, name)
    return dict(ids=host(ids), steps=host(steps), n_masked=host(n_masked), conf=host(conf).reshape(B, S),
                commit=host(commit).reshape(B, S), commit_step=host(cs))


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
        # validity (every sequence): each committed token within 2 delta of the top
        # logit (the oracle's argmax itself unless the top two are that close), and the
        # commit set one that the sampler's rule allows given the confidence tolerance
        tok_ok = r["tok"].copy()
        for j, p_ in enumerate(pos):
            if com[p_]:
                t = gpu["ids"][b][p_]
                assert t != mask and lg[j, t] >= srt[j, -1] - 2 * delta[j], f"b={b} pos={p_}: token {t}"
                if near_tie[j]:
                    tok_ok[p_] = t
        assert gpu["steps"][b] == r["steps"]
        band = np.zeros(S)
        band[pos] = tol * co
        check_decision_validity(gpu["ids"][b], com, ids0[b], tok_ok, r["conf"], mask, kind, gamma,
                                r["k_min"], band, what=f"b={b}")
        assert gpu["n_masked"][b] == pos.size - int(com.sum()), f"b={b}: n_masked"
        if ambiguous:
            excluded += 1
            continue
        assert np.array_equal(gpu["ids"][b], r["ids"]), f"b={b}: ids differ"
        assert np.array_equal(gpu["commit"][b], r["commit"]), f"b={b}: commit differs"
        assert gpu["n_masked"][b] == r["n_masked"], f"b={b}: n_masked"
        assert np.array_equal(gpu["commit_step"][b], r["commit_step"]), f"b={b}: commit_step"
    return excluded
