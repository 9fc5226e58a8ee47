#!/usr/bin/env python
"""Denoise steps/s of one TwoTower denoiser step on B300, plus per-kernel roofline.

One bench step = one denoise step over the whole batch: adaLN(t) prologue, split-KV
attention (context cache + the block's own keys), the synthetic-logits stand-in for
the LM head, and confidence unmasking, all in libtt's CUDA kernels.  Blocks start
fully masked and are decoded with tt_denoise_block_loop (a CUDA graph whose WHILE
node repeats the step on the device until the block is committed); the step counts
per block are deterministic (seeded logits), so an untimed pass first learns them
and the timed region covers exactly --steps denoise steps (whole blocks, then single
tt_denoise_step calls for the remainder).  L2 is flushed before every timed block,
outside the timed events.

Headline workload (--config 4): the ragged paged batch, B=64 sequences with context
lengths uniform on [512, 32768] in shuffled 64-token pages, S=32, 32q/2kv heads,
D=128, H=2688, V=131072, gamma=0.8 - the largest workload that fits one GPU.  The
same JSON line carries one object per other realistic workload (--other-configs,
default 1,2,3: single sequence, batched, long context), each with its own steps/s,
kernel times, rooflines and end-to-end figure.

    python bench.py [--gpus N --steps K --warmup W] [--config C] [--other-configs 1,2,3]
                    [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_wise_mask_tt_b300 import synth  # noqa: E402

METRIC = "denoise steps/s; attention and unmask achieved % of HBM/tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100, help="timed denoise steps")
    ap.add_argument("--warmup", type=int, default=3, help="untimed warm-up denoise steps (>= 3)")
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--other-configs", default="1,2,3",
                    help="comma-separated workloads measured after the headline one and reported "
                         "inside the same JSON line ('' for none)")
    ap.add_argument("--impl", choices=("tt", "reference"), default="tt")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--gamma", type=float, default=None)
    ap.add_argument("--sampler", choices=("confidence", "mock_ar", "predict_noise"),
                    default="confidence",
                    help="unmask rule: confidence unmasking (the main sampler), mock-AR (one "
                         "token per step, left to right) or predict-and-noise (linear schedule)")
    ap.add_argument("--temperature", type=float, default=1.0)
    ap.add_argument("--kernel-reps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-warmup-s", type=float, default=1.5,
                    help="keep warming up for at least this long so the clock sampler sees load")
    ap.add_argument("--kernel-only", choices=("attn", "unmask", "adaln", "logits", "step", "lmhead", "qkv"),
                    default=None,
                    help="profiling aid: run only --reps standalone calls of one entry point on "
                         "the workload (after 3 untimed ones) and print their mean time")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--attn-splits", type=int, default=0,
                    help="context splits per (sequence, kv head) of the attention; 0 = the "
                         "library's choice (a sweep aid for the split cost model)")
    ap.add_argument("--lm-head", action="store_true",
                    help="the step's logits come from the fused LM head over the adaLN output "
                         "(synthetic projection W [V][H]) instead of the hash stand-in")
    ap.add_argument("--qkv-proj", action="store_true",
                    help="every step projects the adaLN output into q, k_blk, v_blk (synthetic "
                         "W_qkv) before the attention, so they follow the timestep")
    ap.add_argument("--no-qkv-leg", action="store_true",
                    help="skip the standalone timing of the query/key/value projection")
    ap.add_argument("--no-lm-head-leg", action="store_true",
                    help="skip the standalone timing of the fused LM head + sampler step")
    ap.add_argument("--generate", type=int, default=32,
                    help="also time tt_generate over this many blocks (Algorithm 1's outer loop: "
                         "decode, append the block to the cache, next block); 0 skips it")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# ------------------------------------------------------------------ replicas
# Sequences are independent, so N GPUs run N replicas with no data-path collective;
# the only communication is the barrier and the max of the timed region.
def replica_seed(base_seed: int, rank: int) -> int:
    """Seed of rank `rank`'s replica (distinct synthetic batches per rank)."""
    return base_seed + 1000 * rank


def max_over_ranks(value: float, dist, device) -> float:
    """Max of a per-rank float over the process group (the job time is the slowest rank's)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(steps_per_rank: int, world: int, elapsed_max_s: float) -> float:
    """Whole-job denoise steps/s: every rank ran steps_per_rank steps in at most elapsed_max_s."""
    return world * steps_per_rank / elapsed_max_s


# Spin (GPU clock cycles, ~1 ms) queued before each standalone timed call, so that the
# host's argument checks, tensor-map encoding and launches are hidden behind work the
# GPU is already doing and never leave it idle between the two events, even when the
# host is briefly slow.
KEEP_BUSY_CYCLES = 2_000_000

# DRAM bytes (read + write) per call, from ncu captures committed as a table in
# profiles/ncu_traffic.md: | workload | call | DRAM bytes per call | source | capture |.
# "source" is the sha256 prefix of the kernel sources the capture ran; when the
# sources have changed since, the figure no longer describes them and reads as null.
TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "ncu_traffic.md")
CALL_SOURCES = {
    "attn": ("attn.cu",),
    "unmask": ("unmask.cu", "unmask_common.cuh"),
    "lmhead": ("lmhead.cu", "unmask_common.cuh"),
}


def sources_sha(call: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in CALL_SOURCES[call]:
        with open(os.path.join(ROOT, "block_wise_mask_tt_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def ncu_traffic(workload_name: str, call: str):
    """(bytes per call or None, note) for one call of a workload."""
    if not os.path.exists(TRAFFIC_TABLE):
        return None, "no committed capture"
    for line in open(TRAFFIC_TABLE):
        cells = [c.strip().strip("`") for c in line.strip().strip("|").split("|")]
        if len(cells) < 4 or cells[0] != workload_name or cells[1] != call:
            continue
        try:
            nbytes = float(cells[2].replace(",", "").replace(" ", ""))
        except ValueError:
            return None, "unparsed capture"
        if cells[3] != sources_sha(call):
            return None, f"kernel changed since the capture (capture {cells[3]}, now {sources_sha(call)})"
        return nbytes, f"ncu capture of sources {cells[3]}, {TRAFFIC_TABLE[len(ROOT) + 1:]}"
    return None, "no committed capture for this workload"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload(args) -> synth.Workload:
    w = synth.WORKLOADS[args.config]
    if args.gamma is not None:
        w = w.replace(gamma=args.gamma)
    return w


def cores_used() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
        return int(n)
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ clocks sampler
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.dev = device_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if not self.lines:
            return None
        sm, smax, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ GPU workload
SAMPLERS = {"confidence": 0, "mock_ar": 1, "predict_noise": 2}


class Workbench:
    """Device-resident inputs, state and buffers for one replica of the workload."""

    def __init__(self, tt, torch, w: synth.Workload, seed: int, sampler: int = 0,
                 temperature: float = 1.0, lm_head: bool = False, qkv_proj: bool = False,
                 attn_splits: int = 0):
        self.tt, self.torch, self.w, self.seed = tt, torch, w, seed
        self.lm_head = lm_head
        self.qkv_proj = qkv_proj
        t0 = time.time()
        self.inp = synth.make_attention_inputs(w, seed)
        self.ad = synth.make_adaln_inputs(w, seed)
        self.w_vocab = self._dev(synth.make_lmhead_weights(w, seed)) if lm_head else None
        self.w_qkv = self._dev(synth.make_qkv_weights(w, seed)) if qkv_proj else None
        self.gen_s = time.time() - t0
        B, S = w.B, w.S
        dev = lambda a: self._dev(a)
        if w.paged:
            kp = self.inp["k_pages"]
            self.dims = tt.attn_dims(B, S, w.Hq, w.Hkv, w.D, 0, w.page_size,
                                     self.inp["page_table"].shape[1], kp.shape[0], w.softmax_scale,
                                     attn_splits)
            kc, vc, pt = dev(kp), dev(self.inp["v_pages"]), dev(self.inp["page_table"])
        else:
            self.dims = tt.attn_dims(B, S, w.Hq, w.Hkv, w.D, self.inp["k_ctx"].shape[1], 0, 0, 0,
                                     w.softmax_scale, attn_splits)
            kc, vc, pt = dev(self.inp["k_ctx"]), dev(self.inp["v_ctx"]), None
        T = torch
        self.t = dict(
            x=dev(self.ad["x"]), shift_table=dev(self.ad["shift_table"]),
            scale_table=dev(self.ad["scale_table"]), q=dev(self.inp["q"]),
            k_blk=dev(self.inp["k_blk"]), v_blk=dev(self.inp["v_blk"]), k_ctx=kc, v_ctx=vc,
            page_table=pt, ctx_len=dev(self.inp["ctx_len"]),
            ids=T.full((B, S), w.mask_id, dtype=T.int32, device="cuda"),
            n_masked=T.full((B,), S, dtype=T.int32, device="cuda"),
            steps=T.zeros(B, dtype=T.int32, device="cuda"),
            commit_step=T.zeros((B, S), dtype=T.uint8, device="cuda"),
            y=T.empty((B, S, w.H), dtype=T.int16, device="cuda"),
            attn_out=T.empty((B, S, w.Hq, w.D), dtype=T.int16, device="cuda"),
            logits=None if lm_head else T.empty((B, S, w.V), dtype=T.float32, device="cuda"),
            conf=T.empty((B, S), dtype=T.float32, device="cuda"),
            commit=T.empty((B, S), dtype=T.uint8, device="cuda"),
            w_vocab=self.w_vocab, w_qkv=self.w_qkv)
        kind = tt.LOGITS_LM_HEAD if lm_head else w.logits_kind
        self.desc = tt.step_desc(self.dims, w.H, w.V, w.mask_id, w.gamma, w.steps_max, w.ln_eps,
                                 seed, 0, kind, w.boost_lo, w.boost_hi, sampler=sampler,
                                 temperature=temperature, qkv_proj=qkv_proj)
        self.ts = tt.step_tensors(**self.t)
        self.ws = tt.workspace(tt.tt_denoise_workspace(self.desc))
        ctx = self.inp["ctx_len"].astype(np.int64)
        self.kv_bytes = int(ctx.sum()) * w.Hkv * w.D * 2 * 2
        self.attn_bytes = (self.kv_bytes + B * S * w.Hq * w.D * 2 * 2 + B * S * w.Hkv * w.D * 2 * 2)
        self.attn_flops = 4 * w.Hq * S * w.D * int((ctx + S).sum())
        self.unmask_bytes_full = B * S * w.V * 4

    def _dev(self, a):
        a = np.ascontiguousarray(a)
        T = self.torch
        return T.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    def reset(self):
        self.t["ids"].fill_(self.w.mask_id)
        self.t["n_masked"].fill_(self.w.S)
        self.t["steps"].zero_()
        self.t["commit_step"].zero_()

    def block(self, block_index: int):
        self.desc.logits.block_index = block_index
        self.tt.tt_denoise_block_loop(self.desc, self.ts, self.ws)

    def step(self, block_index: int):
        self.desc.logits.block_index = block_index
        self.tt.tt_denoise_step(self.desc, self.ts, self.ws)


def plan_blocks(wb: Workbench, first_block: int, need_steps: int):
    """Untimed pass: per-block batched step counts (max over sequences) until need_steps."""
    torch = wb.torch
    plan, total, bi = [], 0, first_block
    while total < need_steps:
        wb.reset()
        wb.block(bi)
        torch.cuda.synchronize()
        n = int(wb.t["steps"].max().item())
        n = max(n, 1)
        take = min(n, need_steps - total)
        plan.append((bi, n, take))
        total += take
        bi += 1
    return plan


def run_timed(wb: Workbench, plan, flush, hist=None):
    """Runs the plan; returns (elapsed seconds summed over blocks, kernel launches).

    hist (optional, int [S][T]): after each whole block, outside its events, adds one
    count per committed position at its commit step (position x step histogram)."""
    torch = wb.torch
    elapsed = 0.0
    launches = 0
    for bi, n, take in plan:
        flush()
        wb.reset()
        torch.cuda._sleep(KEEP_BUSY_CYCLES)  # the block's host-side enqueue hides behind this
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        # adaLN, [projection], split, merge, then logits + unmask or the LM head's 3 kernels
        per_step = (6 if wb.lm_head else 5) + (1 if wb.qkv_proj else 0)
        if take == n:
            wb.block(bi)
            launches += 2 + (per_step + 1) * n  # dyn-slot write + count, then the step and loop_cond
        else:
            for _ in range(take):
                wb.step(bi)
            launches += per_step * take
        e.record()
        e.synchronize()
        elapsed += s.elapsed_time(e) / 1e3
        if hist is not None and take == n:
            cs = wb.t["commit_step"].cpu().numpy().astype(np.int64)
            S, T = hist.shape
            for p_ in range(S):
                k = cs[:, p_]
                k = k[(k >= 1) & (k <= T)]
                np.add.at(hist[p_], k - 1, 1)
    return elapsed, launches


def kernel_times(wb: Workbench, flush, reps: int):
    """Standalone launches of the attention call and the first-step unmask, L2 flushed first."""
    tt, torch, w = wb.tt, wb.torch, wb.w
    B, S = w.B, w.S
    stream = torch.cuda.current_stream()
    att_ws = tt.workspace(tt.tt_denoise_attn_workspace(wb.dims))
    out = torch.empty((B, S, w.Hq, w.D), dtype=torch.int16, device="cuda")
    um_ws = tt.workspace(tt.tt_confidence_unmask_workspace(B, S, w.V))
    ids0 = torch.full((B, S), w.mask_id, dtype=torch.int32, device="cuda")
    ids = ids0.clone()
    steps = torch.zeros(B, dtype=torch.int32, device="cuda")
    spec = tt.tt_logits_spec(wb.seed, 0, w.logits_kind, w.boost_lo, w.boost_hi)
    logits = wb.t["logits"]
    if logits is None:  # the step runs the LM head; the stand-in unmask is timed on its own buffer
        logits = torch.empty((B, S, w.V), dtype=torch.float32, device="cuda")
    tt.tt_synthetic_logits(spec, logits, B, S, w.V, w.mask_id)
    res = {}
    for name in ("attn", "unmask"):
        ts = []
        for r in range(reps + 2):
            flush()
            if name == "unmask":
                ids.copy_(ids0)
                steps.zero_()
            # Keep the GPU busy while the host submits the call, so that host-side
            # argument marshalling never shows up between the two events.
            torch.cuda._sleep(KEEP_BUSY_CYCLES)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            if name == "attn":
                tt.tt_denoise_attn(wb.dims, wb.t["q"], wb.t["k_blk"], wb.t["v_blk"], wb.t["k_ctx"],
                                   wb.t["v_ctx"], wb.t["page_table"], wb.t["ctx_len"], out,
                                   ws=att_ws)
            else:
                tt.tt_confidence_unmask(logits, ids, steps, B, S, w.V, w.mask_id, w.gamma,
                                        w.steps_max, ws=um_ws)
            e.record(stream)
            e.synchronize()
            if r >= 2:
                ts.append(s.elapsed_time(e) / 1e3)
        res[name] = statistics.mean(ts)
    return res


def lmhead_cost(w: synth.Workload, rows: int):
    """Algorithmic FLOPs and bytes of one fused LM-head call over `rows` masked rows:
    2 * rows * H * V multiply-adds; W [V][H] and the hidden rows read once (bf16)."""
    return 2.0 * rows * w.H * w.V, float(w.V * w.H * 2 + rows * w.H * 2)


def run_lmhead(wb: Workbench, flush, reps: int = 5):
    """Standalone tt_lmhead_unmask calls on the workload's shape (every row masked, as
    at the first step of a block), L2 flushed before each; returns the leg's dict."""
    tt, torch, w = wb.tt, wb.torch, wb.w
    B, S = w.B, w.S
    if B * S > 4096:
        return None
    W = wb.w_vocab if wb.w_vocab is not None else wb._dev(synth.make_lmhead_weights(w, wb.seed))
    h = wb._dev(synth.make_hidden(w, wb.seed))
    ids = torch.full((B, S), w.mask_id, dtype=torch.int32, device="cuda")
    steps = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = tt.workspace(tt.tt_lmhead_unmask_workspace(B, S, w.H))
    smp = tt.tt_sampler(int(wb.desc.sampler), w.gamma, float(wb.desc.temperature), w.steps_max)
    stream = torch.cuda.current_stream()
    ts = []
    for r in range(reps + 2):
        flush()
        ids.fill_(w.mask_id)
        steps.zero_()
        torch.cuda._sleep(KEEP_BUSY_CYCLES)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        tt.tt_lmhead_unmask(h, W, ids, steps, B, S, w.H, w.V, w.mask_id, smp, ws=ws)
        e.record(stream)
        e.synchronize()
        if r >= 2:
            ts.append(s.elapsed_time(e) / 1e3)
    if tt.tt_device_status(True) != 0:
        raise RuntimeError("device-side error reported by tt_lmhead_unmask")
    t = statistics.mean(ts)
    flops, byts = lmhead_cost(w, B * S)
    peaks, kind = load_peaks()
    tc, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    bound = "tensor" if flops / (tc * 1e12) >= byts / (hbm * 1e9) else "hbm"
    achieved = flops / t / 1e12 if bound == "tensor" else byts / t / 1e9
    peak = tc if bound == "tensor" else hbm
    return {"us": t * 1e6, "rows": B * S, "H": w.H, "V": w.V, "flops": flops, "algorithmic_bytes": byts,
            "bound": bound, "achieved": achieved, "unit": "TFLOP/s" if bound == "tensor" else "GB/s",
            "peak": peak, "frac": achieved / peak, "peak_source": kind,
            "TFLOP_s": flops / t / 1e12, "GB_s": byts / t / 1e9,
            "roofline_us": max(flops / (tc * 1e12), byts / (hbm * 1e9)) * 1e6,
            "call": "tt_lmhead_unmask, every row masked (first step of a block), L2 flushed"}


def run_qkv(wb: Workbench, flush, reps: int = 5):
    """Standalone tt_qkv_project calls on the workload's shape (every position), L2
    flushed before each; returns the leg's dict with its roofline."""
    tt, torch, w = wb.tt, wb.torch, wb.w
    B, S, N = w.B, w.S, (w.Hq + 2 * w.Hkv) * w.D
    W = wb.w_qkv if wb.w_qkv is not None else wb._dev(synth.make_qkv_weights(w, wb.seed))
    y = wb._dev(synth.make_hidden(w, wb.seed))
    q = torch.empty((B, S, w.Hq, w.D), dtype=torch.int16, device="cuda")
    k = torch.empty((B, S, w.Hkv, w.D), dtype=torch.int16, device="cuda")
    v = torch.empty_like(k)
    stream = torch.cuda.current_stream()
    ts = []
    for r in range(reps + 2):
        flush()
        torch.cuda._sleep(KEEP_BUSY_CYCLES)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        tt.tt_qkv_project(y, W, q, k, v, B, S, w.H, w.Hq, w.Hkv, w.D)
        e.record(stream)
        e.synchronize()
        if r >= 2:
            ts.append(s.elapsed_time(e) / 1e3)
    if tt.tt_device_status(True) != 0:
        raise RuntimeError("device-side error reported by tt_qkv_project")
    t = statistics.mean(ts)
    flops = 2.0 * B * S * w.H * N
    byts = float(N * w.H * 2 + B * S * (w.H + N) * 2)  # W, y read once; q/k/v written once
    peaks, kind = load_peaks()
    tc, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    bound = "tensor" if flops / (tc * 1e12) >= byts / (hbm * 1e9) else "hbm"
    achieved = flops / t / 1e12 if bound == "tensor" else byts / t / 1e9
    peak = tc if bound == "tensor" else hbm
    return {"us": t * 1e6, "rows": B * S, "N": N, "H": w.H, "flops": flops, "algorithmic_bytes": byts,
            "bound": bound, "achieved": achieved, "unit": "TFLOP/s" if bound == "tensor" else "GB/s",
            "peak": peak, "frac": achieved / peak, "peak_source": kind,
            "roofline_us": max(flops / (tc * 1e12), byts / (hbm * 1e9)) * 1e6,
            "call": "tt_qkv_project over every position, L2 flushed"}


def kernel_only(wb: Workbench, which: str, reps: int):
    """Standalone calls of one entry point, for profiler captures (no JSON bench line)."""
    tt, torch, w = wb.tt, wb.torch, wb.w
    B, S = w.B, w.S
    att_ws = tt.workspace(tt.tt_denoise_attn_workspace(wb.dims))
    out = torch.empty((B, S, w.Hq, w.D), dtype=torch.int16, device="cuda")
    um_ws = tt.workspace(tt.tt_confidence_unmask_workspace(B, S, w.V))
    ids0 = torch.full((B, S), w.mask_id, dtype=torch.int32, device="cuda")
    ids = ids0.clone()
    steps = torch.zeros(B, dtype=torch.int32, device="cuda")
    spec = tt.tt_logits_spec(wb.seed, 0, w.logits_kind, w.boost_lo, w.boost_hi)
    logits = wb.t["logits"]
    if logits is None:  # the step runs the LM head; the stand-in unmask is timed on its own buffer
        logits = torch.empty((B, S, w.V), dtype=torch.float32, device="cuda")
    tt.tt_synthetic_logits(spec, logits, B, S, w.V, w.mask_id)
    y = torch.empty((B, S, w.H), dtype=torch.int16, device="cuda")
    if which == "qkv":
        Wq = wb.w_qkv if wb.w_qkv is not None else wb._dev(synth.make_qkv_weights(w, wb.seed))
        hq = wb._dev(synth.make_hidden(w, wb.seed))
        qo = torch.empty((B, S, w.Hq, w.D), dtype=torch.int16, device="cuda")
        ko = torch.empty((B, S, w.Hkv, w.D), dtype=torch.int16, device="cuda")
        vo = torch.empty_like(ko)
    if which == "lmhead":
        W = wb.w_vocab if wb.w_vocab is not None else wb._dev(synth.make_lmhead_weights(w, wb.seed))
        h = wb._dev(synth.make_hidden(w, wb.seed))
        lm_ws = tt.workspace(tt.tt_lmhead_unmask_workspace(B, S, w.H))
        smp = tt.tt_sampler(int(wb.desc.sampler), w.gamma, float(wb.desc.temperature), w.steps_max)

    def call():
        if which == "attn":
            tt.tt_denoise_attn(wb.dims, wb.t["q"], wb.t["k_blk"], wb.t["v_blk"], wb.t["k_ctx"],
                               wb.t["v_ctx"], wb.t["page_table"], wb.t["ctx_len"], out, ws=att_ws)
        elif which == "unmask":
            ids.copy_(ids0)
            steps.zero_()
            tt.tt_confidence_unmask(logits, ids, steps, B, S, w.V, w.mask_id, w.gamma,
                                    w.steps_max, ws=um_ws)
        elif which == "adaln":
            tt.tt_adaln_modulate(wb.t["x"], wb.t["shift_table"], wb.t["scale_table"], y,
                                 eps=w.ln_eps, row_index=wb.t["n_masked"], table_rows=S + 1)
        elif which == "logits":
            tt.tt_synthetic_logits(spec, logits, B, S, w.V, w.mask_id)
        elif which == "qkv":
            tt.tt_qkv_project(hq, Wq, qo, ko, vo, B, S, w.H, w.Hq, w.Hkv, w.D)
        elif which == "lmhead":
            ids.copy_(ids0)
            steps.zero_()
            tt.tt_lmhead_unmask(h, W, ids, steps, B, S, w.H, w.V, w.mask_id, smp, ws=lm_ws)
        else:
            wb.reset()
            wb.step(0)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        call()
    e.record()
    e.synchronize()
    if tt.tt_device_status(True) != 0:
        raise RuntimeError("device-side error reported")
    print(json.dumps({"kernel_only": which, "workload": w.name, "reps": reps,
                      "us_per_call_back_to_back": s.elapsed_time(e) * 1e3 / reps}), flush=True)


def run_e2e(wb: Workbench, plan, torch, tt):
    """Same plan through the public API with host buffers: every block copies its inputs
    from pinned host memory and reads back ids/steps/commit_step."""
    names = ["x", "shift_table", "scale_table", "q", "k_blk", "v_blk", "k_ctx", "v_ctx",
             "page_table", "ctx_len"]
    host = {k: torch.empty(wb.t[k].shape, dtype=wb.t[k].dtype, pin_memory=True).copy_(wb.t[k])
            for k in names if wb.t[k] is not None}
    ids_h = torch.full(wb.t["ids"].shape, wb.w.mask_id, dtype=torch.int32, pin_memory=True)
    out_ids = torch.empty_like(ids_h, pin_memory=True)
    out_steps = torch.empty(wb.t["steps"].shape, dtype=torch.int32, pin_memory=True)
    out_cs = torch.empty(wb.t["commit_step"].shape, dtype=torch.uint8, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values()) + ids_h.numel() * 4
    d2h = out_ids.numel() * 4 + out_steps.numel() * 4 + out_cs.numel()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for bi, n, take in plan:
        for k, v in host.items():
            wb.t[k].copy_(v, non_blocking=True)
        wb.t["ids"].copy_(ids_h, non_blocking=True)
        wb.t["steps"].zero_()
        wb.t["commit_step"].zero_()
        if take == n:
            wb.block(bi)
        else:
            wb.t["n_masked"].fill_(wb.w.S)
            for _ in range(take):
                wb.step(bi)
        out_ids.copy_(wb.t["ids"], non_blocking=True)
        out_steps.copy_(wb.t["steps"], non_blocking=True)
        out_cs.copy_(wb.t["commit_step"], non_blocking=True)
    e.record()
    e.synchronize()
    return s.elapsed_time(e) / 1e3, h2d, d2h


def run_generate(wb: Workbench, n_blocks: int, flush, reps: int = 3):
    """Algorithm 1's outer loop on the device: the prompt cache of the workload with room
    for n_blocks more blocks, then tt_generate (per block: reset, the captured denoise
    loop, tt_append_block) with no end-of-sequence id, so every sequence decodes every
    block.  Returns a dict for the JSON line (best of reps, L2 flushed before each)."""
    tt, torch, w = wb.tt, wb.torch, wb.w
    B, S = w.B, w.S
    L0 = wb.t["k_ctx"].shape[1]
    cap = L0 + n_blocks * S
    kc = torch.zeros((B, cap, w.Hkv, w.D), dtype=torch.int16, device="cuda")
    vc = torch.zeros_like(kc)
    kc[:, :L0].copy_(wb.t["k_ctx"])
    vc[:, :L0].copy_(wb.t["v_ctx"])
    ctx0 = wb.t["ctx_len"].clone()
    dims = tt.attn_dims(B, S, w.Hq, w.Hkv, w.D, cap, 0, 0, 0, w.softmax_scale, 0)
    desc = tt.step_desc(dims, w.H, w.V, w.mask_id, w.gamma, w.steps_max, w.ln_eps, wb.seed, 0,
                        wb.desc.logits.kind, w.boost_lo, w.boost_hi, sampler=wb.desc.sampler,
                        temperature=wb.desc.temperature, qkv_proj=bool(wb.desc.qkv_proj))
    t = dict(wb.t)
    t.update(k_ctx=kc, v_ctx=vc, ctx_len=ctx0.clone())
    ts = tt.step_tensors(**t)
    ws = tt.workspace(tt.tt_denoise_workspace(desc))
    gen = torch.zeros(B, dtype=torch.int32, device="cuda")
    done = torch.zeros(B, dtype=torch.uint8, device="cuda")
    out = torch.empty((B, n_blocks * S), dtype=torch.int32, device="cuda")
    stop = tt.tt_stop_spec(-1, 0, n_blocks * S)

    def reset():
        t["ctx_len"].copy_(ctx0)
        gen.zero_()
        done.zero_()

    best = None
    for _ in range(reps + 1):  # the first call captures the block-loop graph: untimed
        flush()
        reset()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        tt.tt_generate(desc, ts, n_blocks, stop, gen, done, out, ws)
        e.record()
        e.synchronize()
        dt = s.elapsed_time(e) / 1e3
        best = dt if best is None or dt < best else best
    if tt.tt_device_status(True) != 0:
        raise RuntimeError("device-side error reported by tt_generate")
    if t["ctx_len"].tolist() != (ctx0 + n_blocks * S).tolist() or gen.tolist() != [n_blocks * S] * B:
        raise RuntimeError("tt_generate did not decode every block")
    # the append kernel alone (one block into the grown cache, state reset between calls)
    ctx_mid = ctx0 + (n_blocks - 1) * S
    ta = []
    for _ in range(reps + 2):
        t["ctx_len"].copy_(ctx_mid)
        done.zero_()
        flush()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        tt.tt_append_block(dims, t["k_blk"], t["v_blk"], kc, vc, None, t["ctx_len"], t["ids"], stop, gen,
                           done, out, n_blocks * S, 0)
        e.record()
        e.synchronize()
        ta.append(s.elapsed_time(e) / 1e3)
    ta = sorted(ta[2:])[len(ta[2:]) // 2]
    append_bytes = 2 * 2 * B * S * w.Hkv * w.D * 2  # K and V rows, read once and written once
    return {"blocks": n_blocks, "tokens": B * S * n_blocks, "ms": best * 1e3,
            "tokens_per_s": B * S * n_blocks / best, "blocks_per_s": n_blocks / best,
            "cache_rows_start": int(ctx0.max().item()), "eos": "none (every block decoded)",
            "append_block_us": ta * 1e6, "append_block_bytes": append_bytes,
            "append_block_GB_s": append_bytes / ta / 1e9,
            "l2": "flushed before each timed call"}


# ------------------------------------------------------------------ CPU oracle legs
def oracle_block_time(w: synth.Workload, seed: int, block: int, max_steps=None, b_sample=None):
    """The oracle decoding one block of the workload on the host cores.

    Returns (denoise steps done, seconds, sample description).  Each step runs the
    oracle's adaLN, attention (all rows of the sampled sequences), the logits
    generator for the masked rows and the unmask decision."""
    import oracle
    B = w.B if b_sample is None else min(w.B, b_sample)
    ws = w.replace(B=B)
    inp = synth.make_attention_inputs(ws, seed)
    ad = synth.make_adaln_inputs(ws, seed)
    ids = np.full((B, w.S), w.mask_id, np.int64)
    steps = np.zeros(B, np.int64)
    cs = np.zeros((B, w.S), np.uint8)
    n = 0
    t0 = time.perf_counter()
    while np.any(ids == w.mask_id) and (max_steps is None or n < max_steps):
        nm = (ids == w.mask_id).sum(axis=1)
        for b in range(B):
            if nm[b] == 0:
                continue
            oracle.adaln_modulate(ad["x"][b], ad["shift_table"][nm[b]], ad["scale_table"][nm[b]],
                                  w.ln_eps)
        act = [b for b in range(B) if nm[b] > 0]
        rows = [(b, s, h) for b in act for s in range(w.S) for h in range(w.Hq)]
        oracle.denoise_attention_rows(inp, w.softmax_scale, rows)
        for b in act:
            pos = np.flatnonzero(ids[b] == w.mask_id)
            lg = np.zeros((w.S, w.V), np.float32)
            lg[pos] = synth.logits_rows(seed, b, block, int(steps[b]), pos, w.V, w.mask_id,
                                        w.logits_kind, w.boost_lo, w.boost_hi)
            r = oracle.unmask_step(lg, ids[b], int(steps[b]), w.mask_id, w.gamma, w.steps_max, cs[b])
            ids[b], steps[b], cs[b] = r["ids"], r["steps"], r["commit_step"]
        n += 1
    dt = time.perf_counter() - t0
    return n, dt, B


def cpu_baseline(w: synth.Workload, seed: int, budget: float = 20.0):
    """The oracle on the host cores, on a bounded sample: one sequence of the batch,
    decoded step by step (whole blocks while they fit), stopping once about half the
    budget is spent; steps/s scaled to the full batch."""
    steps, secs, block = 0, 0.0, 0
    b_sample = 1 if w.B > 1 else None
    B = 1
    while secs < budget / 2 and block < 64:
        n, dt, B = oracle_block_time(w, seed, block, b_sample=b_sample,
                                     max_steps=None if w.B == 1 and w.L <= 8192 else 2)
        steps += n
        secs += dt
        block += 1
    frac = B / w.B
    # a denoise step of the full batch costs ~1/frac of the sampled one on the CPU
    value = steps / secs * frac
    sample = (f"{steps} denoise steps over {block} block(s) of {B} of {w.B} sequence(s), "
              f"{secs:.1f} s; steps/s scaled by {frac:g} to the full batch")
    return {"value": value, "unit": "denoise steps/s", "cores": cores_used(), "kind": "oracle",
            "sample": sample}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = workload(args)
    b_sample = 1 if w.B > 1 else None
    # warm-up steps
    done, _, _ = oracle_block_time(w, args.seed, 10_000, max_steps=max(args.warmup, 3), b_sample=b_sample)
    steps, secs, block = 0, 0.0, 0
    while steps < args.steps:
        n, dt, B = oracle_block_time(w, args.seed, block, max_steps=args.steps - steps, b_sample=b_sample)
        steps += n
        secs += dt
        block += 1
    frac = B / w.B
    value = steps / secs * frac
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "denoise steps/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": max(args.warmup, 3),
        "ms_per_step": 1e3 / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "gamma": w.gamma, "bench_step": "one denoise step of the batch"},
        "cpu_baseline": {"value": value, "unit": "denoise steps/s", "cores": cores_used(),
                         "kind": "oracle",
                         "sample": f"{steps} denoise steps over {block} block(s) of {B} of {w.B} "
                                   f"sequence(s), scaled by {frac:g}"},
        "e2e": {"value": value, "unit": "denoise steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main
def kernel_rooflines(wb: Workbench, ktimes: dict):
    """Per-kernel figures of the standalone attention and unmask calls, and one roofline
    object per call (algorithmic work / mean duration against the measured peak)."""
    peaks, peak_kind = load_peaks()
    hbm, tc = peaks["hbm_gbs"], peaks["bf16_tflops"]
    w = wb.w
    attn_gbs = wb.attn_bytes / ktimes["attn"] / 1e9
    attn_tfs = wb.attn_flops / ktimes["attn"] / 1e12
    attn_bound = "hbm" if wb.attn_bytes / hbm / 1e9 >= wb.attn_flops / tc / 1e12 else "tensor"
    attn_roof = max(wb.attn_bytes / (hbm * 1e9), wb.attn_flops / (tc * 1e12))
    um_gbs = wb.unmask_bytes_full / ktimes["unmask"] / 1e9
    kernels = {
        "tt_denoise_attn": {"us": ktimes["attn"] * 1e6, "GB_s": attn_gbs, "TFLOP_s": attn_tfs,
                            "bound": attn_bound, "roofline_us": attn_roof * 1e6,
                            "frac": attn_roof / ktimes["attn"], "algorithmic_bytes": wb.attn_bytes,
                            "flops": wb.attn_flops},
        "tt_confidence_unmask": {"us": ktimes["unmask"] * 1e6, "GB_s": um_gbs,
                                 "roofline_us": wb.unmask_bytes_full / (hbm * 1e9) * 1e6,
                                 "frac": um_gbs / hbm, "algorithmic_bytes": wb.unmask_bytes_full},
    }
    if attn_bound == "hbm":
        ra = {"kernel": "tt_denoise_attn (split + combine)", "bound": "hbm", "achieved": attn_gbs,
              "peak": hbm, "unit": "GB/s", "frac": attn_gbs / hbm}
    else:
        ra = {"kernel": "tt_denoise_attn (split + combine)", "bound": "tensor", "achieved": attn_tfs,
              "peak": tc, "unit": "TFLOP/s", "frac": attn_tfs / tc}
    ru = {"kernel": "tt_confidence_unmask (first step, all rows masked)", "bound": "hbm",
          "achieved": um_gbs, "peak": hbm, "unit": "GB/s", "frac": um_gbs / hbm}
    for r, call in ((ra, "attn"), (ru, "unmask")):
        r["traffic"], r["traffic_note"] = ncu_traffic(w.name, call)
        r["traffic_unit"] = "DRAM bytes per call"
        r["algorithmic_bytes"] = wb.attn_bytes if call == "attn" else wb.unmask_bytes_full
        r["peak_source"] = peak_kind
    return kernels, {"tt_denoise_attn": ra, "tt_confidence_unmask": ru}


def l2_note(wb: Workbench) -> str:
    kv = wb.kv_bytes
    lg = 0 if wb.t["logits"] is None else wb.w.B * wb.w.S * wb.w.V * 4
    warm = kv + lg < 126e6
    return ("L2 flushed (512 MiB write) before every timed block, outside the events; within a "
            f"block the context K/V ({kv / 1e6:.1f} MB) and logits ({lg / 1e6:.1f} MB) "
            + ("fit in the 126 MB L2, so steps 2..n of a block find them L2-resident"
               if warm else "exceed the 126 MB L2, so every step streams them from HBM"))


def measure_workload(args, tt, torch, w, seed, flush, world, dist, smi_id, legs: bool):
    """Steps/s of one workload (timed whole blocks), its standalone kernel times and
    rooflines, and the end-to-end figure through host buffers."""
    wb = Workbench(tt, torch, w, seed, SAMPLERS[args.sampler], args.temperature, args.lm_head,
                   args.qkv_proj, args.attn_splits)
    warm_plan = plan_blocks(wb, 100_000, max(args.warmup, 3))
    plan = plan_blocks(wb, 0, args.steps)
    total_steps = sum(t for _, _, t in plan)
    hist = np.zeros((w.S, w.steps_max), np.int64)
    with ClockSampler(smi_id) as clk:
        t_warm = time.time()
        run_timed(wb, warm_plan, flush)
        while time.time() - t_warm < args.min_warmup_s:
            run_timed(wb, warm_plan, flush)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        elapsed, launches = run_timed(wb, plan, flush, hist)
    torch.cuda.synchronize()
    if world > 1:
        elapsed = max_over_ranks(elapsed, dist, "cuda")
        dist.barrier()
    status = tt.tt_device_status(True)
    if status != 0:
        raise RuntimeError(f"device-side error {status} during the timed region ({w.name})")
    ktimes = kernel_times(wb, flush, args.kernel_reps)
    kernels, roofs = kernel_rooflines(wb, ktimes)
    lm = qkv = None
    if legs:
        lm = None if args.no_lm_head_leg and not args.lm_head else run_lmhead(wb, flush)
        if lm is not None:
            kernels["tt_lmhead_unmask"] = {k: lm[k] for k in ("us", "TFLOP_s", "GB_s", "bound", "roofline_us",
                                                               "frac", "algorithmic_bytes", "flops")}
        qkv = None if args.no_qkv_leg and not args.qkv_proj else run_qkv(wb, flush)
        if qkv is not None:
            kernels["tt_qkv_project"] = {k: qkv[k] for k in ("us", "bound", "roofline_us", "frac",
                                                            "algorithmic_bytes", "flops")}
    if args.lm_head and lm is not None and lm["us"] * 1e-6 > ktimes["attn"]:
        roof = {"kernel": "tt_lmhead_unmask (gather + GEMM + decision, first step)", "bound": lm["bound"],
                "achieved": lm["achieved"], "peak": lm["peak"], "unit": lm["unit"], "frac": lm["frac"],
                "peak_source": lm["peak_source"]}
        roof["traffic"], roof["traffic_note"] = ncu_traffic(w.name, "lmhead")
        roof["traffic_unit"] = "DRAM bytes per call"
    else:
        dominant = "tt_denoise_attn" if ktimes["attn"] >= ktimes["unmask"] else "tt_confidence_unmask"
        roof = dict(roofs[dominant])
    e2e = None
    if not args.no_e2e:
        e_el, h2d, d2h = run_e2e(wb, plan, torch, tt)
        if world > 1:
            e_el = max_over_ranks(e_el, dist, "cuda")
        e2e = {"value": job_throughput(total_steps, world, e_el), "unit": "denoise steps/s",
               "h2d_bytes_per_step": int(h2d * len(plan) / total_steps),
               "d2h_bytes_per_step": int(d2h * len(plan) / total_steps)}
    whole = [(bi, n, t) for bi, n, t in plan if t == n]
    res = {
        "workload": w.name, "value": job_throughput(total_steps, world, elapsed),
        "unit": "denoise steps/s", "steps": total_steps,
        "warmup": sum(t for _, _, t in warm_plan), "ms_per_step": 1e3 * elapsed / total_steps,
        "config": {"workload": w.name, "B": w.B, "L": w.L, "L_min": w.L_min, "S": w.S, "Hq": w.Hq,
                   "Hkv": w.Hkv, "D": w.D, "H": w.H, "V": w.V, "gamma": w.gamma, "paged": w.paged,
                   "blocks_timed": len(plan), "whole_blocks": len(whole), "l2": l2_note(wb)},
        "tokens_per_step": (w.B * w.S * len(whole) / max(1, sum(n for _, n, _ in whole))) if whole else None,
        "commit_histogram": {"rows": "block position", "cols": "commit step (1-based)",
                             "counts": hist.tolist()},
        "roofline": roof,
        "rooflines": roofs,
        "kernels": kernels,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    return res, wb, lm, qkv


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    rank, world, local = dist_env()
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from block_wise_mask_tt_b300 import tt

    w = workload(args)
    seed = replica_seed(args.seed, rank)
    if args.kernel_only:
        wb = Workbench(tt, torch, w, seed, SAMPLERS[args.sampler], args.temperature, args.lm_head,
                       args.qkv_proj, args.attn_splits)
        kernel_only(wb, args.kernel_only, args.reps)
        return
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    def flush():
        flush_buf.zero_()

    try:
        smi_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        smi_id = str(local)

    head, wb, lm, qkv = measure_workload(args, tt, torch, w, seed, flush, world, dist, smi_id, legs=True)
    gen_line = None
    others = {}
    other_ids = [int(c) for c in args.other_configs.split(",") if c.strip() != ""]
    other_ids = [c for c in other_ids if c != args.config]
    del wb
    for c in other_ids:
        torch.cuda.empty_cache()
        wc = synth.WORKLOADS[c]
        if args.gamma is not None:
            wc = wc.replace(gamma=args.gamma)
        res, wbc, _, _ = measure_workload(args, tt, torch, wc, seed, flush, world, dist, smi_id, legs=False)
        if gen_line is None and args.generate > 0 and not wc.paged:
            gen_line = run_generate(wbc, args.generate, flush)
            gen_line["workload"] = wc.name
        others[wc.name] = res
        del wbc
    if gen_line is None and args.generate > 0 and not w.paged:
        wbh = Workbench(tt, torch, w, seed, SAMPLERS[args.sampler], args.temperature, args.lm_head,
                        args.qkv_proj)
        gen_line = run_generate(wbh, args.generate, flush)
        gen_line["workload"] = w.name

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(w, seed)
    cfg = dict(head["config"])
    cfg.update({"bench_step": "one denoise step of the whole batch",
                "logits": ("fused LM head over the adaLN output (synthetic W [V][H], resident)"
                           if args.lm_head else "hash stand-in"),
                "qkv": ("projected from the adaLN output every step (synthetic W_qkv, resident)"
                        if args.qkv_proj else "fixed synthetic tensors"),
                "sampler": args.sampler, "temperature": args.temperature,
                "parallelism": f"replicas{world}"})
    line = {
        "metric": METRIC, "value": head["value"], "unit": "denoise steps/s", "n_gpus": world,
        "steps": head["steps"], "warmup": head["warmup"], "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": cfg,
        "tokens_per_step": head["tokens_per_step"],
        "roofline": head["roofline"],
        "rooflines": head["rooflines"],
        "kernels": head["kernels"],
        "cpu_baseline": cpu,
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        "commit_histogram": head["commit_histogram"],
        "configs": others,
        "generate": gen_line,
        "lm_head": lm,
        "qkv_proj": qkv,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
