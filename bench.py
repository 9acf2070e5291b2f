#!/usr/bin/env python3
"""Benchmark of the TwoTower block-diffusion denoise path on one B300 (or N replicas).

Workload (the full block decode): B=64 sequences, context KV length 8192 per sequence, block
S=16, T=16 steps, 6 stacked denoiser attention layers each with its own context-layer KV
cache, d=4096, 32 query / 2 KV heads, head_dim 128, vocabulary 131072, gamma=0.8, bf16.
One bench step = one td_decode_block call on a fresh all-[MASK] block: embedding, adaLN,
QKV projection, fused block attention, gated O projection, LM head + commit, repeated until
every position is committed. Inputs are seeded synthetic tensors created in HBM. The LM-head
weights use the calibrated scale of the workload (logits as sharp as the mid-size step's, so
several positions clear gamma early in a block); the same block with the plain scale (one
commit per sequence and step, the 16-step worst case) is timed as well.

value = committed tokens / s (B*S per block / block wall time), whole job over all ranks.
Also printed: denoised tokens / s (B*S*steps / time), the roofline of the dominant kernel,
the fp64 oracle timed on the host cores on a bounded sample, end-to-end numbers through the
Python API with host buffers, and SM clocks sampled during the timed region.

Multi-GPU: the path shards by sequence and needs no exchange, so N ranks run N independent
replicas (weak scaling); only a barrier and a max of the elapsed time cross ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import select
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

WORKLOAD = dict(workload="block decode loop", B=64, S=16, L=8192, n_layers=6, d=4096, Hq=32,
                Hkv=2, D=128, V=131072, T=16, gamma=0.8)
FALLBACK_W_LM_SIGMA = 0.02   # the plain LM-head scale: no position clears any threshold
MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0)


PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "block_diffusion_lm_denoise_b300", "csrc")


def code_text(src: str) -> str:
    """C/C++/CUDA source with its comments removed and every run of white space turned into
    one space, so that an edit of comments or layout alone keeps a source's hash (string and
    character literals are kept as they are)."""
    out = []
    i, n = 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash(sources) -> str:
    """sha1 over the code text (see code_text) of the given kernel sources, in order."""
    import hashlib
    h = hashlib.sha1()
    for f in sources:
        with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
            h.update(code_text(fh.read()).encode())
        h.update(b"\0")
    return h.hexdigest()


def traffic_per_launch(kernel: str, sources, units: int):
    """DRAM bytes (read + write) per launch of `kernel` from the ncu summaries committed under
    profiles/ ("traffic-record:" lines), scaled from the captured case to `units` (traffic
    grows in proportion to the units processed). None when no record matches the current
    sources (the kernel's code changed since its counters were taken; comments do not
    count)."""
    import glob
    sha = source_hash(sources)
    for path in sorted(glob.glob(os.path.join(PROFILES, "*.md"))):
        with open(path) as fh:
            for line in fh:
                if not line.startswith("traffic-record:"):
                    continue
                f = line.split()
                kv = dict(x.split("=", 1) for x in f[2:] if "=" in x)
                if f[1] == kernel and kv.get("sha1") == sha:
                    return round(int(kv["dram_bytes"]) * units / int(kv["units"]))
    return None


def peaks():
    try:
        with open(MEASURED_PEAKS) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return FALLBACK_PEAKS, "fallback"


# ------------------------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        if self.proc is not None:
            # nvidia-smi needs a while to start: wait for its first sample (taken before the
            # segment, so dropped) so that a short segment still gets samples
            ready, _, _ = select.select([self.proc.stdout], [], [], 5.0)
            if ready:
                self.proc.stdout.readline()
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, ms=None):
        """Median SM clock, its maximum and the throttle reasons seen; with the segment's
        device time `ms`, also time x median clock (kilocycles), which compares segments
        timed at different clocks."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
               "reasons": sorted(reasons), "samples": len(sm)}
        if ms is not None and sm:
            out["kcycles"] = round(ms * statistics.median(sm), 1)
        return out


# ------------------------------------------------------------------------------ oracle sample

class OracleSampler:
    """The fp64 oracle decoding blocks of a few sequences of the workload, step by step
    (a bounded sample: it continues the same block across calls, starting a new block when
    one is fully committed)."""

    def __init__(self, wl, rows=(0,)):
        import numpy as np
        self.np = np
        self.wl = wl
        self.rows = list(rows)
        self.layers = [{k: (v[self.rows].cpu() if k in ("k_ctx", "v_ctx") else v.cpu())
                        for k, v in L.items()} for L in wl.layers]
        self.w, self.emb = wl.w_lm.cpu(), wl.emb.cpu()
        self.pos, self.phi = wl.pos.cpu(), wl.phi_table.cpu()
        self.d = dict(wl.dims.as_dict(), B=len(self.rows))
        self._reset()

    def _reset(self):
        dm = self.wl.dims
        self.tok = self.np.full((len(self.rows), dm.S), dm.V)
        self.msk = self.np.ones((len(self.rows), dm.S), bool)
        self.t = 1

    def step(self) -> int:
        import oracle
        wl = self.wl
        r = oracle.denoise_step(self.d, self.layers, self.phi[self.t - 1], self.w, self.tok,
                                self.msk, wl.gamma, self.t, wl.T, emb=self.emb, pos=self.pos)
        self.tok, self.msk = r["tokens"], r["masked"]
        self.t += 1
        if not self.msk.any() or self.t > wl.T:
            self._reset()
        return int(r["n_committed"].sum())

    def describe(self, steps: int) -> str:
        dm = self.wl.dims
        return (f"fp64 oracle on {len(self.rows)} of {dm.B} sequences: {steps} denoise steps "
                f"of the block loop ({dm.n_layers} layers, L={dm.Lmax}, V={dm.V}); "
                f"committed tokens / wall time")


def oracle_sample(wl, seconds_budget: float, max_steps: int):
    s = OracleSampler(wl)
    committed = steps = 0
    t0 = time.perf_counter()
    while steps < max_steps:
        committed += s.step()
        steps += 1
        if time.perf_counter() - t0 > seconds_budget:
            break
    el = time.perf_counter() - t0
    return committed / el, torch.get_num_threads(), s.describe(steps), steps


def host_cores():
    """(logical cores of the host, threads the oracle's numerical libraries use)."""
    return os.cpu_count(), torch.get_num_threads()


# ------------------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=20.0,
                    help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--loop-graph", default="conditional", choices=["conditional", "flat"],
                    help="form of the decode-loop graph (ncu's launch list sees the kernels "
                         "of the flat form only)")
    ap.add_argument("--only", choices=["attention", "lmhead", "step"],
                    help="launch one kernel family alone, or one denoise step of one layer "
                         "(for profiler captures)")
    ap.add_argument("--sweep", action="store_true",
                    help="time the attention over context lengths and the LM head over row "
                         "counts, one JSON line per case (L2 flushed before every launch)")
    ap.add_argument("--B", type=int, default=32)
    ap.add_argument("--L", type=int, default=8192)
    ap.add_argument("--M", type=int, default=1024)
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()

    world, rank, local = dist_setup()
    from block_diffusion_lm_denoise_b300 import synth

    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.only:
        run_only(args)
        return
    if args.sweep:
        run_sweep(args)
        return

    import block_diffusion_lm_denoise_b300 as td
    td.lib()   # fails loudly if the CUDA library is missing
    if args.loop_graph == "flat":
        td.td_decode_graph_form(td.TD_GRAPH_FLAT)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = synth.decode_loop(dev, seed=4 + rank, w_lm_sigma=synth.DECODE_W_LM_SIGMA)
    dm = wl.dims
    dims = dm.as_dict()
    M = dm.B * dm.S
    ws = td.workspace(dims, td.TD_FN_DECODE_BLOCK, dev)
    tokens = torch.empty_like(wl.tokens)
    masked = torch.empty_like(wl.masked)
    outs = td._outs(dm.B, dm.S, dev, None, None, None, None)

    # the attention alone before anything else runs (the GPU below its power cap): the same
    # launches as the roofline segment after the decode loop, whose clocks the cap lowers
    stream0 = torch.cuda.current_stream()
    q_c = synth.normal((dm.B, dm.S, dm.Hq, dm.D), 1.0, 99, "bench.q", dev)
    kb_c = synth.normal((dm.B, dm.S, dm.Hkv, dm.D), 1.0, 99, "bench.kb", dev)
    vb_c = synth.normal((dm.B, dm.S, dm.Hkv, dm.D), 1.0, 99, "bench.vb", dev)
    o_c = torch.empty_like(q_c)
    aws_c = td.workspace(dims, td.TD_FN_BLOCK_ATTENTION, dev)
    lay0 = wl.layers[0]
    for _ in range(3):
        td.td_block_attention(dims, q_c, kb_c, vb_c, lay0["k_ctx"], lay0["v_ctx"], o=o_c, ws=aws_c)
    torch.cuda.synchronize()
    c_reps = 400
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as cclocks:
        c0.record(stream0)
        for _ in range(c_reps):
            td.td_block_attention(dims, q_c, kb_c, vb_c, lay0["k_ctx"], lay0["v_ctx"], o=o_c,
                                  ws=aws_c)
        c1.record(stream0)
        torch.cuda.synchronize()
    cool_ms = c0.elapsed_time(c1) / c_reps
    del q_c, kb_c, vb_c, o_c, aws_c

    def one_block(w_lm=None):
        tokens.fill_(dm.V)
        masked.fill_(1)
        return td.td_decode_block(dims, wl.layers, wl.emb, wl.pos,
                                  wl.w_lm if w_lm is None else w_lm, wl.phi_table, wl.T,
                                  wl.gamma, tokens, masked, conf=outs[0], pred=outs[1],
                                  n_committed=outs[2], all_done=outs[3], ws=ws)

    for _ in range(max(3, args.warmup)):
        one_block()
    torch.cuda.synchronize()
    assert td.td_device_error() == 0

    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps_taken = []
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        ev0.record(stream)
        for _ in range(args.steps):
            steps_taken.append(one_block())
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, world)
    total_steps = sum(steps_taken)
    value = world * M * args.steps / (ms_max / 1e3)
    denoised = world * M * total_steps / (ms_max / 1e3)

    # ---------------------------------------------------------------- the plain LM-head scale
    # the same block with W_lm ~ N(0, 0.02): no confidence clears gamma, one commit per
    # sequence and step (the fallback), 16 steps per block
    w_plain = synth.normal((dm.V, dm.d), FALLBACK_W_LM_SIGMA, 4 + rank, "w_lm", dev)
    for _ in range(2):
        one_block(w_plain)
    torch.cuda.synchronize()
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as fclocks:
        f0.record(stream)
        fsteps = [one_block(w_plain) for _ in range(args.steps)]
        f1.record(stream)
        torch.cuda.synchronize()
    fms = max_over_ranks(f0.elapsed_time(f1), world)
    fallback = {"w_lm_sigma": FALLBACK_W_LM_SIGMA,
                "committed_tokens_per_s": round(world * M * args.steps / (fms / 1e3), 1),
                "denoised_tokens_per_s": round(world * M * sum(fsteps) / (fms / 1e3), 1),
                "steps_per_block": round(sum(fsteps) / args.steps, 3),
                "ms_per_block": round(fms / args.steps, 3),
                "clocks": fclocks.summary(fms)}
    del w_plain

    # ---------------------------------------------------------------- commit-rule sweep
    # steps per block and committed tokens/s of one block at other thresholds and under the
    # left-to-right rule (the pages: lower gamma commits more per step; mock-AR one per step)
    sweep = []
    hist = None
    for g, rule in ((0.5 / dm.V, td.TD_COMMIT_CONFIDENCE), (0.5, td.TD_COMMIT_CONFIDENCE),
                    (0.8, td.TD_COMMIT_CONFIDENCE), (0.95, td.TD_COMMIT_CONFIDENCE),
                    (0.8, td.TD_COMMIT_LEFT_TO_RIGHT)):
        def blk():
            tokens.fill_(dm.V)
            masked.fill_(1)
            return td.td_decode_block(dims, wl.layers, wl.emb, wl.pos, wl.w_lm, wl.phi_table,
                                      wl.T, g, tokens, masked, conf=outs[0], pred=outs[1],
                                      n_committed=outs[2], all_done=outs[3], ws=ws, rule=rule)
        blk()   # captures this argument set's graph
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        st = blk()
        s1.record(stream)
        torch.cuda.synchronize()
        bms = s0.elapsed_time(s1)
        sweep.append({"gamma": g, "rule": "left_to_right" if rule else "confidence",
                      "steps_per_block": st, "commits_per_step": round(M / st, 2),
                      "committed_tokens_per_s": round(world * M / (bms / 1e3), 1)})

    # ---------------------------------------------------------------- commits per step
    # one block of the headline configuration step by step: positions committed at each step
    # (all sequences), from td_denoise_step's per-sequence counts
    sws = td.workspace(dims, td.TD_FN_DENOISE_STEP, dev)
    tokens.fill_(dm.V)
    masked.fill_(1)
    hist = []
    for t in range(1, wl.T + 1):
        _, _, ncm, dn = td.td_denoise_step(dims, wl.layers, wl.w_lm, wl.phi_table[t - 1], t,
                                           wl.T, wl.gamma, tokens, masked, emb=wl.emb,
                                           pos=wl.pos, ws=sws)
        hist.append(int(ncm.sum().item()))
        if int(dn.item()):
            break
    del sws

    # ---------------------------------------------------------------- end to end (host buffers)
    tok_h = torch.full((dm.B, dm.S), dm.V, dtype=torch.int32).pin_memory()
    msk_h = torch.ones((dm.B, dm.S), dtype=torch.uint8).pin_memory()
    tok_out = torch.empty((dm.B, dm.S), dtype=torch.int32).pin_memory()
    torch.cuda.synchronize()
    barrier(world)
    e0 = time.perf_counter()
    for _ in range(args.steps):
        tokens.copy_(tok_h, non_blocking=True)
        masked.copy_(msk_h, non_blocking=True)
        td.td_decode_block(dims, wl.layers, wl.emb, wl.pos, wl.w_lm, wl.phi_table, wl.T,
                           wl.gamma, tokens, masked, conf=outs[0], pred=outs[1],
                           n_committed=outs[2], all_done=outs[3], ws=ws)
        tok_out.copy_(tokens, non_blocking=True)
        torch.cuda.synchronize()
    e_s = max_over_ranks(time.perf_counter() - e0, world)
    e2e = world * M * args.steps / e_s

    # ---------------------------------------------------------------- roofline (isolated kernels)
    pk, pk_kind = peaks()
    lay = wl.layers[0]
    q = synth.normal((dm.B, dm.S, dm.Hq, dm.D), 1.0, 99, "bench.q", dev)
    kb = synth.normal((dm.B, dm.S, dm.Hkv, dm.D), 1.0, 99, "bench.kb", dev)
    vb = synth.normal((dm.B, dm.S, dm.Hkv, dm.D), 1.0, 99, "bench.vb", dev)
    o = torch.empty_like(q)
    aws = td.workspace(dims, td.TD_FN_BLOCK_ATTENTION, dev)
    for _ in range(3):
        td.td_block_attention(dims, q, kb, vb, lay["k_ctx"], lay["v_ctx"], o=o, ws=aws)
    # back-to-back launches for about half a second, so that the clock sampler (50 ms period)
    # sees the segment; the context K/V (537 MB) is larger than L2
    a_reps = 3000
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(local) as aclocks:
        a0.record(stream)
        for _ in range(a_reps):
            td.td_block_attention(dims, q, kb, vb, lay["k_ctx"], lay["v_ctx"], o=o, ws=aws)
        a1.record(stream)
        torch.cuda.synchronize()
    attn_ms = a0.elapsed_time(a1) / a_reps
    # the same launches with the probabilities carried as hi + lo bf16 pairs (a second P V
    # product per key tile): the cost of the more exact arithmetic
    s_reps = 1000
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        td.td_block_attention(dims, q, kb, vb, lay["k_ctx"], lay["v_ctx"], o=o, ws=aws,
                              precision=td.TD_ATTN_P_SPLIT)
    torch.cuda.synchronize()
    with ClockSampler(local) as sclocks:
        b0.record(stream)
        for _ in range(s_reps):
            td.td_block_attention(dims, q, kb, vb, lay["k_ctx"], lay["v_ctx"], o=o, ws=aws,
                                  precision=td.TD_ATTN_P_SPLIT)
        b1.record(stream)
        torch.cuda.synchronize()
    split_ms = b0.elapsed_time(b1) / s_reps
    kv_bytes = 2 * dm.B * dm.Hkv * dm.Lmax * dm.D * 2
    attn_bytes = kv_bytes + (q.numel() + o.numel() + kb.numel() + vb.numel()) * 2
    attn_gbs = attn_bytes / (attn_ms / 1e3) / 1e9

    h = synth.normal((M, dm.d), 1.0, 99, "bench.h", dev)
    lws = td.workspace(dims, td.TD_FN_LMHEAD_COMMIT, dev)
    tk = torch.empty_like(tokens)
    mk = torch.empty_like(masked)
    for _ in range(3):
        tk.fill_(dm.V); mk.fill_(1)
        td.td_lmhead_commit(dims, h, wl.w_lm, wl.gamma, False, tk, mk, *outs, ws=lws)
    l_reps = 700
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(local) as lclocks:
        l0.record(stream)
        for _ in range(l_reps):
            td.td_lmhead_commit(dims, h, wl.w_lm, wl.gamma, False, tk, mk, *outs, ws=lws)
        l1.record(stream)
        torch.cuda.synchronize()
    lm_ms = l0.elapsed_time(l1) / l_reps
    lm_flops = 2.0 * M * dm.d * dm.V
    lm_tflops = lm_flops / (lm_ms / 1e3) / 1e12
    step_ms = ms / max(1, total_steps)
    attn_share = dm.n_layers * attn_ms / step_ms
    lm_share = lm_ms / step_ms
    attn_kernel = "attn_pair_kernel"   # head_dim 128 with two or more 128-row chunks per unit
    attn_traffic = traffic_per_launch(
        attn_kernel, ["td_ptx.cuh", "td_attention.cuh", "td_attention_pair.cuh"],
        dm.B * dm.Hkv * dm.Lmax)
    lm_kernel = "gemm_pair_kernel<7,EPI_LMHEAD>"   # 256 x 256 tiles on SM pairs (M > 128)
    lm_traffic = traffic_per_launch(lm_kernel, ["td_ptx.cuh", "td_gemm.cuh"], M)
    roof_attn = {"kernel": attn_kernel, "bound": "hbm",
                 "achieved": round(attn_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                 "frac": round(attn_gbs / pk["hbm_gbs"], 4), "traffic": attn_traffic,
                 "algorithmic_bytes_per_launch": attn_bytes, "ms_per_launch": round(attn_ms, 4),
                 "share_of_step": round(attn_share, 3), "peak_source": pk_kind,
                 "clocks": aclocks.summary(attn_ms * a_reps)}
    roof_lm = {"kernel": lm_kernel + " + merge_commit", "bound": "tensor",
               "achieved": round(lm_tflops, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
               "frac": round(lm_tflops / pk["bf16_tflops"], 4), "traffic": lm_traffic,
               "algorithmic_flops_per_launch": lm_flops, "ms_per_launch": round(lm_ms, 4),
               "share_of_step": round(lm_share, 3), "peak_source": pk_kind,
               "clocks": lclocks.summary(lm_ms * l_reps)}
    dominant, other = (roof_attn, roof_lm) if attn_share >= lm_share else (roof_lm, roof_attn)

    # embed, LM row map, 6 x (adaLN, QKV, attention, O-proj), LM head, commit per step; with
    # the loop graph's conditional nodes only the steps that ran launch anything, with the
    # flat graph every step of T launches (those after the block finished return at once)
    launches_per_step = 2 + dm.n_layers * 4 + 2
    graph_form = td.td_decode_graph_form()
    steps_launched = total_steps if graph_form == td.TD_GRAPH_CONDITIONAL else wl.T * args.steps
    result = {
        "metric": "committed tokens/sec (block decode, S=16, gamma=0.8)",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights and context KV of the stated shapes)",
        "config": dict(WORKLOAD, w_lm_sigma=synth.DECODE_W_LM_SIGMA,
                       parallelism=f"replicas x{world}",
                       l2="inputs larger than L2 (3.2 GB of context KV + 1 GB LM head per step)"),
        "denoised_tokens_per_s": round(denoised, 1),
        "denoise_steps_per_block": round(total_steps / args.steps, 3),
        "commits_per_step": hist,
        "fallback_only": fallback,
        "attention_before_decode": {"ms_per_launch": round(cool_ms, 4),
                                    "GB/s": round(attn_bytes / (cool_ms / 1e3) / 1e9, 1),
                                    "frac": round(attn_bytes / (cool_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4),
                                    "clocks": cclocks.summary(cool_ms * c_reps)},
        "attention_split_p": {"ms_per_launch": round(split_ms, 4),
                              "GB/s": round(attn_bytes / (split_ms / 1e3) / 1e9, 1),
                              "frac": round(attn_bytes / (split_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4),
                              "clocks": sclocks.summary(split_ms * s_reps)},
        "commit_sweep": sweep,
        "gpu_launches": launches_per_step * steps_launched,
        "loop_graph": "conditional" if graph_form == td.TD_GRAPH_CONDITIONAL else "flat",
        "clocks": clocks.summary(ms),
        "roofline": dominant,
        "roofline_other": other,
        "e2e": {"value": round(e2e, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": tok_h.numel() * 4 + msk_h.numel(),
                "d2h_bytes_per_step": tok_out.numel() * 4},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, threads, desc, _ = oracle_sample(wl, args.cpu_budget, 64)
        ncpu, _ = host_cores()
        result["cpu_baseline"] = {"value": round(v, 3), "unit": "tokens/s", "cores": threads,
                                  "host_logical_cores": ncpu, "oracle_threads": threads,
                                  "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_only(args):
    """One kernel family on one workload, `reps` launches, no timing: the command that the
    profiler captures (attention: B sequences, context L; lmhead: M rows)."""
    import block_diffusion_lm_denoise_b300 as td
    from block_diffusion_lm_denoise_b300 import synth
    dev = torch.device("cuda", 0)
    if args.only == "attention":
        wl = synth.attention_sweep(args.L, dev, B=args.B)
        lay = wl.layers[0]
        dims = wl.dims.as_dict()
        ws = td.workspace(dims, td.TD_FN_BLOCK_ATTENTION, dev)
        o = torch.empty_like(lay["q"])
        for _ in range(args.reps):
            td.td_block_attention(dims, lay["q"], lay["k_blk"], lay["v_blk"], lay["k_ctx"],
                                  lay["v_ctx"], o=o, ws=ws)
    elif args.only == "step":
        # one denoise step of one layer at the decode-loop widths (d 4096, 32/2 heads, V
        # 131072) with B sequences of context L: every kernel of a step, small on the device
        from block_diffusion_lm_denoise_b300.synth import Dims, _layer, normal, phi_table
        import math
        dm = Dims(B=args.B, S=16, d=4096, Hq=32, Hkv=2, D=128, V=131072, Lmax=args.L,
                  n_layers=1)
        layers = [_layer(7, 0, dm, 1 / math.sqrt(dm.d), 1 / math.sqrt(dm.Hq * dm.D), 1.0, dev)]
        w_lm = normal((dm.V, dm.d), 0.02, 7, "w_lm", dev)
        emb = normal((dm.V + 1, dm.d), 1.0, 7, "emb", dev)
        pos = normal((dm.S, dm.d), 1.0, 7, "pos", dev)
        phi = phi_table(16, dm.d, 7, dev)
        ws = td.workspace(dm.as_dict(), td.TD_FN_DENOISE_STEP, dev)
        for _ in range(args.reps):
            tokens = torch.full((dm.B, dm.S), dm.V, dtype=torch.int32, device=dev)
            masked = torch.ones((dm.B, dm.S), dtype=torch.uint8, device=dev)
            td.td_denoise_step(dm.as_dict(), layers, w_lm, phi[0], 1, 16, 0.8, tokens, masked,
                               emb=emb, pos=pos, ws=ws)
    else:
        wl = synth.lmhead_sweep(args.M, 16, 0.8, dev)
        dims = wl.dims.as_dict()
        ws = td.workspace(dims, td.TD_FN_LMHEAD_COMMIT, dev)
        for _ in range(args.reps):
            wl.tokens.fill_(wl.dims.V)
            wl.masked.fill_(1)
            td.td_lmhead_commit(dims, wl.h, wl.w_lm, 0.8, False, wl.tokens, wl.masked, ws=ws)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    print(json.dumps({"only": args.only, "reps": args.reps, "ok": True}))


def run_sweep(args):
    """Isolated kernel timings over the attention and LM-head workloads: attention with B = 32
    sequences at context L in {512, 2048, 8192, 32768}; LM head + commit at M = B*S rows in
    {16, 256, 1024, 4096} (S = 16, gamma 0.8, all rows masked). Before every timed launch a
    512 MiB buffer is written and then another 256 MiB read, so no input is served from L2
    and no write-back of the flush competes with the launch; each launch is timed with its
    own pair of CUDA events on the launching stream, all launches queued behind a device-side
    spin so that the host is ahead of the device."""
    import block_diffusion_lm_denoise_b300 as td
    from block_diffusion_lm_denoise_b300 import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    pk, pk_kind = peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    clean = torch.ones(256 << 20 >> 3, dtype=torch.int64, device=dev)
    reps = max(args.reps, 10)
    spin = getattr(torch.cuda, "_sleep", None)

    def timed(launch, prep=lambda: None):
        """Mean device time of `launch`; `prep` (state resets) runs outside the events."""
        for _ in range(3):
            prep()
            launch()
        torch.cuda.synchronize()
        # a ~20 ms device-side spin first, so that every launch below is queued before the
        # device reaches it and no event pair includes host-side launch latency
        if spin is not None:
            spin(40_000_000)
        evs = []
        for _ in range(reps):
            flush.fill_(1)
            clean.sum()   # reads 256 MiB: the dirty lines of the write leave L2 before the launch
            prep()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        assert td.td_device_error() == 0
        return sum(a.elapsed_time(b) for a, b in evs) / reps

    for L in (512, 2048, 8192, 32768):
        wl = synth.attention_sweep(L, dev, B=32)
        lay, dims = wl.layers[0], wl.dims.as_dict()
        ws = td.workspace(dims, td.TD_FN_BLOCK_ATTENTION, dev)
        o = torch.empty_like(lay["q"])
        ms = timed(lambda: td.td_block_attention(dims, lay["q"], lay["k_blk"], lay["v_blk"],
                                                 lay["k_ctx"], lay["v_ctx"], o=o, ws=ws))
        dm = wl.dims
        nbytes = 2 * dm.B * dm.Hkv * dm.Lmax * dm.D * 2 + (
            lay["q"].numel() + o.numel() + lay["k_blk"].numel() + lay["v_blk"].numel()) * 2
        gbs = nbytes / (ms / 1e3) / 1e9
        flops = 4.0 * dm.B * dm.Hq * dm.S * (dm.Lmax + dm.S) * dm.D
        print(json.dumps({"sweep": "attention", "B": dm.B, "L": L, "ms": round(ms, 4),
                          "algorithmic_bytes": nbytes, "GB/s": round(gbs, 1),
                          "hbm_frac": round(gbs / pk["hbm_gbs"], 4),
                          "TFLOP/s": round(flops / (ms / 1e3) / 1e12, 1),
                          "peak_source": pk_kind}), flush=True)
        del wl, lay, ws, o
        torch.cuda.empty_cache()

    for M in (16, 256, 1024, 4096):
        wl = synth.lmhead_sweep(M, 16, 0.8, dev)
        dims = wl.dims.as_dict()
        ws = td.workspace(dims, td.TD_FN_LMHEAD_COMMIT, dev)
        dm = wl.dims

        def reset():
            wl.tokens.fill_(dm.V)
            wl.masked.fill_(1)

        ms = timed(lambda: td.td_lmhead_commit(dims, wl.h, wl.w_lm, 0.8, False, wl.tokens,
                                               wl.masked, ws=ws), reset)
        flops = 2.0 * M * dm.d * dm.V
        nbytes = (dm.V * dm.d + M * dm.d) * 2
        tf = flops / (ms / 1e3) / 1e12
        gbs = nbytes / (ms / 1e3) / 1e9
        print(json.dumps({"sweep": "lmhead_commit", "M": M, "S": 16, "ms": round(ms, 4),
                          "TFLOP/s": round(tf, 1), "tensor_frac": round(tf / pk["bf16_tflops"], 4),
                          "GB/s": round(gbs, 1), "hbm_frac": round(gbs / pk["hbm_gbs"], 4),
                          "peak_source": pk_kind}), flush=True)
        del wl, ws
        torch.cuda.empty_cache()


def run_reference(args, world, rank):
    """The fp64 oracle on the host cores, same workload, metric and unit; rank 0 only.
    Each bench step is one oracle denoise step of one sequence's block (bounded sample)."""
    if rank != 0:
        return
    from block_diffusion_lm_denoise_b300 import synth
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    wl = synth.decode_loop(dev, seed=4, w_lm_sigma=synth.DECODE_W_LM_SIGMA)
    smp = OracleSampler(wl)
    for _ in range(args.warmup):
        smp.step()
    committed = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        committed += smp.step()
    el = time.perf_counter() - t0
    value = committed / el
    result = {
        "impl": "reference",
        "metric": "committed tokens/sec (block decode, S=16, gamma=0.8)",
        "value": round(value, 4),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": dict(WORKLOAD, w_lm_sigma=synth.DECODE_W_LM_SIGMA, parallelism="host cores"),
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s",
                         "cores": torch.get_num_threads(),
                         "host_logical_cores": os.cpu_count(),
                         "oracle_threads": torch.get_num_threads(), "kind": "oracle",
                         "sample": smp.describe(args.steps)},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
