#!/usr/bin/env python
"""Throughput benchmark of the GDN segmented forward (one JSON line on rank 0).

A step is one whole gdn_segmented_fwd call -- segment summaries, exclusive scan, and every
segment's chunked forward -- over one batch of the headline workload (B=2, H=32,
T=32768, K=V=128, 4 segments, bf16 inputs, fp32 state and output), inputs already
resident in HBM. Inputs (~0.8 GB) and output (1 GB) are larger than the 129 MB L2, so no
flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the method's plain definition) on the host
cores, a bounded sample of the same workload per step.
Under torchrun (N > 1) every rank runs its own batch (weak scaling; no data-path
collective); timing is max over ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN segmented fwd tokens/s at H32 K=V=128 T=32K bf16; % of roofline"
def varlen_metric(w) -> str:
    """The packed-sequence line's metric: tokens/s of the forward over these lengths and shapes."""
    return (f"GDN packed-sequence fwd tokens/s (lengths {','.join(str(n) for n in w.seq_lens)}) "
            f"at H{w.H} K={w.K} V={w.V} {w.in_dtype}").replace("K=128 V=128", "K=V=128")
KDA_METRIC = "GDN per-channel-gate (KDA) fwd tokens/s at H16 K=V=128 T=8K bf16"
STATE_GRAD_METRIC = ("GDN backward state-gradient path tokens/s (segment summaries M, dS_local, "
                     "reverse M^T scan) at H32 K=V=128 T=32K bf16")
BACKWARD_METRIC = ("GDN backward tokens/s (dq, dk, dv, dg, dbeta, dh0 from dO and dht) at H32 "
                   "K=V=128 T=32K bf16")
# fp32 CUDA-core peak: 152 SMs x 128 fp32 lanes x 2 flops (FMA) x 2.07 GHz maximum SM clock
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
# dense tf32 against dense bf16 on the tensor cores, nominal (1.1 and 2.25 PFLOP/s per GPU): a
# tf32 contraction's peak is the measured bf16 rate times this
TF32_PER_BF16 = 1.1 / 2.25


def metric_of(w) -> str:
    return KDA_METRIC if w.gate_k else METRIC
DEFAULT_WORKLOAD = "cp4_b2_h32_t32k"
L2_BYTES = 129 * 1024 * 1024
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------------------
# distributed plumbing (host logic; tested on CPU with gloo)
# ---------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(backend: str):
    import torch.distributed as dist
    world, rank, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return world, rank


def reduce_max(x: float, device="cpu") -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and str(device).startswith("cuda"):
            dist.barrier(device_ids=[int(str(device).split(":")[1])])
        else:
            dist.barrier()


def aggregate(tokens_per_rank_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: tokens all ranks processed / the slowest rank's time."""
    return tokens_per_rank_step * steps * world / max_seconds


def rank_seed_offset(rank: int) -> int:
    return 0x1000 * rank


# ---------------------------------------------------------------------------------------
# algorithmic model of the path (bytes and flops per launch)
# ---------------------------------------------------------------------------------------
def algorithmic(w, plan=None, out_bytes: int = 4):
    """Compulsory HBM bytes and dense-contraction flops of each stage for workload w under the
    piece plan `plan` = (P, chunks of piece 0, chunks of each later piece) that the library
    reports (default: one equal piece per segment), and of the method itself (the pages' flow:
    summaries of the nseg-1 segments that feed a later one, the scan, the forward).

    Intermediates (the WY factors, per-chunk states) count as zero: the method keeps them on
    chip. The "wy" stage's bytes are this implementation's extra traffic, reported beside the
    stages but not in the executed total."""
    nch = w.T // 64
    if plan is None:
        plan = (w.nseg, nch // w.nseg, nch // w.nseg)
    P, first, rest = plan
    isz = 2 if w.in_dtype == "bf16" else 4
    BH = w.B * w.H
    tok_heads = w.B * w.T * w.H
    chunks = tok_heads // 64
    K, V = w.K, w.V
    kv_state = BH * K * V * 4
    kk_state = BH * K * K * 4
    tc = w.in_dtype == "bf16" and K == 128 and V == 128 and not w.gate_k
    g_tok = (K if w.gate_k else 1) * isz                       # one gate, or one per channel
    fwd_tok = (2 * K + V) * isz + g_tok + isz + V * out_bytes  # q, k, v, g, beta in; o out
    sum_tok = (K + V) * isz + g_tok + isz                      # k, v, g, beta in
    # prep (K K^T, U, W) + state (W H, Kd^T R) + output (Q K^T, Qd H, C R), per chunk
    fwd_flops = (2 * 64 * 64 * K + 2 * 64 * 64 * V + 2 * 64 * 64 * K + 2 * 64 * K * V * 2
                 + 2 * 64 * 64 * K + 2 * 64 * K * V + 2 * 64 * 64 * V)
    # prep (K K^T, U, W) + augmented K x (K+V) state update, per chunk
    sum_flops = (2 * 64 * 64 * K + 2 * 64 * 64 * V + 2 * 64 * 64 * K + 2 * 2 * 64 * K * (K + V))
    ps = max(P - 2, 0)                  # pieces with a summary (1 .. P-2)
    th_first = BH * first * 64          # token-heads of piece 0
    th_rest = BH * rest * 64            # token-heads of each later piece
    stages = {
        # per-chunk WY factors (tensor-core path only): reads k, g, beta; writes the two bf16
        # 64 x 64 factors without their zero blocks above the diagonal, 10 KiB per chunk. An
        # intermediate of this implementation, not of the method, so it is left out of the
        # executed total below.
        "wy": {
            "bytes": (tok_heads * (K * isz + 2 * isz) + chunks * 10240) if tc else 0,
            "flops": chunks * (2 * 64 * 64 * K + 2 * 64 * 64 * 64) if tc else 0,
        },
        # piece 0's forward from h0 (handing its final state on) and the summaries of pieces
        # 1..P-2
        "phase1": {
            "bytes": th_first * fwd_tok + (2 if P > 1 else 1) * kv_state
            + th_rest * ps * sum_tok + ps * (kk_state + kv_state),
            "flops": th_first // 64 * fwd_flops + th_rest * ps // 64 * sum_flops,
        },
        # reads the summaries and the state piece 0 ends in; writes the state entering every
        # later piece and every segment
        "scan": {
            "bytes": (ps * (kk_state + kv_state) + kv_state + ps * kv_state + w.nseg * kv_state
                      if P > 1 else w.nseg * kv_state),
            "flops": ps * BH * 2 * K * K * V,
        },
        # the forward of pieces 1..P-1 from their scanned states
        "phase2": {
            "bytes": (th_rest * (P - 1) * fwd_tok + P * kv_state) if P > 1 else 0,
            "flops": th_rest * (P - 1) // 64 * fwd_flops,
        },
    }
    executed = {"bytes": sum(stages[k]["bytes"] for k in ("phase1", "scan", "phase2")),
                "flops": sum(stages[k]["flops"] for k in ("phase1", "scan", "phase2"))}
    nseg = w.nseg
    method = {
        "bytes": tok_heads * (nseg - 1) // nseg * sum_tok + (nseg - 1) * (kk_state + kv_state)
        + (nseg - 1) * (kk_state + kv_state) + nseg * kv_state + kv_state
        + tok_heads * fwd_tok + nseg * kv_state + kv_state,
        "flops": chunks * (nseg - 1) // nseg * sum_flops + (nseg - 1) * BH * 2 * K * K * V
        + chunks * fwd_flops,
    }
    return stages, executed, method


def literal_algorithmic(w, out_bytes: int = 4):
    """The pages' literal flow as three public calls: every segment's summary (all nseg, as
    every rank forms its own), the scan, every segment's forward from its H_in. Returns the
    per-call bytes/flops (intermediates count as zero; "wy" is this implementation's extra
    traffic, formed once per call that needs it) and the total."""
    isz = 2 if w.in_dtype == "bf16" else 4
    BH = w.B * w.H
    tok_heads = w.B * w.T * w.H
    chunks = tok_heads // 64
    K, V = w.K, w.V
    kv_state = BH * K * V * 4
    kk_state = BH * K * K * 4
    g_tok = (K if w.gate_k else 1) * isz
    fwd_tok = (2 * K + V) * isz + g_tok + isz + V * out_bytes
    sum_tok = (K + V) * isz + g_tok + isz
    fwd_flops = (2 * 64 * 64 * K + 2 * 64 * 64 * V + 2 * 64 * 64 * K + 2 * 64 * K * V * 2
                 + 2 * 64 * 64 * K + 2 * 64 * K * V + 2 * 64 * 64 * V)
    sum_flops = (2 * 64 * 64 * K + 2 * 64 * 64 * V + 2 * 64 * 64 * K + 2 * 2 * 64 * K * (K + V))
    nseg = w.nseg
    calls = {
        "summary": {"bytes": tok_heads * sum_tok + nseg * (kk_state + kv_state),
                    "flops": chunks * sum_flops},
        "scan": {"bytes": (nseg - 1) * (kk_state + kv_state) + kv_state + nseg * kv_state,
                 "flops": (nseg - 1) * BH * 2 * K * K * V},
        "forward": {"bytes": tok_heads * fwd_tok + nseg * kv_state + kv_state,
                    "flops": chunks * fwd_flops},
    }
    total = {"bytes": sum(c["bytes"] for c in calls.values()),
             "flops": sum(c["flops"] for c in calls.values())}
    return calls, total


def wy_tail_beside(w, plan, sms):
    """The library's rule: the last piece's WY tiles are formed beside the first phase when
    that phase leaves at least 8 SMs idle in its last wave (its only one, if it fits one) and
    those tiles take at least one wave of WY CTAs (six per SM)."""
    P, first, rest = plan
    tc = w.in_dtype == "bf16" and w.K == 128 and w.V == 128 and not w.gate_k
    if not tc or P < 2 or w.T == 0 or not sms:
        return False
    bh = w.B * w.H
    last_lo = first + (P - 2) * rest
    chains1 = bh * (P - 1)
    idle1 = sms - chains1 % sms if chains1 % sms else 0
    return idle1 >= 8 and bh * (w.T // 64 - last_lo) >= 6 * sms


def launches_per_step(w, pieces=None, plan=None, sms=None):
    """Kernels one gdn_segmented_fwd call launches: WY factors (tensor-core path) or the
    per-channel-gate pre-pass, piece 0's forward, the piece summaries (3 pieces or more), the
    scan and the second forward (2 pieces or more). When the last piece's WY tiles are formed beside the first phase, that phase is
    one grid (forward and summaries) followed by the WY grid for the last piece."""
    P = pieces or w.nseg
    tc = int(w.in_dtype == "bf16" and w.K == 128 and w.V == 128 and not w.gate_k)
    # per-channel gates at bf16 inputs: the per-chunk factors' pre-pass, as the WY launch
    prep = int(w.in_dtype == "bf16" and bool(w.gate_k))
    n = tc + prep + 1 + (1 if P >= 3 else 0) + (2 if P >= 2 else 0)
    if plan is not None and wy_tail_beside(w, plan, sms):
        n += 0 if P >= 3 else 1
    return n


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# The translation units each recorded kernel is built from (and the headers they include):
# a traffic record stays valid exactly as long as these files are unchanged.
KERNEL_SOURCES = {
    "gdn_forward": ("gdn_tc.cu", "gdn_tc_common.cuh", "gdn_internal.h"),
    "gdn_varlen_forward": ("gdn_tc.cu", "gdn_tc_common.cuh", "gdn_internal.h", "gdn_varlen.cu"),
    "gdn_wy": ("gdn_wy.cu", "gdn_tc_common.cuh", "gdn_internal.h"),
    "state_grad_kernel": ("gdn_bwd.cu", "gdn_internal.h"),
    "chunk_grad_kernel": ("gdn_bwd_chunk.cu", "gdn_internal.h"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources the named kernel is built from (plus the public header)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "context_scan_gb300", "csrc")
    for fn in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, fn), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "gdn.h"), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on the sources the
    kernel is built from now."""
    p = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.txt")
    if not os.path.exists(p) or kernel not in KERNEL_SOURCES:
        return None
    kv = {}
    for line in open(p):
        if ":" in line:
            a, b = line.split(":", 1)
            kv[a.strip()] = b.strip()
    if kv.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open(os.devnull, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            text, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            text, _ = self.proc.communicate()
        rows = list(csv.reader(io.StringIO(text)))
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------
def varlen_algorithmic(w, out_bytes: int = 4):
    """Compulsory HBM bytes and dense-contraction flops of the packed-sequence forward: the WY
    factors (an intermediate of this implementation) and the chunked forward of every sequence
    (its partial last chunk counted as a whole chunk of work, its bytes by tokens)."""
    isz = 2 if w.in_dtype == "bf16" else 4
    K, V, H = w.K, w.V, w.H
    tok_heads = w.T * H
    chunks = H * sum((n + 63) // 64 for n in w.seq_lens)
    states = len(w.seq_lens) * H * K * V * 4
    fwd_tok = (2 * K + V) * isz + 2 * isz + V * out_bytes
    fwd_flops = (2 * 64 * 64 * K + 2 * 64 * 64 * V + 2 * 64 * 64 * K + 2 * 64 * K * V * 2
                 + 2 * 64 * 64 * K + 2 * 64 * K * V + 2 * 64 * 64 * V)
    return {
        "wy": {"bytes": tok_heads * (K * isz + 2 * isz) + chunks * 10240,
               "flops": chunks * (2 * 64 * 64 * K + 2 * 64 * 64 * 64)},
        "forward": {"bytes": tok_heads * fwd_tok + 2 * states, "flops": chunks * fwd_flops},
    }


def pipelined_e2e(torch, host, d, outs, call, n_steps, dev, stream):
    """Seconds for n_steps end-to-end steps through the public API. Every step copies its inputs
    from pinned host memory (`host`, by name; None entries are skipped) into device buffers,
    issues one library call on `stream` (`call(inputs, outputs)`) and reads every output back
    into pinned host memory. Steps are pipelined as a serving loop would run them: two sets of
    device buffers (`d` and `outs` are the first), the host->device copies on one stream, the
    calls on `stream`, the device->host copies on a third, so that one step's copies overlap its
    neighbours' compute and the two copy directions overlap each other (more copy streams per
    direction measured no faster: the host link is the limit)."""
    outs_host = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    dbuf = [d, {n: (None if t is None else torch.empty_like(t)) for n, t in d.items()}]
    obuf = [tuple(outs), tuple(torch.empty_like(t) for t in outs)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]   # inputs of the buffer's step copied in
    used = [torch.cuda.Event() for _ in range(2)]       # the buffer's step computed
    out_read = [torch.cuda.Event() for _ in range(2)]   # its outputs copied out

    def run(n):
        for i in range(n):
            j = i % 2
            di, oi = dbuf[j], obuf[j]
            with torch.cuda.stream(s_in):
                s_in.wait_event(used[j])        # step i-2 no longer reads these inputs
                for nm, t in host.items():
                    if t is not None:
                        di[nm].copy_(t, non_blocking=True)
                in_ready[j].record(s_in)
            stream.wait_event(in_ready[j])
            stream.wait_event(out_read[j])      # step i-2's outputs are out of these buffers
            call(di, oi)
            used[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(used[j])
                for th, td in zip(outs_host, oi):
                    th.copy_(td, non_blocking=True)
                out_read[j].record(s_out)

    run(2)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    s_in.wait_event(a)
    run(n_steps)
    stream.wait_event(out_read[(n_steps - 1) % 2])
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3


def run_varlen(args):
    """The packed-sequence forward (gdn_varlen_fwd) on a seq_lens workload; one step is one call
    over the whole packed batch. Its inputs fit in L2, so a buffer larger than L2 is written
    between timed steps and each step is timed by its own events."""
    import torch

    from context_scan_gb300 import gdn, synth

    world, rank = init_dist("nccl" if args.gpus > 1 else "gloo")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    w0 = synth.WORKLOADS[args.workload]
    w = synth.scaled(w0, seed=w0.seed + rank_seed_offset(rank))
    x = synth.make_inputs(w)
    dt = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
    names = ("q", "k", "v", "g", "beta")
    host = {n: torch.from_numpy(x[n]).to(dt).pin_memory() for n in names}
    host["h0"] = None if x["h0"] is None else torch.from_numpy(x["h0"]).pin_memory()
    d = {n: (None if t is None else t.to(dev)) for n, t in host.items()}
    cu = torch.from_numpy(synth.cu_seqlens(w)).to(dev)
    nseq = len(w.seq_lens)
    o = torch.empty((1, w.T, w.H, w.V), dtype=torch.float32, device=dev)
    hf = torch.empty((nseq, w.H, w.K, w.V), dtype=torch.float32, device=dev)
    prob = gdn.problem(d["k"], d["v"], o, g=d["g"])
    ws = gdn.alloc_varlen_workspace(prob, nseq, device=dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def step(events=None):
        if events is None:
            gdn.gdn_varlen_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, hf, cu, ws,
                               prob=prob, stream=stream)
        else:
            gdn.gdn_varlen_fwd_timed(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, hf,
                                     cu, ws, events, prob=prob, stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    st, detail = gdn.gdn_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {st} detail {detail} during warm-up")
    K = args.steps
    # stage times from a pass of the timed entry point (its events sit between the launches);
    # the timed region runs the plain call, each step between two events of its own
    Ks = min(K, 100)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(Ks)]
    for e5 in ev:
        for e in e5:
            e.record(stream)
    for i in range(Ks):
        flush.fill_(1.0)
        step(ev[i])
    torch.cuda.synchronize()
    pe = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    sampler = ClockSampler(local) if rank == 0 else None
    barrier(dev)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for i in range(K):
        flush.fill_(1.0)   # outside the step's own events
        pe[i][0].record(stream)
        step()
        pe[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    st, detail = gdn.gdn_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {st} detail {detail} in the timed region")
    # stages: the length check, the plan and the WY factors; the first phase (piece 0 of every
    # sequence beside the middle pieces' summaries, or the whole forward when none is cut); the
    # scan; the second phase
    names = ("wy", "phase1", "scan", "phase2")
    avg = {n: sum(e[i].elapsed_time(e[i + 1]) for e in ev) / Ks for i, n in enumerate(names)}
    avg["forward"] = avg["phase1"] + avg["scan"] + avg["phase2"]   # the chains, both phases
    step_s = sum(a.elapsed_time(b) for a, b in pe) / 1e3
    max_s = reduce_max(step_s, device=dev if world > 1 else "cpu")
    barrier(dev)
    stages = varlen_algorithmic(w)
    sms = min(torch.cuda.get_device_properties(dev).multi_processor_count, 256)
    cut_possible = nseq * w.H <= sms and w.T >= 2 * 8 * 64   # gdn_varlen.cu: pieces_possible
    # the length check (with the plan), the WY tiles, the first phase's forwards, the piece
    # summaries, the scan and the second phase; without a possible cut: check, WY, forward
    launches = 6 if (cut_possible and w.in_dtype == "bf16" and w.K == 128 and not w.gate_k) else 3
    peaks, peaks_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    ach = stages["forward"]["bytes"] / (avg["forward"] * 1e-3) / 1e9
    t_roof = max(stages["forward"]["bytes"] / (hbm * 1e9),
                 stages["forward"]["flops"] / (float(peaks["bf16_tflops"]) * 1e12))
    ms_per_step = max_s / K * 1e3
    value = aggregate(w.T, K, world, max_s)

    e2e = None
    if not args.no_e2e:
        n_e2e = max(3, min(K, args.e2e_steps))
        h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
        d2h = o.numel() * o.element_size() + hf.numel() * hf.element_size()

        def call(di, oi):
            gdn.gdn_varlen_fwd(di["q"], di["k"], di["v"], di["g"], di["beta"], di["h0"], oi[0],
                               oi[1], cu, ws, prob=prob, stream=stream)

        e_el = pipelined_e2e(torch, host, d, (o, hf), call, n_e2e, dev, stream)
        e_el = reduce_max(e_el, device=dev if world > 1 else "cpu")
        st, detail = gdn.gdn_check_device_error(ws)
        if st != 0:
            raise RuntimeError(f"device error word {st} detail {detail} in the end-to-end run")
        e2e = {"value": round(aggregate(w.T, n_e2e, world, e_el), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "pipelined": "two buffer sets; copies in and out on their own streams"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_varlen(w, x, budget_s=args.cpu_seconds)
    if rank == 0:
        line = {
            "metric": varlen_metric(w), "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w0.name, "seq_lens": list(w.seq_lens), "B": 1, "H": w.H,
                       "T": w.T, "K": w.K, "V": w.V, "chunk": 64, "in_dtype": w.in_dtype,
                       "out_dtype": "f32", "state_dtype": "f32",
                       "l2": "a 258 MB buffer is written before every step, outside the step's "
                             "events (the inputs fit in L2 at the pages' lengths)",
                       "parallelism": f"weak: {world} rank(s) x one batch each"},
            "roofline": {"bound": "hbm", "achieved": round(ach, 2), "peak": hbm, "unit": "GB/s",
                         "frac": round(ach / hbm, 4),
                         "traffic": recorded_traffic("gdn_varlen_forward", w0.name),
                         "kernel": "gdn_varlen_forward", "kernel_ms": round(avg["forward"], 4),
                         "algorithmic_bytes": stages["forward"]["bytes"],
                         "peak_source": f"{peaks_src} hbm_gbs"},
            "path_roofline": {"t_roof_us": round(t_roof * 1e6, 1),
                              "frac": round(t_roof / (ms_per_step * 1e-3), 4),
                              "bytes": stages["forward"]["bytes"],
                              "flops": stages["forward"]["flops"],
                              "peaks": f"{peaks_src}: hbm {hbm} GB/s, bf16 {peaks['bf16_tflops']} TF/s"},
            "stage_ms": {k: round(v, 4) for k, v in avg.items()},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches * K,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    import torch.distributed as dist
    if dist.is_initialized():
        dist.destroy_process_group()


def state_grad_algorithmic(w):
    """Per launch of the state-gradient kernel over workload w: compulsory HBM bytes (read q, k,
    g, beta in the input dtype and dO in fp32 once; write dS) and fp32 flops per chunk and head
    counted once, every product as a dense tile (the triangular C^T dO and A^T dR alike): K K^T
    and Q K^T (2 * 64*64*K*2), the 64 x 64 inverse (~0.17 M), dR = Kd D + C^T dO (64*K*V*2 +
    64*64*V*2), A^T dR (64*64*V*2), D update (2 * K*64*V*2)."""
    isz = 2 if w.in_dtype == "bf16" else 4
    th = w.B * w.T * w.H
    nbytes = th * (2 * w.K * isz + 2 * isz + w.V * 4) + w.nseg * w.B * w.H * w.K * w.V * 4
    c = 64
    per_chunk = (2 * c * c * w.K * 2 + 0.17e6 + c * w.K * w.V * 2 + c * c * w.V * 2 +
                 c * c * w.V * 2 + 2 * w.K * c * w.V * 2)
    return {"bytes": nbytes, "flops": per_chunk * th / c}


def run_state_grad(args):
    """The backward's state-gradient path ("RFC: HyperParallel Linear Attention Context
    Parallel", section 6.4.3) on the headline workload: one step is the segment summaries M
    (gdn_segment_summary), the per-segment state gradients dS (gdn_state_grad_summary) and the
    reverse scan to dH_in (gdn_state_grad_scan), each bracketed by events on the stream."""
    import numpy as np
    import torch

    import oracle
    from context_scan_gb300 import gdn, synth

    world, rank = init_dist("nccl" if args.gpus > 1 else "gloo")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    w0 = synth.WORKLOADS[args.workload]
    if w0.gate_k or w0.seq_lens is not None:
        raise SystemExit("--path state_grad runs fixed-length scalar-gate workloads only")
    w = synth.scaled(w0, seed=w0.seed + rank_seed_offset(rank))
    if args.T:
        w = synth.scaled(w, T=args.T)
    x = synth.make_inputs(w)
    gr = synth.make_grads(w, dht_sd=0.1)
    dt = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
    d = {n: torch.from_numpy(x[n]).to(dev).to(dt) for n in ("q", "k", "v", "g", "beta")}
    dO = torch.from_numpy(gr["dO"]).to(dev)
    dht = torch.from_numpy(gr["dht"]).to(dev)
    B, H, K, V, nseg = w.B, w.H, w.K, w.V, w.nseg
    M = torch.empty((nseg, B, H, K, K), dtype=torch.float32, device=dev)
    S = torch.empty((nseg, B, H, K, V), dtype=torch.float32, device=dev)
    dS = torch.empty((nseg, B, H, K, V), dtype=torch.float32, device=dev)
    dH_in = torch.empty((nseg, B, H, K, V), dtype=torch.float32, device=dev)
    prob = gdn.problem(d["k"], d["v"])
    gprob = gdn.problem(d["k"], dO, dO)
    ws = gdn.alloc_workspace(prob, 1, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev):
        ev[0].record(stream)
        gdn.gdn_segment_summary(d["k"], d["v"], d["g"], d["beta"], M, S, nseg, ws, prob=prob,
                                stream=stream)
        ev[1].record(stream)
        gdn.gdn_state_grad_summary(d["q"], d["k"], d["g"], d["beta"], dO, dS, nseg, prob=gprob,
                                   stream=stream)
        ev[2].record(stream)
        gdn.gdn_state_grad_scan(M, dS, dht, dH_in, stream=stream)
        ev[3].record(stream)

    def events():
        return [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    for _ in range(args.warmup):
        step(events())
    torch.cuda.synchronize()
    st, detail = gdn.gdn_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {st} detail {detail} during warm-up")
    Ksteps = args.steps
    ev = [events() for _ in range(Ksteps)]
    sampler = ClockSampler(local) if rank == 0 else None
    barrier(dev)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(Ksteps):
        step(ev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    st, detail = gdn.gdn_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {st} detail {detail} in the timed region")
    total_s = t0.elapsed_time(t1) / 1e3
    max_s = reduce_max(total_s, device=dev if world > 1 else "cpu")
    barrier(dev)
    avg = {name: sum(e[a].elapsed_time(e[a + 1]) for e in ev) / Ksteps
           for a, name in enumerate(("summary_M", "state_grad", "scan"))}
    alg = state_grad_algorithmic(w)
    peaks, peaks_src = load_peaks()
    tensor = w.in_dtype == "bf16"   # bf16 inputs take the tensor-core (tf32) instance
    roof = kernel_roofline(alg, avg["state_grad"], float(peaks["hbm_gbs"]),
                           float(peaks["bf16_tflops"]) * TF32_PER_BF16 if tensor else None)
    ms_per_step = max_s / Ksteps * 1e3
    value = aggregate(w.B * w.T, Ksteps, world, max_s)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        heads = [(b, h) for b in range(B) for h in range(H)]
        done, secs = 0, 0.0
        while done < len(heads) and secs < args.cpu_seconds:
            b, h = heads[done]
            xs = {n: np.ascontiguousarray(x[n][b:b + 1, :, h:h + 1])
                  for n in ("q", "k", "v", "g", "beta")}
            dOs = np.ascontiguousarray(gr["dO"][b:b + 1, :, h:h + 1])
            t = time.perf_counter()
            Ms, _ = oracle.summary(xs["k"], xs["v"], xs["g"], xs["beta"], nseg)
            dSs = oracle.state_grad_summary(xs["q"], xs["k"], xs["g"], xs["beta"], dOs, nseg)
            oracle.state_grad_scan(Ms, dSs, gr["dht"][b:b + 1, h:h + 1])
            secs += time.perf_counter() - t
            done += 1
        cpu = {"value": round(B * w.T * done / len(heads) / secs, 1), "unit": "tokens/s",
               "cores": oracle.num_threads(0), "kind": "oracle",
               "sample": f"{done} of {len(heads)} (b,h) heads of {w.name}, all T={w.T} tokens: "
                         f"fp64 segment summaries, per-segment state gradients and the reverse "
                         f"scan; {secs:.1f} s; tokens/s scaled to the whole batch"}
    if rank == 0:
        line = {
            "metric": STATE_GRAD_METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": Ksteps, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32" if w.in_dtype == "f32" else "bf16 in, f32 math",
            "data": "synthetic",
            "config": {"workload": w0.name, "path": "state_grad", "B": B, "H": H, "T": w.T,
                       "K": K, "V": V, "nseg": nseg, "chunk": 64, "in_dtype": w.in_dtype,
                       "dO_dtype": "f32", "l2": "inputs larger than L2 (no flush)",
                       "parallelism": f"weak: {world} rank(s) x one batch each"},
            "roofline": dict(roof, **{
                "traffic": None if args.T else recorded_traffic("state_grad_kernel", w0.name),
                "kernel": "state_grad_kernel", "kernel_ms": round(avg["state_grad"], 4),
                "algorithmic_flops": alg["flops"], "algorithmic_bytes": alg["bytes"],
                "peak_source": (f"{peaks_src} bf16_tflops x {TF32_PER_BF16:.4f} (tf32/bf16 nominal) "
                                f"or hbm_gbs, whichever bounds" if tensor else
                                "fp32 CUDA-core peak: 152 SMs x 128 lanes x 2 x 2.07 GHz")}),
            "stage_ms": {k: round(v, 4) for k, v in avg.items()},
            "cpu_baseline": cpu,
            "e2e": None,
            # WY tiles + tensor-core summary (or one CUDA-core summary), state gradients, scan
            "gpu_launches": (4 if w.in_dtype == "bf16" and K == 128 else 3) * Ksteps,
            "clocks": clocks,
            "peaks_source": peaks_src,
        }
        print(json.dumps(line), flush=True)
    import torch.distributed as dist
    if dist.is_initialized():
        dist.destroy_process_group()


def chunk_grad_algorithmic(w, out_bytes: int = 4):
    """Per launch of the per-chunk gradient kernel over workload w. Bytes: read q, k, v, g, beta
    (input dtype), dO (output dtype), the state entering and the gradient leaving every chunk
    (fp32 K x V each); write dq, dk, dv, dg, dbeta (fp32). Flops per chunk and head, every
    product counted once as a dense tile (triangular ones too, c = 64): K K^T and Q K^T
    (2 c c K 2), the inverse (~0.17 M), W (c c K 2), R = A diag(beta) V - W H (c c V 2 + c K V 2),
    dR = Kd D' + C^T dO (c K V 2 + c c V 2), dQd, dKd, dW (3 c V K 2), dC and dR V^T
    (2 c c V 2), A^T dR (c c V 2), A^T dW and dW Kr^T (2 c c K 2), A^T dA and its product with
    A^T (2 c c c 2), dq and dk from the score gradients (3 c c K 2)."""
    isz = 2 if w.in_dtype == "bf16" else 4
    c, K, V = 64, w.K, w.V
    th = w.B * w.T * w.H
    per_tok = (2 * K + V + 2) * isz + V * out_bytes + (2 * K + V + 2) * 4
    nbytes = th * per_tok + (th // c) * 2 * K * V * 4
    per_chunk = (2 * c * c * K * 2 + 0.17e6 + c * c * K * 2 + c * c * V * 2 + c * K * V * 2 +
                 c * K * V * 2 + c * c * V * 2 + 3 * c * V * K * 2 + 2 * c * c * V * 2 +
                 c * c * V * 2 + 2 * c * c * K * 2 + 2 * c * c * c * 2 + 3 * c * c * K * 2)
    return {"bytes": nbytes, "flops": per_chunk * th / c}


def bwd_pieces(w, sms: int) -> int:
    """The piece count gdn_chunk_bwd gives its state-gradient chains (the library's rule,
    restated to count its launches): 1 when B*H*column-tiles chains fill at most one wave,
    else the largest power of two dividing the chunk count with that many chains per wave."""
    tile = 64 if w.in_dtype == "bf16" else 32
    chains = w.B * w.H * (w.V // tile)
    nch, sms, P = w.T // 64, min(sms, 256), 1
    while nch > 0 and nch % (2 * P) == 0 and chains * 2 * P <= sms:
        P *= 2
    return P


def kernel_roofline(alg, ms, hbm_gbs, tensor_tflops=None):
    """The roofline object of one kernel from its algorithmic work per launch and its average
    launch time: against the tensor-core rate or HBM, whichever bounds it (tensor_tflops given),
    or against the fp32 CUDA-core peak (the CUDA-core instances)."""
    if tensor_tflops is None:
        ach = alg["flops"] / (ms * 1e-3) / 1e12
        return {"bound": "alu", "achieved": round(ach, 3), "peak": round(FP32_ALU_TFLOPS, 2),
                "unit": "TFLOP/s", "frac": round(ach / FP32_ALU_TFLOPS, 4)}
    if alg["flops"] / (tensor_tflops * 1e12) >= alg["bytes"] / (hbm_gbs * 1e9):
        ach = alg["flops"] / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": round(ach, 3), "peak": round(tensor_tflops, 1),
                "unit": "TFLOP/s", "frac": round(ach / tensor_tflops, 4)}
    ach = alg["bytes"] / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(ach, 2), "peak": hbm_gbs, "unit": "GB/s",
            "frac": round(ach / hbm_gbs, 4)}


def backward_compulsory_bytes(w, out_bytes: int = 4):
    """The backward's inputs read once (q, k, v, g, beta, dO, h0, dht) and its gradients
    written once (dq, dk, dv, dg, dbeta fp32, dh0)."""
    isz = 2 if w.in_dtype == "bf16" else 4
    th = w.B * w.T * w.H
    states = w.B * w.H * w.K * w.V * 4
    return th * ((2 * w.K + w.V + 2) * isz + w.V * out_bytes + (2 * w.K + w.V + 2) * 4) + 3 * states


def run_backward(args):
    """The whole backward through gdn_chunk_bwd on one workload: one step is one call, its six
    steps bracketed by events on the stream (forward recomputation, summaries M, per-segment
    state gradients and their reverse scan, the second state-gradient pass, the per-chunk
    gradients)."""
    import numpy as np
    import torch

    import oracle
    from context_scan_gb300 import gdn, synth

    world, rank = init_dist("nccl" if args.gpus > 1 else "gloo")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    w0 = synth.WORKLOADS[args.workload]
    if w0.gate_k or w0.seq_lens is not None:
        raise SystemExit("--path backward runs fixed-length scalar-gate workloads only")
    w = synth.scaled(w0, seed=w0.seed + rank_seed_offset(rank),
                     **({} if args.T is None else {"T": args.T}))
    x = synth.make_inputs(w)
    gr = synth.make_grads(w, dht_sd=0.1)
    dt = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
    host = {n: torch.from_numpy(x[n]).to(dt).pin_memory() for n in ("q", "k", "v", "g", "beta")}
    host["h0"] = None if x["h0"] is None else torch.from_numpy(x["h0"]).pin_memory()
    host["dO"] = torch.from_numpy(gr["dO"]).pin_memory()
    host["dht"] = torch.from_numpy(gr["dht"]).pin_memory()
    d = {n: (None if t is None else t.to(dev)) for n, t in host.items()}
    B, T, H, K, V, nseg = w.B, w.T, w.H, w.K, w.V, w.nseg
    outs = (torch.empty((B, T, H, K), device=dev), torch.empty((B, T, H, K), device=dev),
            torch.empty((B, T, H, V), device=dev), torch.empty((B, T, H), device=dev),
            torch.empty((B, T, H), device=dev), torch.empty((B, H, K, V), device=dev))
    prob = gdn.problem(d["k"], d["v"], d["dO"], g=d["g"])
    ws = gdn.alloc_bwd_workspace(prob, nseg, device=dev)
    stream = torch.cuda.current_stream()
    # the state-gradient chains run one pass (one piece) or two around the summaries and the
    # reverse scan (several pieces): see bwd_pieces
    stage_names = ("forward", "summary_M", "state_grad_1", "state_grad_2", "chunk_grad")

    def call(di, oi, events=None):
        args_ = (di["q"], di["k"], di["v"], di["g"], di["beta"], di["h0"], di["dO"], di["dht"],
                 *oi, nseg, ws)
        if events is None:
            gdn.gdn_chunk_bwd(*args_, prob=prob, stream=stream)
        else:
            gdn.gdn_chunk_bwd_timed(*args_, events, prob=prob, stream=stream)

    for _ in range(args.warmup):
        call(d, outs)
    torch.cuda.synchronize()
    st, detail = gdn.gdn_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {st} detail {detail} during warm-up")
    # stage times from a pass of the timed entry point (its events sit between the launches);
    # the timed region runs the plain call
    K = args.steps
    Ks = min(K, 20)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(Ks)]
    for e6 in ev:
        for e in e6:
            e.record(stream)
    for i in range(Ks):
        call(d, outs, ev[i])
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    barrier(dev)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        call(d, outs)
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    st, detail = gdn.gdn_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {st} detail {detail} in the timed region")
    total_s = t0.elapsed_time(t1) / 1e3
    max_s = reduce_max(total_s, device=dev if world > 1 else "cpu")
    barrier(dev)
    avg = {name: sum(e[a].elapsed_time(e[a + 1]) for e in ev) / Ks
           for a, name in enumerate(stage_names)}
    peaks, peaks_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    # the dominant backward kernel: the second state-gradient pass or the per-chunk gradients
    tensor = w.in_dtype == "bf16"   # bf16 inputs take the tensor-core (tf32) instances
    pieces = bwd_pieces(w, torch.cuda.get_device_properties(dev).multi_processor_count)
    cand = {"state_grad_kernel": (state_grad_algorithmic(synth.scaled(w, nseg=pieces)),
                                  max(avg["state_grad_1"], avg["state_grad_2"])),
            "chunk_grad_kernel": (chunk_grad_algorithmic(w), avg["chunk_grad"])}
    kname = max(cand, key=lambda n: cand[n][1])
    alg, kms = cand[kname]
    roof = kernel_roofline(alg, kms, hbm, float(peaks["bf16_tflops"]) * TF32_PER_BF16 if tensor else None)
    roof.update({"traffic": None if args.T else recorded_traffic(kname, w0.name), "kernel": kname,
                 "kernel_ms": round(kms, 4), "algorithmic_flops": alg["flops"],
                 "algorithmic_bytes": alg["bytes"],
                 "peak_source": (f"{peaks_src} bf16_tflops x {TF32_PER_BF16:.4f} (tf32/bf16 nominal) "
                                 f"or hbm_gbs, whichever bounds" if tensor else
                                 "fp32 CUDA-core peak: 152 SMs x 128 lanes x 2 x 2.07 GHz")})
    ms_per_step = max_s / K * 1e3
    tokens = B * T
    value = aggregate(tokens, K, world, max_s)
    comp = backward_compulsory_bytes(w)
    t_comp = comp / (hbm * 1e9)

    e2e = None
    if not args.no_e2e:
        n_e2e = max(3, min(K, args.e2e_steps))
        h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in outs)
        barrier(dev)
        e_el = pipelined_e2e(torch, host, d, outs, call, n_e2e, dev, stream)
        e_el = reduce_max(e_el, device=dev if world > 1 else "cpu")
        st, detail = gdn.gdn_check_device_error(ws)
        if st != 0:
            raise RuntimeError(f"device error word {st} detail {detail} in the end-to-end run")
        e2e = {"value": round(aggregate(tokens, n_e2e, world, e_el), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "pipelined": "two buffer sets; copies in and out on their own streams"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        heads = [(b, h) for b in range(B) for h in range(H)]
        done, secs = 0, 0.0
        nthreads = oracle.num_threads(0)
        while done < len(heads) and secs < args.cpu_seconds:
            b, h = heads[done]
            xs = {n: np.ascontiguousarray(x[n][b:b + 1, :, h:h + 1])
                  for n in ("q", "k", "v", "g", "beta")}
            h0 = None if x["h0"] is None else np.ascontiguousarray(x["h0"][b:b + 1, h:h + 1])
            t = time.perf_counter()
            oracle.backward(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"],
                            np.ascontiguousarray(gr["dO"][b:b + 1, :, h:h + 1]), h0,
                            np.ascontiguousarray(gr["dht"][b:b + 1, h:h + 1]))
            secs += time.perf_counter() - t
            done += 1
        cpu = {"value": round(tokens * done / len(heads) / secs, 1), "unit": "tokens/s",
               "cores": 1, "kind": "oracle",
               "sample": f"{done} of {len(heads)} (b,h) heads of {w.name}, all T={T} tokens: the "
                         f"fp64 per-token backward (one head is one work unit, so one core of "
                         f"the {nthreads} runs it); {secs:.1f} s; tokens/s scaled to the whole "
                         f"batch"}
    if rank == 0:
        tc = int(w.in_dtype == "bf16" and K == 128 and V == 128)
        fwd_plan = gdn.segmented_plan(prob, T // 64) if T else (1, 0, 0)
        launches = launches_per_step(synth.scaled(w, nseg=T // 64 or 1), fwd_plan[0], fwd_plan,
                                     torch.cuda.get_device_properties(dev).multi_processor_count) + \
            (1 + 1 if pieces == 1 else (tc + 1) + 3 + 1 + 1)
        line = {
            "metric": BACKWARD_METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32" if w.in_dtype == "f32" else "bf16 in, f32 math",
            "data": "synthetic",
            "config": {"workload": w0.name, "path": "backward", "B": B, "H": H, "T": T, "K": K,
                       "V": V, "nseg": nseg, "state_grad_pieces": pieces, "chunk": 64,
                       "in_dtype": w.in_dtype,
                       "dO_dtype": "f32", "grad_dtype": "f32",
                       "l2": "inputs larger than L2 (no flush)",
                       "parallelism": f"weak: {world} rank(s) x one batch each"},
            "roofline": roof,
            "path_roofline": {"t_roof_us": round(t_comp * 1e6, 1),
                              "frac": round(t_comp / (ms_per_step * 1e-3), 4),
                              "bytes": comp,
                              "counts": "compulsory HBM bytes only: inputs, dO and dht read "
                                        "once, the gradients written once",
                              "peaks": f"{peaks_src}: hbm {hbm} GB/s"},
            "stage_ms": {k: round(v, 4) for k, v in avg.items()},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches * K,
            "clocks": clocks,
            "peaks_source": peaks_src,
        }
        print(json.dumps(line), flush=True)
    import torch.distributed as dist
    if dist.is_initialized():
        dist.destroy_process_group()


def workload_metric(w0) -> str:
    """The headline metric names its own workload; the other workloads carry their shape."""
    if w0.name == DEFAULT_WORKLOAD:
        return METRIC
    if w0.gate_k:
        return KDA_METRIC
    return (f"GDN segmented fwd tokens/s at B{w0.B} H{w0.H} K=V={w0.K} T={w0.T} "
            f"{w0.nseg} segments {w0.in_dtype}; % of roofline")


def run_ours(args):
    import numpy as np
    import torch

    from context_scan_gb300 import gdn, synth

    if synth.WORKLOADS[args.workload].seq_lens is not None:
        return run_varlen(args)

    world, rank = init_dist("nccl" if args.gpus > 1 else "gloo")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    w0 = synth.WORKLOADS[args.workload]
    w = synth.scaled(w0, seed=w0.seed + rank_seed_offset(rank),
                     per_sequence_seed=(None if w0.per_sequence_seed is None
                                        else w0.per_sequence_seed + rank_seed_offset(rank)),
                     **({} if args.T is None else {"T": args.T}))
    literal = args.schedule == "literal"
    x = synth.make_inputs(w)
    dt = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
    names = ("q", "k", "v", "g", "beta")
    host = {n: torch.from_numpy(x[n]).to(dt).pin_memory() for n in names}
    host["h0"] = None if x["h0"] is None else torch.from_numpy(x["h0"]).pin_memory()
    d = {n: (None if t is None else t.to(dev, non_blocking=False)) for n, t in host.items()}
    o = torch.empty((w.B, w.T, w.H, w.V), dtype=torch.float32, device=dev)
    hf = torch.empty((w.B, w.H, w.K, w.V), dtype=torch.float32, device=dev)
    prob = gdn.problem(d["k"], d["v"], o, g=d["g"])
    if prob.gate_k != int(w.gate_k):
        raise RuntimeError("the problem's gate layout does not match the workload")
    stream = torch.cuda.current_stream()
    if literal:
        # the pages' flow from three public calls: every segment's summary, the in-order
        # apply, every segment's forward from its H_in
        plan = (w.nseg, w.T // 64 // w.nseg, w.T // 64 // w.nseg)
        ws = gdn.alloc_workspace(prob, 1, device=dev)
        Mb = torch.empty((w.nseg, w.B, w.H, w.K, w.K), dtype=torch.float32, device=dev)
        Sb = torch.empty((w.nseg, w.B, w.H, w.K, w.V), dtype=torch.float32, device=dev)
        Hin = torch.empty((w.nseg, w.B, w.H, w.K, w.V), dtype=torch.float32, device=dev)
        stage_names = ("summary", "scan", "forward")
    else:
        plan = gdn.segmented_plan(prob, w.nseg)
        ws = gdn.alloc_workspace(prob, w.nseg, device=dev)
        stage_names = ("wy", "phase1", "scan", "phase2")
    pieces = plan[0]

    def call(di, oi):
        if literal:
            gdn.gdn_segment_summary(di["k"], di["v"], di["g"], di["beta"], Mb, Sb, w.nseg, ws,
                                    prob=prob, stream=stream)
            gdn.gdn_summary_scan(Mb, Sb, di["h0"], Hin, stream=stream)
            gdn.gdn_segment_fwd(di["q"], di["k"], di["v"], di["g"], di["beta"], Hin, oi[0],
                                oi[1], w.nseg, ws, prob=prob, stream=stream)
        else:
            gdn.gdn_segmented_fwd(di["q"], di["k"], di["v"], di["g"], di["beta"], di["h0"],
                                  oi[0], oi[1], w.nseg, ws, prob=prob, stream=stream)

    def step(events=None):
        if events is None:
            call(d, (o, hf))
        elif literal:
            events[0].record(stream)
            gdn.gdn_segment_summary(d["k"], d["v"], d["g"], d["beta"], Mb, Sb, w.nseg, ws,
                                    prob=prob, stream=stream)
            events[1].record(stream)
            gdn.gdn_summary_scan(Mb, Sb, d["h0"], Hin, stream=stream)
            events[2].record(stream)
            gdn.gdn_segment_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], Hin, o, hf, w.nseg,
                                ws, prob=prob, stream=stream)
            events[3].record(stream)
        else:
            gdn.gdn_segmented_fwd_timed(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o,
                                        hf, w.nseg, ws, events, prob=prob, stream=stream)

    # Inputs and output that fit in L2 twice over could be served from it in the next step:
    # then a buffer larger than L2 is written between the timed steps, outside their events.
    in_mb = total_input_mb(w)
    touched = in_mb * 2**20 + w.B * w.T * w.H * w.V * 4
    flush = (torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
             if touched < 2 * L2_BYTES else None)

    for _ in range(args.warmup):
        if flush is not None:
            flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    st, detail = gdn.gdn_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {st} detail {detail} during warm-up")

    K = args.steps
    nev = len(stage_names) + 1
    # The stage times come from the library's own events recorded inside each step. Outside
    # the literal flow (whose step is several calls) they are taken in a pass of their own:
    # the timed region then runs the plain call a user makes, with nothing recorded between
    # its kernels (events there would keep its grids from overlapping their neighbours).
    Ks = K if literal else min(K, 100)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(Ks)]
    for e4 in ev:        # torch creates the CUDA event on first record; the library then
        for e in e4:     # re-records the same handles inside each step
            e.record(stream)
    if not literal:
        for i in range(Ks):
            if flush is not None:
                flush.fill_(1.0)
            step(ev[i])
        torch.cuda.synchronize()
    pe = ([[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
          if flush is not None and not literal else None)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if rank == 0 else None
    barrier(dev)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)   # let the sampler start before the timed region
    t0.record(stream)
    for i in range(K):
        if flush is not None:
            flush.fill_(1.0)   # outside the step's own events
        if literal:
            step(ev[i])
        else:
            if pe is not None:
                pe[i][0].record(stream)
            step()
            if pe is not None:
                pe[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier(dev)
    if flush is None:
        elapsed = t0.elapsed_time(t1) / 1e3
    elif literal:
        elapsed = sum(e[0].elapsed_time(e[-1]) for e in ev) / 1e3
    else:
        elapsed = sum(a.elapsed_time(b) for a, b in pe) / 1e3
    max_elapsed = reduce_max(elapsed, device=dev if world > 1 else "cpu")
    st, detail = gdn.gdn_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {st} detail {detail} in the timed region")

    stage_ms = {n: [] for n in stage_names}
    for e in ev:
        for i, name in enumerate(stage_names):
            stage_ms[name].append(e[i].elapsed_time(e[i + 1]))
    avg = {k: sum(v) / len(v) for k, v in stage_ms.items()}
    _, _, method = algorithmic(w, plan)
    if literal:
        stages, executed = literal_algorithmic(w)
        kernel_name = {"summary": "gdn_summary_call", "scan": "gdn_scan",
                       "forward": "gdn_segment_fwd"}
    else:
        stages, executed, _ = algorithmic(w, plan)
        kernel_name = {"wy": "gdn_wy", "phase1": "gdn_phase1", "scan": "gdn_scan",
                       "phase2": "gdn_forward"}
    # the dominant kernel: the longest stage that times one kernel (with the last piece's WY
    # tiles formed beside it, the first phase's stage holds two grids)
    one_kernel = dict(avg)
    if not literal and wy_tail_beside(w, plan, torch.cuda.get_device_properties(dev).multi_processor_count):
        one_kernel.pop("phase1")
    dominant = max(one_kernel, key=one_kernel.get)
    peaks, peaks_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    bf16_peak = float(peaks["bf16_tflops"])
    ach = stages[dominant]["bytes"] / (avg[dominant] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(ach, 2), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4),
                "traffic": recorded_traffic(kernel_name[dominant], w0.name),
                "kernel": kernel_name[dominant], "kernel_ms": round(avg[dominant], 4),
                "algorithmic_bytes": stages[dominant]["bytes"],
                "peak_source": f"{peaks_src} hbm_gbs"}
    ms_per_step = max_elapsed / K * 1e3
    tokens = w.B * w.T
    value = aggregate(tokens, K, world, max_elapsed)

    def path(total, what):
        t_roof = max(total["bytes"] / (hbm * 1e9), total["flops"] / (bf16_peak * 1e12))
        return {"t_roof_us": round(t_roof * 1e6, 1),
                "frac": round(t_roof / (ms_per_step * 1e-3), 4),
                "bytes": total["bytes"], "flops": total["flops"], "counts": what,
                "peaks": f"{peaks_src}: hbm {hbm} GB/s, bf16 {peaks['bf16_tflops']} TF/s"}

    path_roofline = path(executed, "the work this schedule runs: every pass it makes over the "
                                   "inputs, summaries and states (intermediates such as the WY "
                                   "tiles count as zero)")
    method_roofline = path(method, f"the pages' method: summaries of the {w.nseg - 1} segments "
                                   f"that feed a later one, the scan, the forward")

    # ---- end to end through the public API (pinned host -> device, call, device -> host)
    e2e = None
    if not args.no_e2e:
        n_e2e = max(3, min(K, args.e2e_steps))
        h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
        d2h = o.numel() * o.element_size() + hf.numel() * hf.element_size()
        barrier(dev)
        e_el = pipelined_e2e(torch, host, d, (o, hf), call, n_e2e, dev, stream)
        e_el = reduce_max(e_el, device=dev if world > 1 else "cpu")
        st, detail = gdn.gdn_check_device_error(ws)
        if st != 0:
            raise RuntimeError(f"device error word {st} detail {detail} in the end-to-end run")
        e2e = {"value": round(aggregate(tokens, n_e2e, world, e_el), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "pipelined": "two buffer sets; copies in and out on their own streams"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, x, budget_s=args.cpu_seconds)

    if rank == 0:
        tc = int(w.in_dtype == "bf16" and w.K == 128 and w.V == 128 and not w.gate_k)
        launches = (2 * tc + 3) if literal else launches_per_step(
            w, pieces, plan, torch.cuda.get_device_properties(dev).multi_processor_count)
        l2 = (f"inputs larger than L2 ({in_mb:.0f} MB in + "
              f"{w.B * w.T * w.H * w.V * 4 / 2**20:.0f} MB out > 129 MB); no flush"
              if flush is None else
              f"inputs fit in L2 ({in_mb:.0f} MB): a {2 * L2_BYTES / 2**20:.0f} MB buffer is "
              f"written before every step, outside the step's events")
        line = {
            "metric": workload_metric(w0), "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w0.name, "B": w.B, "H": w.H, "T": w.T, "K": w.K, "V": w.V,
                       "nseg": w.nseg, "schedule": args.schedule,
                       "pieces": {"P": plan[0], "first_chunks": plan[1], "rest_chunks": plan[2]},
                       "chunk": 64, "in_dtype": w.in_dtype,
                       "gates": "per key channel" if w.gate_k else "per token",
                       "out_dtype": "f32", "state_dtype": "f32", "l2": l2,
                       "parallelism": f"weak: {world} rank(s) x one batch each"},
            "roofline": roofline,
            "path_roofline": path_roofline,
            "method_roofline": method_roofline,
            "stage_ms": {k: round(v, 4) for k, v in avg.items()},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches * K,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    import torch.distributed as dist
    if dist.is_initialized():
        dist.destroy_process_group()


def total_input_mb(w):
    isz = 2 if w.in_dtype == "bf16" else 4
    g = w.K if w.gate_k else 1
    return w.B * w.T * w.H * ((2 * w.K + w.V) * isz + (g + 1) * isz) / 2**20


# ---------------------------------------------------------------------------------------
# the oracle timed on the host cores (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------------------
def oracle_heads(w, x, heads, nthreads=0):
    """Run the oracle recurrence (o, h_final and the state entering every segment) on the
    given (b, h) heads; returns seconds."""
    import oracle
    t = time.perf_counter()
    for b, h in heads:
        xs = {n: x[n][b:b + 1, :, h:h + 1] for n in ("q", "k", "v", "g", "beta")}
        h0 = None if x["h0"] is None else x["h0"][b:b + 1, h:h + 1]
        rec = oracle.kda_recurrence if w.gate_k else oracle.recurrence
        rec(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"], h0,
            seg_len=w.seg_len, col_block=8, nthreads=nthreads)
    return time.perf_counter() - t


def cpu_baseline(w, x, budget_s=12.0):
    import oracle
    cores = oracle.num_threads(0)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    done, secs = 0, 0.0
    while done < len(heads) and secs < budget_s:
        secs += oracle_heads(w, x, [heads[done]])
        done += 1
    value = w.B * w.T * done / len(heads) / secs
    return {"value": round(value, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} of {len(heads)} (b,h) heads of {w.name}, all T={w.T} tokens, "
                      f"fp64 per-token recurrence with the state entering each of the "
                      f"{w.nseg} segments; {secs:.1f} s; tokens/s scaled to the whole batch"}


def cpu_baseline_varlen(w, x, budget_s=12.0):
    import oracle
    from context_scan_gb300 import synth
    cores = oracle.num_threads(0)
    cu = synth.cu_seqlens(w)
    done, secs = 0, 0.0
    while done < w.H and secs < budget_s:
        h = done
        xs = {n: x[n][:, :, h:h + 1] for n in ("q", "k", "v", "g", "beta")}
        h0 = None if x["h0"] is None else x["h0"][:, h:h + 1]
        t = time.perf_counter()
        oracle.varlen_recurrence(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"], cu, h0)
        secs += time.perf_counter() - t
        done += 1
    value = w.T * done / w.H / secs
    return {"value": round(value, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} of {w.H} heads of {w.name}, every packed sequence, fp64 per-token "
                      f"recurrence; {secs:.1f} s; tokens/s scaled to all heads"}


def run_reference_varlen(args, w, x):
    import oracle
    from context_scan_gb300 import synth
    cores = oracle.num_threads(0)
    cu = synth.cu_seqlens(w)

    def head(h):
        xs = {n: x[n][:, :, h:h + 1] for n in ("q", "k", "v", "g", "beta")}
        h0 = None if x["h0"] is None else x["h0"][:, h:h + 1]
        t = time.perf_counter()
        oracle.varlen_recurrence(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"], cu, h0)
        return time.perf_counter() - t

    for i in range(args.warmup):
        head(i % w.H)
    secs = sum(head((args.warmup + i) % w.H) for i in range(args.steps))
    value = w.T * args.steps / w.H / secs   # one step = one head of the packed batch
    line = {
        "impl": "reference", "metric": varlen_metric(w), "value": round(value, 1),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "seq_lens": list(w.seq_lens), "B": 1, "H": w.H,
                   "T": w.T, "K": w.K, "V": w.V, "in_dtype": w.in_dtype},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"each step: one head of {w.name} (every packed sequence), "
                                   f"fp64 per-token recurrence on {cores} host threads"},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from context_scan_gb300 import synth
    import oracle
    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w)
    if w.seq_lens is not None:
        return run_reference_varlen(args, w, x)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    cores = oracle.num_threads(0)
    for i in range(args.warmup):
        oracle_heads(w, x, [heads[i % len(heads)]])
    secs = 0.0
    for i in range(args.steps):
        secs += oracle_heads(w, x, [heads[(args.warmup + i) % len(heads)]])
    # one step = one of the B*H heads; tokens/s scaled to the whole batch
    value = w.B * w.T * args.steps / len(heads) / secs
    line = {
        "impl": "reference", "metric": metric_of(w), "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "K": w.K, "V": w.V,
                   "nseg": w.nseg, "in_dtype": w.in_dtype},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"each step: one (b,h) head of {w.name} ({w.T} tokens), "
                                   f"fp64 per-token recurrence on {cores} host threads"},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def record_traffic(csv_path: str, kernel: str, workload: str, command: str, grid=None,
                   scale_note: str = "", scale=None, out_dir=None) -> str:
    """Write profiles/traffic_<kernel>_<workload>.txt from an ncu CSV of one capture of the
    kernel (metrics dram__bytes_read.sum and dram__bytes_write.sum; with several launches in
    the CSV, the one whose grid is `grid`, or with grid "sum" the sum over every launch in it:
    the launches of one call of a stage that runs several). The record carries the hash of the
    sources the kernel is built from now, so bench.py trusts it exactly until one of them
    changes.
    scale = (factor, fixed_bytes): per-launch bytes = (captured - fixed) * factor + fixed, for
    a capture of a smaller case of the same kernel."""
    units = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}
    launches = {}
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    rd = csv.DictReader(io.StringIO("".join(lines)))
    for r in rd:
        name = r.get("Metric Name", "")
        if name not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        key = (r.get("ID"), r.get("Kernel Name", ""), r.get("Grid Size", ""))
        v = float(r["Metric Value"].replace(",", "")) * units.get(r.get("Metric Unit", "byte"), 1.0)
        launches.setdefault(key, {})[name] = v
    if grid == "sum":
        if not launches:
            raise SystemExit(f"no launch in {csv_path}")
        v = {m: sum(x.get(m, 0.0) for x in launches.values())
             for m in ("dram__bytes_read.sum", "dram__bytes_write.sum")}
        kname = " + ".join(f"{k[1].split('(')[0].strip()} grid {k[2]}" for k in launches)
        kname, kgrid = f"{len(launches)} launches: {kname}", "(one call)"
    else:
        picked = [(k, v) for k, v in launches.items() if grid is None or k[2] == grid]
        if len(picked) != 1:
            raise SystemExit(f"expected one launch{' with grid ' + grid if grid else ''} in "
                             f"{csv_path}, found {len(picked)}")
        (lid, kname, kgrid), v = picked[0]
    captured = v["dram__bytes_read.sum"] + v["dram__bytes_write.sum"]
    per_launch = captured
    if scale is not None:
        factor, fixed = scale
        per_launch = (captured - fixed) * factor + fixed
    out = os.path.join(out_dir or os.path.join(ROOT, "profiles"), f"traffic_{kernel}_{workload}.txt")
    with open(out, "w") as f:
        name = kname if grid == "sum" else kname.split('(')[0].strip()
        f.write(f"kernel: {name} grid {kgrid} on {workload}\n")
        f.write(f"kernel_source_hash: {kernel_source_hash(kernel)}\n")
        f.write(f"dram_bytes_per_launch: {per_launch:.0f}\n")
        f.write(f"captured: dram__bytes_read.sum {v['dram__bytes_read.sum']:.0f} + "
                f"dram__bytes_write.sum {v['dram__bytes_write.sum']:.0f} = {captured:.0f}\n")
        if scale is not None:
            f.write(f"scaled: (captured - {scale[1]:.0f}) x {scale[0]:.4f} + {scale[1]:.0f}"
                    f"{'; ' + scale_note if scale_note else ''}\n")
        f.write(f"command: {command}\n")
        f.write(f"hash covers: {', '.join(KERNEL_SOURCES[kernel])}, include/gdn.h\n")
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--path", choices=["forward", "state_grad", "backward"], default="forward",
                    help="forward: the segmented forward (the headline line); state_grad: the "
                         "backward's state-gradient path on the same workload; backward: the "
                         "whole backward (gdn_chunk_bwd)")
    ap.add_argument("--schedule", choices=["pieces", "literal"], default="pieces",
                    help="pieces: one gdn_segmented_fwd call (the library's piece plan; the "
                         "headline line); literal: the pages' flow from three public calls -- "
                         "gdn_segment_summary over every segment, gdn_summary_scan, "
                         "gdn_segment_fwd")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--T", type=int, default=None,
                    help="run the workload at this sequence length instead (a smaller case of "
                         "the same kernels for profiler captures; not a bench line)")
    ap.add_argument("--record-traffic", metavar="NCU_CSV", default=None,
                    help="write profiles/traffic_<--traffic-kernel>_<--workload>.txt from an ncu "
                         "CSV of dram__bytes_read.sum and dram__bytes_write.sum (no GPU needed)")
    ap.add_argument("--traffic-kernel", default="gdn_forward", choices=sorted(KERNEL_SOURCES))
    ap.add_argument("--traffic-grid", default=None,
                    help='the captured launch\'s grid, e.g. "(128, 1, 1)", or "sum": every '
                         'launch in the CSV (one call of a stage that runs several)')
    ap.add_argument("--traffic-command", default="", help="the command line the CSV came from")
    args = ap.parse_args(argv)
    if args.record_traffic:
        print(record_traffic(args.record_traffic, args.traffic_kernel, args.workload,
                             args.traffic_command, grid=args.traffic_grid))
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.path == "state_grad":
        run_state_grad(args)
    elif args.path == "backward":
        run_backward(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
