#!/usr/bin/env python
"""Benchmark of the csgmv LoRA path on GB300.

One step = one pass of the whole path over one batch: the device batch builder
(chunk size, stable token permutation, segments) followed by the
shrink->expand call (csgmv_qkv, given an h workspace as a caller would).  The
default workload is the largest configuration that fits one GPU: prefill
gate_up, 32 requests of U[64, 2048] tokens (~33.8k tokens), K = 4096,
c = 2 slices of 14336 columns, 16 slots with ranks from {8, 16, 32, 64} on a
Zipf(1.1) assignment.  Steps rotate over enough independent input sets (own
x, A, B, base and batch) that the data a step touches is not in L2.

Besides the headline line, every other configuration is measured in the same
run under `per_config` (CUDA-event time of the csgmv_qkv or embedding call
and of the builder, its roofline fraction and tokens/s): tiny, decode QKV,
skewed down_proj at chunk 16 / 32 / 64 / 128, lm_head decode, pruned lm_head
and the embedding gather.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead,
on bounded token samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from segmented_gather_gemm_gb300 import workloads as wl  # noqa: E402

METRIC = "csgmv shrink+expand tokens/s at 1 GB300; % of HBM/tensor roofline vs CPU oracle"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# The configurations measured next to the headline workload: (label, workload,
# chunk override), and the roofline fraction each one is held to.
PER_CONFIG = [
    ("tiny", "tiny", 0),
    ("decode_qkv", "decode_qkv", 0),
    ("skewed_down_proj_chunk16", "skewed_down_proj", 16),
    ("skewed_down_proj_chunk32", "skewed_down_proj", 32),
    ("skewed_down_proj_chunk64", "skewed_down_proj", 64),
    ("skewed_down_proj_chunk128", "skewed_down_proj", 128),
    ("lm_head_decode", "lm_head_decode", 0),
    ("lm_head_pruned", "lm_head_pruned", 0),
    ("embedding", "embedding", 0),
    ("embedding_transposed", "embedding_transposed", 0),
]
TARGET_FRAC = {"prefill_gate_up": 0.70, "skewed_down_proj": 0.70, "decode_qkv": 0.60, "lm_head_decode": 0.60}


# --------------------------------------------------------------------------- workloads

def make_workload(name: str, seed: int, chunk: int, scale: float = 1.0, bs: int = 0):
    if name == "decode_qkv":
        return wl.decode_qkv(seed=seed, bs=bs or 256)
    if name == "prefill_gate_up":
        return wl.prefill_gate_up(seed=seed, scale_tokens=scale)
    if name == "skewed_down_proj":
        return wl.skewed_down_proj(seed=seed, chunk=chunk, scale_tokens=scale)
    if name == "lm_head_decode":
        return wl.lm_head_decode(seed=seed, bs=bs or 512)
    if name == "lm_head_pruned":
        return wl.lm_head_pruned(seed=seed, bs=bs or 64)
    if name == "tiny":
        return wl.tiny_single_slice(seed=seed)
    if name == "embedding":
        return wl.embedding_gather(seed=seed)
    if name == "embedding_transposed":  # the same gather from the load-time (L, V, R) table
        w = wl.embedding_gather(seed=seed)
        w.transposed = True
        w.name = w.name.replace("embedding_lora_a", "embedding_lora_a_transposed")
        return w
    raise SystemExit(f"unknown workload {name}")


def token_ranks(w) -> np.ndarray:
    """Rank of the slot of every token (request slot repeated per token)."""
    return np.repeat(w.ranks[w.req_adapter], w.req_lens)


def algorithmic(w, chunk: int) -> dict:
    """Bytes and FLOPs the path must move / do for workload w: x rows of tokens
    with a rank > 0, A rows c*r_a*K and B columns N*r_a of every used slot with
    r_a > 0, base read + write of covered columns for those tokens, and the
    int32 indices the kernel reads.  h is not counted: the fused kernel keeps it
    on chip, and the workspace path's fp32 round trip is the implementation's own."""
    if isinstance(w, wl.EmbeddingWorkload):
        rt = token_ranks(w)
        s = w.s
        nseg = sum(-(-int(n) // chunk) for n in np.bincount(np.repeat(w.req_adapter, w.req_lens)) if n)
        b = s * 4 + s * w.R * 2 + int(rt.sum()) * 2 + 4 * (s + 2 * nseg + 1)
        return {"bytes": b, "flops": 0, "tokens": s, "active": int((rt > 0).sum())}
    rt = token_ranks(w)
    act = rt > 0
    ncov = int(w.offsets[-1] - w.offsets[0])
    used = np.unique(np.repeat(w.req_adapter, w.req_lens)[act])
    ra = w.ranks[used].astype(np.int64)
    counts = np.bincount(np.repeat(w.req_adapter, w.req_lens), minlength=w.L)
    nseg = int(sum(-(-int(n) // chunk) for n in counts if n))
    b = (int(act.sum()) * w.K * 2 + int((w.c * ra * w.K * 2).sum()) + int((ncov * ra * 2).sum())
         + int(act.sum()) * ncov * 4 + 4 * (w.s + 2 * nseg + 1))
    flops = int((2 * rt.astype(np.int64) * (w.c * w.K + ncov)).sum())
    return {"bytes": b, "flops": flops, "tokens": w.s, "active": int(act.sum())}


WIDE_COLS = 32768  # the library's kWideCols
DECODE_CAPS = {"segments": 512, "loras": 256, "tokens": 2048}  # the decode kernels' table capacities


def qkv_kernels(w, bi) -> int:
    """Kernels one csgmv_qkv call launches when given a workspace: two (shrink,
    expand) where the library takes its two-kernel path, else one.  The path
    is taken by 16- / 32-token tiles (the decode kernels when the batch info's
    capacities fit their tables, the small-tile kernel with at least WIDE_COLS
    output columns) and by 128-token tiles with a buffer rank R >= 16.
    With a built batch info `bi` this is the library's own answer
    (csgmv_qkv_path with csgmv_qkv_workspace_bytes of workspace); without one
    the rule is applied here with the bench's capacities (max_segments =
    tokens + 1), which a host test checks against the library."""
    if isinstance(w, wl.EmbeddingWorkload):
        return 1
    if bi is not None and bi.c.num_tokens >= 0:
        from segmented_gather_gemm_gb300 import binding as B
        ws = B.csgmv_qkv_workspace_bytes(bi, w.c)
        return 1 if B.csgmv_qkv_path(bi, w.K, w.N, w.offsets, w.c, ws) == "fused" else 2
    slots = max(1, min(max(w.bs, 1), w.L))
    tm = 16 if w.s // slots <= 16 else (32 if w.s // slots <= 48 else 128)
    if tm <= 32:
        max_segments = bi.c.max_segments if bi is not None else w.s + 1
        max_loras = bi.c.max_loras if bi is not None else w.L
        decode = (max_segments <= DECODE_CAPS["segments"] and max_loras <= DECODE_CAPS["loras"]
                  and w.s <= DECODE_CAPS["tokens"])
        split = int(w.offsets[-1]) - int(w.offsets[0]) >= WIDE_COLS or decode
    else:
        split = w.R >= 16
    return 2 if split else 1


def set_bytes(w) -> int:
    if isinstance(w, wl.EmbeddingWorkload):
        return w.ids.nbytes + w.A_emb.nbytes
    return w.x.nbytes + w.A.nbytes + w.B.nbytes + w.base.nbytes


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Sources of the kernels behind each recorded traffic figure, with their
# launcher and shared headers: the decode kernels, the small-tile shrink and
# the wide expand for lm_head, the streaming tcgen05 kernels for prefill.
_SHARED_SOURCES = ("lora_tma.cuh", "lora_launch.cu", "device_utils.cuh", "csgmv_internal.h")
KERNEL_SOURCES = {
    "decode_qkv": ("lora_decode.cuh", "lora_decode.cu") + _SHARED_SOURCES,
    "lm_head_decode": ("lora_small.cuh", "lora_small.cu", "lora_wide.cuh", "lora_wide.cu") + _SHARED_SOURCES,
    "prefill_gate_up": ("lora_stream.cuh", "lora_stream.cu", "lora_sshrink.cu") + _SHARED_SOURCES,
    "skewed_down_proj": ("lora_stream.cuh", "lora_stream.cu", "lora_sshrink.cu") + _SHARED_SOURCES,
}


def kernel_source_hash(workload: str | None = None) -> str:
    """Hash of the kernel sources a recorded traffic figure belongs to (those
    of `workload`, else every LoRA kernel source), with comments and
    whitespace removed, so that an edit of a comment keeps the record."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "segmented_gather_gemm_gb300", "csrc")
    wanted = KERNEL_SOURCES.get(workload)
    for f in sorted(os.listdir(csrc)):
        if (f in wanted) if wanted else (f.startswith("lora_") or f in ("device_utils.cuh", "csgmv_internal.h")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                text = fh.read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            text = re.sub(r"//[^\n]*", " ", text)
            h.update(f.encode() + b"\0" + " ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    summary, if it was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash(workload):
        return None
    return e.get("bytes_per_launch")


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        load = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(load)}


# --------------------------------------------------------------------------- GPU arm

class DeviceSet:
    """One independent input set resident in HBM, with its own batch info.
    `share` reuses another set's device tensors (same data, another chunk
    size)."""

    def __init__(self, w, chunk_override: int, max_rank: int, share: "DeviceSet | None" = None):
        import torch

        from segmented_gather_gemm_gb300 import binding as B
        self.w = w

        def bf(b):
            return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()

        self.lens = torch.from_numpy(w.req_lens).cuda()
        self.ad = torch.from_numpy(w.req_adapter).cuda()
        self.ranks = torch.from_numpy(w.ranks).cuda()
        if isinstance(w, wl.EmbeddingWorkload):
            self.scal = torch.ones(w.L, dtype=torch.float32, device="cuda")
            self.ids = share.ids if share else torch.from_numpy(w.ids).cuda()
            # the transposed table is made once, as a caller does when it loads an adapter
            self.A = share.A if share else (B.csgmv_transpose_embedding(bf(w.A_emb)) if w.transposed
                                            else bf(w.A_emb))
            self.out = torch.zeros((w.s, w.R), dtype=torch.bfloat16, device="cuda")
            self.bi = B.BatchInfo.for_batch(len(w.req_lens), w.s, w.L, w.R)
        else:
            self.scal = torch.from_numpy(w.scalings).cuda()
            if share:
                self.x, self.A, self.B, self.y = share.x, share.A, share.B, share.y
            else:
                self.x, self.A, self.B, self.y = bf(w.x), bf(w.A), bf(w.B), bf(w.base)
            if w.meta.get("builder") == "lm_head":  # runs in request order: room for one segment per token
                self.bi = B.BatchInfo(w.bs, w.s, w.s + 1, max_loras=w.L, max_rank=w.R)
            else:
                self.bi = B.BatchInfo.for_batch(w.bs, w.s, w.L, w.R, min_chunk=min(16, chunk_override or 16))
            self.widest = int(np.max(np.diff(w.offsets)))
            # h workspace: csgmv_qkv takes its two-kernel path where that is faster
            self.ws = share.ws if share else torch.empty(B.csgmv_qkv_workspace_bytes(self.bi, w.c) // 4,
                                                         dtype=torch.float32, device="cuda")
        self.chunk_override = chunk_override

    def build(self):
        from segmented_gather_gemm_gb300 import binding as B
        w = self.w
        if getattr(w, "meta", {}).get("builder") == "lm_head":
            B.csgmv_build_lm_head_batch_info(self.bi, self.lens, self.ad, w.s, self.ranks, self.scal,
                                             max_chunk_size=w.max_chunk_size, use_cuda_graph=True)
            return
        B.csgmv_build_batch_info(self.bi, self.lens, self.ad, w.s, self.ranks, self.scal,
                                 max_chunk_size=w.max_chunk_size, chunk_size_override=self.chunk_override,
                                 use_cuda_graph=True)

    def compute(self):
        from segmented_gather_gemm_gb300 import binding as B
        w = self.w
        if isinstance(w, wl.EmbeddingWorkload):
            if w.transposed:
                B.embedding_lora_a_transposed(self.ids, self.A, w.V, None, self.out, self.bi)
            else:
                B.embedding_lora_a(self.ids, self.A, w.V, self.out, self.bi)
        else:
            B.csgmv_qkv(self.x, self.A, self.B, w.offsets, w.c, self.widest, self.y, self.bi, workspace=self.ws)

    def step(self):
        self.build()
        self.compute()


def capture(torch, fn_list):
    """One CUDA graph that runs fn_list in order on the capture stream."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for fn in fn_list:
            fn()
    return g


def timed_graphs(torch, sets, n, kind, max_graph=1200):
    """Graphs that together run exactly n steps, rotating over the sets."""
    def fns(start, count):
        pick = {"step": "step", "compute": "compute", "build": "build"}[kind]
        return [getattr(sets[i % len(sets)], pick) for i in range(start, start + count)]
    if n <= max_graph:
        return [capture(torch, fns(0, n))]
    g_len = max(1, max_graph // len(sets)) * len(sets)
    full, rem = divmod(n, g_len)
    plan = [capture(torch, fns(0, g_len))] * full
    if rem:
        plan.append(capture(torch, fns(full * g_len, rem)))
    return plan


def time_plan(torch, plan, dist=None):
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    start.record()
    for g in plan:
        g.replay()
    end.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return start.elapsed_time(end) / 1e3


def max_over_ranks(seconds: float, dist, device: str) -> float:
    """The slowest rank's elapsed time (every rank gets it)."""
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, steps: int, tokens_per_step: float, elapsed: float) -> float:
    """Tokens of all replicas / the slowest replica's time (weak scaling:
    every rank runs its own batches)."""
    return world * steps * tokens_per_step / elapsed


def sets_needed(per_set: int) -> int:
    """Input sets to rotate so that a step never finds its data in L2: one
    set when a set alone is over twice the L2, else enough sets to exceed it."""
    if per_set >= 2 * L2_BYTES:
        return 1
    return -(-2 * L2_BYTES // per_set) + 1


def roofline_of(alg: dict, seconds: float, peaks: dict) -> dict:
    """Achieved bytes (or flops) per second of one call against the measured
    peak, on whichever of HBM bytes or tensor flops bounds the call."""
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    t_hbm = alg["bytes"] / (hbm * 1e9)
    t_tc = alg["flops"] / (tc * 1e12)
    if t_hbm >= t_tc:
        ach = alg["bytes"] / seconds / 1e9
        r = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4)}
    else:
        ach = alg["flops"] / seconds / 1e12
        r = {"bound": "tensor", "achieved": round(ach, 2), "peak": tc, "unit": "TFLOP/s", "frac": round(ach / tc, 4)}
    r["roofline_us"] = round(max(t_hbm, t_tc) * 1e6, 3)
    return r


def time_kind(torch, sets, kind: str, target_s: float = 0.05, cap: int = 2400):
    """Average CUDA-event seconds of one `kind` call ("compute" or "build"),
    replayed from graphs that rotate over the sets for about target_s."""
    n0 = len(sets)
    probe = timed_graphs(torch, sets, n0, kind)
    time_plan(torch, probe)
    est = time_plan(torch, probe) / n0
    reps = int(min(cap, max(n0, target_s / max(est, 1e-7))))
    reps = -(-reps // n0) * n0
    plan = timed_graphs(torch, sets, reps, kind)
    time_plan(torch, plan[:1])
    return time_plan(torch, plan) / reps, reps


def measure_config(torch, label: str, workload: str, chunk: int, peaks: dict, scale: float = 1.0) -> dict:
    """One configuration on its own input sets: the csgmv_qkv (or embedding)
    call and the builder, each timed with CUDA events over graph replays, the
    call's roofline fraction and its tokens/s."""
    w0 = make_workload(workload, 0, chunk or 128, scale)
    nsets = sets_needed(set_bytes(w0))
    ws = [w0] + [make_workload(workload, s, chunk or 128, scale) for s in range(1, nsets)]
    sets = [DeviceSet(w, chunk, w.R) for w in ws]
    for s in sets:
        s.step()
    torch.cuda.synchronize()
    status = [s.bi.device_status() for s in sets]
    if any(status):
        raise SystemExit(f"{label}: device status {status}")
    t_call, reps = time_kind(torch, sets, "compute")
    t_build, _ = time_kind(torch, sets, "build")
    chunk_used = sets[0].bi.chunk_size
    algs = [algorithmic(w, chunk_used) for w in ws]
    alg = {k: float(np.mean([a[k] for a in algs])) for k in ("bytes", "flops", "tokens")}
    r = roofline_of(alg, t_call, peaks)
    out = {
        "workload": w0.name, "call_us": round(t_call * 1e6, 3), "build_us": round(t_build * 1e6, 3),
        "tokens": alg["tokens"], "tokens_per_s": round(alg["tokens"] / t_call, 1),
        "step_tokens_per_s": round(alg["tokens"] / (t_call + t_build), 1),
        "algorithmic_bytes": int(alg["bytes"]), "algorithmic_flops": int(alg["flops"]),
        "kernels_per_call": qkv_kernels(w0, sets[0].bi), "chunk_size": chunk_used,
        "input_sets": nsets, "timed_calls": reps,
    }
    out.update({k: r[k] for k in ("bound", "achieved", "unit", "frac", "roofline_us")})
    out["target_frac"] = TARGET_FRAC.get(workload)
    del sets
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import torch

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from segmented_gather_gemm_gb300 import build as sgb
    sgb.build()
    from segmented_gather_gemm_gb300 import binding as B
    B.lib()

    w0 = make_workload(args.workload, 0, args.chunk, args.scale, args.bs)
    per_set = set_bytes(w0)
    nsets = args.sets or sets_needed(per_set)
    seeds = [1000 * rank + i for i in range(nsets)]
    ws = [w0 if s == 0 else make_workload(args.workload, s, args.chunk, args.scale, args.bs) for s in seeds]
    chunk_override = args.chunk if args.workload == "skewed_down_proj" else 0
    sets = [DeviceSet(w, chunk_override, w.R) for w in ws]
    torch.cuda.synchronize()

    # warm-up: every set once, then W steps
    for s in sets:
        s.step()
    for i in range(args.warmup):
        sets[i % nsets].step()
    torch.cuda.synchronize()
    status = [s.bi.device_status() for s in sets]
    if any(status):
        raise SystemExit(f"device status {status}")

    plan = timed_graphs(torch, sets, args.steps, "step")
    time_plan(torch, plan[:1])  # graph upload / first replay

    with ClockSampler(local) as clk:
        # keep the GPU busy on the same steps for a while so the clock samples
        # describe this workload, then the timed region
        t_end = time.time() + args.soak_seconds
        while time.time() < t_end:
            time_plan(torch, plan[:1])
        elapsed = time_plan(torch, plan, dist)
    clocks = clk.summary()
    if dist is not None:
        elapsed = max_over_ranks(elapsed, dist, "cuda")

    peaks, peak_src = load_peaks()
    t_compute, k_compute = time_kind(torch, sets, "compute")
    t_build, _ = time_kind(torch, sets, "build")

    k_steps = args.steps
    chunk = sets[0].bi.chunk_size
    algs = [algorithmic(w, chunk) for w in ws]
    tokens_per_step = float(np.mean([a["tokens"] for a in algs]))
    alg = {k: float(np.mean([a[k] for a in algs])) for k in ("bytes", "flops", "tokens")}
    value = whole_job_rate(world, k_steps, tokens_per_step, elapsed)

    breakdown = {"build_batch_info": round(t_build * 1e6, 3), "csgmv_qkv": round(t_compute * 1e6, 3),
                 "step": round(elapsed / k_steps * 1e6, 3)}
    kernels = qkv_kernels(w0, sets[0].bi)
    if kernels == 2 and not isinstance(w0, wl.EmbeddingWorkload):
        breakdown.update(time_split_kernels(torch, sets))

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(torch, ws[0], chunk_override, min(args.steps, 200), world)
    del sets
    torch.cuda.empty_cache()

    roofline = roofline_of(alg, t_compute, peaks)
    tr = recorded_traffic(args.workload)
    roofline["traffic"] = tr
    roofline["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    roofline["kernel"] = ("embedding_lora_a" if isinstance(w0, wl.EmbeddingWorkload) else
                          "csgmv_qkv call (" + ("shrink + expand kernels through the workspace"
                                                if kernels == 2 else "one fused kernel") + ")")
    roofline["algorithmic_bytes_per_launch"] = int(alg["bytes"])
    roofline["algorithmic_flops_per_launch"] = int(alg["flops"])
    roofline["kernel_us"] = round(t_compute * 1e6, 3)
    roofline["timed_calls"] = k_compute

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed / k_steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w0.name, "tokens_per_step": tokens_per_step, "chunk_size": chunk,
                   "input_sets": nsets, "set_bytes": per_set,
                   "l2": (f"rotating {nsets} input sets ({nsets * per_set / 1e6:.0f} MB > 2x L2) instead of a flush"
                          if nsets > 1 else f"one input set of {per_set / 1e6:.0f} MB (> 2x L2) instead of a flush"),
                   "step": "csgmv_build_batch_info + " + ("embedding_lora_a" if isinstance(w0, wl.EmbeddingWorkload)
                                                          else "csgmv_qkv"),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "roofline": roofline,
        "breakdown_us": breakdown,
        "gpu_launches": (1 + kernels) * k_steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_per_config:
        per = {}
        with ClockSampler(local) as clk2:
            for label, workload, ch in PER_CONFIG:
                if workload == args.workload and ch == chunk_override:
                    continue
                per[label] = measure_config(torch, label, workload, ch, peaks)
        per["clocks"] = clk2.summary()
        line["per_config"] = per
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(ws, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def time_split_kernels(torch, sets) -> dict:
    """CUDA-event time of the two kernels of the workspace path on their own:
    csgmv_shrink into an fp32 h buffer, then csgmv_expand from it (the same
    kernels csgmv_qkv launches there)."""
    from segmented_gather_gemm_gb300 import binding as B
    hs = []
    for s in sets:
        w = s.w
        hs.append(s.ws[: w.s * w.c * w.R].view(w.s, w.c * w.R))

    class _Shrink:
        def __init__(self, s, h):
            self.s, self.h = s, h

        def compute(self):
            s = self.s
            B.csgmv_shrink(s.x, s.A, s.w.c, self.h, s.bi)

    class _Expand(_Shrink):
        def compute(self):
            s = self.s
            B.csgmv_expand(self.h, s.B, s.w.offsets, s.w.c, s.widest, s.y, True, s.bi)

    t_s, _ = time_kind(torch, [_Shrink(s, h) for s, h in zip(sets, hs)], "compute")
    t_e, _ = time_kind(torch, [_Expand(s, h) for s, h in zip(sets, hs)], "compute")
    return {"shrink": round(t_s * 1e6, 3), "expand": round(t_e * 1e6, 3)}


def run_e2e(torch, w, chunk_override, steps, world):
    """Same step through the public API with pinned HOST inputs: copy the
    step's inputs in, build + compute, copy the result out, every step.  Two
    sets of device buffers and three streams let step i's device-to-host copy
    overlap step i+1's host-to-device copy (the copy engines run both
    directions at once), as a serving loop would; every copy of every step is
    inside the timed region."""
    from segmented_gather_gemm_gb300 import binding as B
    if isinstance(w, wl.EmbeddingWorkload):
        return None

    def pin(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            t = t.view(dtype)
        return t.pin_memory()

    hx = pin(w.x.view(np.int16), torch.bfloat16)
    hbase = pin(w.base.view(np.int16), torch.bfloat16)
    hlens, had = pin(w.req_lens), pin(w.req_adapter)
    hranks, hscal = pin(w.ranks), pin(w.scalings)
    hy = [torch.empty_like(hbase).pin_memory() for _ in range(2)]
    dA = torch.from_numpy(w.A.view(np.int16)).view(torch.bfloat16).cuda()
    dB = torch.from_numpy(w.B.view(np.int16)).view(torch.bfloat16).cuda()
    lm_head = w.meta.get("builder") == "lm_head"
    widest = int(np.max(np.diff(w.offsets)))

    class Set:
        def __init__(self):
            self.dx = torch.empty(hx.shape, dtype=torch.bfloat16, device="cuda")
            self.dy = torch.empty(hbase.shape, dtype=torch.bfloat16, device="cuda")
            self.dl = torch.empty_like(hlens, device="cuda")
            self.da = torch.empty_like(had, device="cuda")
            self.dr = torch.empty_like(hranks, device="cuda")
            self.ds = torch.empty_like(hscal, device="cuda")
            self.bi = B.BatchInfo(w.bs, w.s, w.s + 1, max_loras=w.L, max_rank=w.R) if lm_head \
                else B.BatchInfo.for_batch(w.bs, w.s, w.L, w.R)
            self.ws = torch.empty(B.csgmv_qkv_workspace_bytes(self.bi, w.c) // 4, dtype=torch.float32,
                                  device="cuda")
            self.h2d_done, self.comp_done, self.d2h_done = (torch.cuda.Event() for _ in range(3))
            self.d2h_done.record()

    sets = [Set(), Set()]
    s_h2d, s_comp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def one(i):
        b = sets[i & 1]
        with torch.cuda.stream(s_h2d):
            s_h2d.wait_event(b.d2h_done)  # this set's last result has left the device
            b.dx.copy_(hx, non_blocking=True)
            b.dy.copy_(hbase, non_blocking=True)
            b.dl.copy_(hlens, non_blocking=True)
            b.da.copy_(had, non_blocking=True)
            b.dr.copy_(hranks, non_blocking=True)
            b.ds.copy_(hscal, non_blocking=True)
            b.h2d_done.record(s_h2d)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(b.h2d_done)
            if lm_head:
                B.csgmv_build_lm_head_batch_info(b.bi, b.dl, b.da, w.s, b.dr, b.ds, max_chunk_size=w.max_chunk_size)
            else:
                B.csgmv_build_batch_info(b.bi, b.dl, b.da, w.s, b.dr, b.ds, max_chunk_size=w.max_chunk_size,
                                         chunk_size_override=chunk_override)
            B.csgmv_qkv(b.dx, dA, dB, w.offsets, w.c, widest, b.dy, b.bi, workspace=b.ws)
            b.comp_done.record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(b.comp_done)
            hy[i & 1].copy_(b.dy, non_blocking=True)
            b.d2h_done.record(s_d2h)

    for i in range(5):
        one(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    h2d = hx.nbytes + hbase.nbytes + hlens.nbytes + had.nbytes + hranks.nbytes + hscal.nbytes
    return {"value": round(world * steps * w.s / el, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(hy[0].nbytes), "steps": steps,
            "how": "wall clock over the steps (host API calls, pinned H2D + D2H copies, builder + csgmv_qkv); "
                   "two buffer sets on three streams, so one step's D2H copy overlaps the next step's H2D copy"}


# --------------------------------------------------------------------------- CPU (oracle) arm

def oracle_step(w, rows):
    """The oracle on `rows` of workload w: builder over the whole batch, then the
    fused per-token fp64 path on the sampled tokens."""
    import oracle
    if isinstance(w, wl.EmbeddingWorkload):
        chunk = oracle.chunk_size(w.s, w.max_chunk_size)
        oracle.build_batch_info(w.req_lens, w.req_adapter, chunk)
        ta = oracle.token_adapter(w.req_lens, w.req_adapter)
        oracle.embedding(w.ids[rows], w.A_emb, ta[rows], w.ranks)
        return
    chunk = w.chunk_override or oracle.chunk_size(w.s, w.max_chunk_size)
    if w.meta.get("builder") == "lm_head":
        oracle.build_lm_head_batch_info(w.req_lens, w.req_adapter, chunk)
    else:
        oracle.build_batch_info(w.req_lens, w.req_adapter, chunk)
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    oracle.fused(w.x[rows], w.A, w.B, w.offsets, w.c, ta[rows], w.ranks, w.scalings, w.base[rows])


def cpu_baseline(ws, seconds: float):
    """The oracle as it stands on all host cores, on growing token samples of
    the workload until about `seconds` of CPU work."""
    import oracle
    oracle.build()
    w = ws[0]
    n = 8
    t_total, tok_total = 0.0, 0
    i = 0
    while t_total < seconds:
        wi = ws[i % len(ws)]
        rows = np.arange(min(n, wi.s))
        t0 = time.perf_counter()
        oracle_step(wi, rows)
        dt = time.perf_counter() - t0
        t_total += dt
        tok_total += len(rows)
        if dt < seconds / 10 and n < wi.s:
            n = min(wi.s, n * 2)
        i += 1
    return {"value": round(tok_total / t_total, 2), "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{tok_total} tokens of {w.name} over {i} oracle calls "
                      f"(full batch builder + fp64 fused per token), {t_total:.1f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = make_workload(args.workload, 0, args.chunk, args.scale, args.bs)
    # size each step's token sample so the whole run stays within ~2 minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows_n = 1
    t0 = time.perf_counter()
    oracle_step(w, np.arange(1))
    per_tok = max(time.perf_counter() - t0, 1e-6)
    rows_n = int(max(1, min(w.s, budget / per_tok)))
    rows = np.arange(rows_n)
    for _ in range(args.warmup):
        oracle_step(w, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, rows)
    el = time.perf_counter() - t0
    value = args.steps * rows_n / el
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "tokens_per_step": rows_n,
                   "step": "oracle batch builder + fp64 fused per token on a token sample"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": f"{rows_n} of {w.s} tokens per step, {args.steps} steps"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill_gate_up",
                    choices=["decode_qkv", "prefill_gate_up", "skewed_down_proj", "lm_head_decode", "lm_head_pruned",
                             "tiny", "embedding", "embedding_transposed"])
    ap.add_argument("--chunk", type=int, default=128, help="chunk size of skewed_down_proj")
    ap.add_argument("--scale", type=float, default=1.0, help="token scale of the prefill workloads")
    ap.add_argument("--bs", type=int, default=0, help="requests of the decode workloads (0 = default)")
    ap.add_argument("--sets", type=int, default=0, help="input sets to rotate (0 = enough to defeat L2)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the other configurations")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--soak-seconds", type=float, default=1.0,
                    help="seconds of untimed steps before the timed region, under the clock sampler")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
