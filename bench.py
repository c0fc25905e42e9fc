#!/usr/bin/env python
"""Fused GQA attention forward benchmark on GB300.

One step = one launch of the fused attention forward over the long causal GQA
prefill workload (B=1, Hq=32, Hkv=8, N=32768, D=128, bf16) with inputs
resident in HBM.  Prints one JSON line (rank 0):
  value      TFLOP/s over all ranks, FLOPs counted 2*B*Hq*N^2*D (causal);
  roofline   the kernel's achieved TFLOP/s against the measured bf16 peak;
  e2e        the same metric with host->device input copies and the
             device->host read of O and LSE inside the timed region;
  cpu_baseline  the float64 oracle timed on the host cores on a row sample.
``--all`` prints that line first and then one line for each of the other
benchmarked workloads (the short and L2-resident ones timed both with L2
flushed between launches, which gives ``value``, and warm).
``--impl reference`` times the float64 oracle alone (CPU) on the same metric.
Under torchrun the (batch, kv head) groups of the problem are split into
contiguous ranges, one per rank, with no collective on the data path: by
default the job is a batch of one workload per rank (weak scaling);
``--partition strong`` splits the groups of one workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gqa_attention_forward_gb300 import workloads  # noqa: E402

METRIC = "attention fwd TFLOP/s (causal FLOPs) on 1 GB300; % of dense FP16/BF16 peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "long_prefill_causal_gqa_bf16_n32768"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(workloads.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--graph", action="store_true",
                    help="time replays of a CUDA graph holding one step (launch-overhead path)")
    ap.add_argument("--all", action="store_true",
                    help="after the headline line, one line for each workload in ALL_WORKLOADS")
    ap.add_argument("--partition", choices=["weak", "strong"], default="weak",
                    help="weak: each rank takes the groups of its own batch entries of a batch "
                         "that grows with the ranks; strong: the ranks split one workload")
    ap.add_argument("--item-order", type=int, choices=[0, 1], default=None,
                    help="work-item order of the persistent kernel (library default if unset)")
    ap.add_argument("--launch-only", type=int, default=0, metavar="N",
                    help="only N launches of the workload, each after a 256 MB L2 flush, and no "
                         "output (a target for ncu: -s N-1 -c 1 captures the last launch)")
    return ap.parse_args()


# the headline workload first, then the other configurations and next-step workloads
ALL_WORKLOADS = [DEFAULT_WORKLOAD, "tiny_causal_gqa_f16", "pages_shape_causal_gqa_f16",
                 "noncausal_gqa_bf16_n4096", "tail_stress_causal_gqa_bf16_n2000",
                 "chunked_prefill_causal_gqa_bf16_q4096_k32768", "decode_gqa_bf16_b1_q1_k32768",
                 "decode_gqa_bf16_b16_q1_k8192", "short_chunk_gqa_bf16_q16_k32768",
                 "noncausal_gqa_bf16_n4096_split", "chunked_prefill_causal_gqa_bf16_q4096_k32768_split"]
L2_BYTES = 126 * 2 ** 20  # GB300 L2 (129 MB as the device reports it)
FLUSH_BYTES = 256 * 2 ** 20


def group_range(total: int, world: int, rank: int):
    """Contiguous range [g0, g1) of `total` (batch, kv head) groups owned by `rank`:
    the ranges of ranks 0..world-1 cover every group exactly once, in order, and
    differ in size by at most one."""
    base, extra = divmod(total, world)
    g0 = rank * base + min(rank, extra)
    return g0, g0 + base + (1 if rank < extra else 0)


def slice_groups(w, x: dict, g0: int, g1: int) -> dict:
    """The inputs of groups [g0, g1) of workload w: a (b, kv head) group's G query
    heads, its keys and its values are contiguous in [B, H, N, D], so a group range
    is a plain slice of each tensor, laid out as a problem with B = g1 - g0, Hq = G
    and Hkv = 1."""
    G = w.Hq // w.Hkv
    return {"q": x["q"].reshape(w.B * w.Hkv, G, w.N, w.D)[g0:g1],
            "k": x["k"].reshape(w.B * w.Hkv, 1, w.n_keys, w.D)[g0:g1],
            "v": x["v"].reshape(w.B * w.Hkv, 1, w.n_keys, w.D)[g0:g1]}


def rank_problem(w, partition: str, world: int, rank: int):
    """(sub-workload, inputs, global FLOPs per step) of this rank.

    weak: the job is a batch of `world` copies of w; rank r's groups are those of
    its own copy, drawn from seed w.seed + r.  strong: the job is w itself; rank r
    takes group_range(B*Hkv, world, r) of it (possibly none)."""
    if partition == "weak" or world == 1:
        seed = w.seed + rank
        return w, workloads.make_inputs(w, seed=seed), w.flops * world
    total = w.B * w.Hkv
    g0, g1 = group_range(total, world, rank)
    sub = w.with_(name=w.name, B=g1 - g0, Hq=w.Hq // w.Hkv, Hkv=1)
    return sub, slice_groups(w, workloads.make_inputs(w), g0, g1), w.flops


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(x: float, device=None) -> float:
    """The largest of the ranks' values (every rank gets it); x itself on one rank."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step_per_rank: float, steps: int, world: int, max_ms: float) -> float:
    """Units all ranks processed over the slowest rank's time (weak scaling)."""
    return world * flops_per_step_per_rank * steps / (max_ms / 1e3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ CPU oracle
def row_flops(w, rows: np.ndarray) -> float:
    """Counted FLOPs of the selected output rows: 4*D per allowed key (query row i
    of a causal block of N rows over Nk keys sees i + Nk - N + 1 keys)."""
    i = rows % w.N
    keys = (i + w.n_keys - w.N + 1) if w.causal else np.full_like(i, w.n_keys)
    return float(4.0 * w.D * keys.sum())


class OracleSampler:
    """Times the float64 oracle on random output rows of a workload."""

    def __init__(self, w, seed: int = 4242):
        import oracle

        self.oracle = oracle
        self.w = w
        x = workloads.make_inputs(w)
        self.q = x["q"].reshape(-1, w.D)
        self.k = oracle.widen(x["k"], w.dtype)
        self.v = oracle.widen(x["v"], w.dtype)
        self.rng = np.random.default_rng(seed)
        self.threads = 0

    def run(self, n_rows: int):
        w = self.w
        rows = np.sort(self.rng.integers(0, w.B * w.Hq * w.N, size=n_rows))
        q_rows = self.oracle.widen(self.q[rows], w.dtype)
        t0 = time.perf_counter()
        _, _, self.threads = self.oracle.attention_rows(q_rows, rows, self.k, self.v, w.Hq, w.scale,
                                                        w.causal, Nq=w.N)
        return row_flops(w, rows), time.perf_counter() - t0


def cpu_baseline(w, seconds: float):
    s = OracleSampler(w)
    flops, secs, rows = 0.0, 0.0, 0
    n = 64
    while secs < seconds:
        f, t = s.run(n)
        flops, secs, rows = flops + f, secs + t, rows + n
        if t < seconds / 8:
            n *= 2
    return {"value": flops / secs / 1e12, "unit": UNIT, "cores": s.threads, "kind": "oracle",
            "sample": f"{rows} random output rows of {w.name} (float64 C oracle, "
                      f"{secs:.1f} s, {flops / 1e9:.1f} GFLOP counted 4*D per allowed key)"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        with open(self.tmp.name) as f:
            lines = [ln.strip() for ln in f if ln.strip()]
        os.unlink(self.tmp.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm
# the files that hold the persistent prefill kernel's code (attn_fwd_ws_kernel)
KERNEL_SOURCES = ("gqa_attention_forward_gb300/csrc/attn_fwd_ws.cuh",
                  "gqa_attention_forward_gb300/csrc/kernel_common.cuh",
                  "gqa_attention_forward_gb300/csrc/sm103_ptx.cuh")
PROFILES = os.path.join(ROOT, "profiles")


def kernel_source_digest() -> str:
    """sha256 over the kernel's source files (file name + bytes, in a fixed order)."""
    import hashlib

    files = [os.path.join(ROOT, f) for f in KERNEL_SOURCES]
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the persistent kernel from a committed ncu summary
    (any file under profiles/ whose 'workload:' line names this workload), if it
    was taken with the current kernel sources; otherwise None."""
    try:
        names = sorted(os.listdir(PROFILES))
    except OSError:
        return None
    digest = None
    for name in names:
        if not name.endswith(".md"):
            continue
        try:
            with open(os.path.join(PROFILES, name)) as fh:
                kv = dict(line.split(": ", 1) for line in fh.read().splitlines() if ": " in line)
        except OSError:
            continue
        if kv.get("workload", "").strip() != workload or "dram_bytes_per_launch" not in kv:
            continue
        digest = digest or kernel_source_digest()
        if kv.get("kernel_source_sha256", "").strip() == digest:
            return int(kv["dram_bytes_per_launch"])
    return None


def to_dev(bits, dtype, device):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16).to(device)


def algorithmic_bytes(w) -> int:
    """Q, K, V read once, O written once, LSE written once."""
    return 2 * w.B * w.D * (2 * w.Hq * w.N + 2 * w.Hkv * w.n_keys) + 4 * w.B * w.Hq * w.N


def measure(w_full, args, rank, world, device):
    """Times one workload on this rank; returns rank 0's JSON line (None elsewhere)."""
    import torch
    import torch.distributed as dist

    from gqa_attention_forward_gb300 import binding

    w, x, job_flops = rank_problem(w_full, args.partition, world, rank)
    has_work = w.B > 0
    flops_rank = w.flops if has_work else 0.0
    q, k, v = (to_dev(x[n], w.dtype, device) for n in "qkv")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    dcode = binding.ATTN_BF16 if w.dtype == "bf16" else binding.ATTN_F16
    square = w.n_keys == w.N
    decode = w.entry == "attn_fwd_decode"
    split = w.entry == "attn_fwd_kv_split"
    workspace, ws_bytes = None, 0
    if decode and has_work:
        st, ws_bytes = binding.attn_fwd_decode_workspace(w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D)
        if st != binding.ATTN_OK:
            raise binding.AttnError(st, "attn_fwd_decode_workspace")
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=device)
    if split and has_work:
        st, ws_bytes = binding.attn_fwd_kv_split_workspace(w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D,
                                                           w.causal)
        if st != binding.ATTN_OK:
            raise binding.AttnError(st, "attn_fwd_kv_split_workspace")
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)

    def launch():
        if not has_work:
            return
        s_now = torch.cuda.current_stream(device)  # the capture stream while capturing
        if decode:
            st = binding.attn_fwd_decode(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D,
                                         w.scale, w.causal, dcode, workspace, ws_bytes, s_now)
        elif split:
            st = binding.attn_fwd_kv_split(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D,
                                           w.scale, w.causal, dcode, workspace, ws_bytes, s_now)
        elif square:
            st = binding.attn_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.D, w.scale, w.causal,
                                  dcode, s_now)
        else:
            st = binding.attn_fwd_kv(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D,
                                     w.scale, w.causal, dcode, s_now)
        if st != binding.ATTN_OK:
            raise binding.AttnError(st, w.entry if (decode or split) else
                                    ("attn_fwd" if square else "attn_fwd_kv"))

    step = launch
    host_us = None
    launch()  # the first call of a variant configures the kernel (and, in graph mode,
    torch.cuda.synchronize()  # must come before the capture)
    if args.graph and has_work:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            launch()
        step = graph.replay

    for _ in range(max(args.warmup, 3)):
        step()
    if not args.graph and has_work:
        # host cost of one call through the Python binding (validation + launch), on
        # warm calls queued back to back
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(20):
            launch()
        host_us = (time.perf_counter() - t0) / 20 * 1e6
        torch.cuda.synchronize()
    st = binding.attn_last_device_error(stream)
    if st != binding.ATTN_OK:
        raise binding.AttnError(st, "warm-up")

    # Inputs and outputs that fit in L2 would stay there between launches: such a
    # workload is timed with L2 flushed before every launch (a 256 MB write outside
    # the timed events), which gives `value`, and warm as well.
    in_l2 = 2 * w_full.B * w_full.D * (w_full.Hq * w_full.N + 2 * w_full.Hkv * w_full.n_keys) <= L2_BYTES
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device) if in_l2 else None
    K = args.steps

    def timed(flushed: bool):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        clocks = ClockSampler(device.index if world == 1 else int(os.environ.get("LOCAL_RANK", 0)))
        clocks.start()
        # A spin kernel ahead of the timed launches lets the host queue all of them
        # before the GPU reaches the first, so short launches are not timed waiting
        # for the host (it runs before the first start event, outside the timing).
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(int(2000 * max(2000, 40 * K)))  # cycles: ~2 GHz x microseconds
        for i in range(K):
            if flushed:
                flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        clock_info = clocks.stop()
        if world > 1:
            dist.barrier()
        st = binding.attn_last_device_error(stream)
        if st != binding.ATTN_OK:
            raise binding.AttnError(st, "timed region")
        per_launch = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        # inputs larger than L2: first start to last end; L2-resident inputs: the sum of
        # the launches alone (warm: back to back; flushed: a flush between launches)
        span = float(np.sum(per_launch)) if in_l2 else starts[0].elapsed_time(ends[-1])
        return max_over_ranks(span, device), float(np.mean(per_launch)), clock_info

    warm = None
    if in_l2:
        warm_ms, warm_kern, _ = timed(False)
        warm = {"ms_per_step": round(warm_ms / K, 5),
                "value": round(job_flops * K / (warm_ms / 1e3) / 1e12, 2)}
        total_ms, kern_ms, clock_info = timed(True)
    else:
        total_ms, kern_ms, clock_info = timed(False)
    value = job_flops * K / (total_ms / 1e3) / 1e12
    achieved = flops_rank / (kern_ms / 1e3) / 1e12 if has_work else 0.0

    # ---- end to end: pinned host inputs -> device -> attention -> O, LSE back to host
    hq, hk, hv = (torch.from_numpy(np.ascontiguousarray(x[n]).view(np.int16)).pin_memory()
                  for n in "qkv")
    ho = torch.empty(o.numel(), dtype=torch.int16).pin_memory()
    hl = torch.empty(lse.numel(), dtype=torch.float32).pin_memory()
    dq, dk, dv = (t.view(torch.int16).view(-1) for t in (q, k, v))
    do = o.view(torch.int16).view(-1)
    E = max(1, min(args.e2e_steps, K))

    def e2e_step():
        if not has_work:
            return
        if decode or split:
            dq.copy_(hq.view(-1), non_blocking=True)
            dk.copy_(hk.view(-1), non_blocking=True)
            dv.copy_(hv.view(-1), non_blocking=True)
            step()
            ho.copy_(do, non_blocking=True)
            hl.copy_(lse.view(-1), non_blocking=True)
            return
        # one C-ABI call with host buffers: chunked copies in and out overlap the compute
        st = binding.attn_fwd_host(hq, hk, hv, ho, hl, q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N,
                                   w.n_keys, w.D, w.scale, w.causal, dcode, stream)
        if st != binding.ATTN_OK:
            raise binding.AttnError(st, "attn_fwd_host")

    e2e_step()  # first call creates the library's copy streams
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / E, device)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * 2 + hl.numel() * 4
    if rank != 0:
        return None

    algo_bytes = algorithmic_bytes(w)
    peaks, peak_src = load_peaks()
    long_region = total_ms > 1000.0
    gbs = algo_bytes / (kern_ms / 1e3) / 1e9 if has_work else 0.0
    if decode:
        # streams K and V once: bound by HBM bandwidth, not the tensor core
        roofline = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                    "traffic": profiled_traffic(w_full.name), "algorithmic_bytes": algo_bytes,
                    "peak_source": f"{peak_src} copy bandwidth",
                    "kernel": "gqa::attn_fwd_decode_kernel"
                              + (" + gqa::attn_combine_kernel" if ws_bytes else ""),
                    "kernel_ms": round(kern_ms, 5), "tflops": round(achieved, 2)}
    else:
        peak = peaks["bf16_tflops_sustained" if long_region else "bf16_tflops"]
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                    "unit": UNIT, "frac": round(achieved / peak, 4),
                    "traffic": profiled_traffic(w_full.name), "algorithmic_bytes": algo_bytes,
                    "peak_source": f"{peak_src} {'sustained' if long_region else 'burst'} bf16",
                    "kernel": "gqa::attn_fwd_ws_kernel", "kernel_ms": round(kern_ms, 5),
                    "frac_of_2250_nominal": round(achieved / 2250.0, 4),
                    # the algorithmic bytes over the same launch time, against the copy bandwidth
                    "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4)}
    if args.partition == "strong" and world > 1:
        parallelism = f"groups of one problem split over {world} ranks"
    else:
        parallelism = f"batch of {world} x the workload, (b, kv head) groups split by rank"
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True,
        "scaling": "strong" if (args.partition == "strong" and world > 1) else "weak",
        "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded i.i.d. normal, see workloads.py)",
        "config": {"workload": w_full.name, "B": w_full.B, "Hq": w_full.Hq, "Hkv": w_full.Hkv,
                   "N": w_full.N, "Nk": w_full.n_keys, "D": w_full.D, "causal": w_full.causal,
                   "flops_per_step": job_flops,
                   "flop_convention": "2*B*Hq*N^2*D causal, 4*B*Hq*N^2*D non-causal "
                                      "(N query rows over Nk keys: 4*B*Hq*D*(N*Nk - N^2/2) "
                                      "causal, 4*B*Hq*D*N*Nk non-causal)",
                   "l2": ("inputs fit in L2: flushed (256 MB write) before every timed launch"
                          if in_l2 else "inputs larger than L2 (no flush)"),
                   "parallelism": parallelism},
        "roofline": roofline,
        "e2e": {"value": round(job_flops / (e2e_ms / 1e3) / 1e12, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "path": (f"torch copies around {w.entry}" if (decode or split) else
                         "attn_fwd_host: pinned host buffers, chunked copies overlapping compute")},
        "gpu_launches": K * (2 if (decode and ws_bytes) else 1) * (1 if has_work else 0),
        "launch": {"mode": "cuda_graph_replay" if args.graph else "direct",
                   "host_us_per_call": None if host_us is None else round(host_us, 2)},
        "clocks": clock_info,
    }
    if warm is not None:
        line["l2_warm"] = warm
    return line


def run_ours(args):
    import torch
    import torch.distributed as dist

    from gqa_attention_forward_gb300 import binding

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    if args.item_order is not None:
        binding.load().attn_test_set_item_order(args.item_order)
    names = ALL_WORKLOADS if args.all else [args.workload]
    if args.all and args.workload != DEFAULT_WORKLOAD:
        names = [args.workload] + [n for n in ALL_WORKLOADS if n != args.workload]
    for i, name in enumerate(names):
        w = workloads.WORKLOADS[name]
        line = measure(w, args, rank, world, device)
        if rank == 0:
            if not args.no_cpu_baseline and world == 1:  # rank 0 at N = 1 only
                secs = args.cpu_seconds if i == 0 else min(args.cpu_seconds, 5.0)
                line["cpu_baseline"] = cpu_baseline(w, secs)
            print(json.dumps(line), flush=True)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = workloads.WORKLOADS[args.workload]
    s = OracleSampler(w)
    rows_per_step = 256 if w.causal else 64
    for _ in range(max(args.warmup, 1)):
        s.run(16)
    flops = secs = 0.0
    for _ in range(args.steps):
        f, t = s.run(rows_per_step)
        flops += f
        secs += t
    value = flops / secs / 1e12
    sample = (f"{args.steps} steps x {rows_per_step} random output rows of {w.name} "
              f"(float64 C oracle on the host cores)")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded i.i.d. normal)", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N,
                       "Nk": w.n_keys, "D": w.D, "causal": w.causal},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": s.threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_launch_only(args):
    """N launches of the workload's C entry point with L2 flushed before each."""
    import torch

    from gqa_attention_forward_gb300 import binding

    w = workloads.WORKLOADS[args.workload]
    device = torch.device("cuda", torch.cuda.current_device())
    x = workloads.make_inputs(w)
    q, k, v = (to_dev(x[n], w.dtype, device) for n in "qkv")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=device)
    s = torch.cuda.current_stream(device)
    dcode = binding.ATTN_BF16 if w.dtype == "bf16" else binding.ATTN_F16
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    ws, nbytes = None, 0
    if w.entry == "attn_fwd_kv_split":
        st, nbytes = binding.attn_fwd_kv_split_workspace(w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D, w.causal)
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    elif w.entry == "attn_fwd_decode":
        st, nbytes = binding.attn_fwd_decode_workspace(w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
    for _ in range(args.launch_only):
        flush.zero_()
        if w.entry == "attn_fwd_kv_split":
            st = binding.attn_fwd_kv_split(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D,
                                           w.scale, w.causal, dcode, ws, nbytes, s)
        elif w.entry == "attn_fwd_decode":
            st = binding.attn_fwd_decode(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D,
                                         w.scale, w.causal, dcode, ws, nbytes, s)
        else:
            st = binding.attn_fwd_kv(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D,
                                     w.scale, w.causal, dcode, s)
        if st != binding.ATTN_OK:
            raise binding.AttnError(st, w.entry)
    torch.cuda.synchronize()
    st = binding.attn_last_device_error(s)
    if st != binding.ATTN_OK:
        raise binding.AttnError(st, "launch-only")


def main():
    args = parse_args()
    if args.launch_only > 0:
        run_launch_only(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
