#!/usr/bin/env python3
"""Benchmark: absorbed MLA decode on B300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]
    python bench.py --projections   (rows a1/a8: absorb_q and out_proj alone)

A step is one decode step of the hot path over one synthetic batch: the
paged absorbed attention kernel and, when the batch is cut across SMs, its
log-sum-exp combine kernel (both launched by one mla_decode_attn call).  The
K timed steps are captured into one CUDA graph and replayed once.  The
default workload is 64 sequences x 128 heads x 4096 cached positions
(d_c = 512, d_r = 64, bf16, pages of 64 rows at a random permutation of the
pool).  Inputs are generated on the device before timing; the 302 MB cache is
larger than the 126 MB L2, so no flush is inserted between steps.

value   : whole-job TFLOP/s = 2*(d_c+d_r) + 2*d_c FLOPs per (query, head,
          visible cached row), summed over all ranks, / max-over-ranks time.
e2e     : the same metric through the same call with the step's inputs
          (q_lat, q_pe, seq_lens, page_table) copied from pinned host memory
          and the result (o, lse) copied back, inside the timed region.
roofline: the attention kernel alone, timed with CUDA events recorded around
          it by the library (mla_set_decode_events), against the measured HBM
          bandwidth (cache bytes) or bf16 tensor peak, whichever bound is
          slower for this workload.

With N > 1 (torchrun) every rank runs an independent replica on its own GPU
(the decode path has no exchange step): weak scaling, no collective on the
data path.  --impl reference times the fp64 CPU oracle on the host cores on
a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_latent_kv_71_b300 import workloads  # noqa: E402

METRIC = ("MLA absorbed decode TFLOP/s + cache GB/s, % of B300 roofline "
          "(B=64,H=128,L=4096)")
DEFAULT_WORKLOAD = "decode_b64_h128_l4096"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def work_of(case: workloads.DecodeCase):
    """(FLOPs, cache bytes) of one decode step: per visible (query, head, row)
    2*(d_c+d_r) + 2*d_c FLOPs; every cached row (d_c + d_r bf16) read once."""
    B, T, H, d_c = case.q_lat.shape
    d_r = case.q_pe.shape[3]
    lens = case.seq_lens.cpu().tolist()
    rows = 0
    for n in lens:
        for t in range(T):
            rows += max(0, n - (T - 1 - t)) if case.causal else n
    flops = rows * H * (2 * (d_c + d_r) + 2 * d_c)
    cache_bytes = sum(lens) * (d_c + d_r) * case.pool.element_size()
    return flops, cache_bytes


class ClockSampler:
    """SM clock and throttle reasons sampled during the timed region: through
    NVML when the Python binding is importable, else by an nvidia-smi process
    polling every 50 ms."""

    REASONS = {
        "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
        "hw_power_brake_slowdown": 0x80, "sw_power_cap": 0x4,
    }

    def __init__(self, device_index: int):
        self.samples, self.reasons = [], set()
        self.err = ""
        self.max_mhz = None
        self.mode = None
        self.device_index = device_index
        try:
            import pynvml
            pynvml.nvmlInit()
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
            try:
                self.h = pynvml.nvmlDeviceGetHandleByUUID(uuid)
            except Exception:
                self.h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.nv = pynvml
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:
            self.err = repr(e)
            import shutil
            if shutil.which("nvidia-smi"):
                self.mode = "smi"
        self._stop = threading.Event()

    def _run_nvml(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
                mask = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for name, bit in self.REASONS.items():
                    if mask & bit:
                        self.reasons.add(name)
            except Exception as e:
                self.err = repr(e)
            time.sleep(0.002)

    def __enter__(self):
        if self.mode == "nvml":
            self.t = threading.Thread(target=self._run_nvml, daemon=True)
            self.t.start()
        elif self.mode == "smi":
            import subprocess
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            idx = vis.split(",")[self.device_index] if vis else str(self.device_index)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", idx, "--query-gpu=clocks.sm,clocks.max.sm,"
                 "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # let the first sample land before the timed work starts
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self.mode == "nvml":
            self.t.join()
        elif self.mode == "smi":
            time.sleep(0.1)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            for line in out.splitlines():
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 3:
                    continue
                try:
                    self.samples.append(float(parts[0]))
                    self.max_mhz = float(parts[1])
                    mask = int(parts[2], 16)
                except ValueError:
                    continue
                for name, bit in self.REASONS.items():
                    if mask & bit:
                        self.reasons.add(name)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "note": "no clock samples: " + self.err}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": self.mode}


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
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


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


def traffic_record(kernel_src_sha: str, workload: str):
    """DRAM bytes per launch of the attention kernel from a committed ncu
    capture, or None if absent, taken on a different kernel source, or on a
    different workload."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_src_sha256") != kernel_src_sha:
        return None, "stale"
    if d.get("workload") != workload:
        return None, "other workload"
    return d.get("dram_bytes_per_launch"), d.get("source")


def code_only(src: str) -> str:
    """C++ source without comments and blank lines (the traffic record is
    keyed by the code, so that editing a comment does not void it)."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_sha() -> str:
    h = hashlib.sha256()
    for name in ("decode_bf16.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "mla_latent_kv_71_b300", "csrc", name)) as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()


def compact_sample(case: workloads.DecodeCase, nb: int):
    """First nb sequences of a case with their pages gathered into a small
    CPU pool (for timing the CPU oracle without copying the whole cache)."""
    table = case.page_table[:nb]
    used = table[table >= 0].long()
    pool = case.pool[used.to(case.pool.device)].cpu()
    new_table = torch.full_like(table.cpu(), -1)
    new_table[(table >= 0).cpu()] = torch.arange(used.numel(), dtype=torch.int32)
    return workloads.DecodeCase(case.q_lat[:nb].cpu(), case.q_pe[:nb].cpu(), pool, new_table,
                                case.seq_lens[:nb].cpu(), case.scale, case.causal)


def time_oracle(sample: workloads.DecodeCase):
    import oracle
    lib = oracle.load()
    t0 = time.perf_counter()
    oracle.decode_attn(sample.q_lat, sample.q_pe, sample.pool, sample.page_table,
                       sample.seq_lens, sample.scale, causal=sample.causal, lib=lib)
    return time.perf_counter() - t0


def oracle_threads() -> int:
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n and n.isdigit() else (os.cpu_count() or 1)


def cpu_baseline(case: workloads.DecodeCase, budget_s: float = 15.0):
    """The oracle as it stands on the host cores, on the first sequences of
    the workload (calibrated to about budget_s of CPU work)."""
    B = case.q_lat.shape[0]
    one = compact_sample(case, 1)
    t1 = time_oracle(one)
    nb = max(1, min(B, int(budget_s / max(t1, 1e-3))))
    sample = compact_sample(case, nb) if nb > 1 else one
    t = time_oracle(sample) if nb > 1 else t1
    flops, _ = work_of(sample)
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": oracle_threads(),
            "kind": "oracle",
            "sample": f"first {nb} of {B} sequences (all heads, all positions), fp64, "
                      f"{t:.2f} s"}


# ------------------------------------------------------------------ our arm

def run_ours(args, rank, world, local):
    from mla_latent_kv_71_b300 import mla
    dev = torch.device("cuda", local)
    case = workloads.make_workload(args.workload, device=dev)
    B, T, H, d_c = case.q_lat.shape
    flops, cache_bytes = work_of(case)
    o = torch.empty_like(case.q_lat)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, mla.decode_workspace_size(B, T, H, d_c, case.q_lat.dtype)),
                     dtype=torch.uint8, device=dev)
    lens_host = case.seq_lens.cpu()

    def step():
        mla.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table, case.seq_lens,
                        case.scale, causal=case.causal, o=o, lse=lse, workspace=ws,
                        seq_lens_host=lens_host)

    # kernels per step: attention + combine when the plan cuts a sequence
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)

    # The K timed steps are captured once into a CUDA graph and replayed, as
    # a serving loop would run its decode step: the GPU then runs the kernels
    # back to back instead of waiting on the host's per-call work.  Events the
    # library records around each step's attention kernel are captured too.
    ev_attn = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    for a, b in ev_attn:  # torch creates events lazily: record once so the handles exist
        a.record(s)
        b.record(s)
    torch.cuda.synchronize(dev)
    # Two graphs of the K steps: the timed one as a serving loop would run
    # it, and a second with the library's events recorded around each step's
    # attention kernel (the per-kernel figure; event nodes between the
    # kernels would otherwise sit inside the timed steps).
    graph = torch.cuda.CUDAGraph()
    launches0 = mla.launch_count()
    with torch.cuda.graph(graph, stream=s):
        for i in range(args.steps):
            step()
    launches = mla.launch_count() - launches0  # kernels one replay launches
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=s):
        for i in range(args.steps):
            mla.set_decode_events(*ev_attn[i])
            step()
    mla.set_decode_events(None, None)
    with torch.cuda.stream(s):
        graph.replay()  # untimed: first replays of the graphs
        graph_ev.replay()
    torch.cuda.synchronize(dev)
    # The graph of K steps is replayed R times back to back inside the
    # clock-sampled region (R so that the region lasts about half a second
    # and the clock samples fall under load), each replay between its own
    # CUDA events; the step time is the median replay's time over K.
    with torch.cuda.stream(s):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s)
        graph.replay()
        t1.record(s)
    torch.cuda.synchronize(dev)
    one_ms = max(t0.elapsed_time(t1), 1e-3)
    replays = int(max(5, min(2000, 500.0 / one_ms)))
    ev_rep = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(replays)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    with clocks, torch.cuda.stream(s):
        for a, b in ev_rep:
            a.record(s)
            graph.replay()
            b.record(s)
        torch.cuda.synchronize(dev)
    barrier(world)
    rep_ms = [a.elapsed_time(b) for a, b in ev_rep]
    step_ms = statistics.median(rep_ms) / args.steps
    step_ms = max_over_ranks(step_ms, world)
    # the attention kernel's own time: the median over the K steps of the
    # events around it, from three replays of the events graph
    attn_samples = []
    for _ in range(3):
        with torch.cuda.stream(s):
            graph_ev.replay()
        torch.cuda.synchronize(dev)
        attn_samples += [a.elapsed_time(b) for a, b in ev_attn]
    attn_ms = statistics.median(attn_samples)
    code, detail = mla.get_device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} detail {detail:#x}")

    # ---- end to end through the same call: every step uploads its inputs
    # from pinned host memory and downloads o and lse, inside the timed
    # region.  Two device buffer sets and one stream each for uploads,
    # kernels and downloads let step k's kernels overlap step k+1's upload
    # and step k-1's download, as a serving loop would pipeline them; events
    # keep a buffer from being overwritten while still in use.
    names = (case.q_lat, case.q_pe, case.seq_lens, case.page_table)
    h_in = [t.cpu().pin_memory() for t in names]
    h_out = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(),
              torch.empty(lse.shape, dtype=lse.dtype).pin_memory()) for _ in range(2)]
    d_in = [[torch.empty_like(t) for t in names] for _ in range(2)]
    d_out = [(torch.empty_like(o), torch.empty_like(lse)) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()
    s_up, s_dn = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]   # buffer b's inputs are on the device
    ev_run = [torch.cuda.Event() for _ in range(2)]  # buffer b's kernels are done
    ev_dn = [torch.cuda.Event() for _ in range(2)]   # buffer b's outputs are on the host

    def e2e_steps(n):
        for k in range(n):
            b = k % 2
            s_up.wait_event(ev_run[b])  # the kernels of step k-2 no longer read buffer b
            with torch.cuda.stream(s_up):
                for d_t, h_t in zip(d_in[b], h_in):
                    d_t.copy_(h_t, non_blocking=True)
            ev_up[b].record(s_up)
            s.wait_event(ev_up[b])
            s.wait_event(ev_dn[b])  # step k-2's outputs have left buffer b
            q, pe, lens, table = d_in[b]
            mla.decode_attn(q, pe, case.pool, table, lens, case.scale, causal=case.causal,
                            o=d_out[b][0], lse=d_out[b][1], workspace=ws, seq_lens_host=h_in[2],
                            stream=s)
            ev_run[b].record(s)
            s_dn.wait_event(ev_run[b])
            with torch.cuda.stream(s_dn):
                h_out[b][0].copy_(d_out[b][0], non_blocking=True)
                h_out[b][1].copy_(d_out[b][1], non_blocking=True)
            ev_dn[b].record(s_dn)

    for ev in ev_run + ev_dn:
        ev.record(s)
    e2e_steps(max(3, args.warmup))
    torch.cuda.synchronize(dev)
    e_steps = max(50, min(args.steps * 10, 400))
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    h0 = time.perf_counter()
    e2e_steps(e_steps)
    host_ms = (time.perf_counter() - h0) * 1e3 / e_steps  # the host's enqueue time per step
    s_dn.wait_event(ev_run[(e_steps - 1) % 2])
    e1.record(s_dn)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, world)
    if not torch.equal(h_out[(e_steps - 1) % 2][0], o.cpu()):
        raise RuntimeError("end-to-end output differs from the timed step's")

    pk, pk_kind = peaks()
    t_flop = flops / (pk["bf16_tflops"] * 1e12)
    t_hbm = cache_bytes / (pk["hbm_gbs"] * 1e9)
    attn_s = attn_ms * 1e-3
    traffic, _ = traffic_record(kernel_sha(), args.workload)
    if t_hbm >= t_flop:
        roof = {"bound": "hbm", "achieved": cache_bytes / attn_s / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / attn_s / 1e12, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = traffic
    roof["kernel"] = "decode_bf16_kernel"
    roof["peak_kind"] = f"{pk_kind} (burst)"
    roof["algorithmic_bytes_per_launch"] = cache_bytes
    roof["algorithmic_flops_per_launch"] = flops
    roof["attn_us"] = attn_ms * 1e3
    roof["roofline_us"] = max(t_flop, t_hbm) * 1e6
    roof["pct_roofline_attn"] = max(t_flop, t_hbm) / attn_s
    roof["pct_roofline_step"] = max(t_flop, t_hbm) / (step_ms * 1e-3)
    roof["tensor_frac_attn"] = flops / attn_s / 1e12 / pk["bf16_tflops"]

    value = flops * world / (step_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "T": T, "H": H, "d_c": d_c,
                   "d_r": case.q_pe.shape[3], "page": case.pool.shape[1],
                   "cached_positions": int(case.seq_lens.sum()),
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (cache %.0f MB > 126 MB); no flush" %
                         (cache_bytes / 1e6)},
        "cache_gbs": cache_bytes * world / (step_ms * 1e-3) / 1e9,
        "pct_roofline": max(t_flop, t_hbm) / (step_ms * 1e-3),
        "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "steps": e_steps, "host_enqueue_ms_per_step": host_ms, "pipelining": "uploads, kernels and downloads on three streams, "
                                                "two device buffer sets"},
        "timing": {"replays": replays, "steps_per_replay": args.steps,
                   "replay_ms_min": min(rep_ms), "replay_ms_max": max(rep_ms)},
        "gpu_launches": launches,
        "roofline": roof,
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case)
    return line


# ------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    """The fp64 oracle on the host cores, on a bounded sample per step."""
    spec = workloads.WORKLOADS[args.workload]
    full = workloads.make_workload(args.workload, device="cpu", B=1)
    t1 = time_oracle(full)
    B = spec["B"]
    nb = max(1, min(B, int(args.ref_step_s / max(t1, 1e-3))))
    sample = workloads.make_workload(args.workload, device="cpu", B=nb)
    flops, _ = work_of(sample)
    for _ in range(args.warmup if args.warmup < 2 else 1):
        time_oracle(sample)
    times = [time_oracle(sample) for _ in range(args.steps)]
    t = statistics.mean(times)
    value = flops / t / 1e12
    lens = workloads.workload_lens(spec)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "T": spec["T"], "H": spec["H"],
                   "d_c": spec["d_c"], "d_r": spec["d_r"], "page": workloads.PAGE,
                   "cached_positions": int(sum(lens)), "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle_threads(),
                         "kind": "oracle",
                         "sample": f"each step: first {nb} of {B} sequences, all heads, fp64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def time_alone(fn, s, flush, steps: int, warmup: int) -> float:
    """Median device time (us) of one call of fn on stream s, L2 flushed
    before each: fn is captured once in a CUDA graph and the graph replayed,
    so the host's submission work (argument checks, tensor maps) stays
    outside the timed region, as in the decode step's timing."""
    with torch.cuda.stream(s):
        for _ in range(warmup):
            fn()
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fn()
    times = []
    with torch.cuda.stream(s):
        for _ in range(steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            graph.replay()
            b.record(s)
            b.synchronize()
            times.append(a.elapsed_time(b) * 1e3)
    return statistics.median(times)


def time_stream(fns, s, steps: int, warmup: int) -> float:
    """Per-call device time (us) of calls streamed back to back, as in a
    decode step: the calls fns, each over its own copy of the inputs (the
    copies together larger than L2, so that no call finds its weights left
    in L2 by the one before), are captured in order in one CUDA graph; the
    graph is replayed between CUDA events and the median replay time is
    divided by the number of calls.  Unlike time_alone this leaves out the
    launch of a lone graph, which a step of many kernels pays once."""
    with torch.cuda.stream(s):
        for _ in range(warmup):
            for f in fns:
                f()
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for f in fns:
            f()
    times = []
    with torch.cuda.stream(s):
        graph.replay()
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            graph.replay()
            b.record(s)
            b.synchronize()
            times.append(a.elapsed_time(b) * 1e3)
    return statistics.median(times) / len(fns)


def run_projections(args, local):
    """The query absorption (q_lat = W^UK^T q_nope) and the output projection
    (out = W^O concat_i W^UV_i o_i) at the two-token workload's sizes (64
    query rows x 128 heads, d_h 128, d_c 512, d 7168).  Each is timed two
    ways: streamed back to back over rotating copies of its inputs larger
    than L2 together (time_stream: "us", the figure the roofline fraction
    uses), and alone (time_alone: one call in a CUDA graph, L2 flushed by a
    256 MB write before each replay: "us_alone", which adds the launch of a
    lone graph).  Both are bound by their weight bytes (16.8 MB W^UK;
    16.8 MB W^UV + 235 MB W^O) against the measured HBM rate."""
    from mla_latent_kv_71_b300 import mla
    dev = torch.device("cuda", local)
    spec = workloads.WORKLOADS["mtp_b32_t2_l8192"]
    B, T, H, d_h, d_c, d = spec["B"], spec["T"], spec["H"], spec["d_h"], spec["d_c"], spec["d"]
    rows = B * T
    bf = torch.bfloat16
    w_uk, w_uv, w_o = workloads.projection_weights(H, d_h, d_c, d, seed=spec["seed"] + 4000, device=dev,
                                                   dtype=bf)
    qn = workloads.q_nope(B, T, H, d_h, seed=spec["seed"] + 3000, device=dev, dtype=bf).reshape(rows, H, d_h)
    g = torch.Generator(device=dev).manual_seed(spec["seed"] + 5000)
    o = torch.randn((rows, H, d_c), generator=g, device=dev).to(bf)
    q_lat = torch.empty((rows, H, d_c), dtype=bf, device=dev)
    v_tmp = torch.empty((rows, H * d_h), dtype=bf, device=dev)
    out = torch.empty((rows, d), dtype=bf, device=dev)
    ws = torch.zeros(max(1, mla.out_proj_workspace_size(rows, H, d_h, d, bf)), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)

    def timed(fn):
        return time_alone(fn, s, flush, args.steps, args.warmup)

    # rotating copies: 8 x 27 MB for the query absorption, 2 x 265 MB for
    # the output projection
    absorb_sets = [(qn.clone(), w_uk.clone(), torch.empty_like(q_lat)) for _ in range(8)]
    out_sets = [(o.clone(), w_uv.clone(), w_o.clone(), torch.empty_like(v_tmp), torch.empty_like(out),
                 torch.zeros_like(ws)) for _ in range(2)]
    pk, pk_kind = peaks()
    res = {"metric": "MLA decode projections, weight GB/s vs measured HBM", "rows": rows, "H": H,
           "d_h": d_h, "d_c": d_c, "d": d, "dtype": "bf16", "data": "synthetic",
           "timing": (f"us: median of {args.steps} replays of a graph of calls back to back over "
                      f"rotating input copies larger than L2, per call; us_alone: median of "
                      f"{args.steps} graph replays of one call, L2 flushed before each"),
           "peak_hbm_gbs": pk["hbm_gbs"], "peak_kind": pk_kind}
    for name, fn, fns, wbytes, other, flops in (
            ("absorb_q", lambda: mla.absorb_q(qn, w_uk, q_lat, stream=s),
             [(lambda a=a: mla.absorb_q(a[0], a[1], a[2], stream=s)) for a in absorb_sets],
             w_uk.numel() * 2, (qn.numel() + q_lat.numel()) * 2, 2 * rows * H * d_h * d_c),
            ("out_proj", lambda: mla.out_proj(o, w_uv, w_o, v_tmp, out, ws, stream=s),
             [(lambda a=a: mla.out_proj(*a, stream=s)) for a in out_sets],
             (w_uv.numel() + w_o.numel()) * 2, (o.numel() + 2 * v_tmp.numel() + out.numel()) * 2,
             2 * rows * H * d_h * d_c + 2 * rows * d * H * d_h)):
        us = time_stream(fns, s, args.steps, args.warmup)
        us_alone = timed(fn)
        gbs = (wbytes + other) / (us * 1e-6) / 1e9
        res[name] = {"us": us, "us_alone": us_alone, "weight_bytes": wbytes, "bytes": wbytes + other,
                     "gbs": gbs, "frac_hbm": gbs / pk["hbm_gbs"], "tflops": flops / (us * 1e-6) / 1e12}
    code, detail = mla.get_device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} detail {detail:#x}")
    return res


def run_prefill(args, local):
    """Training-form prefill (row f3) of one 4096-token sequence with the
    DeepSeek-shaped attention (128 heads, d_h 128, d_c 512, d_r 64, d 7168),
    each call timed alone like --projections (median of graph replays, L2
    flushed before each).  The attention is bound by the tensor cores: its
    work is the causal count of (query, key, head) triples x 640 FLOPs
    (2 (d_h + d_r) for the score, 2 d_h for the weighted sum), against the
    bf16 tensor peak.  The expansion (W^UK c, W^UV c) and W^O are GEMMs."""
    from mla_latent_kv_71_b300 import mla
    dev = torch.device("cuda", local)
    B, L, H, d_h, d_c, d_r, d = 1, 4096, 128, 128, 512, 64, 7168
    case = workloads.prefill_case(B, L, H, d=d, seed=111, device=dev)
    rows = B * L
    bf = torch.bfloat16
    k = torch.empty((rows, H, d_h), dtype=bf, device=dev)
    v = torch.empty_like(k)
    u = torch.empty_like(k)
    lse = torch.empty((rows, H), dtype=torch.float32, device=dev)
    out = torch.empty((rows, d), dtype=bf, device=dev)
    need = int(mla.library().mla_prefill_workspace_size(rows, H, d_h, d, mla.MLA_BF16))
    ws = torch.zeros(max(1, need), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)
    pk, pk_kind = peaks()
    triples = H * B * L * (L + 1) // 2
    attn_flops = triples * (2 * (d_h + d_r) + 2 * d_h)
    res = {"metric": "MLA training-form prefill attention TFLOP/s vs bf16 tensor peak",
           "workload": f"prefill_b{B}_l{L}_h{H}", "B": B, "L": L, "H": H, "d_h": d_h, "d_c": d_c,
           "d_r": d_r, "d": d, "causal": True, "dtype": "bf16", "data": "synthetic",
           "timing": f"median of {args.steps} graph replays of one call, L2 flushed before each",
           "peak_bf16_tflops": pk["bf16_tflops"], "peak_kind": pk_kind}
    us = time_alone(lambda: mla.prefill_expand(case.kv, case.w_uk, case.w_uv, k, v, stream=s), s, flush,
                    args.steps, args.warmup)
    fl = 2 * 2 * rows * H * d_h * d_c
    res["expand"] = {"us": us, "flops": fl, "tflops": fl / (us * 1e-6) / 1e12,
                     "frac_tensor": fl / (us * 1e-6) / 1e12 / pk["bf16_tflops"]}
    us = time_alone(lambda: mla.prefill_attn(case.q_nope, case.q_pe, k, case.kv, v, L, case.scale, True,
                                             u, lse, stream=s), s, flush, args.steps, args.warmup)
    tf = attn_flops / (us * 1e-6) / 1e12
    res["attention"] = {"us": us, "flops": attn_flops, "tflops": tf, "frac_tensor": tf / pk["bf16_tflops"]}
    us = time_alone(lambda: mla.prefill_out(u, case.w_o, out, ws, stream=s), s, flush, args.steps,
                    args.warmup)
    fl = 2 * rows * d * H * d_h
    res["out"] = {"us": us, "flops": fl, "tflops": fl / (us * 1e-6) / 1e12,
                  "frac_tensor": fl / (us * 1e-6) / 1e12 / pk["bf16_tflops"]}
    code, detail = mla.get_device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} detail {detail:#x}")
    return res


def run_prologue(args, local):
    """The steps before the decode, each timed like --projections (streamed
    over rotating input copies, and alone): the
    cache write of one new token per sequence of the headline batch (64
    tokens at position 4096: c = W^DKV h and k^R = RoPE(W^KR h) from d = 7168
    into the paged pool) and the query of those tokens (W^Q c^Q from the
    1536-wide compressed query to 128 heads x [128 content ; 64 RoPE],
    RoPE part rotated).  Both are bound by their weight bytes (8.3 MB and
    75.5 MB) against the measured HBM rate."""
    from mla_latent_kv_71_b300 import mla
    dev = torch.device("cuda", local)
    B, pos, d, d_c, d_r, H, d_h, d_q = 64, 4096, 7168, 512, 64, 128, 128, 1536
    bf = torch.bfloat16
    g = torch.Generator(device=dev).manual_seed(6000)
    w_dkv = workloads.weight((d_c, d), d, g, dev, bf)
    w_kr = workloads.weight((d_r, d), d, g, dev, bf)
    w_q = workloads.weight((H * (d_h + d_r), d_q), d_q, g, dev, bf)
    h = torch.randn((B, d), generator=g, device=dev).to(bf)
    c_q = torch.randn((B, d_q), generator=g, device=dev).to(bf)
    seq_ids = torch.arange(B, dtype=torch.int32, device=dev)
    positions = torch.full((B,), pos, dtype=torch.int32, device=dev)
    max_pages = pos // workloads.PAGE + 1
    table = torch.full((B, max_pages), -1, dtype=torch.int32, device=dev)
    table[:, pos // workloads.PAGE] = torch.arange(B, dtype=torch.int32, device=dev)
    pool = torch.zeros((B, workloads.PAGE, d_c + d_r), dtype=bf, device=dev)
    ws_kv = torch.zeros(max(1, mla.cache_append_workspace_size(B, d, d_c, bf)), dtype=torch.uint8,
                        device=dev)
    ws_q = torch.zeros(max(1, mla.project_q_workspace_size(B, H, d_h, d_r, d_q, bf)),
                       dtype=torch.uint8, device=dev)
    q_nope = torch.empty((B, H, d_h), dtype=bf, device=dev)
    q_pe = torch.empty((B, H, d_r), dtype=bf, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)

    def timed(fn):
        return time_alone(fn, s, flush, args.steps, args.warmup)

    # rotating copies: 16 x 8.3 MB of W^DKV, W^KR; 3 x 75.5 MB of W^Q
    kv_sets = [(w_dkv.clone(), w_kr.clone(), torch.zeros_like(ws_kv)) for _ in range(16)]
    q_sets = [(w_q.clone(), torch.zeros_like(ws_q)) for _ in range(3)]
    pk, pk_kind = peaks()
    res = {"metric": "MLA decode prologue, GB/s vs measured HBM", "tokens": B, "position": pos,
           "d": d, "d_c": d_c, "d_r": d_r, "H": H, "d_h": d_h, "d_q": d_q, "dtype": "bf16",
           "data": "synthetic",
           "timing": (f"us: median of {args.steps} replays of a graph of calls back to back over "
                      f"rotating weight copies larger than L2, per call; us_alone: median of "
                      f"{args.steps} graph replays of one call, L2 flushed before each"),
           "peak_hbm_gbs": pk["hbm_gbs"], "peak_kind": pk_kind}
    for name, fn, fns, wbytes, other, flops, launches in (
            ("cache_append",
             lambda: mla.cache_append(h, w_dkv, w_kr, seq_ids, positions, table, pool, workspace=ws_kv,
                                      stream=s),
             [(lambda a=a: mla.cache_append(h, a[0], a[1], seq_ids, positions, table, pool, workspace=a[2],
                                             stream=s)) for a in kv_sets],
             (w_dkv.numel() + w_kr.numel()) * 2, h.numel() * 2 + B * (d_c + d_r) * 2,
             2 * B * (d_c + d_r) * d, 2),
            ("project_q",
             lambda: mla.project_q(c_q, w_q, positions, H, d_h, d_r, q_nope, q_pe, workspace=ws_q,
                                   stream=s),
             [(lambda a=a: mla.project_q(c_q, a[0], positions, H, d_h, d_r, q_nope, q_pe, workspace=a[1],
                                          stream=s)) for a in q_sets],
             w_q.numel() * 2, c_q.numel() * 2 + (q_nope.numel() + q_pe.numel()) * 2,
             2 * B * H * (d_h + d_r) * d_q, 2)):
        us = time_stream(fns, s, args.steps, args.warmup)
        us_alone = timed(fn)
        gbs = (wbytes + other) / (us * 1e-6) / 1e9
        res[name] = {"us": us, "us_alone": us_alone, "weight_bytes": wbytes, "bytes": wbytes + other,
                     "gbs": gbs, "frac_hbm": gbs / pk["hbm_gbs"], "tflops": flops / (us * 1e-6) / 1e12,
                     "launches_per_call": launches}
    code, detail = mla.get_device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} detail {detail:#x}")
    return res


def run_merged(args, local):
    """The output projection two ways at the two-token workload's sizes (64
    rows, 128 heads, d_h 128, d_c 512, d 7168), each timed like
    --projections: W^UV and W^O kept apart (mla_out_proj, 252 MB of
    weights) and merged ahead of time (mla_out_proj_merged, one 7168 x 65536
    matrix, 940 MB) -- the trade the pages weigh; and the query side the same
    way (W^UQ and W^UK apart, 92 MB with W^Q's RoPE rows, against the folded
    W^UK^T W^UQ, 201 MB)."""
    from mla_latent_kv_71_b300 import mla
    dev = torch.device("cuda", local)
    spec = workloads.WORKLOADS["mtp_b32_t2_l8192"]
    B, T, H, d_h, d_c, d = spec["B"], spec["T"], spec["H"], spec["d_h"], spec["d_c"], spec["d"]
    rows = B * T
    bf = torch.bfloat16
    _, w_uv, w_o = workloads.projection_weights(H, d_h, d_c, d, seed=spec["seed"] + 4000, device=dev,
                                                dtype=bf)
    g = torch.Generator(device=dev).manual_seed(spec["seed"] + 5000)
    o = torch.randn((rows, H, d_c), generator=g, device=dev).to(bf)
    w_merged = mla.fold_out_weights(w_uv, w_o)
    v_tmp = torch.empty((rows, H * d_h), dtype=bf, device=dev)
    out = torch.empty((rows, d), dtype=bf, device=dev)
    ws = torch.zeros(max(1, mla.out_proj_workspace_size(rows, H, d_h, d, bf)), dtype=torch.uint8, device=dev)
    ws_m = torch.zeros(max(1, int(mla.library().mla_out_proj_merged_workspace_size(rows, H, d_c, d, 0))),
                       dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)
    pk, pk_kind = peaks()
    res = {"metric": "MLA output projection, weights kept apart vs merged, GB/s vs measured HBM",
           "rows": rows, "H": H, "d_h": d_h, "d_c": d_c, "d": d, "dtype": "bf16", "data": "synthetic",
           "timing": f"median of {args.steps} graph replays of one call, L2 flushed before each",
           "peak_hbm_gbs": pk["hbm_gbs"], "peak_kind": pk_kind}
    for name, fn, wbytes, other, flops in (
            ("out_proj", lambda: mla.out_proj(o, w_uv, w_o, v_tmp, out, ws, stream=s),
             (w_uv.numel() + w_o.numel()) * 2, (o.numel() + 2 * v_tmp.numel() + out.numel()) * 2,
             2 * rows * H * d_h * d_c + 2 * rows * d * H * d_h),
            ("out_proj_merged", lambda: mla.out_proj_merged(o, w_merged, out, ws_m, stream=s),
             w_merged.numel() * 2, (o.numel() + out.numel()) * 2, 2 * rows * d * H * d_c)):
        us = time_alone(fn, s, flush, args.steps, args.warmup)
        gbs = (wbytes + other) / (us * 1e-6) / 1e9
        res[name] = {"us": us, "weight_bytes": wbytes, "bytes": wbytes + other, "gbs": gbs,
                     "frac_hbm": gbs / pk["hbm_gbs"], "tflops": flops / (us * 1e-6) / 1e12}
    res["merged_over_apart_time"] = res["out_proj_merged"]["us"] / res["out_proj"]["us"]
    # The query side: c^Q (1536 wide) -> q_lat, W^UQ then W^UK apart
    # (mla_project_q's content and RoPE rows, then mla_absorb_q) against the
    # folded W^UK^T W^UQ (mla_absorb_q_merged; the RoPE rows of W^Q are
    # still needed for q^R and are timed on their own here, as a project_q of
    # a W^Q with only those rows per head would cost).
    d_q, d_r = 1536, 64
    gq = torch.Generator(device=dev).manual_seed(spec["seed"] + 6000)
    w_q = workloads.weight((H * (d_h + d_r), d_q), d_q, gq, dev, bf)
    w_uk = workloads.weight((H, d_h, d_c), d_c, gq, dev, bf)
    c_q = torch.randn((rows, d_q), generator=gq, device=dev).to(bf)
    pos = torch.full((rows,), 4096, dtype=torch.int32, device=dev)
    wq_m = mla.fold_q_weights(w_uk, w_q, d_r)
    q_nope = torch.empty((rows, H, d_h), dtype=bf, device=dev)
    q_pe = torch.empty((rows, H, d_r), dtype=bf, device=dev)
    q_lat = torch.empty((rows, H, d_c), dtype=bf, device=dev)
    ws_q = torch.zeros(max(1, mla.project_q_workspace_size(rows, H, d_h, d_r, d_q)), dtype=torch.uint8,
                       device=dev)
    t_pq = time_alone(lambda: mla.project_q(c_q, w_q, pos, H, d_h, d_r, q_nope, q_pe, workspace=ws_q,
                                            stream=s), s, flush, args.steps, args.warmup)
    t_ab = time_alone(lambda: mla.absorb_q(q_nope, w_uk, q_lat.view(rows, H, d_c), stream=s), s, flush,
                      args.steps, args.warmup)
    t_m = time_alone(lambda: mla.absorb_q_merged(c_q, wq_m, q_lat, stream=s), s, flush, args.steps,
                     args.warmup)
    apart_w = (w_q.numel() + w_uk.numel()) * 2
    merged_w = wq_m.numel() * 2
    res["query_apart"] = {"us": t_pq + t_ab, "project_q_us": t_pq, "absorb_q_us": t_ab,
                          "weight_bytes": apart_w, "gbs": apart_w / ((t_pq + t_ab) * 1e-6) / 1e9}
    res["query_merged_content"] = {"us": t_m, "weight_bytes": merged_w,
                                   "gbs": merged_w / (t_m * 1e-6) / 1e9,
                                   "frac_hbm": merged_w / (t_m * 1e-6) / 1e9 / pk["hbm_gbs"],
                                   "note": "content part only; q^R still needs the RoPE rows of W^Q"}
    res["query_merged_over_apart_time"] = t_m / (t_pq + t_ab)
    code, detail = mla.get_device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} detail {detail:#x}")
    return res


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--projections", action="store_true",
                    help="time mla_absorb_q and mla_out_proj alone (rows a1/a8)")
    ap.add_argument("--prologue", action="store_true",
                    help="time mla_cache_append and mla_project_q alone (the cache write before the path)")
    ap.add_argument("--merged", action="store_true",
                    help="time mla_out_proj against mla_out_proj_merged (W^O W^UV merged ahead of time)")
    ap.add_argument("--prefill", action="store_true",
                    help="time the training-form prefill (expansion, causal attention, W^O) of 4096 tokens")
    ap.add_argument("--ref-step-s", type=float, default=5.0,
                    help="reference arm: CPU seconds per step (sample size)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank, world, local = dist_setup()
    if args.projections:
        if rank == 0:
            print(json.dumps(run_projections(args, local)), flush=True)
        return
    if args.prologue:
        if rank == 0:
            print(json.dumps(run_prologue(args, local)), flush=True)
        return
    if args.merged:
        if rank == 0:
            print(json.dumps(run_merged(args, local)), flush=True)
        return
    if args.prefill:
        if rank == 0:
            print(json.dumps(run_prefill(args, local)), flush=True)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    line = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
