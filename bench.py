#!/usr/bin/env python
"""Benchmark of the paged serving-attention hot path on GB300.

A step is one pass of the whole path over one batch: the host plan (lengths,
tile, chunking, longest-first CTA queues, reduction map) and one persistent
kernel launch (page gather, attention, in-kernel merge of split rows).

  value  -- decode KV GB/s of the Llama-3-8B-shaped batch (128 requests, 32/8
            heads, page 16, KV ~ U[1,4096]) with inputs resident in HBM: KV
            bytes per step / device time per step (CUDA events around K launches
            on the launching stream; the plan is built once, as it is reused
            across layers).
  e2e    -- same metric through the C ABI from host buffers: every step plans
            from host index arrays (pinned copy inside), copies q host->device
            from pinned memory, runs, and reads o and lse back.  Steps alternate
            between two workspaces on two streams, so one step's host planning
            and copies overlap the other's kernel (the serial time is reported
            beside it).
  configs -- the other workloads (tiny, skewed long-context, causal prefill,
            shared prefix) timed the same way, each with its own unit.

`--impl reference` times the float64 CPU oracle on a bounded sample of the same
workload (the reference arm of this build).  Multi-GPU runs are independent
replicas (no collective on the data path): value sums over ranks, time is the
max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s (% of GB300 HBM peak); prefill TFLOPS (% bf16 peak); µs/batch"
PRIMARY = "llama3_8b_decode"
L2_BYTES = 129 * 2 ** 20


# ----------------------------------------------------------------------------------------------
# workload accounting
# ----------------------------------------------------------------------------------------------

def lengths(b):
    qo = b.qo_indptr.astype(np.int64)
    kv = b.kv_indptr.astype(np.int64)
    n_p = np.diff(kv)
    l_kv = np.where(n_p > 0, (n_p - 1) * b.page_size + b.last_page_len, 0)
    return np.diff(qo), l_kv


def kv_bytes(b):
    _, l_kv = lengths(b)
    elem = b.k_pages.dtype.itemsize  # 2 for bf16 bits, 1 for e4m3 codes
    return int(l_kv.sum()) * b.num_kv_heads * b.head_dim * elem * 2


def algorithmic_bytes(b):
    """KV read + q read + o/lse written + page indices read (bytes one launch must move)."""
    rows = b.total_q * b.num_qo_heads
    return kv_bytes(b) + rows * b.head_dim * 2 * 2 + rows * 4 + int(b.kv_indptr[-1]) * 4


def visible_pairs(b, window_left=-1):
    l_q, l_kv = lengths(b)
    if window_left >= 0:  # causal with a sliding window: token t sees keys p - w .. p, p = l_kv - l_q + t
        tot = 0
        for lq, lk in zip(l_q.tolist(), l_kv.tolist()):
            p = lk - lq + np.arange(lq)
            tot += int(np.clip(np.minimum(p + 1, window_left + 1), 0, None).sum())
        return tot
    tot = 0
    for lq, lk in zip(l_q.tolist(), l_kv.tolist()):
        if b.causal:
            t = np.arange(lq)
            tot += int(np.clip(lk - lq + t + 1, 0, lk).sum())
        else:
            tot += lq * lk
    return tot


def flops(b, window_left=-1):
    return 4 * b.head_dim * visible_pairs(b, window_left) * b.num_qo_heads


# ----------------------------------------------------------------------------------------------
# device helpers
# ----------------------------------------------------------------------------------------------

def to_dev(a, torch, dev):
    if a.dtype == np.uint8:  # e4m3 codes
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


class Case:
    """One batch resident on the device with its workspace and plan."""

    def __init__(self, b, torch, dev, num_ctas=0, variant=None):
        from serving_attention_plan_gb300 import binding as B
        self.variant = variant
        self.b = b
        self.torch = torch
        self.q, self.k, self.v = to_dev(b.q, torch, dev), to_dev(b.k_pages, torch, dev), to_dev(b.v_pages, torch, dev)
        self.o = torch.empty((b.total_q, b.num_qo_heads, b.head_dim), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((b.total_q, b.num_qo_heads), dtype=torch.float32, device=dev)
        self.ws = B.Workspace(b.batch_size, b.total_q, int(b.kv_indptr[-1]), b.num_qo_heads, b.num_kv_heads,
                              b.head_dim, num_ctas)
        if variant:
            variant = dict(variant)
            kv_dtype = variant.pop("kv_dtype", None)
            if kv_dtype:
                self.ws.set_kv_dtype(*kv_dtype)
            if variant:
                self.ws.set_variant(**variant)
        self.plan()

    def plan(self):
        b = self.b
        self.ws.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.page_size, b.causal)

    def run(self):
        self.ws.run(self.q, self.k, self.v, self.o, self.lse)


E2E_CONTEXTS = 3  # workspaces / streams the end-to-end steps rotate through


def time_launches(torch, fn, steps, warmup, barrier=None):
    """Device time of `steps` back-to-back calls (CUDA events on the current stream), after warm-up."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps  # ms per step


def time_launches_cold(torch, fn, steps, warmup):
    """Device time of one call with a cold L2: before each call a buffer twice the L2 size is written,
    then another one of that size is read (outside the timed events), so L2 holds none of the call's
    data and no dirty lines whose write-back the call would pay for; the CUDA events bracket the call
    alone.  Mean over `steps`."""
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device="cuda")
    clean = torch.ones(2 * L2_BYTES // 4, dtype=torch.int32, device="cuda")
    for _ in range(warmup):
        flush.fill_(1)
        clean.sum()
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    ev = []
    for i in range(steps):
        flush.fill_(i)
        clean.sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        fn()
        e1.record(s)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / steps  # ms per call


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.idx)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        loaded = [r[0] for r in rows if r[2] > 200.0] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(r[2] for r in rows)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs"), d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged since."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d:
        return None
    h = hashlib.sha256()
    for f in d.get("sources", []):
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return d.get("dram_bytes_per_launch") if h.hexdigest() == d.get("sources_sha256") else None


# ----------------------------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------------------------

def cpu_oracle_sample(b, budget_s=15.0):
    """Time the float64 oracle over whole requests of `b` until ~budget_s; returns (GB/s, sample text, s)."""
    from oracle import attention as A
    order = list(range(b.batch_size))
    t0 = time.perf_counter()
    done = []
    for i in order:
        A.batch_attention(b, requests=[i])
        done.append(i)
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    _, l_kv = lengths(b)
    nbytes = int(l_kv[done].sum()) * b.num_kv_heads * b.head_dim * 4
    return nbytes / dt / 1e9, f"{len(done)} of {b.batch_size} requests ({int(l_kv[done].sum())} KV tokens)", dt


def reference_arm(args):
    from serving_attention_plan_gb300 import workloads as W
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    b = W.by_name(args.config)
    if hasattr(b, "flat"):
        b = b.flat
    for _ in range(args.warmup):
        cpu_oracle_sample(b, budget_s=2.0)
    vals = []
    samples = ""
    for _ in range(args.steps):
        v, samples, _ = cpu_oracle_sample(b, budget_s=max(2.0, 60.0 / max(args.steps, 1)))
        vals.append(v)
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_config(args.config, b), parallelism="host cores (CPU oracle)"),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": samples + " per step, float64 NumPy oracle"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks (the slowest replica sets the whole job's time); identity at N = 1."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, seconds: float, world: int) -> float:
    """Whole-job throughput of `world` independent replicas: all ranks' units over the slowest rank's time."""
    return world * units_per_rank / seconds


def workload_config(name, b):
    l_q, l_kv = lengths(b)
    return {
        "workload": name, "batch": b.batch_size, "num_qo_heads": b.num_qo_heads, "num_kv_heads": b.num_kv_heads,
        "head_dim": b.head_dim, "page_size": b.page_size, "causal": bool(b.causal),
        "kv_tokens": int(l_kv.sum()), "q_tokens": int(l_q.sum()),
        "l2": "inputs larger than L2" if kv_bytes(b) > L2_BYTES else "inputs fit in L2 (no flush)",
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--config", default=PRIMARY)
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--batch", type=int, default=0, help="smaller batch of the decode workload (profiling captures)")
    ap.add_argument("--only", default="", help="time only this other workload or variant line (profiling captures)")
    args = ap.parse_args()
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        barrier = dist.barrier

    import __graft_entry__
    __graft_entry__.build()
    from serving_attention_plan_gb300 import workloads as W

    hbm_peak, bf16_peak, bf16_sus, peak_src = measured_peaks()
    if args.only:
        print(json.dumps({"only": args.only, **bench_other(args.only, torch, dev, hbm_peak, bf16_peak, args.steps,
                                                          args.warmup)}))
        return
    if args.batch and args.config == PRIMARY:
        b = W.llama3_8b_decode(batch=args.batch)
    elif args.batch and args.config == "ragged_causal_prefill":
        b = W.ragged_causal_prefill(batch=args.batch)
    else:
        b = W.by_name(args.config)
    case = Case(b, torch, dev)
    nbytes = kv_bytes(b)
    abytes = algorithmic_bytes(b)

    with ClockSampler(local) as clk:
        ms = time_launches(torch, case.run, args.steps, args.warmup, barrier)
    clocks = clk.summary()
    device_errors = case.ws.get_error()  # a timed-out pipeline wait or a skipped page would show here
    if device_errors:
        print(f"bench: device error bits {device_errors:#x} during the timed launches", file=sys.stderr)
    ms = max_over_ranks(ms, dev)
    hdr = case.ws.info()
    kernel_name = f"decode_kernel<R={int(hdr[3])}>" if hdr[1] == 0 else "prefill_kernel"
    value = replica_throughput(nbytes, ms * 1e-3, world) / 1e9
    achieved = abytes / (ms * 1e-3) / 1e9

    # host time of fi_plan (planning + enqueueing the upload) with the device idle, and the launch
    # replayed from a CUDA graph (fi_run is capturable; the plan stays in the workspace)
    plan_us = []
    for _ in range(30):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        case.plan()
        plan_us.append((time.perf_counter() - t0) * 1e6)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        case.run()
    graph_ms = time_launches(torch, graph.replay, min(args.steps, 500), 10)

    # end to end through the C ABI from host buffers
    q_host = torch.from_numpy(np.ascontiguousarray(b.q).view(np.int16)).pin_memory()
    o_host = torch.empty((b.total_q, b.num_qo_heads, b.head_dim), dtype=torch.int16).pin_memory()
    lse_host = torch.empty((b.total_q, b.num_qo_heads), dtype=torch.float32).pin_memory()
    q_dev16 = case.q.view(torch.int16)
    o_dev16 = case.o.view(torch.int16)

    def e2e_step():
        case.plan()
        q_dev16.copy_(q_host, non_blocking=True)
        case.run()
        o_host.copy_(o_dev16, non_blocking=True)
        lse_host.copy_(case.lse, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    e2e_steps = max(10, min(args.steps // 10, 200))
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    serial_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps

    # The same steps pipelined: E2E_CONTEXTS workspaces, each with its own q/o/lse buffers and
    # stream.  Step i runs on context i % E2E_CONTEXTS; before reusing a context the host waits for
    # its previous step's completion event, i.e. for that step's o and lse to be in host memory.
    from serving_attention_plan_gb300 import binding as B

    class _Ctx:
        pass

    ctxs = []
    for _ in range(E2E_CONTEXTS):
        c = _Ctx()
        c.ws = B.Workspace(b.batch_size, b.total_q, int(b.kv_indptr[-1]), b.num_qo_heads, b.num_kv_heads,
                           b.head_dim)
        c.q, c.o, c.lse = torch.empty_like(case.q), torch.empty_like(case.o), torch.empty_like(case.lse)
        c.o_host, c.lse_host = torch.empty_like(o_host).pin_memory(), torch.empty_like(lse_host).pin_memory()
        c.stream, c.done, c.busy = torch.cuda.Stream(), torch.cuda.Event(), False
        ctxs.append(c)

    def e2e_step_pipelined(i):
        c = ctxs[i % E2E_CONTEXTS]
        if c.busy:
            c.done.synchronize()
        c.ws.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.page_size, b.causal, stream=c.stream)
        with torch.cuda.stream(c.stream):
            c.q.view(torch.int16).copy_(q_host, non_blocking=True)
        c.ws.run(c.q, case.k, case.v, c.o, c.lse, stream=c.stream)
        with torch.cuda.stream(c.stream):
            c.o_host.copy_(c.o.view(torch.int16), non_blocking=True)
            c.lse_host.copy_(c.lse, non_blocking=True)
        c.done.record(c.stream)
        c.busy = True

    for i in range(4):
        e2e_step_pipelined(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step_pipelined(i)
    for c in ctxs:
        c.done.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
    e2e_same = all(torch.equal(c.o_host, o_host) and torch.equal(c.lse_host, lse_host) for c in ctxs)
    e2e_errors = [c.ws.get_error() for c in ctxs]
    if any(e2e_errors):
        print(f"bench: device error bits {e2e_errors} during the end-to-end steps", file=sys.stderr)
    plan_bytes = 4 * (16 + int(hdr[5]) + 1 + 8 * int(hdr[6]) + 8 * int(hdr[7]) + int(hdr[8]) + int(b.kv_indptr[-1]))
    h2d = int(b.q.nbytes) + plan_bytes
    d2h = int(o_host.numel() * 2 + lse_host.numel() * 4)

    extra = {}
    if not args.no_extra:
        for name in ("tiny_decode", "skewed_long_decode", "ragged_causal_prefill", "shared_prefix_decode") + \
                W.KERNEL_DIST_WORKLOADS + tuple(VARIANT_WORKLOADS):
            try:
                extra[name] = bench_other(name, torch, dev, hbm_peak, bf16_peak)
            except Exception as e:  # report, never hide
                extra[name] = {"error": f"{type(e).__name__}: {e}"}

    cpu = None
    if not args.no_cpu and rank == 0 and world == 1:
        v, sample, dt = cpu_oracle_sample(b, budget_s=15.0)
        cpu = {"value": v, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": sample + f", {dt:.1f} s, float64 NumPy oracle (BLAS threads default)"}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "us_per_batch": ms * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(args.config, b), parallelism=f"replicas x{world}"),
        "frac_of_hbm_peak": value / world / hbm_peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                     "traffic": ncu_traffic(f"{kernel_name}/{args.config}"), "kernel": kernel_name,
                     "algorithmic_bytes_per_launch": abytes},
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "pipelining": f"{E2E_CONTEXTS} workspaces / {E2E_CONTEXTS} streams", "outputs_equal_serial": e2e_same,
                "serial_ms_per_step": serial_ms,
                "serial_value": world * nbytes / (serial_ms * 1e-3) / 1e9},
        "breakdown": {"plan_host_us_median": float(np.median(plan_us)), "graph_replay_us": graph_ms * 1e3,
                      "note": "fi_plan on the host with the device idle; one fi_run captured in a CUDA graph and "
                              "replayed back to back"},
        "gpu_launches": args.steps,
        "device_errors": device_errors,
        "clocks": clocks,
        "plan": {"path": int(hdr[1]), "rows_tile": int(hdr[3]), "num_ctas": int(hdr[5]), "items": int(hdr[6]),
                 "split_rows": int(hdr[7]), "l_kv_chunk": int(hdr[9])},
        "configs": extra,
        "cpu_baseline": cpu,
    }
    # last key, compact: every workload's headline number and its fraction of the measured roofline
    line["targets"] = targets_summary(args.config, value / world, ms, hbm_peak, bf16_peak, peak_src, extra)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


# ncu DRAM-traffic entries (profiles/ncu_traffic.json) of the dominant kernel of each target workload
TRAFFIC_KEYS = {"skewed_long_decode": "decode_kernel<R=8>/skewed_long_decode",
                "ragged_causal_prefill": "prefill_kernel/ragged_causal_prefill",
                "variant_llama3_8b_decode_fp8_e4m3": "decode_kernel_fp8<R=4>/llama3_8b_decode_fp8_e4m3"}


def targets_summary(name, gbs, ms, hbm_peak, bf16_peak, peak_src, extra):
    """One short entry per workload (µs per batch, rate, fraction of the measured peak, the goal)."""
    r3 = lambda x: None if x is None else round(float(x), 3)
    out = {name: {"us": r3(ms * 1e3), "GB/s": r3(gbs), "frac_hbm": r3(gbs / hbm_peak), "goal": ">=0.75 hbm"}}
    goals = {"skewed_long_decode": ">=0.75 hbm", "ragged_causal_prefill": ">=0.50 bf16",
             "shared_prefix_decode": "reported", "variant_llama3_8b_decode_fp8_e4m3": "reported",
             "variant_ragged_causal_prefill_fp8_e4m3": "reported",
             "tiny_decode": "latency"}
    for k, goal in goals.items():
        e = extra.get(k)
        if not e or "error" in e:
            out[k] = {"error": (e or {}).get("error", "not run")}
            continue
        t = {"us": r3(e["us_per_batch"])}
        if "tflops" in e or "tflops_visible_pairs" in e:
            t.update({"TFLOP/s": r3(e.get("tflops", e.get("tflops_visible_pairs"))),
                      "frac_bf16": r3(e["frac_of_bf16_peak"])})
        elif "kv_gbs_unique" in e:
            t.update({"GB/s_unique_kv": r3(e["kv_gbs_unique"]), "frac_hbm": r3(e["frac_of_hbm_peak"]),
                      "launches": e.get("launches_per_step")})
        elif "kv_gbs" in e:
            t.update({"GB/s": r3(e["kv_gbs"]), "frac_hbm": r3(e["frac_of_hbm_peak"])})
        if k in TRAFFIC_KEYS:
            t["traffic"] = ncu_traffic(TRAFFIC_KEYS[k])  # DRAM bytes of one launch (ncu), null if stale
        t["goal"] = goal
        out[k] = t
    out["peaks"] = {"hbm_gbs": hbm_peak, "bf16_tflops": bf16_peak, "source": peak_src}
    return out


# Attention variants (sliding window, logit soft-cap, NHD pages) on two of the workloads
VARIANT_WORKLOADS = {
    "variant_llama3_8b_decode_nhd_softcap50": ("llama3_8b_decode", dict(logits_soft_cap=50.0, kv_layout="NHD")),
    "variant_ragged_causal_prefill_window1024_softcap50": ("ragged_causal_prefill",
                                                            dict(window_left=1024, logits_soft_cap=50.0)),
    "variant_llama3_8b_decode_fp8_e4m3": ("llama3_8b_decode", dict(kv_dtype=("e4m3", 0.5, 0.5))),
    "variant_ragged_causal_prefill_fp8_e4m3": ("ragged_causal_prefill", dict(kv_dtype=("e4m3", 0.25, 0.25))),
}


def bench_variant(name, torch, dev, hbm_peak, bf16_peak, steps=200, warmup=10):
    import dataclasses
    from serving_attention_plan_gb300 import workloads as W
    base, var = VARIANT_WORKLOADS[name]
    w = W.by_name(base)
    if var.get("kv_dtype"):
        w = W.as_e4m3(w, var["kv_dtype"][1], var["kv_dtype"][2])
    if var.get("kv_layout") == "NHD":
        w = dataclasses.replace(w, k_pages=np.ascontiguousarray(w.k_pages.transpose(0, 2, 1, 3)),
                                v_pages=np.ascontiguousarray(w.v_pages.transpose(0, 2, 1, 3)))
    c = Case(w, torch, dev, variant=var)
    ms = time_launches(torch, c.run, steps, warmup)
    hdr = c.ws.info()
    out = {"us_per_batch": ms * 1e3, "path": path_name(w, hdr), "variant": var,
           "config": dict(workload_config(base, w), l2="inputs larger than L2"), "device_errors": c.ws.get_error()}
    if hdr[1] == 1:
        tf = flops(w, var.get("window_left", -1)) / (ms * 1e-3) / 1e12
        out.update({"tflops_visible_pairs": tf, "frac_of_bf16_peak": tf / bf16_peak})
    else:
        gbs = kv_bytes(w) / (ms * 1e-3) / 1e9
        out.update({"kv_gbs": gbs, "frac_of_hbm_peak": gbs / hbm_peak})
    return out


def bench_other(name, torch, dev, hbm_peak, bf16_peak, steps=200, warmup=10):
    from serving_attention_plan_gb300 import binding as B
    from serving_attention_plan_gb300 import workloads as W
    if name in VARIANT_WORKLOADS:
        return bench_variant(name, torch, dev, hbm_peak, bf16_peak, steps, warmup)
    w = W.by_name(name)
    if name == "shared_prefix_decode":
        # one composable plan: the prefix block row (tensor cores, chunks to slots) and the suffix rows
        # (decode tiles, each merging its chunks and the prefix slots of its rows): two launches
        pre = Case(w.prefix, torch, dev)
        ws = B.Workspace(w.suffix.batch_size, w.suffix.total_q, max(int(w.suffix.kv_indptr[-1]),
                                                                   int(w.prefix.kv_indptr[-1])), 32, 8)
        ws.plan_composable((w.prefix.qo_indptr, w.prefix.kv_indptr, w.prefix.kv_indices, w.prefix.last_page_len),
                           (w.suffix.qo_indptr, w.suffix.kv_indptr, w.suffix.kv_indices, w.suffix.last_page_len),
                           16, False)
        o, lse = torch.empty_like(pre.o), torch.empty_like(pre.lse)

        def step():
            ws.run(pre.q, pre.k, pre.v, o, lse)

        ms = time_launches(torch, step, steps, warmup)
        errs = ws.get_error()
        # the same step as two plans (prefix attention + its contraction, then the suffix decode with
        # the prefix state folded in by fi_run_merge): three launches
        suf = Case.__new__(Case)
        suf.b, suf.torch, suf.q, suf.k, suf.v = w.suffix, torch, pre.q, pre.k, pre.v
        suf.o, suf.lse = torch.empty_like(pre.o), torch.empty_like(pre.lse)
        suf.ws = B.Workspace(w.suffix.batch_size, w.suffix.total_q, int(w.suffix.kv_indptr[-1]), 32, 8)
        suf.plan()

        def two_plans():
            pre.run()
            suf.ws.run_merge(suf.q, suf.k, suf.v, pre.o, pre.lse, suf.o, suf.lse)

        ms_two = time_launches(torch, two_plans, steps, warmup)
        nbytes = kv_bytes(w.prefix) + kv_bytes(w.suffix)
        return {"us_per_batch": ms * 1e3, "kv_gbs_unique": nbytes / (ms * 1e-3) / 1e9,
                "frac_of_hbm_peak": nbytes / (ms * 1e-3) / 1e9 / hbm_peak, "launches_per_step": 2,
                "plan": "one composable plan (fi_plan_composable): prefix on tcgen05 tiles, suffix decode merging "
                        "the prefix slots", "device_errors": errs,
                "us_two_plans_three_launches": ms_two * 1e3, "composable_plan": ws.info().tolist()[:10]}
    c = Case(w, torch, dev)
    cold = kv_bytes(w) < 2 * L2_BYTES  # inputs that L2 could hold: flush it before every launch
    ms = (time_launches_cold if cold else time_launches)(torch, c.run, steps, warmup)
    hdr = c.ws.info()
    errs = c.ws.get_error()
    out = {"us_per_batch": ms * 1e3, "path": path_name(w, hdr),
           "config": dict(workload_config(name, w), l2="flushed before every launch (2x L2 written, then 2x L2 of other data read)" if cold else
                          "inputs larger than L2"),
           "device_errors": errs}
    if cold:
        out["us_per_batch_hot_l2"] = time_launches(torch, c.run, steps, warmup) * 1e3
    if hdr[1] == 1:
        tf = flops(w) / (ms * 1e-3) / 1e12
        out.update({"tflops": tf, "frac_of_bf16_peak": tf / bf16_peak})
    else:
        gbs = kv_bytes(w) / (ms * 1e-3) / 1e9
        out.update({"kv_gbs": gbs, "frac_of_hbm_peak": gbs / hbm_peak})
    return out


def path_name(w, hdr) -> str:
    """Which kernel body the plan runs: 256-row items (two 128-row MMA tiles) on tcgen05, or <= 8-row
    decode tiles whose consumer is warp-level MMA (16-byte-copy loader, power-of-two pages) or CUDA
    cores (bulk loader)."""
    if hdr[1] == 1:
        return "256-row items, tcgen05"
    ps = int(w.page_size)
    return f"{int(hdr[3])}-row tiles, " + ("mma.sync" if ps & (ps - 1) == 0 else "CUDA cores")


if __name__ == "__main__":
    main()
