#!/usr/bin/env python3
"""Benchmark of decode-step attention over a paged KV cache on GB300.

One step = one pass of the decode hot path over one synthetic batch:
ts_kv_append (one new token per sequence) followed by ts_paged_decode_attn
(page gather + GQA scores + online softmax + PV, split-KV across all SMs and
the LSE merge of cut sequences). The default workload is the Llama-3-8B-shaped
decode layer: B=64, 32 query / 8 kv heads, head dim 128, bf16 K/V with fp32
accumulation, page size 16, lengths U[512, 4096], pool 1.25x the need.

metric: achieved HBM GB/s of paged decode attention = algorithmic K+V bytes
read per step (tokens attended x H_kv x 2 x D x 2 B) / step time; query
tokens/s (= B / step time) is reported beside it.

Timing: CUDA events on the launching stream, W warm-up steps, then exactly K
timed steps between barriers + synchronizes; max over ranks. Two rotated
copies of the K/V pool (each larger than L2) defeat L2 reuse between steps.
``--impl reference`` times the fp64 CPU oracle instead (on the host cores).
With N > 1 GPUs (torchrun) every rank runs its own replica (weak scaling).
"""

from __future__ import annotations

import os
import sys

# The CPU oracle runs single-threaded: pin BLAS threads before numpy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import ctypes
import hashlib
import json
import math
import re
import statistics
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged decode-attn achieved HBM GB/s (% of ~8 TB/s) and query tokens/s, 1 GB300"
UNIT = "GB/s"


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["llama3_8b_layer", "mixed_lengths"], default="llama3_8b_layer")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="profiling run for ncu: one pool copy, no e2e / CPU baseline / clock sampling")
    return ap.parse_args()


def build_workload(name: str, device):
    if name == "llama3_8b_layer":
        return workloads.llama3_8b_layer(device=device)
    if name == "mixed_lengths":
        return workloads.mixed_lengths(device=device)
    raise ValueError(name)


# --------------------------------------------------------------------------
# Clock sampling through NVML (read-only queries)
# --------------------------------------------------------------------------

class ClockSampler:
    """Samples SM clock and clock-event reasons of one GPU every ``period_s``."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, index: int, period_s: float = 0.002):
        self.ok = False
        self.samples = []
        self.period = period_s
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.handle)) != 0:
                return
            mx = ctypes.c_uint()
            self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))  # 1 = SM clock
            self.max_mhz = int(mx.value)
            self.ok = True
        except OSError:
            return

    def _sample(self):
        clk = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk))
        self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.handle, ctypes.byref(reasons))
        return time.perf_counter(), int(clk.value), int(reasons.value)

    def start(self):
        if not self.ok:
            return
        self._stop = threading.Event()

        def loop():
            while not self._stop.is_set():
                self.samples.append(self._sample())
                time.sleep(self.period)
        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()

    def stop(self):
        if self.ok:
            self._stop.set()
            self._thread.join()

    def summary(self, t0: float, t1: float):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        inside = [s for s in self.samples if t0 <= s[0] <= t1] or self.samples[-3:]
        mhz = statistics.median([s[1] for s in inside]) if inside else None
        bits = 0
        for s in inside:
            bits |= s[2]
        reasons = [name for bit, name in self.REASONS.items() if bits & bit and name != "gpu_idle"]
        return {"sm_mhz": mhz, "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(inside)}


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_traffic(profile_name: str, source: str):
    """dram bytes per launch recorded by an ncu capture of the current kernel source, else None."""
    path = os.path.join(ROOT, "profiles", profile_name)
    src = os.path.join(ROOT, "paged_kv_cache_46_gb300", "csrc", source)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*\(source sha256 ([0-9a-f]+)", text)
    if m and m.group(2) == sha:
        return float(m.group(1))
    return None


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return rank, world, local, dist
    return 0, 1, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x: float, dist, device) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# --------------------------------------------------------------------------

def oracle_pass(view, case):
    import oracle
    kp, vp = view["k_pool"], view["v_pool"]
    if case.append:
        kp, vp = oracle.kv_append(kp, vp, view["k_new"], view["v_new"], view["block_table"],
                                  view["positions"], case.page_size)
    return oracle.decode_attention(view["q"], kp, vp, view["block_table"], view["seq_lens"], case.scale)


def sample_bytes(case, idx):
    esize = 4 if case.dtype == "f32" else 2
    return int(case.attn_lens[idx].astype(np.int64).sum()) * case.H_kv * (case.D + case.Dv) * esize


def cpu_baseline(case, budget_s: float = 12.0):
    """The oracle on the full batch, repeated until ~budget_s of CPU time."""
    view = workloads.oracle_view(case)
    idx = np.arange(case.B)
    nbytes = sample_bytes(case, idx)
    reps, t_total = 0, 0.0
    while t_total < budget_s and reps < 1000:
        t = time.perf_counter()
        oracle_pass(view, case)
        t_total += time.perf_counter() - t
        reps += 1
    sec = t_total / reps
    return {"value": nbytes / sec / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"full batch ({case.B} sequences, {int(case.attn_lens.sum())} tokens) x {reps} passes, "
                      f"fp64 numpy, 1 BLAS thread", "query_tokens_per_s": case.B / sec, "ms_per_pass": sec * 1e3}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    case = build_workload(args.workload, "cpu")
    view_all = workloads.oracle_view(case)
    # size each step's sample so the whole run stays within ~2 minutes
    t = time.perf_counter()
    oracle_pass(workloads.oracle_view(case, [0]), case)
    per_seq = max(time.perf_counter() - t, 1e-4)
    n_seq = int(max(1, min(case.B, 120.0 / max(1, args.steps + args.warmup) / per_seq)))
    views = []
    for s in range(min(case.B, 8)):
        idx = (np.arange(n_seq) + s * n_seq) % case.B
        views.append((idx, workloads.oracle_view(case, idx)))
    del view_all
    for i in range(args.warmup):
        oracle_pass(views[i % len(views)][1], case)
    total_bytes, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        idx, v = views[i % len(views)]
        oracle_pass(v, case)
        total_bytes += sample_bytes(case, idx)
    el = time.perf_counter() - t0
    value = total_bytes / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": case.name, "B": case.B, "H_q": case.H_q, "H_kv": case.H_kv,
                                        "D": case.D, "page_size": case.page_size,
                                        "sample_sequences_per_step": n_seq},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{n_seq} of {case.B} sequences per step, fp64 numpy, 1 BLAS thread"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def run_ours(args):
    rank, world, local, dist = dist_setup(args.gpus)
    import paged_kv_cache_46_gb300 as ts
    from paged_kv_cache_46_gb300 import build as ts_build
    if rank == 0:
        ts_build.build()
    barrier(dist)
    if world > 1 and rank != 0:
        ts_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    case = build_workload(args.workload, dev)
    bt = torch.from_numpy(case.block_table).to(dev)
    lens = torch.from_numpy(case.attn_lens).to(dev)
    pos = torch.from_numpy(case.positions).to(dev)
    # second copy of the pools: consecutive steps read different memory
    if args.profile:
        args.no_e2e = args.no_cpu_baseline = True
        pools = [(case.k_pool, case.v_pool)] * 2
    else:
        pools = [(case.k_pool, case.v_pool), (case.k_pool.clone(), case.v_pool.clone())]
    out = torch.empty_like(case.q)
    lse = torch.empty(case.B, case.H_q, dtype=torch.float32, device=dev)
    ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(case.B, case.H_q, case.D), dev)
    stream = torch.cuda.current_stream()
    nbytes = case.kv_bytes_read()
    launches_per_step = 3 if case.append else 2

    def step(i, ev=None):
        kp, vp = pools[i % 2]
        if case.append:
            ts.ts_kv_append(case.k_new, case.v_new, kp, vp, bt, pos, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        ts.ts_paged_decode_attn(case.q, kp, vp, bt, lens, case.scale, out=out, lse=lse, workspace=ws,
                                stream=stream)
        if ev is not None:
            ev[1].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    if args.profile:
        sampler.ok = False
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.start()
    barrier(dist)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    start.record(stream)
    for i in range(args.steps):
        step(i, evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    barrier(dist)
    sampler.stop()
    ms_total = start.elapsed_time(end)
    ms_total = max_over_ranks(ms_total, dist, dev)
    ms_step = ms_total / args.steps
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    err_word = ts.ts_read_device_error(ws)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        h_q = case.q.cpu().pin_memory()
        h_kn = case.k_new.cpu().pin_memory() if case.append else None
        h_vn = case.v_new.cpu().pin_memory() if case.append else None
        h_bt = torch.from_numpy(case.block_table).pin_memory()
        h_lens = torch.from_numpy(case.attn_lens).pin_memory()
        h_pos = torch.from_numpy(case.positions).pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        d_q, d_kn, d_vn = torch.empty_like(case.q), torch.empty_like(case.k_new), torch.empty_like(case.v_new)
        d_bt, d_lens, d_pos = torch.empty_like(bt), torch.empty_like(lens), torch.empty_like(pos)
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_kn, h_vn, h_bt, h_lens, h_pos) if t is not None)
        d2h = h_out.numel() * h_out.element_size()

        def e2e_step(i):
            kp, vp = pools[i % 2]
            d_q.copy_(h_q, non_blocking=True)
            d_bt.copy_(h_bt, non_blocking=True)
            d_lens.copy_(h_lens, non_blocking=True)
            if case.append:
                d_kn.copy_(h_kn, non_blocking=True)
                d_vn.copy_(h_vn, non_blocking=True)
                d_pos.copy_(h_pos, non_blocking=True)
                ts.ts_kv_append(d_kn, d_vn, kp, vp, d_bt, d_pos, stream=stream)
            ts.ts_paged_decode_attn(d_q, kp, vp, d_bt, d_lens, case.scale, out=out, lse=lse, workspace=ws,
                                    stream=stream)
            h_out.copy_(out, non_blocking=True)

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier(dist)
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        for i in range(args.steps):
            e2e_step(i)
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(s2.elapsed_time(e2), dist, dev) / args.steps
        e2e = {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "query_tokens_per_s": world * case.B / (e2e_ms * 1e-3)}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    peak, peak_kind = measured_peaks()
    achieved = nbytes / (attn_ms * 1e-3) / 1e9
    value = world * nbytes / (ms_step * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if case.dtype == "bf16" else "f32", "accumulate": "f32",
        "data": "synthetic",
        "config": {"workload": case.name, "B": case.B, "H_q": case.H_q, "H_kv": case.H_kv, "D": case.D,
                   "page_size": case.page_size, "tokens_attended": int(case.attn_lens.sum()),
                   "kv_bytes_per_step": nbytes, "append": case.append, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: two rotated copies of the K/V pool "
                         f"({2 * case.k_pool.numel() * case.k_pool.element_size() / 1e9:.2f} GB each)"},
        "query_tokens_per_s": world * case.B / (ms_step * 1e-3),
        "hbm_frac_of_8tbs": value / world / 8000.0,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs (copy)",
                     "kernel": "ts_paged_decode_attn (split-KV kernel + LSE merge kernel)",
                     "traffic": kernel_traffic(f"paged_decode_{case.name}.md", "ts_paged_decode.cu")},
        "gpu_launches": launches_per_step * args.steps,
        "device_error_word": err_word,
        "clocks": sampler.summary(t_wall0, t_wall1),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(case)
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
