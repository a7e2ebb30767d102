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

# The CPU oracle runs one sequence chunk per host thread, each with a
# single-threaded BLAS: pin BLAS threads before numpy loads.
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
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged decode-attn achieved HBM GB/s (% of ~8 TB/s) and query tokens/s, 1 GB300"
UNIT = "GB/s"
WORKLOADS = ["llama3_8b_layer", "mixed_lengths", "cascade", "mla", "spec_verify_q2", "spec_verify_q4",
             "llama3_8b_layer_fp8", "cascade_nested", "sliding_window", "mla_fp8", "mla_spec_q4", "spec_tree"]
# measured workloads whose kernels are tensor-bound: dense-peak ratio to bf16
# of their operand type (e4m3 runs at twice the bf16 rate)
FP8_TENSOR = ("mla_fp8",)


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default="llama3_8b_layer")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only --workload (the default line also times every other workload)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="profiling run for ncu: one pool copy, no e2e / CPU baseline / clock sampling")
    ap.add_argument("--batch-scale", type=float, default=1.0,
                    help="scale the batch (sequences / groups) down for small profiling captures")
    return ap.parse_args()


# --------------------------------------------------------------------------
# Clock sampling through NVML (read-only queries)
# --------------------------------------------------------------------------

class ClockSampler:
    """Samples SM clock and clock-event reasons of one GPU every ``period_s``."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, index: int, period_s: float = 0.0005):
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


def device_clock(a, b):
    """Median over SMs of the average SM clock between two clock-stamp
    calls (cycle difference / timer difference, matched by SM)."""
    first = {}
    for sm, clk, ns in a.cpu().tolist():
        first.setdefault(sm, (clk, ns))
    mhz, window = [], []
    for sm, clk, ns in b.cpu().tolist():
        if sm in first and ns > first[sm][1]:
            mhz.append((clk - first[sm][0]) / (ns - first[sm][1]) * 1e3)
            window.append((ns - first[sm][1]) / 1e3)
            del first[sm]
    if not mhz:
        return {"sm_mhz_device": None}
    return {"sm_mhz_device": round(statistics.median(mhz), 1), "sm_mhz_device_min": round(min(mhz), 1),
            "device_sms": len(mhz), "device_window_us": round(statistics.median(window), 1)}


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
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:  # host-only ranks (tests of the multi-rank plumbing)
            dist.init_process_group("gloo")
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
# Workloads: algorithmic bytes / flops, device steps, CPU oracle samples
# --------------------------------------------------------------------------

def build_workload(name: str, device, small: bool = False, scale: float = 1.0):
    """The named workload at full size (or a small instance with the same
    per-sequence distributions, for CPU-side oracle timing; `scale` shrinks the
    batch for profiling captures)."""
    def n(full):
        return max(1, int(round(full * scale)))
    if name == "llama3_8b_layer":
        return workloads.llama3_8b_layer(device=device, B=8 if small else n(64))
    if name == "mixed_lengths":
        return workloads.mixed_lengths(device=device, repeat=2 if small else n(32))
    if name == "cascade":
        return workloads.shared_prefix_cascade(device=device, groups=1 if small else n(16),
                                               members=32 if small else 1024)
    if name == "mla":
        return workloads.absorbed_mla(device=device, B=2 if small else n(64))
    if name == "cascade_nested":
        return workloads.nested_prefix_cascade(device=device, members=8 if small else n(256))
    if name == "llama3_8b_layer_fp8":
        return workloads.llama3_8b_layer_fp8(device=device, B=8 if small else n(64))
    if name == "sliding_window":
        return workloads.sliding_window(device=device, B=4 if small else n(64))
    if name.startswith("spec_verify_q"):
        return workloads.speculative_verify(device=device, B=8 if small else n(64), q_len=int(name[13:]))
    if name == "mla_fp8":
        return workloads.absorbed_mla_fp8(device=device, B=2 if small else n(64))
    if name == "mla_spec_q4":
        return workloads.absorbed_mla_multi(device=device, B=2 if small else n(64))
    if name == "spec_tree":
        case, parents = workloads.speculative_tree(device=device, B=8 if small else n(64))
        case.meta["parents"] = parents
        return case
    raise ValueError(name)


def algorithmic(case, groups=None):
    """(bytes, tensor flops) one decode pass must move / compute.

    Paged GQA: every attended token's K and V rows once. Cascade: each group's
    prefix once plus every sequence's own rows. MLA: every latent row once;
    flops of Q.C^T over 576 dims and P.V over 512."""
    es = 2 if case.dtype == "bf16" else 4
    tokens = int(case.attended_lens.astype(np.int64).sum())
    if case.mla:  # every query row of every token (q_len of them per sequence)
        return case.kv_bytes_read(), tokens * case.q_len * case.H_q * (case.D + case.Dv) * 2
    if case.kv_fp8:
        return case.kv_bytes_read(), 0
    row = case.H_kv * (case.D + case.Dv) * es
    if groups is not None and groups["num_groups"] > 0:
        prefix_tokens = int(groups["prefix_len"].astype(np.int64).sum())
        members = np.diff(groups["member_indptr"])
        shared = int((groups["prefix_len"].astype(np.int64) * members).sum())
        flops = 4 * int((groups["prefix_len"].astype(np.int64) * members).sum()) * case.H_q * case.D
        return (tokens - shared + prefix_tokens) * row, flops
    return tokens * row, 0


def forest_as_groups(forest):
    """The per-node view algorithmic() needs: each node's own tokens and its
    members, and every sequence's shared tokens (its deepest node's path)."""
    N = int(forest["num_nodes"])
    own = np.diff(forest["prefix_indptr"]).astype(np.int64) * 16
    members = np.diff(forest["member_indptr"]).astype(np.int64)
    deep = forest["group_of"]
    shared = int(forest["prefix_len"][deep[deep >= 0]].astype(np.int64).sum()) if N else 0
    return {"num_groups": N, "own_tokens": own, "members": members, "shared_tokens": shared}


def algorithmic_forest(case, fg):
    """Nested cascade: each node's own pages once plus every sequence's own
    rows past its deepest node; prefix flops over every (member, node token)."""
    es = 2
    tokens = int(case.attn_lens.astype(np.int64).sum())
    row = case.H_kv * (case.D + case.Dv) * es
    distinct = int(fg["own_tokens"].sum())
    flops = 4 * int((fg["own_tokens"] * fg["members"]).sum()) * case.H_q * case.D
    return (tokens - fg["shared_tokens"] + distinct) * row, flops, (tokens - fg["shared_tokens"]) * row


def suffix_bytes(case, groups):
    """Algorithmic bytes of the paged (suffix) kernel of a cascade call: every
    sequence's own rows past its group's shared prefix."""
    es = 2 if case.dtype == "bf16" else 4
    tokens = int(case.attn_lens.astype(np.int64).sum())
    members = np.diff(groups["member_indptr"])
    shared = int((groups["prefix_len"].astype(np.int64) * members).sum())
    return (tokens - shared) * case.H_kv * (case.D + case.Dv) * es


def oracle_pass(view, case):
    import oracle
    if case.mla and case.kv_fp8:
        return oracle.mla_decode_attention_fp8(view["q"], view["q_scale"], view["k_pool"], view["k_scale"],
                                               view["block_table"], view["seq_lens"], case.scale, case.Dv)
    if case.mla and case.q_len > 1:
        return oracle.mla_multi_query_decode_attention(view["q"], view["k_pool"], view["block_table"],
                                                       view["seq_lens"], case.scale, case.Dv)
    if case.mla:
        return oracle.mla_decode_attention(view["q"], view["k_pool"], view["block_table"], view["seq_lens"],
                                           case.scale, case.Dv)
    if "parents" in case.meta:
        return oracle.tree_verify_decode_attention(view["q"], view["k_pool"], view["v_pool"], view["block_table"],
                                                   view["seq_lens"], view["parents"], case.scale)
    kp, vp = view["k_pool"], view["v_pool"]
    if case.kv_fp8:
        ks, vs = view["k_scale"], view["v_scale"]
        if case.append:
            kp, vp, ks, vs = oracle.kv_append_fp8(kp, vp, ks, vs, view["k_new"], view["v_new"], view["block_table"],
                                                  view["positions"], case.page_size)
        return oracle.decode_attention_fp8(view["q"], kp, vp, ks, vs, view["block_table"], view["seq_lens"],
                                           case.scale)
    if case.q_len > 1:
        return oracle.multi_query_decode_attention(view["q"], kp, vp, view["block_table"], view["seq_lens"],
                                                   case.scale)
    if case.window > 0:
        return oracle.decode_attention_window(view["q"], kp, vp, view["block_table"], view["seq_lens"], case.scale,
                                              case.window)
    if case.append:
        kp, vp = oracle.kv_append(kp, vp, view["k_new"], view["v_new"], view["block_table"],
                                  view["positions"], case.page_size)
    return oracle.decode_attention(view["q"], kp, vp, view["block_table"], view["seq_lens"], case.scale)


def sample_bytes(case, idx):
    """Flat (ungrouped) algorithmic bytes of the sampled sequences."""
    es = 4 if case.dtype == "f32" else 2
    tokens = int(case.attended_lens[idx].astype(np.int64).sum())
    if case.mla:
        return tokens * (case.D + 4) if case.kv_fp8 else tokens * case.D * es
    if case.kv_fp8:
        return tokens * case.H_kv * (case.D + case.Dv) + tokens * case.H_kv * 2 * 4
    return tokens * case.H_kv * (case.D + case.Dv) * es


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, else the Arm
    implementer / part codes)."""
    try:
        text = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    m = re.search(r"^model name\s*:\s*(.+)$", text, re.M)
    if m:
        return m.group(1).strip()
    imp = re.search(r"^CPU implementer\s*:\s*(\S+)", text, re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)", text, re.M)
    if imp and part:
        return f"Arm CPU implementer {imp.group(1)} part {part.group(1)}"
    return "unknown"


class OraclePool:
    """The oracle over a sample of sequences on all host threads: the sample
    is split into one chunk per thread, and numpy's BLAS calls and array
    operations (which release the interpreter lock) run concurrently."""

    def __init__(self, case, idx, threads: int):
        self.case = case
        chunks = [c for c in np.array_split(np.asarray(idx), max(1, min(threads, len(idx)))) if len(c)]
        self.views = [workloads.oracle_view(case, c) for c in chunks]
        self.ex = ThreadPoolExecutor(max_workers=len(self.views))
        self.threads = len(self.views)

    def run(self):
        list(self.ex.map(lambda v: oracle_pass(v, self.case), self.views))

    def close(self):
        self.ex.shutdown()


def time_oracle(case, idx, budget_s: float, threads: int = 1):
    """Seconds per oracle pass over sequences idx (repeated up to budget_s)."""
    pool = OraclePool(case, idx, threads)
    reps, t_total = 0, 0.0
    while (t_total < budget_s or reps == 0) and reps < 1000:
        t = time.perf_counter()
        pool.run()
        t_total += time.perf_counter() - t
        reps += 1
    pool.close()
    return t_total / reps, reps


def cpu_baseline(case, budget_s: float = 12.0):
    """The oracle (fp64 numpy) on all host threads over a bounded sample of the workload."""
    threads = host_threads()
    t1, _ = time_oracle(case, [int(np.argmin(case.attended_lens))], 0.0)
    per_seq_est = max(t1, 1e-4) * case.attended_lens.mean() / max(1, case.attended_lens.min())
    n = int(max(min(case.B, threads), min(case.B, threads * budget_s / 3 / per_seq_est)))
    idx = workloads.sample_sequences(case, n)[:n] if n < case.B else np.arange(case.B)
    sec, reps = time_oracle(case, idx, budget_s, threads)
    used = min(threads, len(idx))
    nbytes = sample_bytes(case, idx)
    return {"value": nbytes / sec / 1e9, "unit": UNIT, "cores": used, "kind": "oracle", "cpu": host_cpu_model(),
            "host_threads": threads,
            "sample": f"{len(idx)} of {case.B} sequences ({int(case.attended_lens[idx].sum())} tokens) x {reps} passes, "
                      f"fp64 numpy split over {used} threads (one BLAS thread each); bytes counted flat "
                      f"(no prefix sharing)",
            "query_tokens_per_s": len(idx) * case.q_len / sec}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    case = build_workload(args.workload, "cpu", small=args.workload in ("cascade", "mla", "cascade_nested",
                                                                        "mla_spec_q4", "spec_tree") or
                          args.workload.startswith("spec_verify") or args.workload.endswith("fp8"))
    # size each step's sample so the whole run stays within ~2 minutes, on
    # all host threads (one chunk of the step's sequences each)
    threads = host_threads()
    t1, _ = time_oracle(case, [0], 0.0)
    per_seq = max(t1, 1e-4)
    n_seq = int(max(1, min(case.B, threads * 120.0 / max(1, args.steps + args.warmup) / per_seq)))
    pools = []
    for s in range(min(case.B, 8)):
        idx = (np.arange(n_seq) + s * n_seq) % case.B
        pools.append((idx, OraclePool(case, idx, threads)))
    for i in range(args.warmup):
        pools[i % len(pools)][1].run()
    total_bytes, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        idx, pool = pools[i % len(pools)]
        pool.run()
        total_bytes += sample_bytes(case, idx)
    el = time.perf_counter() - t0
    used = pools[0][1].threads
    for _, pool in pools:
        pool.close()
    value = total_bytes / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": case.name, "B": case.B, "H_q": case.H_q, "H_kv": case.H_kv,
                                        "D": case.D, "page_size": case.page_size,
                                        "sample_sequences_per_step": n_seq},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle", "cpu": host_cpu_model(),
                         "sample": f"{n_seq} of {case.B} sequences per step, fp64 numpy split over {used} "
                                   f"threads (one BLAS thread each)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

class DeviceStep:
    """One decode pass of a workload on the device, through the C ABI."""

    def __init__(self, ts, case, dev, rotate: int):
        self.ts, self.case, self.dev = ts, case, dev
        c = case
        self.bt = torch.from_numpy(c.block_table).to(dev)
        self.lens = torch.from_numpy(c.attn_lens).to(dev)
        self.pos = torch.from_numpy(c.positions).to(dev)
        rows = (c.B, c.H_q) if c.q_len == 1 else (c.B, c.q_len, c.H_q)
        out_dtype = torch.bfloat16 if c.q.dtype == torch.uint8 else c.q.dtype
        self.out = torch.empty(*rows, c.Dv, dtype=out_dtype, device=dev)
        self.parents = (torch.from_numpy(c.meta["parents"]).to(dev) if "parents" in c.meta else None)
        self.lse = torch.empty(*rows, dtype=torch.float32, device=dev)
        pools = [(c.k_pool, c.v_pool)]
        for _ in range(rotate - 1):
            pools.append((c.k_pool.clone(), c.v_pool.clone() if c.v_pool is not None else None))
        self.pools = pools
        # fp8 caches: each rotated pool copy has its own scale arrays
        def clone(t):
            return t.clone() if t is not None else None
        self.scales = [(c.k_scale, c.v_scale)] + [(clone(c.k_scale), clone(c.v_scale))
                                                  for _ in range(rotate - 1)] if c.kv_fp8 else None
        self.groups = None
        self.gdev = None
        self.forest = None
        if c.name.startswith("nested_cascade"):
            t = time.perf_counter()
            self.forest = ts.ts_group_prefixes_nested(c.block_table, c.seq_lens, c.page_size, 2)
            self.group_ms = (time.perf_counter() - t) * 1e3
            self.gdev = ts.forest_to_device(self.forest, dev)
            ws_bytes = ts.ts_cascade_decode_workspace_size(c.B, c.H_q, c.D)
        elif c.name.startswith("cascade"):
            t = time.perf_counter()
            self.groups = ts.ts_group_prefixes(c.block_table, c.seq_lens, c.page_size, 2)
            self.group_ms = (time.perf_counter() - t) * 1e3
            self.gdev = ts.groups_to_device(self.groups, dev)
            ws_bytes = ts.ts_cascade_decode_workspace_size(c.B, c.H_q, c.D)
        elif c.mla:
            ws_bytes = ts.ts_mla_multi_workspace_size(c.B, c.q_len, c.H_q, c.Dv)
        elif self.parents is not None:
            ws_bytes = 256
        elif c.q_len > 1:
            ws_bytes = ts.ts_paged_decode_multi_workspace_size(c.B, c.q_len, c.H_q, c.D)
        else:
            ws_bytes = ts.ts_paged_decode_workspace_size(c.B, c.H_q, c.D)
        self.ws = ts.new_workspace(ws_bytes, dev)

    def attention(self, i, q=None, bt=None, lens=None, stream=None, gdev=None, out=None, q_scale=None):
        ts, c = self.ts, self.case
        kp, vp = self.pools[i % len(self.pools)]
        out = self.out if out is None else out
        q = c.q if q is None else q
        bt = self.bt if bt is None else bt
        lens = self.lens if lens is None else lens
        if self.forest is not None:
            ts.ts_cascade_nested_decode_attn(q, kp, vp, gdev or self.gdev, bt, lens, c.scale, out=out,
                                             lse=self.lse, workspace=self.ws, stream=stream)
        elif self.groups is not None:
            ts.ts_cascade_decode_attn(q, kp, vp, gdev or self.gdev, bt, lens, c.scale, out=out, lse=self.lse,
                                      workspace=self.ws, stream=stream)
        elif c.mla and c.kv_fp8:
            ks, _ = self.scales[i % len(self.scales)]
            ts.ts_mla_paged_decode_fp8(q, q_scale if q_scale is not None else c.meta["q_scale"], kp, ks, bt, lens,
                                       c.scale, d_v=c.Dv, out=out, lse=self.lse, workspace=self.ws, stream=stream)
        elif c.mla and c.q_len > 1:
            ts.ts_mla_paged_decode_multi(q, kp, bt, lens, c.scale, d_v=c.Dv, out=out, lse=self.lse,
                                         workspace=self.ws, stream=stream)
        elif c.mla:
            ts.ts_mla_paged_decode(q, kp, bt, lens, c.scale, d_v=c.Dv, out=out, lse=self.lse,
                                   workspace=self.ws, stream=stream)
        elif self.parents is not None:
            ts.ts_paged_decode_tree_attn(q, kp, vp, bt, lens, self.parents, c.scale, out=out, lse=self.lse,
                                         workspace=self.ws, stream=stream)
        elif c.window > 0:
            ts.ts_paged_decode_window_attn(q, kp, vp, bt, lens, c.scale, c.window, out=out, lse=self.lse,
                                           workspace=self.ws, stream=stream)
        elif c.q_len > 1:
            ts.ts_paged_decode_multi_attn(q, kp, vp, bt, lens, c.scale, out=out, lse=self.lse,
                                          workspace=self.ws, stream=stream)
        elif c.kv_fp8:
            ks, vs = self.scales[i % len(self.scales)]
            ts.ts_paged_decode_fp8_attn(q, kp, vp, ks, vs, bt, lens, c.scale, out=out, lse=self.lse,
                                        workspace=self.ws, stream=stream)
        else:
            ts.ts_paged_decode_attn(q, kp, vp, bt, lens, c.scale, out=out, lse=self.lse, workspace=self.ws,
                                    stream=stream)

    def step(self, i, ev=None, stream=None, inputs=None):
        ts, c = self.ts, self.case
        kp, vp = self.pools[i % len(self.pools)]
        inputs = inputs or {}
        if c.append and c.kv_fp8:
            ks, vs = self.scales[i % len(self.scales)]
            ts.ts_kv_append_fp8(inputs.get("k_new", c.k_new), inputs.get("v_new", c.v_new), kp, vp, ks, vs,
                                inputs.get("bt", self.bt), inputs.get("pos", self.pos), stream=stream)
        elif c.append:
            ts.ts_kv_append(inputs.get("k_new", c.k_new), inputs.get("v_new", c.v_new), kp, vp,
                            inputs.get("bt", self.bt), inputs.get("pos", self.pos), stream=stream)
        if ev is not None:
            ev[0].record(stream)
        self.attention(i, q=inputs.get("q"), bt=inputs.get("bt"), lens=inputs.get("lens"), stream=stream,
                       gdev=inputs.get("gdev"), out=inputs.get("out"), q_scale=inputs.get("q_scale"))
        if ev is not None:
            ev[1].record(stream)


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
    if args.profile:
        args.no_e2e = args.no_cpu_baseline = True
    line = measure(ts, args, args.workload, args.steps, args.warmup, dev, rank, world, dist, headline=True)
    # Every other workload in the same process (the default invocation, one
    # GPU): each entry is timed like the headline (warm-up, K timed steps with
    # CUDA events, inputs larger than L2, clocks sampled during the timed
    # region, the launch trace in a separate pass), without the end-to-end and
    # CPU legs.
    if line is not None and world == 1 and not args.profile and not args.no_extra and \
            args.workload == "llama3_8b_layer":
        extra = {}
        for w in WORKLOADS:
            if w == args.workload:
                continue
            torch.cuda.empty_cache()
            d = measure(ts, args, w, min(args.steps, 50), max(3, min(args.warmup, 5)), dev, rank, world, dist,
                        headline=False)
            extra[w] = {k: d[k] for k in ("ms_per_step", "value", "unit", "query_tokens_per_s", "roofline",
                                          "kernels", "clocks", "config", "gpu_launches", "device_error_word",
                                          "tensor", "flat_equivalent_gbs", "dtype") if k in d}
            extra[w]["steps"] = min(args.steps, 50)
            extra[w]["warmup"] = max(3, min(args.warmup, 5))
        line["workloads"] = extra
    if line is not None:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def measure(ts, args, workload, steps, warmup, dev, rank, world, dist, headline):
    """Time one workload on this rank; returns the bench line (rank 0) or None."""
    case = build_workload(workload, dev, scale=args.batch_scale)
    pool_bytes = case.k_pool.numel() * case.k_pool.element_size() * (2 if case.v_pool is not None else 1)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    rotate = 1 if args.profile else max(2, int(math.ceil(4 * l2 / pool_bytes)) if pool_bytes < 4 * l2 else 2)
    if pool_bytes > 2 * 1e9:
        rotate = 1  # already many times larger than L2
    runner = DeviceStep(ts, case, dev, rotate)
    stream = torch.cuda.current_stream()
    if runner.forest is not None:
        fg = forest_as_groups(runner.forest)
        nbytes, flops, forest_suffix = algorithmic_forest(case, fg)
    else:
        nbytes, flops = algorithmic(case, runner.groups)

    for i in range(warmup):
        runner.step(i, stream=stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    if args.profile:
        sampler.ok = False
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # per-SM clock stamps right before and after the timed work (outside its
    # events): each SM's average clock over the timed region
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    stamps = [torch.zeros(2 * n_sm, 3, dtype=torch.int64, device=dev) for _ in range(2)]
    sampler.start()
    barrier(dist)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    ts.ts_clock_stamp(stamps[0], stream)
    start.record(stream)
    for i in range(steps):
        # no events between steps: consecutive kernels may overlap through
        # programmatic dependent launch, as in a serving loop
        runner.step(i, stream=stream)
    end.record(stream)
    ts.ts_clock_stamp(stamps[1], stream)
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    barrier(dist)
    sampler.stop()
    ms_step = max_over_ranks(start.elapsed_time(end), dist, dev) / steps
    err_word = ts.ts_read_device_error(runner.ws)

    # per-kernel device times: a second timed pass with the library's launch
    # trace on (CUDA events recorded around each of its launches, on the
    # launching stream); kept apart from the pass above, whose step time the
    # extra event records would perturb
    n_tr = min(steps, 50)
    ts.ts_trace_collect()
    ts.ts_trace_enable(True)
    for i in range(n_tr):
        runner.step(i, stream=stream)
    torch.cuda.synchronize()
    ts.ts_trace_enable(False)
    per_kernel = {}
    for name, ms in ts.ts_trace_collect(capacity=64 * n_tr):
        per_kernel.setdefault(name, []).append(ms)
    kernels = {k: {"launches_per_step": len(v) / n_tr, "mean_ms": statistics.mean(v),
                   "share": sum(v) / sum(sum(x) for x in per_kernel.values())}
               for k, v in per_kernel.items()}
    launches_per_step = sum(len(v) for v in per_kernel.values()) / n_tr

    # end to end through the public API with host buffers (pinned): the step's
    # inputs go up, its output comes back, every step
    e2e = None
    if headline and not args.no_e2e:
        hin = {"q": case.q.cpu().pin_memory(), "bt": torch.from_numpy(case.block_table).pin_memory(),
               "lens": torch.from_numpy(case.attn_lens).pin_memory()}
        if case.append:
            hin.update(k_new=case.k_new.cpu().pin_memory(), v_new=case.v_new.cpu().pin_memory(),
                       pos=torch.from_numpy(case.positions).pin_memory())
        if case.mla and case.kv_fp8:
            hin["q_scale"] = case.meta["q_scale"].cpu().pin_memory()
        # all of a step's inputs travel in one pinned buffer and one copy
        offs, total = {}, 0
        for k, v in hin.items():
            offs[k] = total
            total += (v.numel() * v.element_size() + 255) // 256 * 256
        h_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
        for k, v in hin.items():
            nb = v.numel() * v.element_size()
            h_pack[offs[k]:offs[k] + nb].copy_(v.reshape(-1).view(torch.uint8))
        # two device copies of the inputs and of the output: step i+1's inputs
        # go up, and step i-1's output comes back, while step i computes
        d_packs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]

        def views(dp):
            return {k: dp[offs[k]:offs[k] + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                    for k, v in hin.items()}
        dins = [views(dp) for dp in d_packs]
        d_outs = [runner.out, torch.empty_like(runner.out)]
        h_outs = [torch.empty(runner.out.shape, dtype=runner.out.dtype).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in hin.values())
        d2h = h_outs[0].numel() * h_outs[0].element_size()
        host_group_ms = []

        def group_on_host():
            """The user's call sequence for a cascade step: group on the host."""
            t = time.perf_counter()
            if runner.forest is not None:
                g = ts.ts_group_prefixes_nested(case.block_table, case.seq_lens, case.page_size, 2)
            else:
                g = ts.ts_group_prefixes(case.block_table, case.seq_lens, case.page_size, 2)
            host_group_ms.append((time.perf_counter() - t) * 1e3)
            return g

        def e2e_step(i, st, groups=None):
            """One step: inputs up, (cascade: the step's groups up), attend,
            output back. For cascade, returns the next step's groups, formed
            on the host while this step's kernels run."""
            d_packs[0].copy_(h_pack, non_blocking=True)
            inputs = dict(dins[0])
            if groups is not None:
                inputs["gdev"] = (ts.forest_to_device(groups, dev) if runner.forest is not None
                                  else ts.groups_to_device(groups, dev))
            runner.step(i, stream=st, inputs=inputs)
            h_outs[0].copy_(runner.out, non_blocking=True)
            return group_on_host() if groups is not None else None

        UNROLL = 8
        cp = torch.cuda.Stream(device=dev)
        ev_h2d, ev_comp, ev_d2h = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

        def pipelined_steps(st, n=UNROLL, groups=None):
            """n decode steps, each with its own input upload and output
            read-back, on two streams: uploads and read-backs run on `cp`
            beside the previous / next step's kernels (double-buffered). With
            `groups` (cascade) each step also uploads its groups and forms the
            next step's on the host while its kernels run; returns the groups
            formed last."""
            cp.wait_stream(st)
            with torch.cuda.stream(cp):
                d_packs[0].copy_(h_pack, non_blocking=True)
            ev_h2d[0].record(cp)
            for k in range(n):
                b = k & 1
                if k + 1 < n:
                    if k >= 1:
                        cp.wait_event(ev_comp[b ^ 1])  # step k-1 has read its inputs
                    with torch.cuda.stream(cp):
                        d_packs[b ^ 1].copy_(h_pack, non_blocking=True)
                    ev_h2d[b ^ 1].record(cp)
                st.wait_event(ev_h2d[b])
                if k >= 2:
                    st.wait_event(ev_d2h[b])  # step k-2's output is back on the host
                inputs = dict(dins[b], out=d_outs[b])
                if groups is not None:
                    with torch.cuda.stream(st):
                        inputs["gdev"] = (ts.forest_to_device(groups, dev) if runner.forest is not None
                                          else ts.groups_to_device(groups, dev))
                runner.step(k, stream=st, inputs=inputs)
                ev_comp[b].record(st)
                cp.wait_event(ev_comp[b])
                with torch.cuda.stream(cp):
                    h_outs[b].copy_(d_outs[b], non_blocking=True)
                ev_d2h[b].record(cp)
                if groups is not None:
                    groups = group_on_host()
            st.wait_stream(cp)
            return groups

        regroups = runner.groups is not None or runner.forest is not None
        n_e2e = min(steps, 50) if regroups else (steps + UNROLL - 1) // UNROLL * UNROLL
        groups = group_on_host() if regroups else None
        for i in range(min(warmup, 3)):
            groups = e2e_step(i, stream, groups)
        torch.cuda.synchronize()
        # A serving loop replays its decode steps from a CUDA graph: capture
        # UNROLL pipelined steps (uploads, library calls, read-backs) once and
        # replay them. Cascade regroups on the host every step and runs the
        # same pipeline eagerly: each step's grouping runs on the host while
        # the previous step's kernels run on the device.
        graph = None
        if not regroups:
            cap = torch.cuda.Stream(device=dev)
            cap.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                pipelined_steps(cap)
            stream.wait_stream(cap)
            for _ in range(2):
                graph.replay()
            torch.cuda.synchronize()
        barrier(dist)
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        s2.record(stream)
        if graph is not None:
            for _ in range(n_e2e // UNROLL):
                graph.replay()
        else:
            groups = pipelined_steps(stream, n_e2e, groups)
        e2.record(stream)
        torch.cuda.synchronize()
        wall_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
        e2e_ms = max(max_over_ranks(s2.elapsed_time(e2), dist, dev) / n_e2e, wall_ms)
        e2e = {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": n_e2e,
               "query_tokens_per_s": world * case.B * case.q_len / (e2e_ms * 1e-3),
               "cuda_graph": graph is not None,
               "copies_overlap_compute": True}
        if host_group_ms:
            e2e["host_grouping_ms"] = statistics.median(host_group_ms)

    if rank != 0:
        return None
    peaks = {}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        peaks = json.load(open(path))
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    tc_peak = float(peaks.get("bf16_tflops", 1900.0))
    peak_kind = "measured" if peaks else "fallback"
    value = world * nbytes / (ms_step * 1e-3) / 1e9
    # the dominant kernel and its algorithmic work per launch
    dom = max(kernels, key=lambda k: kernels[k]["share"])
    dom_ms = kernels[dom]["mean_ms"]
    dom_bytes, dom_flops = nbytes, flops
    if runner.groups is not None and dom == "paged_decode_kernel":
        dom_bytes, dom_flops = suffix_bytes(case, runner.groups), 0
    if runner.forest is not None and dom == "paged_decode_kernel":
        dom_bytes, dom_flops = forest_suffix, 0
    # the file holding the dominant kernel's device code (its hash ties a
    # recorded DRAM-traffic figure to the code that produced it)
    source = {"mla_decode_kernel": "ts_mla.cu", "cascade_prefix_kernel": "ts_cascade.cu",
              "mq_tc_kernel": "ts_mq_tc.cu"}.get(dom, "ts_paged_decode_kernel.cuh")
    hbm_achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = kernel_traffic(f"{dom}__{workload}.md", source)
    if case.mla:
        tflops = dom_flops / (dom_ms * 1e-3) / 1e12
        fp8 = workload in FP8_TENSOR
        peak = tc_peak * (2.0 if fp8 else 1.0)
        roofline = {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                    "frac": tflops / peak,
                    "peak_source": (f"{peak_kind} bf16_tflops (burst) x 2 (e4m3 / bf16 nominal dense ratio)"
                                    if fp8 else f"{peak_kind} bf16_tflops (burst)"),
                    "kernel": dom, "kernel_ms": dom_ms, "flops_per_launch": dom_flops, "traffic": traffic,
                    "hbm": {"achieved": hbm_achieved, "peak": hbm_peak, "unit": "GB/s",
                            "frac": hbm_achieved / hbm_peak, "bytes_per_launch": dom_bytes}}
    else:
        roofline = {"bound": "hbm", "achieved": hbm_achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": hbm_achieved / hbm_peak, "peak_source": f"{peak_kind} hbm_gbs (copy)",
                    "kernel": dom, "kernel_ms": dom_ms, "bytes_per_launch": dom_bytes, "traffic": traffic}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ("e4m3 q and latent" if case.kv_fp8 and case.mla else
                                       "e4m3 K/V, bf16 q" if case.kv_fp8 else
                                       "bf16" if case.dtype == "bf16" else "f32"), "accumulate": "f32",
        "data": "synthetic",
        "config": {"workload": case.name, "B": case.B, "H_q": case.H_q, "H_kv": case.H_kv, "D": case.D,
                   "Dv": case.Dv, "page_size": case.page_size, "tokens_attended": int(case.attended_lens.sum()),
                   "kv_bytes_per_step": nbytes, "append": case.append, "q_len": case.q_len,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {rotate} rotated pool cop{'y' if rotate == 1 else 'ies'} of "
                         f"{pool_bytes / 1e9:.2f} GB (L2 {l2 / 1e6:.0f} MB)"},
        "query_tokens_per_s": world * case.B * case.q_len / (ms_step * 1e-3),
        "hbm_frac_of_8tbs": value / world / 8000.0,
        "roofline": roofline,
        "kernels": kernels,
        "gpu_launches": int(round(launches_per_step * steps)),
        "device_error_word": err_word,
        "clocks": {**sampler.summary(t_wall0, t_wall1), **device_clock(stamps[0], stamps[1])},
    }
    if flops and "cascade_prefix_kernel" in kernels:
        # all prefix launches of a step (one per level of a nested forest)
        pms = kernels["cascade_prefix_kernel"]["mean_ms"] * kernels["cascade_prefix_kernel"]["launches_per_step"]
        tflops = flops / (pms * 1e-3) / 1e12
        line["tensor"] = {"kernel": "cascade_prefix_kernel", "achieved": tflops, "peak": tc_peak,
                          "unit": "TFLOP/s", "frac": tflops / tc_peak, "flops_per_step": flops,
                          "launches_per_step": kernels["cascade_prefix_kernel"]["launches_per_step"],
                          "kernel_ms": pms, "peak_source": f"{peak_kind} bf16_tflops (burst)"}
    if runner.forest is not None:
        flat = sample_bytes(case, np.arange(case.B))
        line["config"]["flat_kv_bytes"] = flat
        line["config"]["forest_nodes"] = int(runner.forest["num_nodes"])
        line["config"]["forest_levels"] = int(runner.forest["num_levels"])
        line["flat_equivalent_gbs"] = flat / (ms_step * 1e-3) / 1e9
    if runner.groups is not None:
        flat = sample_bytes(case, np.arange(case.B))
        line["config"]["flat_kv_bytes"] = flat
        line["config"]["groups"] = int(runner.groups["num_groups"])
        line["flat_equivalent_gbs"] = flat / (ms_step * 1e-3) / 1e9
    if e2e is not None:
        line["e2e"] = e2e
    if headline and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(case)
    return line


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
