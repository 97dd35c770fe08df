"""Benchmark: cascade verify on the pages' example shape (one GPU per rank).

One step is one cpa_cascade_verify call: Pass A (prefix, read once per
request) + Pass B (own-branch drafts) + merge for B=64 requests, topk=4
branches of S=5 drafts, prefix L=2000, H_q=32, H_kv=8, head_dim=128, page 16
-- one decoder layer's verify attention.  The metric is unique KV bytes
(B*L + B*topk*S tokens x 4096 B) per second; naive expand is timed on the
same inputs for the us/step comparison.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own batch (weak scaling, no collective on
the data path); rank 0 prints one JSON line.  `--impl reference` times the
fp64 CPU oracle on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "cascade verify: KV GB/s vs ~8 TB/s HBM; us/step vs naive expand"
WORKLOAD = ("pages' example verify: B=64, topk=4, S=5, L=2000, H_q=32, H_kv=8, d_head=128, "
            "bf16 N(0,1), page size 16, random page table, chain-per-branch mask")
CFG = "pages_example"
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = ["cascade_paged_attention_gb300/csrc/cpa_attn.cuh",
                  "cascade_paged_attention_gb300/csrc/cpa_device.cuh",
                  "cascade_paged_attention_gb300/csrc/cpa_api.cu"]
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "cascade_verify_pages_example.json")


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_sample(wl, n_requests: int, threads: int = 0, min_seconds: float = 0.0):
    """Time the oracle on the first n_requests requests of the workload (all their rows),
    repeated until at least min_seconds have passed.  Returns (GB/s, seconds, passes)."""
    import oracle

    rows_per_req = wl.topk * wl.S * wl.H_q
    rows = np.arange(n_requests * rows_per_req, dtype=np.int64)
    kv_bytes = (int(wl.prefix_lens[:n_requests].sum()) + n_requests * wl.topk * wl.S) \
        * wl.kv_bytes_per_token()
    passes = 0
    t0 = time.perf_counter()
    while True:
        oracle.verify_wl(wl, rows=rows, threads=threads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return kv_bytes * passes / dt / 1e9, dt, passes


def reduce_max(x: float, pg=None, device=None) -> float:
    """The largest x over all ranks (x itself without a process group)."""
    if pg is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_gbs(bytes_per_rank: float, world: int, steps: int, total_ms: float) -> float:
    """Whole-job GB/s: every rank moved bytes_per_rank per step; the job took the
    slowest rank's time."""
    return bytes_per_rank * world * steps / (total_ms * 1e-3) / 1e9


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import cpa_synth
    import oracle.build

    oracle.build.build()
    wl = cpa_synth.make_verify(**cpa_synth.VERIFY_CONFIGS[CFG])
    cores = os.cpu_count() or 1
    # one step: every row of n_req of the 64 requests (about 16 ms each on 16 cores),
    # sized so that the whole run stays within a couple of minutes for any --steps
    n_req = max(1, min(wl.B, round(3000 / max(1, args.steps + args.warmup))))
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, n_req)
    vals, times = [], []
    for _ in range(args.steps):
        v, dt, _ = cpu_oracle_sample(wl, n_req)
        vals.append(v)
        times.append(dt)
    total_bytes = (int(wl.prefix_lens[:n_req].sum()) + n_req * wl.topk * wl.S) \
        * wl.kv_bytes_per_token() * args.steps
    value = total_bytes / sum(times) / 1e9
    sample = f"{n_req} of {wl.B} requests (all {wl.topk * wl.S * wl.H_q} rows each) per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local):
    import torch

    import cascade_paged_attention_gb300 as cpa
    import cpa_synth

    cpa.build_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    wl = cpa_synth.make_verify(**cpa_synth.VERIFY_CONFIGS[CFG])
    B, topk, S, H_q, H_kv, P = wl.B, wl.topk, wl.S, wl.H_q, wl.H_kv, wl.page_size
    d = wl.head_dim

    def host(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(dtype) if dtype is not None else t).pin_memory()

    h_q = host(wl.q, torch.bfloat16)
    h_k = host(wl.k_pages, torch.bfloat16)
    h_v = host(wl.v_pages, torch.bfloat16)
    h_ppt = host(wl.prefix_page_table)
    h_dpt = host(wl.draft_page_table)
    h_lens = host(wl.prefix_lens)
    q, kp, vp = h_q.to(dev), h_k.to(dev), h_v.to(dev)
    ppt, dpt, lens = h_ppt.to(dev), h_dpt.to(dev), h_lens.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], H_q, dtype=torch.float32, device=dev)
    o_n = torch.empty_like(q)
    lse_n = torch.empty_like(lse)
    ws = torch.zeros(cpa.cpa_cascade_verify_workspace_size(B, topk, S, H_q, H_kv, d, P),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    mpl = wl.max_prefix_len

    def cascade():
        cpa.cpa_cascade_verify(q, kp, vp, ppt, dpt, lens, topk, S, max_prefix_len=mpl, o=o,
                               lse=lse, workspace=ws)

    def naive():
        cpa.cpa_naive_expand_verify(q, kp, vp, ppt, dpt, lens, topk, S, max_prefix_len=mpl,
                                    o=o_n, lse=lse_n, workspace=ws)

    unique_bytes = wl.unique_kv_tokens() * wl.kv_bytes_per_token()
    naive_bytes = wl.naive_kv_tokens() * wl.kv_bytes_per_token()

    def barrier():
        if pg is not None:
            pg.barrier()

    def max_over_ranks(x: float) -> float:
        return reduce_max(x, pg, dev)

    def timed(fn, steps, per_launch=False):
        """Time `steps` calls: total ms (events around the whole run) and per-call ms."""
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        evs[0].record(stream)
        for i in range(steps):
            fn()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
        return evs[0].elapsed_time(evs[-1]), per

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    total_ms, per_ms = timed(cascade, args.steps)
    clock_info = clocks.stop()
    total_ms = max_over_ranks(total_ms)
    ms_per_step = total_ms / args.steps
    value = weak_scaling_gbs(unique_bytes, world, args.steps, total_ms)
    launch_ms = statistics.mean(per_ms)
    achieved = unique_bytes / (launch_ms * 1e-3) / 1e9

    naive_total, _ = timed(naive, args.steps)
    naive_total = max_over_ranks(naive_total)
    naive_ms = naive_total / args.steps

    # end to end through the public API: host inputs -> device, call, result -> host
    h_o = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_ppt, h_dpt, h_lens))
    d2h = h_o.numel() * 2 + h_lse.numel() * 4

    def e2e_step():
        q.copy_(h_q, non_blocking=True)
        kp.copy_(h_k, non_blocking=True)
        vp.copy_(h_v, non_blocking=True)
        ppt.copy_(h_ppt, non_blocking=True)
        dpt.copy_(h_dpt, non_blocking=True)
        lens.copy_(h_lens, non_blocking=True)
        cascade()
        h_o.copy_(o, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 10))
    e2e_total, _ = timed(e2e_step, e2e_steps)
    e2e_total = max_over_ranks(e2e_total)
    e2e_value = weak_scaling_gbs(unique_bytes, world, e2e_steps, e2e_total)

    peak, peak_kind = measured_peaks()
    traffic = None
    if os.path.exists(PROFILE_SUMMARY):
        with open(PROFILE_SUMMARY) as f:
            prof = json.load(f)
        if prof.get("kernel_hash") == kernel_hash():
            traffic = prof.get("dram_bytes_per_launch")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle.build

        oracle.build.build()
        n_req = wl.B
        v, dt, passes = cpu_oracle_sample(wl, n_req, min_seconds=10.0)
        cpu = {"value": v, "unit": "GB/s", "cores": os.cpu_count() or 1, "kind": "oracle",
               "sample": f"all {n_req} requests, all rows, {passes} passes ({dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "per_gpu_batch": B,
                       "l2": f"inputs larger than L2 (KV pool {kp.numel() * 2 * 2 / 2**20:.0f} MiB"
                             f" vs {L2_BYTES // 2**20} MiB L2), no flush"},
            "us_per_step": ms_per_step * 1e3,
            "naive_expand": {"us_per_step": naive_ms * 1e3,
                             "kv_gbs_unique": unique_bytes / (naive_ms * 1e-3) / 1e9,
                             "kv_gbs_read": naive_bytes / (naive_ms * 1e-3) / 1e9,
                             "speedup_cascade_vs_naive": naive_ms / ms_per_step},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": unique_bytes,
                         "launch_us": launch_ms * 1e3},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "us_per_step": e2e_total / e2e_steps * 1e3},
            "gpu_launches": args.steps,
            "clocks": clock_info,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_init()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
