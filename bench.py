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


def recorded_traffic(path: str, current_hash: str):
    """DRAM bytes per launch from a committed capture summary, or None when the
    file is missing or was taken on other kernel sources (its hash differs)."""
    if not os.path.exists(path):
        return None
    with open(path) as f:
        prof = json.load(f)
    if prof.get("kernel_hash") != current_hash:
        return None
    return prof.get("dram_bytes_per_launch")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_bf16_tflops():
    """Burst bf16 dense peak (a kernel timed alone), measured if recorded."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1900.0


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


def pct(xs, q):
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q))


def launch_stats(per_ms):
    """Per-launch CUDA-event times (ms) -> mean / median / p10 / p90 in us."""
    return {"mean": 1e3 * float(np.mean(per_ms)), "median": 1e3 * pct(per_ms, 50),
            "p10": 1e3 * pct(per_ms, 10), "p90": 1e3 * pct(per_ms, 90), "n": len(per_ms)}


class Timer:
    """CUDA-event timing on one stream, with an optional L2 flush before every call."""

    def __init__(self, torch, stream, flush_bytes: int):
        self.torch = torch
        self.stream = stream
        # writing a buffer twice the size of L2 evicts every line a call could reuse
        self.flush_buf = torch.empty(flush_bytes, dtype=torch.uint8, device=stream.device)

    def flush(self):
        self.flush_buf.fill_(1)

    def back_to_back(self, fn, steps, warmup, barrier=lambda: None):
        """`steps` calls back to back: (total ms, per-call ms)."""
        torch = self.torch
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        evs[0].record(self.stream)
        for i in range(steps):
            fn()
            evs[i + 1].record(self.stream)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
        return evs[0].elapsed_time(evs[-1]), per

    def cold(self, fn, iters, warmup=3):
        """Per-call ms of `iters` calls, each after an L2 flush (flush not timed)."""
        torch = self.torch
        for _ in range(warmup):
            fn()
        per = []
        for _ in range(iters):
            self.flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(self.stream)
            fn()
            b.record(self.stream)
            b.synchronize()
            per.append(a.elapsed_time(b))
        return per


def to_device(torch, dev, a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(dtype) if dtype is not None else t).to(dev)


def verify_config_row(torch, cpa, cpa_synth, timer, dev, name, peak, iters, cpu, rows_budget):
    """Cascade and naive expand on one verify workload (cold L2), and the oracle beside them."""
    wl = cpa_synth.make_verify(**cpa_synth.VERIFY_CONFIGS[name])
    q = to_device(torch, dev, wl.q, torch.bfloat16)
    kp = to_device(torch, dev, wl.k_pages, torch.bfloat16)
    vp = to_device(torch, dev, wl.v_pages, torch.bfloat16)
    ppt, dpt, lens = (to_device(torch, dev, a) for a in (wl.prefix_page_table,
                                                         wl.draft_page_table, wl.prefix_lens))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], wl.H_q, dtype=torch.float32, device=dev)
    mpl = wl.max_prefix_len

    def cascade():
        cpa.cpa_cascade_verify(q, kp, vp, ppt, dpt, lens, wl.topk, wl.S, max_prefix_len=mpl,
                               o=o, lse=lse)

    def naive():
        cpa.cpa_naive_expand_verify(q, kp, vp, ppt, dpt, lens, wl.topk, wl.S,
                                    max_prefix_len=mpl, o=o, lse=lse)

    unique = wl.unique_kv_tokens() * wl.kv_bytes_per_token()
    c = launch_stats(timer.cold(cascade, iters))
    n = launch_stats(timer.cold(naive, max(50, iters // 2)))
    row = {
        "config": name, "unique_kv_bytes": unique,
        "naive_kv_bytes": wl.naive_kv_tokens() * wl.kv_bytes_per_token(),
        "cascade_us": c, "naive_us": n,
        "cascade_gbs": unique / (c["median"] * 1e-6) / 1e9,
        "frac_of_hbm_peak": unique / (c["median"] * 1e-6) / 1e9 / peak,
        "speedup_cascade_vs_naive": n["median"] / c["median"],
    }
    del q, kp, vp
    torch.cuda.empty_cache()
    if cpu:
        import oracle

        n_rows = wl.n_tokens * wl.H_q
        rows = np.arange(min(n_rows, rows_budget), dtype=np.int64)
        t0 = time.perf_counter()
        oracle.verify_wl(wl, rows=rows)
        dt = time.perf_counter() - t0
        # unique KV bytes scaled by the share of (row, key) pairs the sample covered
        keys = (wl.prefix_lens.astype(np.int64) + wl.S).repeat(wl.topk * wl.S * wl.H_q)
        share = float(keys[:len(rows)].sum()) / float(keys.sum())
        row["oracle"] = {"value": unique * share / dt / 1e9, "unit": "GB/s",
                         "cores": os.cpu_count() or 1, "kind": "oracle", "seconds": dt,
                         "sample": f"first {len(rows)} of {n_rows} (token, head) rows"}
    return row


def prefill_rows(torch, cpa, cpa_synth, timer, dev, peak_tf, iters, cpu):
    """Prefix-hit prefill (B=8, N=8192) at h = 0, 0.5, 0.75: time, TFLOP/s of visible
    pairs, T(h)/T(0) beside 1 - h^2, and the oracle on sampled rows."""
    c = dict(cpa_synth.PREFILL_CONFIG)
    hits = c.pop("hits")
    out, t_zero = [], None
    for h in hits:
        H = int(h * c["N"])
        wl = cpa_synth.make_prefill(H=H, **c)
        q = to_device(torch, dev, wl.q, torch.bfloat16)
        kp = to_device(torch, dev, wl.k_pages, torch.bfloat16)
        vp = to_device(torch, dev, wl.v_pages, torch.bfloat16)
        pt = to_device(torch, dev, wl.page_table)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[0], wl.H_q, dtype=torch.float32, device=dev)

        def call():
            cpa.cpa_prefill_hit(q, kp, vp, pt, wl.B, wl.N, wl.H, o=o, lse=lse)

        st = launch_stats(timer.cold(call, iters))
        flops = 4.0 * wl.head_dim * wl.H_q * wl.B * wl.visible_pairs()
        tf = flops / (st["median"] * 1e-6) / 1e12
        if t_zero is None:
            t_zero = st["median"]
        row = {"config": f"prefill_hit h={h}", "B": wl.B, "N": wl.N, "H": wl.H,
               "us": st, "flops": flops, "tflops": tf, "frac_of_bf16_peak": tf / peak_tf,
               "t_over_t0": st["median"] / t_zero,
               "pair_ratio": 1.0 - (wl.H * (wl.H + 1)) / (wl.N * (wl.N + 1))}
        del q, kp, vp
        torch.cuda.empty_cache()
        if cpu:
            import oracle

            M = wl.N - wl.H
            rng = np.random.default_rng(7)
            toks = np.sort(rng.choice(wl.B * M, size=64, replace=False))
            rows = (toks[:, None] * wl.H_q + np.arange(wl.H_q)[None, :]).reshape(-1)
            t0 = time.perf_counter()
            oracle.prefill_wl(wl, rows=rows)
            dt = time.perf_counter() - t0
            keys = float(sum(wl.H + (int(t) % M) + 1 for t in toks) * wl.H_q)
            row["oracle"] = {"value": 4.0 * wl.head_dim * keys / dt / 1e12, "unit": "TFLOP/s",
                             "cores": os.cpu_count() or 1, "kind": "oracle", "seconds": dt,
                             "sample": f"64 random suffix tokens x all {wl.H_q} heads",
                             "extrapolated_full_s": dt * flops / (4.0 * wl.head_dim * keys)}
        out.append(row)
    return out


def next_rows(torch, cpa, cpa_synth, timer, dev, peak, iters, bf16_us):
    """The built 'next' paths on the pages' example request shape (cold L2):
    FP8 KV pages, one draft tree per request, a system prompt shared by all."""
    out = []
    # FP8 E4M3 pools with per-channel scales
    wl = cpa_synth.make_verify_fp8(scales="channel", **cpa_synth.VERIFY_CONFIGS[CFG])
    q = to_device(torch, dev, wl.q, torch.bfloat16)
    kp, vp = (to_device(torch, dev, a) for a in (wl.k_pages, wl.v_pages))
    ks, vs = (to_device(torch, dev, np.ascontiguousarray(a, dtype=np.float32))
              for a in (wl.k_scale, wl.v_scale))
    ppt, dpt, lens = (to_device(torch, dev, a) for a in (wl.prefix_page_table,
                                                         wl.draft_page_table, wl.prefix_lens))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], wl.H_q, dtype=torch.float32, device=dev)

    def fp8():
        cpa.cpa_cascade_verify_fp8(q, kp, vp, ks, vs, ppt, dpt, lens, wl.topk, wl.S,
                                   max_prefix_len=wl.max_prefix_len, o=o, lse=lse)

    st = launch_stats(timer.cold(fp8, iters))
    b = wl.unique_kv_tokens() * wl.kv_bytes_per_token()
    out.append({"config": "pages_example, FP8 E4M3 KV pages (per-channel scales)",
                "unique_kv_bytes": b, "us": st,
                "gbs": b / (st["median"] * 1e-6) / 1e9,
                "frac_of_hbm_peak": b / (st["median"] * 1e-6) / 1e9 / peak,
                "time_vs_bf16_cascade": st["median"] / bf16_us})
    del q, kp, vp
    # one 20-node draft tree per request
    tw = cpa_synth.make_tree_verify(**cpa_synth.TREE_CONFIGS["tree_pages_example"])
    q, kp, vp = (to_device(torch, dev, a, torch.bfloat16) for a in (tw.q, tw.k_pages, tw.v_pages))
    ppt, tpt, lens, par = (to_device(torch, dev, a) for a in (
        tw.prefix_page_table, tw.tree_page_table, tw.prefix_lens, tw.parents))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], tw.H_q, dtype=torch.float32, device=dev)

    def tree():
        cpa.cpa_tree_verify(q, kp, vp, ppt, tpt, lens, par, max_prefix_len=tw.max_prefix_len,
                            o=o, lse=lse)

    st = launch_stats(timer.cold(tree, iters))
    b = tw.unique_kv_tokens() * tw.kv_bytes_per_token()
    out.append({"config": "tree_pages_example: B=64, one 20-node draft tree each, L=2000",
                "unique_kv_bytes": b, "us": st,
                "gbs": b / (st["median"] * 1e-6) / 1e9,
                "frac_of_hbm_peak": b / (st["median"] * 1e-6) / 1e9 / peak,
                "time_vs_chain_cascade": st["median"] / bf16_us})
    del q, kp, vp
    # multi-level: 1024 shared + 976 own prefix tokens
    sw = cpa_synth.make_shared_verify(**cpa_synth.SHARED_CONFIGS["shared_pages_example"])
    q, kp, vp = (to_device(torch, dev, a, torch.bfloat16) for a in (sw.q, sw.k_pages, sw.v_pages))
    spt, ppt, dpt, lens = (to_device(torch, dev, a) for a in (
        sw.shared_page_table, sw.prefix_page_table, sw.draft_page_table, sw.prefix_lens))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], sw.H_q, dtype=torch.float32, device=dev)

    def shared():
        cpa.cpa_cascade_verify_shared(q, kp, vp, spt, sw.shared_len, ppt, dpt, lens, sw.topk,
                                      sw.S, max_prefix_len=sw.max_prefix_len, o=o, lse=lse)

    st = launch_stats(timer.cold(shared, iters))
    b = sw.unique_kv_tokens() * sw.kv_bytes_per_token()
    out.append({"config": "shared_pages_example: B=64, 1024 shared + 976 own prefix tokens, "
                          "topk=4, S=5",
                "unique_kv_bytes": b, "us": st,
                "gbs": b / (st["median"] * 1e-6) / 1e9,
                "frac_of_hbm_peak": b / (st["median"] * 1e-6) / 1e9 / peak,
                "time_vs_single_level_cascade": st["median"] / bf16_us})
    del q, kp, vp
    torch.cuda.empty_cache()
    return out


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
    timer = Timer(torch, stream, 2 * L2_BYTES)

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

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    total_ms, per_ms = timer.back_to_back(cascade, args.steps, args.warmup, barrier)
    clock_info = clocks.stop()
    total_ms = max_over_ranks(total_ms)
    ms_per_step = total_ms / args.steps
    value = weak_scaling_gbs(unique_bytes, world, args.steps, total_ms)
    ls = launch_stats(per_ms)
    launch_ms = ls["mean"] * 1e-3
    achieved = unique_bytes / (launch_ms * 1e-3) / 1e9

    naive_total, _ = timer.back_to_back(naive, args.steps, args.warmup, barrier)
    naive_total = max_over_ranks(naive_total)
    naive_ms = naive_total / args.steps

    # the same call with L2 flushed before every launch (cold-L2 figure)
    cold = launch_stats(timer.cold(cascade, args.cold_iters))
    cold_naive = launch_stats(timer.cold(naive, max(50, args.cold_iters // 2)))

    # end to end through the public API: host inputs -> device, call, result -> host.
    # The two KV pools go up on two streams at once (one copy stream does not fill
    # the host link); the call waits for both.
    h_o = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_ppt, h_dpt, h_lens))
    d2h = h_o.numel() * 2 + h_lse.numel() * 4
    side = torch.cuda.Stream(dev)

    def e2e_step():
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            vp.copy_(h_v, non_blocking=True)
        q.copy_(h_q, non_blocking=True)
        kp.copy_(h_k, non_blocking=True)
        ppt.copy_(h_ppt, non_blocking=True)
        dpt.copy_(h_dpt, non_blocking=True)
        lens.copy_(h_lens, non_blocking=True)
        stream.wait_stream(side)
        cascade()
        h_o.copy_(o, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 10))
    e2e_total, _ = timer.back_to_back(e2e_step, e2e_steps, args.warmup, barrier)
    e2e_total = max_over_ranks(e2e_total)
    e2e_value = weak_scaling_gbs(unique_bytes, world, e2e_steps, e2e_total)

    peak, peak_kind = measured_peaks()
    peak_tf = measured_bf16_tflops()
    traffic = recorded_traffic(PROFILE_SUMMARY, kernel_hash())

    do_cpu = rank == 0 and not args.no_cpu_baseline
    configs = []
    if rank == 0 and args.configs == "all":
        for name in ("llama3_8b", "long_variable"):
            configs.append(verify_config_row(torch, cpa, cpa_synth, timer, dev, name, peak,
                                             args.cold_iters, do_cpu, rows_budget=4096))
        configs.extend(prefill_rows(torch, cpa, cpa_synth, timer, dev, peak_tf,
                                    max(50, args.cold_iters // 2), do_cpu))
        configs.extend(next_rows(torch, cpa, cpa_synth, timer, dev, peak, args.cold_iters,
                                 cold["median"]))

    cpu = None
    if do_cpu:
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
                             f" vs {L2_BYTES // 2**20} MiB L2), no flush between the timed "
                             f"steps; cold_l2 flushes L2 before every launch"},
            "us_per_step": ms_per_step * 1e3,
            "naive_expand": {"us_per_step": naive_ms * 1e3,
                             "kv_gbs_unique": unique_bytes / (naive_ms * 1e-3) / 1e9,
                             "kv_gbs_read": naive_bytes / (naive_ms * 1e-3) / 1e9,
                             "speedup_cascade_vs_naive": naive_ms / ms_per_step},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": unique_bytes,
                         "launch_us": ls["mean"], "launch_us_median": ls["median"],
                         "launch_us_p10": ls["p10"], "launch_us_p90": ls["p90"]},
            "cold_l2": {"cascade_us": cold, "naive_us": cold_naive,
                        "cascade_gbs": unique_bytes / (cold["median"] * 1e-6) / 1e9,
                        "frac": unique_bytes / (cold["median"] * 1e-6) / 1e9 / peak,
                        "speedup_cascade_vs_naive": cold_naive["median"] / cold["median"]},
            "configs": configs,
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
    ap.add_argument("--configs", choices=["all", "none"], default="all",
                    help="also time the other verify configs and the prefill (cold L2)")
    ap.add_argument("--cold-iters", type=int, default=100,
                    help="launches timed one by one after an L2 flush")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_init()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
