"""Run one entry point of libcpa.so on a named workload, for profiling.

    python -m cascade_paged_attention_gb300.profile_case --case cascade \
        --config pages_example --warmup 2 --iters 3

Generates the seeded workload, runs `warmup` untimed and `iters` timed calls
on the current stream and prints the mean time per call (CUDA events).  Meant
to be wrapped by ncu (one kernel name, a few launches).

With ``--trace OUT.json`` it loads the diagnostic build (trace hooks compiled
in), runs one more call with the trace buffer attached and writes every CTA's
start, end, producer-done, MMA-done and epilogue-done times (ns from the
launch's first start) and its tile and unit counts, with a summary of how
the CTAs' end times spread.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import cascade_paged_attention_gb300 as cpa  # noqa: E402
import cpa_synth  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=["cascade", "naive", "pass_a", "pass_b", "prefill", "tree",
                                       "tree_pass_b", "shared", "cascade_fp8"],
                    default="cascade")
    ap.add_argument("--config", default="pages_example")
    ap.add_argument("--hit", type=float, default=0.5, help="prefill: cached fraction h")
    ap.add_argument("--scales", default="channel", help="cascade_fp8: tensor or channel")
    ap.add_argument("--batch", type=int, default=0, help="override B")
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--graph", action="store_true",
                    help="also replay the iters calls from one captured CUDA graph")
    ap.add_argument("--trace", default="",
                    help="write per-CTA times of one call (diagnostic build) to this JSON file")
    args = ap.parse_args()

    if args.trace:
        from cascade_paged_attention_gb300 import build as cbuild

        os.environ["CPA_LIBRARY"] = cbuild.build(trace=True)
    cpa.build_library()
    dev = torch.device("cuda:0")

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(dev)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    if args.case == "prefill":
        c = dict(cpa_synth.PREFILL_CONFIG)
        c.pop("hits")
        if args.batch:
            c["B"] = args.batch
        H = int(args.hit * c["N"])
        wl = cpa_synth.make_prefill(H=H, **c)
        q, kp, vp, pt = bf(wl.q), bf(wl.k_pages), bf(wl.v_pages), i32(wl.page_table)

        def call():
            cpa.cpa_prefill_hit(q, kp, vp, pt, wl.B, wl.N, wl.H)
        work = f"prefill B={wl.B} N={wl.N} H={wl.H}: {wl.visible_pairs() * wl.B * wl.H_q} pairs"
    elif args.case == "cascade_fp8":
        cfg = dict(cpa_synth.VERIFY_CONFIGS[args.config])
        if args.batch:
            cfg["B"] = args.batch
        wl = cpa_synth.make_verify_fp8(scales=args.scales, **cfg)
        q = bf(wl.q)
        kp = torch.from_numpy(np.ascontiguousarray(wl.k_pages)).to(dev)
        vp = torch.from_numpy(np.ascontiguousarray(wl.v_pages)).to(dev)
        ks = torch.from_numpy(np.ascontiguousarray(wl.k_scale, dtype=np.float32)).to(dev)
        vs = torch.from_numpy(np.ascontiguousarray(wl.v_scale, dtype=np.float32)).to(dev)
        ppt, dpt, lens = i32(wl.prefix_page_table), i32(wl.draft_page_table), i32(wl.prefix_lens)
        mpl = wl.max_prefix_len

        def call():
            cpa.cpa_cascade_verify_fp8(q, kp, vp, ks, vs, ppt, dpt, lens, wl.topk, wl.S, mpl)
        work = (f"{args.config} FP8 ({args.scales} scales): unique KV "
                f"{wl.unique_kv_tokens() * wl.kv_bytes_per_token() / 1e6:.1f} MB")
    elif args.case == "shared":
        cfg = dict(cpa_synth.SHARED_CONFIGS[args.config])
        wl = cpa_synth.make_shared_verify(**cfg)
        q, kp, vp = bf(wl.q), bf(wl.k_pages), bf(wl.v_pages)
        spt, ppt = i32(wl.shared_page_table), i32(wl.prefix_page_table)
        dpt, lens = i32(wl.draft_page_table), i32(wl.prefix_lens)
        mpl = wl.max_prefix_len

        def call():
            cpa.cpa_cascade_verify_shared(q, kp, vp, spt, wl.shared_len, ppt, dpt, lens, wl.topk,
                                          wl.S, mpl)
        work = (f"{args.config}: unique KV {wl.unique_kv_tokens() * wl.kv_bytes_per_token() / 1e6:.1f}"
                f" MB")
    elif args.case in ("tree", "tree_pass_b"):
        cfg = dict(cpa_synth.TREE_CONFIGS[args.config])
        if args.batch:
            cfg["B"] = args.batch
        wl = cpa_synth.make_tree_verify(**cfg)
        q, kp, vp = bf(wl.q), bf(wl.k_pages), bf(wl.v_pages)
        ppt, tpt, lens = i32(wl.prefix_page_table), i32(wl.tree_page_table), i32(wl.prefix_lens)
        par = i32(wl.parents)
        mpl = wl.max_prefix_len

        def call():
            if args.case == "tree":
                cpa.cpa_tree_verify(q, kp, vp, ppt, tpt, lens, par, mpl)
            else:
                cpa.cpa_tree_pass_b(q, kp, vp, tpt, par)
        work = (f"{args.config}: unique KV {wl.unique_kv_tokens() * wl.kv_bytes_per_token() / 1e6:.1f}"
                f" MB")
    else:
        cfg = dict(cpa_synth.VERIFY_CONFIGS[args.config])
        if args.batch:
            cfg["B"] = args.batch
        wl = cpa_synth.make_verify(**cfg)
        q, kp, vp = bf(wl.q), bf(wl.k_pages), bf(wl.v_pages)
        ppt, dpt, lens = i32(wl.prefix_page_table), i32(wl.draft_page_table), i32(wl.prefix_lens)
        mpl = wl.max_prefix_len

        def call():
            if args.case == "cascade":
                cpa.cpa_cascade_verify(q, kp, vp, ppt, dpt, lens, wl.topk, wl.S, mpl)
            elif args.case == "naive":
                cpa.cpa_naive_expand_verify(q, kp, vp, ppt, dpt, lens, wl.topk, wl.S, mpl)
            elif args.case == "pass_a":
                cpa.cpa_cascade_pass_a(q, kp, vp, ppt, lens, wl.topk, wl.S, mpl)
            else:
                cpa.cpa_cascade_pass_b(q, kp, vp, dpt, wl.B, wl.topk, wl.S)
        work = (f"{args.config}: unique KV {wl.unique_kv_tokens() * wl.kv_bytes_per_token() / 1e6:.1f}"
                f" MB")

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.iters):
        call()
    e.record()
    torch.cuda.synchronize()
    print(f"{args.case} {work}: {s.elapsed_time(e) / args.iters * 1e3:.1f} us/call")
    if args.graph:
        # the same calls without host gaps between them: the kernel time alone
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(args.iters):
                call()
        g.replay()
        torch.cuda.synchronize()
        s.record()
        g.replay()
        e.record()
        torch.cuda.synchronize()
        print(f"{args.case} {work}: {s.elapsed_time(e) / args.iters * 1e3:.1f} us/call (graph)")
    if args.trace:
        trace_one_call(call, args.trace, work)


def trace_one_call(call, out_path: str, work: str):
    """Run `call` once with the trace buffer attached; summarise per-CTA times."""
    import ctypes
    import json

    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    base, per = 4 * 64 * 1024, 8
    buf = torch.zeros(base + per * n_sm, dtype=torch.int64, device="cuda:0")
    L = cpa.lib()
    L.cpa_trace_set_buffer.restype = ctypes.c_int
    L.cpa_trace_set_buffer.argtypes = [ctypes.c_void_p]
    if L.cpa_trace_set_buffer(ctypes.c_void_p(buf.data_ptr())) != 0:
        raise RuntimeError("cpa_trace_set_buffer failed")
    call()
    torch.cuda.synchronize()
    L.cpa_trace_set_buffer(None)
    cta = buf[base:].view(n_sm, per).cpu().numpy().astype(np.int64)
    # the per-tile event rows of CTAs 0..3 (clock64 stamps), for a closer look
    np.save(os.path.splitext(out_path)[0] + "_events.npy",
            buf[:base].view(4, 64, 1024).cpu().numpy())
    used = cta[:, 5] > 0
    t0 = int(cta[used, 0].min())
    rel = lambda col: [int(x - t0) if u else None for x, u in zip(cta[:, col], used)]
    ends = np.array([int(x - t0) for x, u in zip(cta[:, 1], used) if u])
    starts = np.array([int(x - t0) for x, u in zip(cta[:, 0], used) if u])
    summary = {
        "work": work, "ctas_with_work": int(used.sum()),
        "start_ns": {"min": int(starts.min()), "max": int(starts.max())},
        "end_ns": {"min": int(ends.min()), "p10": float(np.percentile(ends, 10)),
                   "median": float(np.median(ends)), "p90": float(np.percentile(ends, 90)),
                   "max": int(ends.max())},
        "tail_ns": int(ends.max() - np.median(ends)),
        "slowest_ctas": [int(i) for i in np.argsort(-np.where(used, cta[:, 1], 0))[:8]],
    }
    out = {"summary": summary,
           "per_cta": {"start": rel(0), "end": rel(1), "producer_done": rel(2),
                       "mma_done": rel(3), "epilogue_done": rel(4),
                       "tiles": [int(x) for x in cta[:, 5]], "units": [int(x) for x in cta[:, 6]]}}
    with open(out_path, "w") as f:
        json.dump(out, f)
    print(json.dumps(summary))


if __name__ == "__main__":
    main()
