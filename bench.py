#!/usr/bin/env python
"""Decode-step benchmark of the sparse-MLA path on one GB300 (or N, weak scaling).

One step = indexer score -> top-K -> fused resolve -> sparse MLA decode of the
4 MLA layers of one IndexShare group, captured in a CUDA graph and replayed.
Workload (default): full residency, 32 requests x 65,536 tokens, top-K 2048,
64x128 E4M3 indexer, 128 MLA heads over 576-dim latent rows stored as 656-B
FP8 rows, page 64, 4 layers.  Synthetic seeded inputs, resident in HBM
before the timed region; L2 is flushed (256 MiB write, then a 256 MiB read of a
second buffer, so no dirty lines carry into the step) before every timed step.

Output: one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(the only reference implementation there is) on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("resolved top-K rows/s & decode-step µs per layer at 1 GB300; "
          "% of HBM/host-link peak")

WORKLOAD = dict(name="full_residency_32x65536_k2048", B=32, N=65536, nq=1, K=2048, Hi=64, Di=128,
                H=128, L=4, P=64, seed=0)

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p["bf16_tflops_sustained"]),
                    sm_max=float(p.get("sm_max_mhz", 2070.0)), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, sm_max=2070.0, src="fallback")


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # nvidia-smi is sampling before the timed region starts
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
def setup_pool(w, device):
    import torch
    from sparse_mla_kv_fp8_gb300 import hs
    from sparse_mla_kv_fp8_gb300 import workload as wl
    B, N, P, L = w["B"], w["N"], w["P"], w["L"]
    pages = B * ((N + P - 1) // P)
    cfg = hs.make_config(max_requests=B, max_tokens=N, page_tokens=P, top_k=w["K"],
                         num_spec=w["nq"] - 1, tail_tokens=0, num_mla_layers=L,
                         mla_heads=w["H"], idx_heads=w["Hi"], idx_dim=w["Di"],
                         row_fmt=hs.HS_ROW_E4M3_656, idx_fmt=hs.HS_IDX_E4M3,
                         gpu_blocks=pages, host_blocks=0)
    pool = hs.Pool(cfg, device=device)
    for b in range(B):
        pool.open(b, hs.HS_FULL)
        for t0 in range(0, N, 16384):
            n = min(16384, N - t0)
            rows = wl.mla_rows(w["seed"], b, t0, n, L, wl.ROW_E4M3_656, device=device)
            keys = wl.idx_keys(w["seed"], b, t0, n, w["Di"], wl.IDX_E4M3, device=device)
            pool.append(b, rows, keys)
            del rows, keys
    torch.cuda.synchronize()
    return pool


def step_inputs(w, s, device):
    import torch
    from sparse_mla_kv_fp8_gb300 import workload as wl
    B, nq = w["B"], w["nq"]
    q = torch.stack([wl.idx_query(w["seed"], b, s, nq, w["Hi"], w["Di"], wl.IDX_E4M3, device)
                     for b in range(B)]).contiguous()
    wt = torch.stack([wl.idx_weights(w["seed"], b, s, nq, w["Hi"], device) for b in range(B)]).contiguous()
    qm = wl.mla_query(w["seed"], s, B, nq, w["H"], w["L"], device).contiguous()
    return q, wt, qm


def algorithmic(w):
    """Algorithmic bytes / flops the method must move per launch of each stage."""
    B, N, nq, K, Hi, Di, H, R = w["B"], w["N"], w["nq"], w["K"], w["Hi"], w["Di"], w["H"], 656
    return {
        "indexer": dict(bytes=B * N * (Di + 4) + B * nq * Hi * (Di + 4), flops=2 * B * nq * N * Hi * Di),
        "topk": dict(bytes=B * nq * K * 4, flops=0),
        "resolve": dict(bytes=B * nq * K * 4 * 3, flops=0),
        "attention": dict(bytes=B * nq * K * R + B * nq * H * 576 * 2 + B * nq * H * 512 * 2,
                          flops=2 * B * nq * K * H * 1088),
    }


def max_over_ranks(x: float, device) -> float:
    """The slowest rank's value (every rank gets it)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rows_per_s(world: int, rows_per_step_per_rank: int, ms_per_step: float) -> float:
    """Weak scaling: every rank resolves and attends its own requests' rows;
    the job's rate is all ranks' rows over the slowest rank's step time."""
    return world * rows_per_step_per_rank / (ms_per_step / 1e3)


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    from sparse_mla_kv_fp8_gb300 import hs

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    w = dict(WORKLOAD)
    if args.requests:
        w["B"] = args.requests
    B, nq, K, L, H = w["B"], w["nq"], w["K"], w["L"], w["H"]
    pool = setup_pool(w, device)
    tau = 1.0 / math.sqrt(576)
    n_inputs = 4
    inputs = [step_inputs(w, s + 1, device) for s in range(n_inputs)]
    q = inputs[0][0].clone()
    wt = inputs[0][1].clone()
    qm = inputs[0][2].clone()
    out = torch.empty((L, B, nq, H, 512), dtype=torch.bfloat16, device=device)
    topk = torch.empty((B, nq, K), dtype=torch.int32, device=device)
    rid = torch.empty((B, nq, K), dtype=torch.int32, device=device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    scrub = torch.zeros(256 << 20, dtype=torch.uint8, device=device)

    def flush_l2():
        flush.zero_()  # write a buffer larger than L2 ...
        scrub.max()    # ... then read another, so the write-back of those dirty lines lands here

    stream = torch.cuda.Stream(device)
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        pool.step(B, nq, q, wt, qm, tau, out, topk, rid, stream=stream)  # eager warm-up
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            pool.step(B, nq, q, wt, qm, tau, out, topk, rid, stream=stream)
    torch.cuda.synchronize()
    if pool.get_error() != hs.HS_OK:
        raise RuntimeError("device error during warm-up")

    def load(i):
        a, b_, c = inputs[i % n_inputs]
        q.copy_(a)
        wt.copy_(b_)
        qm.copy_(c)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            load(i)
            graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: graph replays, L2 flushed before each step ----
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    with ClockSampler(local_rank) as clk:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                load(i)
                flush_l2()
                starts[i].record(stream)
                graph.replay()
                ends[i].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t_wall = time.perf_counter() - t_wall
        # ---- per-stage timing (same step, eager, events between the stages) ----
        stage = stage_times(pool, w, inputs, q, wt, qm, out, topk, rid, flush_l2, stream,
                            min(args.steps, 50))
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    if pool.get_error() != hs.HS_OK:
        raise RuntimeError("device error in the timed region")
    if world > 1:
        total_ms = max_over_ranks(total_ms, device)
    ms_per_step = total_ms / args.steps
    rows_per_step = B * nq * K * L
    value = whole_job_rows_per_s(world, rows_per_step, ms_per_step)

    # ---- end to end: host inputs in, result out, through the public API ----
    e2e = end_to_end(pool, w, inputs, stream, args.steps, device)

    peaks = _peaks()
    alg = algorithmic(w)
    roof, roof_all = roofline(stage, alg, peaks, w)
    step_bytes = alg["indexer"]["bytes"] + alg["topk"]["bytes"] + alg["resolve"]["bytes"] + L * alg["attention"]["bytes"]
    res = {
        "metric": METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "us_per_layer": ms_per_step * 1e3 / L,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "dtype_note": "indexer: E4M3 MMA operands, fp32 accumulate; attention (the dominant kernel): E4M3 rows dequantised to fp16 MMA operands with fp16 queries and probabilities, fp32 accumulate and softmax",
        "data": "synthetic (seeded; indexer values m/8 in E4M3, latent N(0,1) quantised to E4M3 + fp32 group scales)",
        "config": {"workload": w["name"], "requests_per_gpu": B, "tokens_per_request": w["N"],
                   "queries_per_request": nq, "top_k": K, "indexer": f"{w['Hi']}x{w['Di']} e4m3",
                   "mla_heads": H, "latent": 576, "row_bytes": 656, "mla_layers": L,
                   "page_tokens": w["P"], "residency": "full", "graph": "cuda graph replay",
                   "l2": "flushed before each timed step (256 MiB write, then a 256 MiB read of a second buffer)"},
        "stage_us": {k: v * 1e3 for k, v in stage.items()},
        "hbm_frac_step": (step_bytes / (ms_per_step / 1e3)) / (peaks["hbm"] * 1e9),
        "roofline": roof,
        "stage_roofline": roof_all,
        "host_link": host_link(device) if not args.no_host_link else None,
        "e2e": e2e,
        "gpu_launches": pool.step_kernel_count(B, nq) * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": t_wall,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    pool.close()
    return res


HOLD_CYCLES = 1_000_000  # ~0.5 ms of SM clock: longer than enqueueing one step's stages


def stage_times(pool, w, inputs, q, wt, qm, out, topk, rid, flush_l2, stream, steps):
    """Average ms per launch of each stage, CUDA events on the launching stream
    (the stages are queued behind a spin kernel, so they run back to back)."""
    import torch
    B, nq, L = w["B"], w["nq"], w["L"]
    tau = 1.0 / math.sqrt(576)
    acc = {"indexer": 0.0, "topk": 0.0, "resolve": 0.0, "attention": 0.0}
    scores = pool_scores = None
    stride = w["N"]
    scores = torch.empty((B, nq, stride), dtype=torch.float32, device=q.device)
    for i in range(steps):
        a, b_, c = inputs[i % len(inputs)]
        q.copy_(a)
        wt.copy_(b_)
        qm.copy_(c)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4 + L)]
        with torch.cuda.stream(stream):
            flush_l2()
            # hold the stream while the host enqueues every stage, so that the
            # spans below time the kernels and not the host's launch calls
            torch.cuda._sleep(HOLD_CYCLES)
            ev[0].record(stream)
            pool.indexer_score(q, wt, B, nq, scores, stride, stream=stream)
            ev[1].record(stream)
            pool.topk(scores, stride, B, nq, topk, stream=stream)
            ev[2].record(stream)
            pool.resolve(topk, B, nq, rid, stream=stream)
            ev[3].record(stream)
            for l in range(L):
                pool.sparse_mla_decode(l, qm[l], rid, B, nq, tau, out[l], None, stream=stream)
                ev[4 + l].record(stream)
        torch.cuda.synchronize()
        acc["indexer"] += ev[0].elapsed_time(ev[1])
        acc["topk"] += ev[1].elapsed_time(ev[2])
        acc["resolve"] += ev[2].elapsed_time(ev[3])
        acc["attention"] += ev[3].elapsed_time(ev[3 + L]) / L
    del pool_scores
    return {k: v / steps for k, v in acc.items()}


# DRAM bytes per launch from one ncu capture of 16 requests (scaled x2 to 32
# requests), valid only for the kernel sources they were taken
# on (the kernel's .cu and the shared device header, hashed together).
TRAFFIC = {"attention": (("attention.cu", "tc.cuh"), "b1be9eaf94bcde78", 2 * (27643264 + 3392)),
           "indexer": (("indexer.cu", "tc.cuh"), "9a84ea0a9b297437", 2 * (138577152 + 2479616)),
           "topk": (("topk.cu", "tc.cuh"), "cf9fadfe87a5a0c2", 2 * 4227328)}


def _traffic(stage, w):
    import hashlib
    # the figures are per launch of the 32-request workload only
    if stage not in TRAFFIC or w != WORKLOAD:
        return None
    files, sha, nbytes = TRAFFIC[stage]
    h = hashlib.sha256()
    for fname in files:
        with open(os.path.join(ROOT, "sparse_mla_kv_fp8_gb300", "csrc", fname), "rb") as f:
            h.update(f.read())
    return nbytes if h.hexdigest()[:16] == sha else None


KERNELS = {"indexer": "indexer_tc_kernel", "topk": "topk_cluster_kernel",
           "resolve": "resolve_plan_kernel", "attention": "attn_tc_kernel"}


def roofline(stage, alg, peaks, w):
    """Roofline of every stage; the one with the largest share of the step is
    the headline.  The attention is a bf16 tensor-core contraction above the
    ridge (425 flop/B vs ~285 for the measured peaks): tensor-bound against the
    sustained bf16 peak (it is timed inside a long step).  The indexer, top-K
    and resolve are memory-bound against the measured HBM copy bandwidth."""
    L = w["L"]
    share = {"indexer": stage["indexer"], "topk": stage["topk"], "resolve": stage["resolve"],
             "attention": stage["attention"] * L}
    tot = sum(share.values())
    out = {}
    for k in share:
        ms = stage[k]
        a = alg[k]
        gbs = a["bytes"] / (ms / 1e3) / 1e9
        if k == "attention":
            tf = a["flops"] / (ms / 1e3) / 1e12
            out[k] = {"kernel": KERNELS[k], "bound": "tensor", "achieved": tf, "peak": peaks["bf16_sus"],
                      "unit": "TFLOP/s", "frac": tf / peaks["bf16_sus"], "traffic": _traffic(k, w),
                      "peak_source": peaks["src"] + " bf16 sustained (fp16 operands: the same dense rate)",
                      "hbm_achieved_gbs": gbs, "hbm_frac": gbs / peaks["hbm"],
                      "share_of_step": share[k] / tot, "us_per_launch": ms * 1e3}
        else:
            out[k] = {"kernel": KERNELS[k], "bound": "hbm", "achieved": gbs, "peak": peaks["hbm"],
                      "unit": "GB/s", "frac": gbs / peaks["hbm"], "traffic": _traffic(k, w),
                      "peak_source": peaks["src"], "share_of_step": share[k] / tot,
                      "us_per_launch": ms * 1e3}
    dom = max(share, key=share.get)
    return out[dom], out


def host_link(device, steps=10):
    """Miss traffic over the host link: a zero-residency batch (4 requests x
    65,536 tokens, 4 layers) whose hot buffers are emptied before every call,
    so each hs_resolve copies 4 x 2048 rows x 4 layers from pinned host memory.
    Peak: a pinned-host -> device cudaMemcpyAsync of 1 GiB."""
    import numpy as np
    import torch
    from sparse_mla_kv_fp8_gb300 import hs
    from sparse_mla_kv_fp8_gb300 import workload as wl
    B, N, K, L, P = 4, 65536, 2048, 4, 64
    pages = N // P
    cfg = hs.make_config(max_requests=B, max_tokens=N, page_tokens=P, top_k=K, num_spec=0,
                         tail_tokens=0, num_mla_layers=L, mla_heads=128, idx_heads=64,
                         idx_dim=128, row_fmt=hs.HS_ROW_E4M3_656, idx_fmt=hs.HS_IDX_E4M3,
                         gpu_blocks=B * (2 * K // P) + 8, host_blocks=B * pages)
    pool = hs.Pool(cfg, device=device)
    for b in range(B):
        pool.open(b, hs.HS_ZERO)
        pool.append(b, wl.mla_rows(7, b, 0, N, L, wl.ROW_E4M3_656, device=device),
                    torch.zeros((N, 128), dtype=torch.uint8, device=device))
    idx = np.stack([wl.drawn_topk(7, b, 1, 0, N, K, P, "uniform_zipf")[None] for b in range(B)])
    topk = torch.from_numpy(idx).to(device)
    rid = torch.empty_like(topk)
    empty_map = np.full(N, -1, np.int32)
    empty_slots = np.full(pool.C, -1, np.int32)
    zero_stamp = np.zeros(pool.C, np.uint32)
    times = []
    for i in range(steps + 2):
        for b in range(B):
            pool.load_state(b, empty_map, empty_slots, zero_stamp, 0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(HOLD_CYCLES)  # the copy kernels start without waiting for the host
        e0.record()
        pool.resolve(topk, B, 1, rid)
        e1.record()
        torch.cuda.synchronize()
        if i >= 2:
            times.append(e0.elapsed_time(e1))
    st = pool.stats()
    pool.close()
    misses_per_call = B * K
    nbytes = misses_per_call * L * 656
    ms = statistics.median(times)
    src = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(1 << 30, dtype=torch.uint8, device=device)
    pk = []
    for i in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        pk.append((1 << 30) / (e0.elapsed_time(e1) / 1e3) / 1e9)
    peak = max(pk)
    ach = nbytes / (ms / 1e3) / 1e9
    del src, dst
    return {"workload": "zero residency, 4 requests x 65,536 tokens, 4 layers, hot buffers emptied "
                        "before each call: 8192 misses x 4 layers x 656 B per hs_resolve",
            "bytes_per_call": nbytes, "us_per_call": ms * 1e3, "achieved_gbs": ach,
            "peak_gbs": peak, "peak_source": "measured cudaMemcpyAsync pinned host -> device, 1 GiB",
            "frac": ach / peak, "timed": "resolve plan + miss copy (events around hs_resolve)",
            "misses_counted": int(st["misses"])}


def end_to_end(pool, w, inputs, stream, steps, device):
    """Same metric through the public API with pinned-host inputs and a
    device->host read of the step's output inside the timed region.  Every
    step copies its own inputs in and its own output back; the copies run on
    two copy streams (the two copy engines) so that step i+1's inputs and
    step i-1's output move while step i computes (double-buffered device
    inputs and outputs, ordered by events)."""
    import torch
    B, nq, K, L, H = w["B"], w["nq"], w["K"], w["L"], w["H"]
    tau = 1.0 / math.sqrt(576)
    host_in = [(a.cpu().pin_memory(), b.cpu().pin_memory(), c.cpu().pin_memory()) for a, b, c in inputs]
    dev_in = [tuple(torch.empty_like(t) for t in inputs[0]) for _ in range(2)]
    outs = [torch.empty((L, B, nq, H, 512), dtype=torch.bfloat16, device=device) for _ in range(2)]
    topk = torch.empty((B, nq, K), dtype=torch.int32, device=device)
    rid = torch.empty_like(topk)
    host_out = torch.empty(outs[0].shape, dtype=outs[0].dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in[0])
    d2h = host_out.numel() * host_out.element_size()
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event(enable_timing=False)
    in_done = [ev() for _ in range(steps)]
    comp_done = [ev() for _ in range(steps)]
    out_done = [ev() for _ in range(steps)]
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(s_in)
    stream.wait_event(ev0)
    s_out.wait_event(ev0)
    for i in range(steps):
        q, wt, qm = dev_in[i % 2]
        out = outs[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(comp_done[i - 2])  # step i-2 has finished with these inputs
            a, b_, c = host_in[i % len(host_in)]
            q.copy_(a, non_blocking=True)
            wt.copy_(b_, non_blocking=True)
            qm.copy_(c, non_blocking=True)
            in_done[i].record(s_in)
        stream.wait_event(in_done[i])
        if i >= 2:
            stream.wait_event(out_done[i - 2])  # step i-2's output has left this buffer
        pool.step(B, nq, q, wt, qm, tau, out, topk, rid, stream=stream)
        comp_done[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[i])
            host_out.copy_(out, non_blocking=True)
            out_done[i].record(s_out)
    s_out.wait_event(comp_done[steps - 1])
    ev1.record(s_out)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    return {"value": B * nq * K * L / (ms / 1e3), "unit": "rows/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "step i+1's inputs and step i-1's output are copied on two copy streams while step i runs"}


# ---------------------------------------------------------------------------
# CPU oracle timing
# ---------------------------------------------------------------------------
def oracle_request_step(w, b, s):
    """One request x one step of the workload through the CPU oracle: indexer
    over all N tokens, top-K, resolve (full residency), attention of the L
    layers.  Returns (seconds, rows)."""
    import numpy as np
    import oracle
    from sparse_mla_kv_fp8_gb300 import workload as wl
    N, nq, K, L, H, P = w["N"], w["nq"], w["K"], w["L"], w["H"], w["P"]
    keys = wl.idx_keys(w["seed"], b, 0, N, w["Di"], wl.IDX_E4M3).numpy()
    q = wl.idx_query(w["seed"], b, s, nq, w["Hi"], w["Di"], wl.IDX_E4M3).numpy()
    wt = wl.idx_weights(w["seed"], b, s, nq, w["Hi"]).numpy()
    qm = wl.mla_query(w["seed"], s, 1, nq, H, L).view(__import__("torch").int16).numpy().view(np.uint16)
    sigma = np.ones(N, np.float32)
    hot = oracle.HotState(2 * K, N)
    resident = oracle.page_resident(oracle.FULL, N, 0, P)
    t0 = time.perf_counter()
    s_all = oracle.indexer_scores(oracle.IDX_E4M3, q, wt, keys, sigma, N)
    idx = np.stack([oracle.topk(s_all[j], oracle.visible(N, nq, j), K) for j in range(nq)])
    t_sel = time.perf_counter() - t0
    r = hot.resolve(resident, P, N, idx)
    assert r["status"] == 0
    # the rows the selection reads (input preparation, not timed)
    sel = np.unique(idx[idx >= 0])
    rows = {}
    for t in sel.tolist():
        rows[t] = None
    import torch
    needed = torch.from_numpy(sel).long()
    blocks = sorted(set((needed // 1024).tolist()))
    allrows = {}
    for blk in blocks:
        chunk = wl.mla_rows(w["seed"], b, blk * 1024, min(1024, N - blk * 1024), L, wl.ROW_E4M3_656)
        for t in sel[(sel >= blk * 1024) & (sel < blk * 1024 + 1024)].tolist():
            allrows[t] = chunk[t - blk * 1024]
    t1 = time.perf_counter()
    tau = 1.0 / math.sqrt(576)
    for j in range(nq):
        ids = idx[j][idx[j] >= 0]
        for l in range(L):
            rr = np.stack([allrows[t][l].numpy() for t in ids.tolist()])
            oracle.attention(oracle.ROW_E4M3_656, qm[l, 0, j], rr, tau)
    t_att = time.perf_counter() - t1
    return t_sel + t_att, nq * K * L


def cpu_baseline(w, budget_s=20.0):
    import oracle
    secs, rows, n = 0.0, 0, 0
    while n == 0 or secs < budget_s * 0.5:
        dt, r = oracle_request_step(w, n % w["B"], 1 + n)
        secs += dt
        rows += r
        n += 1
        if secs > budget_s:
            break
    return {"value": rows / secs, "unit": "rows/s", "cores": oracle.omp_threads(), "kind": "oracle",
            "sample": f"{n} request-step(s) of the workload (indexer over {w['N']} tokens, "
                      f"top-{w['K']}, resolve, {w['L']} layers x {w['H']} heads attention), "
                      f"rows/s = selected rows x layers / oracle seconds"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    w = dict(WORKLOAD)
    for i in range(args.warmup):
        oracle_request_step(w, i % w["B"], 1000 + i)
    secs, rows = 0.0, 0
    for i in range(args.steps):
        dt, r = oracle_request_step(w, i % w["B"], 1 + i)
        secs += dt
        rows += r
    value = rows / secs
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w["name"], "requests_per_gpu": w["B"],
                       "tokens_per_request": w["N"], "top_k": w["K"], "mla_layers": w["L"],
                       "sample": "one request per step"},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": oracle.omp_threads(),
                             "kind": "oracle",
                             "sample": "each step = 1 request x 1 decode step of the workload"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)  # ~0.6 s timed: several clock samples
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--requests", type=int, default=0, help="override requests per GPU")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-host-link", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
