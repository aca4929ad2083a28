#!/usr/bin/env python3
"""Benchmark of the paged GQA attention path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config batch|long|...]

Default workload: batch decode, 128 requests, 32 q heads / 8 kv heads, head_dim 128,
page_size 16, kv lengths U[512, 4096] (seed 0), a 32-layer cache
[32, pages, 2, 16, 8, 128] bf16 of 42.7 GB.  One step = plan (host) + for each of the
32 layer slices: last-page append and batched decode, in one launch
(pkv_run_decode_append; --separate-append issues pkv_kv_append_planned + pkv_run_decode).  The
metric is KV GB/s: the K and V bytes of every visible token per layer, over the device
time of the step.
The cache streamed per step is far larger than L2, so no flush is needed.

Printed: one JSON line (rank 0).  `--impl reference` times the CPU oracle on a bounded
sample of the same workload instead (host cores only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_kv_attention_gqa_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attn KV GB/s vs HBM peak; paged prefill TFLOP/s vs bf16 peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=["batch", "long", "long_window", "tiny", "prefill", "mixed"], default="batch",
                    help="batch (default): the decode step; prefill / mixed: those steps' own lines")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-secondary", action="store_true", help="skip the prefill / mixed / long-decode lines")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--separate-append", action="store_true",
                    help="decode workloads: pkv_kv_append_planned + pkv_run_decode per layer instead of the fused call")
    ap.add_argument("--layers", type=int, default=0, help="fewer cache layers (profiling a small case)")
    ap.add_argument("--heads", default=None,
                    help="Hq/Hkv/head_dim for --config prefill or batch (the same lengths on another head shape, "
                         "e.g. 16/8/256 or 8/1/128)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- plumbing

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    except Exception:
        return dict(hbm_gbs=FALLBACK_HBM_GBS, bf16_tflops=FALLBACK_BF16_TFLOPS, bf16_tflops_sustained=1700.0,
                    source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            try:
                uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
                cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
            except Exception:
                pass
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9], float(parts[9])))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r, _ in rows for i, v in enumerate(r) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "mem_mhz": statistics.median(r[3] for r in rows), "reasons": reasons, "samples": len(rows)}


def kernel_traffic(kernel_file: str, summary: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    source of the kernel (its sha256 is recorded beside the figure); else None."""
    path = os.path.join(ROOT, "profiles", summary)
    src = os.path.join(ROOT, "paged_kv_attention_gqa_gb300", "csrc", kernel_file)
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        rec = {}
        for line in text.splitlines():
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                rec[k.strip()] = v.strip().strip("`")
        if rec.get("source sha256") != sha:
            return None
        return float(rec["dram bytes per launch"])
    except Exception:
        return None


def make_handle(pb, B, sm_count=0):
    return B.Handle(num_qo_heads=pb.num_qo_heads, num_kv_heads=pb.num_kv_heads, head_dim=pb.head_dim,
                    page_size=pb.page_size, max_batch=pb.batch, max_total_tokens=max(pb.num_tokens, pb.batch),
                    max_num_pages=len(pb.kv_indices), num_cache_pages=pb.max_pages,
                    max_prefill_rows=max(pb.max_prefill_rows, 0), sm_count=sm_count, sink_page=pb.sink_page)


def decode_kv_bytes(pb, window_left=-1):
    """K+V bytes of every visible token of a decode pass over one layer."""
    tot = 0
    for L in pb.kv_lens:
        L = int(L)
        lo = max(0, L - 1 - window_left) if window_left >= 0 else 0
        tot += (L - lo)
    return tot * pb.num_kv_heads * pb.head_dim * 2 * 2


def prefill_flops(pb, causal=True, window_left=-1):
    pairs = 0
    for L, n in zip(pb.kv_lens, pb.qo_lens):
        L, n = int(L), int(n)
        c = L - n
        for i in range(n):
            p = c + i
            hi = p if causal else L - 1
            lo = max(0, p - window_left) if window_left >= 0 else 0
            pairs += hi - lo + 1
    return 4.0 * pb.head_dim * pb.num_qo_heads * pairs


# ----------------------------------------------------------------------------- our arm

def decode_workload(args):
    if args.config == "batch":
        pb = wl.config_batch_decode(seed=args.seed, num_layers=args.layers or 32)
        if args.heads:
            hq, hkv, d = (int(v) for v in args.heads.split("/"))
            pb = wl.custom(args.seed, pb.kv_lens, pb.qo_lens, num_qo_heads=hq, num_kv_heads=hkv, head_dim=d,
                           page_size=pb.page_size, num_layers=pb.num_layers, q_scale=pb.q_scale)
        window = -1
    elif args.config == "tiny":
        pb = wl.config_tiny(seed=args.seed)
        window = -1
    else:
        window = 4096 if args.config == "long_window" else -1
        pb = wl.config_long(seed=args.seed, window_left=window)
    return pb, window


def run_ours(args, rank, world):
    from paged_kv_attention_gqa_gb300 import binding as B
    B.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    pb, window = decode_workload(args)
    L = pb.num_layers
    x = wl.make_inputs(pb, device=dev, seed=args.seed, unused="randn")
    cache = x["kv_cache"]
    h = make_handle(pb, B)
    ws = torch.empty(h.workspace_size(B.MODE_DECODE), dtype=torch.uint8, device=dev)
    out = torch.empty_like(x["q"])
    lse = torch.empty(pb.batch, pb.num_qo_heads, dtype=torch.float32, device=dev)
    kvp, kvi, lpl = pb.kv_indptr, pb.kv_indices, pb.last_page_len
    h.plan(B.MODE_DECODE, None, kvp, kvi, lpl, workspace=ws, window_left=window)
    # launches per layer: the decode kernel (which also appends the layer's new tokens, or
    # append + decode with --separate-append), + the merge kernel when some row is cut
    tiles, _ = h.decode_split(kvp, lpl, window)
    cut = bool((tiles[:, 3] >= 0).any())
    launches_per_layer = (2 if args.separate_append else 1) + (1 if cut else 0)

    ev_pairs = []

    def layer(l, q, k, v, o, ls):
        if args.separate_append:
            h.kv_append_planned(k, v, cache[l], workspace=ws)
            h.run_decode(q, cache[l], o, ls, workspace=ws)
        else:
            h.run_decode_append(q, k, v, cache[l], o, ls, workspace=ws)

    def step(record, i=0):
        # record: time one layer's launch per step with events on the launching stream (layer
        # i mod L, so every layer is sampled), keeping event records out of the other gaps
        h.plan(B.MODE_DECODE, None, kvp, kvi, lpl, workspace=ws, window_left=window)
        for l in range(L):
            if record and l == i % L:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                layer(l, x["q"], x["k_new"], x["v_new"], out, lse)
                b.record(stream)
                ev_pairs.append((a, b))
            else:
                layer(l, x["q"], x["k_new"], x["v_new"], out, lse)

    for _ in range(max(args.warmup, 3)):
        step(False)
    torch.cuda.synchronize()
    assert h.check_device_error(ws) == 0
    clocks = ClockSampler()
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(True, i)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_step = max_over_ranks(t0.elapsed_time(t1) / args.steps, world)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_pairs)
    assert h.check_device_error(ws) == 0

    kv_layer_bytes = decode_kv_bytes(pb, window)
    step_bytes = kv_layer_bytes * L
    value = world * step_bytes / (ms_step * 1e-3) / 1e9
    achieved = kv_layer_bytes / (launch_ms * 1e-3) / 1e9
    traffic = (kernel_traffic("decode.cu", "decode_batch128_traffic.md") if args.config == "batch" and not args.heads
               else None)

    # end to end through host buffers: per step the host index arrays (plan), and per
    # layer q / new K / new V in from pinned host memory, out + lse back to it
    e2e = None
    if not args.no_e2e:
        qh = torch.empty((L,) + tuple(x["q"].shape), dtype=torch.bfloat16, pin_memory=True)
        kh = torch.empty((L,) + tuple(x["k_new"].shape), dtype=torch.bfloat16, pin_memory=True)
        vh = torch.empty_like(kh, pin_memory=True)
        oh = torch.empty_like(qh, pin_memory=True)
        lh = torch.empty((L,) + tuple(lse.shape), dtype=torch.float32, pin_memory=True)
        qh.copy_(x["q"].cpu().unsqueeze(0).expand_as(qh))
        kh.copy_(x["k_new"].cpu().unsqueeze(0).expand_as(kh))
        vh.copy_(x["v_new"].cpu().unsqueeze(0).expand_as(vh))
        # two device staging sets, one per step in flight: a step's inputs (all layers) are
        # copied in on one stream while the previous step computes, its outputs copied out on
        # another while the next step computes; the step's 32 launches stay back to back
        qd = [torch.empty_like(qh, device=dev) for _ in range(2)]
        kd = [torch.empty_like(kh, device=dev) for _ in range(2)]
        vd = [torch.empty_like(vh, device=dev) for _ in range(2)]
        od = [torch.empty_like(oh, device=dev) for _ in range(2)]
        ld = [torch.empty_like(lh, device=dev) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        e2e_count = [0]

        def e2e_step():
            b = e2e_count[0] & 1
            e2e_count[0] += 1
            s_in.wait_event(ev_done[b])  # the step two back has read set b
            with torch.cuda.stream(s_in):
                qd[b].copy_(qh, non_blocking=True)
                kd[b].copy_(kh, non_blocking=True)
                vd[b].copy_(vh, non_blocking=True)
            ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])  # and its outputs have been copied out
            h.plan(B.MODE_DECODE, None, kvp, kvi, lpl, workspace=ws, window_left=window)
            for l in range(L):
                layer(l, qd[b][l], kd[b][l], vd[b][l], od[b][l], ld[b][l])
            ev_done[b].record(stream)
            s_out.wait_event(ev_done[b])
            with torch.cuda.stream(s_out):
                oh.copy_(od[b], non_blocking=True)
                lh.copy_(ld[b], non_blocking=True)
            ev_out[b].record(s_out)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        k2 = max(10, args.steps // 4)
        s0 = time.perf_counter()
        for _ in range(k2):
            e2e_step()
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - s0) * 1e3 / k2, world)
        h2d = L * (x["q"].numel() + 2 * x["k_new"].numel()) * 2 + 4 * (len(kvp) + len(kvi) + len(lpl))
        d2h = L * (out.numel() * 2 + lse.numel() * 4)
        e2e = {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "copies": "pinned host buffers; per step one H2D of every layer's q / new K / new V on one "
                         "stream and one D2H of every layer's out / lse on another, overlapped with the "
                         "neighbouring steps' kernels (two device staging sets)"}
        # the last step's outputs came back: check them against the device results
        torch.cuda.synchronize()
        assert torch.equal(oh.to(dev), od[(e2e_count[0] - 1) & 1]), "e2e output copy mismatch"
        del qh, kh, vh, oh, lh, qd, kd, vd, od, ld

    # host plan cost (the pages quote ~2 us/row iterating a tensor row, 0.1 us via numpy)
    reps = 200
    s0 = time.perf_counter()
    for _ in range(reps):
        h.plan(B.MODE_DECODE, None, kvp, kvi, lpl, workspace=ws, window_left=window)
    plan_us_row = (time.perf_counter() - s0) * 1e6 / reps / pb.batch
    torch.cuda.synchronize()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; N(0,1) bf16 q/K/V)",
        "config": {"workload": f"{pb.name}: {pb.batch} requests, Hq {pb.num_qo_heads} / Hkv {pb.num_kv_heads}, "
                               f"head_dim {pb.head_dim}, page_size {pb.page_size}, {L} layers, window_left {window}",
                   "kv_cache_bytes": int(cache.numel() * 2), "kv_bytes_per_step": int(step_bytes),
                   "step": (f"plan + {L} x (pkv_kv_append_planned + pkv_run_decode)" if args.separate_append else
                            f"plan + {L} x pkv_run_decode_append (append fused into the decode launch)"),
                   "l2": "inputs larger than L2: every step streams the whole cache",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "e2e": e2e,
        "gpu_launches": int(args.steps * L * launches_per_layer),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "kernel": ("decode_kernel (+ merge_kernel when a row is cut; one run_decode)"
                                if args.separate_append else
                                "decode_kernel with the append fused (+ merge_kernel when a row is cut; one "
                                "run_decode_append)"),
                     "launch_ms": round(launch_ms, 5), "peak_source": peaks["source"],
                     # launch_ms: one launch timed alone (events on both sides break the chain of
                     # programmatic launches); inside the step each launch's prologue overlaps the
                     # previous launch's tail, so a layer takes ms_per_step / layers
                     "layer_ms_in_step": round(ms_step / L, 5)},
        "clocks": clk,
        "plan_us_per_row": round(plan_us_row, 3),
        "tokens_per_s": round(world * pb.batch * L / (ms_step * 1e-3), 1),
    }
    del x, cache
    torch.cuda.empty_cache()
    if not args.no_secondary:
        line["secondary"] = secondary(B, dev, peaks, args.seed)
    if rank == 0 and not args.no_e2e:
        line["cpu_baseline"] = cpu_baseline(pb, args.seed, window)
    return line


def run_step_primary(args, rank, world):
    """--config prefill | mixed: one step = append + the attention pass on one layer slice,
    timed per step with a 256 MB L2 flush between steps (the slice is ~0.2-1.8 GB)."""
    from paged_kv_attention_gqa_gb300 import binding as B
    B.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    pb = wl.config_prefill(seed=args.seed) if args.config == "prefill" else wl.config_mixed(seed=args.seed)
    if args.config == "prefill" and args.heads:
        hq, hkv, d = (int(v) for v in args.heads.split("/"))
        pb = wl.custom(args.seed, pb.kv_lens, pb.qo_lens, num_qo_heads=hq, num_kv_heads=hkv, head_dim=d,
                       page_size=pb.page_size)
    mode = B.MODE_PREFILL if args.config == "prefill" else B.MODE_MIXED
    x = wl.make_inputs(pb, device=dev, seed=args.seed, unused="randn")
    kv = x["kv_cache"][0]
    h = make_handle(pb, B)
    ws = torch.empty(h.workspace_size(mode), dtype=torch.uint8, device=dev)
    out = torch.empty_like(x["q"])
    lse = torch.empty(x["q"].shape[:2], dtype=torch.float32, device=dev)
    run = h.run_prefill if mode == B.MODE_PREFILL else h.run_mixed
    h.plan(mode, pb.qo_indptr, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
    flush = l2_flush_buffer(dev)
    step_ms, run_ms = [], []
    for it in range(max(args.warmup, 3) + args.steps):
        flush()
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(stream)
        h.kv_append_planned(x["k_new"], x["v_new"], kv, workspace=ws)
        b.record(stream)
        run(x["q"], kv, out, lse, workspace=ws)
        c.record(stream)
        torch.cuda.synchronize()
        if it >= max(args.warmup, 3):
            step_ms.append(a.elapsed_time(c))
            run_ms.append(b.elapsed_time(c))
    assert h.check_device_error(ws) == 0
    ms = max_over_ranks(statistics.median(step_ms), world)
    kms = statistics.median(run_ms)
    if args.config == "prefill":
        fl = prefill_flops(pb)
        value, unit = world * fl / (ms * 1e-3) / 1e12, "TFLOP/s"
        achieved = fl / (kms * 1e-3) / 1e12
        wide = pb.head_dim == 256
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": (kernel_traffic("prefill_wide.cuh", "prefill_ragged16_d256.md") if wide
                            else kernel_traffic("prefill_pair.cuh", "prefill_ragged16_pair.md")),
                "kernel": "prefill_wide_kernel" if wide else "prefill_pair_kernel",
                "launch_ms": round(kms, 5), "peak_source": peaks["source"]}
        launches = 2
    else:
        dec = [r for r in range(pb.batch) if pb.qo_lens[r] == 1]
        dec_bytes = sum(int(pb.kv_lens[r]) for r in dec) * pb.num_kv_heads * pb.head_dim * 4
        value, unit = world * dec_bytes / (ms * 1e-3) / 1e9, "GB/s"
        roof = {"bound": "hbm", "achieved": round(dec_bytes / (kms * 1e-3) / 1e9, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(dec_bytes / (kms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4), "traffic": None,
                "kernel": "decode pass + prefill pass (run_mixed)", "launch_ms": round(kms, 5),
                "peak_source": peaks["source"]}
        launches = 3
    return {"metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; N(0,1) bf16 q/K/V)",
            "config": {"workload": f"{pb.name}: {pb.batch} rows, {pb.num_tokens} new tokens, Hq {pb.num_qo_heads} / "
                                   f"Hkv {pb.num_kv_heads}, head_dim {pb.head_dim}, page_size {pb.page_size}",
                       "l2": "256 MB written between steps"},
            "e2e": None, "gpu_launches": launches * args.steps, "roofline": roof}


class L2Flush:
    """Evicts L2 between timed calls: writes a 256 MB buffer (the flush), then reads another
    256 MB buffer, so that L2 holds only clean lines when the timed call starts and the
    write-back of the flush's dirty lines is not charged to it."""

    def __init__(self, dev):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.fill_(1)
        self.r.sum()


def l2_flush_buffer(dev):
    return L2Flush(dev)


def time_runs(fn, flush, iters=20, warm=3):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(iters):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def secondary(B, dev, peaks, seed):
    """Prefill (TFLOP/s vs bf16 peak), mixed step, the batch workload's append and long-context
    decode, each timed per call with an L2 flush between calls."""
    res = {}
    flush = l2_flush_buffer(dev)
    # ragged causal prefill with cached prefix
    pb = wl.config_prefill(seed=seed)
    x = wl.make_inputs(pb, device=dev, seed=seed, unused="randn")
    h = make_handle(pb, B)
    ws = torch.empty(h.workspace_size(B.MODE_PREFILL), dtype=torch.uint8, device=dev)
    h.plan(B.MODE_PREFILL, pb.qo_indptr, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
    kv = x["kv_cache"][0]
    out = torch.empty_like(x["q"])
    lse = torch.empty(x["q"].shape[:2], dtype=torch.float32, device=dev)
    h.kv_append_planned(x["k_new"], x["v_new"], kv, workspace=ws)
    ms = time_runs(lambda: h.run_prefill(x["q"], kv, out, lse, workspace=ws), flush)
    app_ms = time_runs(lambda: h.kv_append_planned(x["k_new"], x["v_new"], kv, workspace=ws), flush)
    fl = prefill_flops(pb)
    tf = fl / (ms * 1e-3) / 1e12
    res["prefill"] = {"workload": "16 rows, new U[128,2048], prefix U[0,4096], 32/8/128, causal",
                      "ms": round(ms, 4), "tflops": round(tf, 1), "peak_tflops": peaks["bf16_tflops"],
                      "frac": round(tf / peaks["bf16_tflops"], 4), "tokens_per_s": round(pb.num_tokens / (ms * 1e-3)),
                      "append_ms": round(app_ms, 4),
                      # DRAM bytes of one launch from the committed ncu capture (None once the
                      # kernel source differs from the captured one)
                      "traffic": kernel_traffic("prefill_pair.cuh", "prefill_ragged16_pair.md")}
    del x, kv
    # mixed step
    pb = wl.config_mixed(seed=seed)
    x = wl.make_inputs(pb, device=dev, seed=seed, unused="randn")
    h = make_handle(pb, B)
    ws = torch.empty(h.workspace_size(B.MODE_MIXED), dtype=torch.uint8, device=dev)
    h.plan(B.MODE_MIXED, pb.qo_indptr, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
    kv = x["kv_cache"][0]
    out = torch.empty_like(x["q"])
    lse = torch.empty(x["q"].shape[:2], dtype=torch.float32, device=dev)
    h.kv_append_planned(x["k_new"], x["v_new"], kv, workspace=ws)
    ms = time_runs(lambda: h.run_mixed(x["q"], kv, out, lse, workspace=ws), flush)
    dec = [r for r in range(pb.batch) if pb.qo_lens[r] == 1]
    dec_bytes = sum(int(pb.kv_lens[r]) for r in dec) * pb.num_kv_heads * pb.head_dim * 4
    pf_rows = [r for r in range(pb.batch) if pb.qo_lens[r] >= 2]
    sub = wl.PagedBatch("p", pb.num_qo_heads, pb.num_kv_heads, pb.head_dim, 16, pb.kv_lens[pf_rows],
                        pb.qo_lens[pf_rows], [pb.page_table[r] for r in pf_rows], pb.max_pages)
    pf_fl = prefill_flops(sub)
    bound_ms = (dec_bytes / (peaks["hbm_gbs"] * 1e9) + pf_fl / (peaks["bf16_tflops"] * 1e12)) * 1e3
    res["mixed"] = {"workload": "96 decode rows + 4 prompt rows, 32/8/128", "ms": round(ms, 4),
                    "roofline_ms": round(bound_ms, 4), "frac": round(bound_ms / ms, 4),
                    "decode_kv_gb": round(dec_bytes / 1e9, 3), "prefill_tflop": round(pf_fl / 1e12, 4)}
    del x, kv
    # the batch-decode workload's append of its 128 new tokens into one layer slice, alone:
    # at the plan's write locations, and from device index arrays (no plan)
    pb = wl.config_batch_decode(seed=seed, num_layers=1)
    x = wl.make_inputs(pb, device=dev, seed=seed, unused="randn", layers=1)
    h = make_handle(pb, B)
    ws = torch.empty(h.workspace_size(B.MODE_DECODE), dtype=torch.uint8, device=dev)
    h.plan(B.MODE_DECODE, None, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
    kv = x["kv_cache"][0]
    idx = [torch.as_tensor(np.asarray(a, np.int32), device=dev) for a in (pb.kv_indptr, pb.kv_indices, pb.last_page_len)]
    planned_ms = time_runs(lambda: h.kv_append_planned(x["k_new"], x["v_new"], kv, workspace=ws), flush)
    indexed_ms = time_runs(lambda: h.kv_append(x["k_new"], x["v_new"], pb.batch, kv, None, *idx, pb.batch), flush)
    app_bytes = 2 * pb.batch * pb.num_kv_heads * pb.head_dim * 2 * 2  # K and V rows read and written
    res["append_batch"] = {"workload": "128 new tokens (one per row) into one layer slice, 8 kv heads, head_dim 128",
                           "planned_us": round(planned_ms * 1e3, 2), "indexed_us": round(indexed_ms * 1e3, 2),
                           "bytes": app_bytes}
    del x, kv
    # long-context split-KV decode, full and windowed
    for window in (-1, 4096):
        pb = wl.config_long(seed=seed, window_left=window)
        x = wl.make_inputs(pb, device=dev, seed=seed, unused="randn")
        h = make_handle(pb, B)
        ws = torch.empty(h.workspace_size(B.MODE_DECODE), dtype=torch.uint8, device=dev)
        h.plan(B.MODE_DECODE, None, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws, window_left=window)
        kv = x["kv_cache"][0]
        out = torch.empty_like(x["q"])
        lse = torch.empty(x["q"].shape[:2], dtype=torch.float32, device=dev)
        ms = time_runs(lambda: h.run_decode(x["q"], kv, out, lse, workspace=ws), flush)
        gbs = decode_kv_bytes(pb, window) / (ms * 1e-3) / 1e9
        res["long_decode" + ("_window4096" if window >= 0 else "")] = {
            "workload": "8 rows, L U[65536,131072], 64/8/128", "ms": round(ms, 4), "gbs": round(gbs, 1),
            "frac": round(gbs / peaks["hbm_gbs"], 4)}
        del x, kv
    torch.cuda.empty_cache()
    res["shapes"] = shape_lines(B, dev, peaks, seed, flush)
    return res


def shape_lines(B, dev, peaks, seed, flush):
    """The batch-decode and ragged-prefill workloads' lengths on other page sizes, head
    dims, group sizes and kv-head counts (one layer each, per call after an L2 flush)."""
    out = []
    base = wl.config_batch_decode(seed=seed, num_layers=1)
    ones = np.ones(base.batch, np.int64)
    for P, Hq, Hkv, D in [(1, 32, 8, 128), (8, 32, 8, 128), (64, 32, 8, 128), (16, 16, 8, 256), (16, 32, 16, 128),
                          (16, 28, 4, 128), (16, 16, 2, 128), (16, 8, 1, 128)]:
        pb = wl.custom(seed, base.kv_lens, ones, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P)
        x = wl.make_inputs(pb, device=dev, seed=seed, unused="randn", layers=1)
        h = make_handle(pb, B)
        ws = torch.empty(h.workspace_size(B.MODE_DECODE), dtype=torch.uint8, device=dev)
        h.plan(B.MODE_DECODE, None, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
        kv = x["kv_cache"][0]
        o = torch.empty_like(x["q"])
        ls = torch.empty(x["q"].shape[:2], dtype=torch.float32, device=dev)
        ms = time_runs(lambda: h.run_decode(x["q"], kv, o, ls, workspace=ws), flush)
        gbs = decode_kv_bytes(pb) / (ms * 1e-3) / 1e9
        out.append({"pass": "decode", "shape": f"P {P}, {Hq}/{Hkv}/{D}, 128 rows L U[512,4096]",
                    "ms": round(ms, 4), "gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4)})
        del x, kv
    base = wl.config_prefill(seed=seed)
    for P, Hq, Hkv, D in [(1, 32, 8, 128), (64, 32, 8, 128), (16, 16, 8, 256), (16, 28, 4, 128)]:
        pb = wl.custom(seed, base.kv_lens, base.qo_lens, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P)
        x = wl.make_inputs(pb, device=dev, seed=seed, unused="randn", layers=1)
        h = make_handle(pb, B)
        ws = torch.empty(h.workspace_size(B.MODE_PREFILL), dtype=torch.uint8, device=dev)
        h.plan(B.MODE_PREFILL, pb.qo_indptr, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
        kv = x["kv_cache"][0]
        o = torch.empty_like(x["q"])
        ls = torch.empty(x["q"].shape[:2], dtype=torch.float32, device=dev)
        ms = time_runs(lambda: h.run_prefill(x["q"], kv, o, ls, workspace=ws), flush)
        tf = prefill_flops(pb) / (ms * 1e-3) / 1e12
        out.append({"pass": "prefill", "shape": f"P {P}, {Hq}/{Hkv}/{D}, 16 rows as the ragged-prefill workload",
                    "ms": round(ms, 4), "tflops": round(tf, 1), "frac": round(tf / peaks["bf16_tflops"], 4)})
        del x, kv
    torch.cuda.empty_cache()
    return out


def cpu_baseline(pb, seed, window, seconds=10.0, one_core_seconds=5.0):
    """The oracle as it stands on the host cores, on one layer of the same workload: passes
    over that layer repeated for about `seconds` on all host threads, and for about
    `one_core_seconds` on one thread."""
    import oracle
    x = wl.make_inputs(pb, device="cuda" if torch.cuda.is_available() else "cpu", seed=seed, unused="randn",
                       layers=1)
    qb, kvb = wl.bf16_bits(x["q"]), wl.bf16_bits(x["kv_cache"][0])
    del x

    def timed(threads, budget):
        passes, s0 = 0, time.perf_counter()
        while True:
            oracle.attention(qb, kvb, pb.qo_indptr, pb.kv_indptr, pb.kv_indices, pb.last_page_len,
                             num_qo_heads=pb.num_qo_heads, num_kv_heads=pb.num_kv_heads, head_dim=pb.head_dim,
                             page_size=pb.page_size, window_left=window, threads=threads)
            passes += 1
            el = time.perf_counter() - s0
            if el >= budget or passes >= 1000:
                return passes, el

    layer_bytes = decode_kv_bytes(pb, window)
    threads = os.cpu_count() or 1
    n, el = timed(threads, seconds)
    n1, el1 = timed(1, one_core_seconds)
    return {"value": round(layer_bytes * n / el / 1e9, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"layer 0 of {pb.num_layers} ({pb.batch} rows), {n} passes in {el:.1f} s, rows split over "
                      f"{threads} threads",
            "one_core": {"value": round(layer_bytes * n1 / el1 / 1e9, 3), "unit": "GB/s", "cores": 1,
                         "sample": f"the same layer, {n1} passes in {el1:.1f} s on one thread"}}


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    """The oracle, timed on the host cores, on the same workload: each step is one layer of
    the decode step (every row), the bounded sample the oracle finishes in about a second."""
    import oracle
    pb, window = decode_workload(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = wl.make_inputs(pb, device=dev, seed=args.seed, unused="randn", layers=1)
    qb, kvb = wl.bf16_bits(x["q"]), wl.bf16_bits(x["kv_cache"][0])
    del x
    threads = os.cpu_count() or 1
    steps, warm = max(1, min(args.steps, 10)), min(args.warmup, 1)

    def one():
        oracle.attention(qb, kvb, pb.qo_indptr, pb.kv_indptr, pb.kv_indices, pb.last_page_len,
                         num_qo_heads=pb.num_qo_heads, num_kv_heads=pb.num_kv_heads, head_dim=pb.head_dim,
                         page_size=pb.page_size, window_left=window, threads=threads)

    for _ in range(warm):
        one()
    s0 = time.perf_counter()
    for _ in range(steps):
        one()
    ms = (time.perf_counter() - s0) * 1e3 / steps
    gbs = decode_kv_bytes(pb, window) / (ms * 1e-3) / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded)",
            "config": {"workload": f"{pb.name}: {pb.batch} requests, Hq {pb.num_qo_heads} / Hkv {pb.num_kv_heads}, "
                                   f"head_dim {pb.head_dim}, page_size {pb.page_size}, one layer slice per step",
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"one of {pb.num_layers} layers per step, all {pb.batch} rows"},
            "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    args = parse()
    rank, world = dist_setup(args)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    line = run_step_primary(args, rank, world) if args.config in ("prefill", "mixed") else run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
