"""Throughput of the hot path: causal bf16 attention forward + backward at 128K
tokens (B=1, H=32, N=131072, d=128, chunks of 4096), on N GPUs of one node.

One step = attn_chunked_fwd (persistent forward over every visible chunk
pair) + attn_chunked_bwd (row dot, dK/dV kernel, dQ kernel) on resident,
seeded synthetic inputs.  Each rank runs its own full problem (the heads and
sequences of a batch are independent), so N GPUs do N times the work: weak
scaling, no data-path collective.

FLOP convention: only visible (causal) query-key pairs count; a forward is two
GEMMs over them (2 * B * H * N^2 * d for the causal square), a backward 2.5x
that.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  --impl reference times the fp64 oracle on the
host cores on a bounded sample of the same workload (the reference arm).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal bf16 attn fwd+bwd TFLOP/s at 128K tokens, % of tensor peak"
UNIT = "TFLOP/s"
WORKLOAD = "causal_128k_balanced"
L2_BYTES = 129 * 10**6  # GB300 L2 size


PKG = os.path.join(ROOT, "long_sequence_exact_gb300")
# Source files whose text fixes each tensor-core kernel's code: a DRAM figure
# taken by ncu is used only while the hash of these files is the one recorded
# beside it (profiles/*.md, "traffic:" lines), so a changed kernel reports no
# stale traffic.
KERNEL_SOURCES = {
    "fwd_tc": ("csrc/fwd_tc.cu", "csrc/fwd_split.h", "csrc/ptx.cuh", "csrc/internal.h",
               "csrc/tma_host.h"),
    "bwd_fused_tc": ("csrc/bwd_tc.cu", "csrc/bwd_split.h", "csrc/ptx.cuh", "csrc/internal.h",
                     "csrc/tma_host.h"),
    "bwd_dkdv_tc": ("csrc/bwd_tc.cu", "csrc/bwd_split.h", "csrc/ptx.cuh", "csrc/internal.h",
                    "csrc/tma_host.h"),
    "bwd_dq_tc": ("csrc/bwd_tc.cu", "csrc/bwd_split.h", "csrc/ptx.cuh", "csrc/internal.h",
                  "csrc/tma_host.h"),
}
TRACE_KERNELS = {0: "fwd_tc", 1: "bwd_dkdv_tc", 2: "bwd_dq_tc", 12: "bwd_fused_tc"}


def _code_only(text):
    """Source text without comments and with whitespace runs collapsed, so
    that editing a comment does not count as changing the kernel."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(name):
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[name]:
        with open(os.path.join(PKG, rel)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def tile_pairs(b, h, n, causal=True):
    """(query tile, key tile) pairs of 128 x 128 that the kernels visit."""
    t = (n + 127) // 128
    return b * h * (t * (t + 1) // 2 if causal else t * t)


def recorded_traffic(name, units, d, causal):
    """DRAM bytes per launch of kernel `name` scaled to `units` tile pairs,
    from a committed ncu summary of the same kernel source, head dimension
    and masking (each head dimension is its own instantiation, with its own
    traffic); None when there is none (never taken, or the kernel has
    changed since).  A profiles/*.md line reads
      traffic: kernel=<name> source=<hash16> d=<head dim> causal=<0|1>
               bytes=<dram read+write> units=<tile pairs>
    (on one line)."""
    import glob
    want = kernel_source_hash(name)
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                if not line.lstrip().startswith("traffic:"):
                    continue
                kv = dict(t.split("=", 1) for t in line.split()[1:] if "=" in t)
                if (kv.get("kernel") == name and kv.get("source") == want
                        and kv.get("d") == str(d) and kv.get("causal") == str(int(causal))
                        and "bytes" in kv and "units" in kv):
                    return {"bytes": float(kv["bytes"]) / float(kv["units"]) * units,
                            "source": os.path.relpath(path, ROOT), "captured_units": float(kv["units"])}
    return None


def parse_trace(words):
    """Per-launch records written by the persistent kernels (lsx_trace_enable):
    [kid, G, items] then (start_ns, end_ns, items) per CTA.  Returns a list of
    dicts with the SM idle fraction 1 - sum(busy) / (G * makespan)."""
    out, i = [], 0
    while i + 3 <= len(words):
        kid, g, items = int(words[i]), int(words[i + 1]), int(words[i + 2])
        if g <= 0 or i + 3 + 3 * g > len(words):
            break
        cta = [(int(words[i + 3 + 3 * c]), int(words[i + 4 + 3 * c]), int(words[i + 5 + 3 * c]))
               for c in range(g)]
        t0 = min(c[0] for c in cta)
        t1 = max(c[1] for c in cta)
        span = max(t1 - t0, 1)
        busy = sum(c[1] - c[0] for c in cta)
        ends = sorted(c[1] - t0 for c in cta)
        out.append({"kernel": TRACE_KERNELS.get(kid, str(kid)), "ctas": g, "items": items,
                    "items_run": sum(c[2] for c in cta),
                    "makespan_ms": round(span / 1e6, 3),
                    "idle_fraction": round(1.0 - busy / (g * span), 4),
                    "first_cta_done_ms": round(ends[0] / 1e6, 3),
                    "median_cta_done_ms": round(ends[g // 2] / 1e6, 3)})
        i += 3 + 3 * g
    return out


def traced(step, dev):
    """Runs `step` once with the schedule trace on; returns parse_trace's list."""
    import torch
    from long_sequence_exact_gb300 import _lib
    lib = _lib.load()
    buf = torch.zeros(1 << 17, dtype=torch.int64, device=dev)
    torch.cuda.synchronize()
    _lib.check(lib.lsx_trace_enable(buf.data_ptr(), buf.numel() * 8), "lsx_trace_enable")
    try:
        step()
        torch.cuda.synchronize()
        used = lib.lsx_trace_used() // 8
    finally:
        lib.lsx_trace_enable(None, 0)
    words = buf[:used].cpu().tolist()
    return parse_trace(words)


def job_throughput(ms_local, work_per_step, steps, world, device="cpu"):
    """Whole-job rate over N ranks that each did `steps` steps of
    `work_per_step` units in `ms_local` ms: the slowest rank's time (a MAX
    all-reduce when world > 1) sets it.  Returns (ms_max, units per second / 1e12)."""
    import torch
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, world * work_per_step * steps / (ms_max / 1e3) / 1e12


def flops(b, h, n, d, causal=True):
    pairs = n * (n + 1) / 2 if causal else n * n
    fwd = 4.0 * b * h * pairs * d
    return fwd, 2.5 * fwd


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        clk = (m.get("clocks_under_load") or {}).get("sm_mhz_median")
        return {"hbm_gbs": m["hbm_gbs"], "bf16": m["bf16_tflops"],
                "bf16_sustained": m["bf16_tflops_sustained"], "source": "measured",
                "sustained_sm_mhz": clk}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback",
            "sustained_sm_mhz": None}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons, watts = [], None, set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            try:
                watts.append(float(parts[3]))
            except ValueError:
                pass
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "power_w": statistics.median(watts) if watts else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_times(lib_mod):
    import ctypes
    lib = lib_mod.load()
    buf = ctypes.create_string_buffer(4096)
    n = lib.lsx_timing_report(buf, 4096)
    out = {}
    if n > 0:
        for line in buf.value.decode().strip().splitlines():
            name, cnt, tot = line.split()
            out[name] = (int(cnt), float(tot))
    return out


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import long_sequence_exact_gb300 as lsx
    from long_sequence_exact_gb300 import _lib
    from long_sequence_exact_gb300.inputs import WORKLOADS, make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = WORKLOADS[args.workload or WORKLOAD]
    workload = WORKLOAD
    if args.workload or args.n or args.heads:
        w = w.with_(N=args.n or w.N, Hq=args.heads or w.Hq, Hkv=args.heads or w.Hkv)
        workload = (f"{w.name}_n{w.N}_h{w.Hq}_profiling" if args.workload
                    else f"causal_{w.N}_h{w.Hq}_profiling")
    if args.deterministic:
        lsx.set_deterministic(True)  # (before the workspace sizes: no split in this mode)
        workload += "_deterministic"
    x = make_inputs(w, device=dev, seed=w.seed + rank)
    q, k, v, d_o = x["q"], x["k"], x["v"], x["d_o"]
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    import ctypes
    vq_, vk_ = _lib.view(q), _lib.view(k)
    ws_bytes = _lib.load().attn_chunked_bwd_workspace_size(ctypes.byref(vq_), ctypes.byref(vk_),
                                                           w.chunk, 1)
    ws = torch.empty(int(ws_bytes), dtype=torch.uint8, device=dev)
    ws_f = torch.empty(int(_lib.load().attn_chunked_fwd_workspace_size(
        ctypes.byref(vq_), ctypes.byref(vk_), w.chunk, 1)), dtype=torch.uint8, device=dev)

    def step():
        lsx.chunked_fwd(q, k, v, w.chunk, causal=w.causal, out=o, lse=lse, workspace=ws_f)
        lsx.chunked_bwd(q, k, v, o, lse, d_o, w.chunk, causal=w.causal, dq=dq, dk=dk, dv=dv,
                        workspace=ws)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if lsx.sync_status() != 0:
        raise RuntimeError("device status after warm-up")

    lib = _lib.load()
    lib.lsx_timing_reset()
    lib.lsx_timing_enable(1)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
    lib.lsx_timing_enable(0)
    ms = e0.elapsed_time(e1)
    ktimes = kernel_times(_lib)
    lib.lsx_timing_reset()
    if lsx.sync_status() != 0:
        raise RuntimeError("device status after the timed steps")

    f_fwd, f_bwd = flops(w.B, w.Hq, w.N, w.D, w.causal)
    step_flops = f_fwd + f_bwd
    in_bytes = q.numel() * q.element_size()
    ms_max, value = job_throughput(ms, step_flops, args.steps, world, dev)

    # end to end through the same C ABI: every step copies its inputs in from
    # pinned host memory and all of its outputs (O, LSE, dQ, dK, dV) back.
    # The copies run on two copy streams, double-buffered on the device: the
    # inputs of step s+1 go in and the outputs of step s-1 come out while
    # step s computes.  The timed region starts before the first input copy
    # and ends after the last output copy.
    e2e = None
    if not args.no_e2e:
        host_in = [t_.cpu().pin_memory() for t_ in (q, k, v, d_o)]
        host_out = [torch.empty_like(t_, device="cpu").pin_memory() for t_ in (o, lse, dq, dk, dv)]
        h2d = sum(t_.numel() * t_.element_size() for t_ in host_in)
        d2h = sum(t_.numel() * t_.element_size() for t_ in host_out)
        bufs = [((q, k, v, d_o), (o, lse, dq, dk, dv)),
                (tuple(torch.empty_like(t_) for t_ in (q, k, v, d_o)),
                 tuple(torch.empty_like(t_) for t_ in (o, lse, dq, dk, dv)))]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        def e2e_run(n):
            ev = lambda: torch.cuda.Event()  # noqa: E731
            ready, done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
            start_ev = ev()
            start_ev.record(stream)

            def copy_in(step_no):
                ins = bufs[step_no % 2][0]
                s_in.wait_event(start_ev)
                if step_no >= 2:  # the step that last read these buffers
                    s_in.wait_event(done[step_no % 2])
                with torch.cuda.stream(s_in):
                    for d_, h_ in zip(ins, host_in):
                        d_.copy_(h_, non_blocking=True)
                ready[step_no % 2].record(s_in)

            copy_in(0)
            for step_no in range(n):
                (xq, xk, xv, xdo), (xo, xl, xdq, xdk, xdv) = bufs[step_no % 2]
                if step_no + 1 < n:
                    copy_in(step_no + 1)
                stream.wait_event(ready[step_no % 2])
                if step_no >= 2:  # step_no - 2's outputs (same buffers) are copied out
                    stream.wait_event(out_done[step_no % 2])
                lsx.chunked_fwd(xq, xk, xv, w.chunk, causal=w.causal, out=xo, lse=xl,
                                workspace=ws_f)
                lsx.chunked_bwd(xq, xk, xv, xo, xl, xdo, w.chunk, causal=w.causal, dq=xdq, dk=xdk,
                                dv=xdv, workspace=ws)
                done[step_no % 2].record(stream)
                s_out.wait_event(done[step_no % 2])
                with torch.cuda.stream(s_out):
                    for h_, d_ in zip(host_out, (xo, xl, xdq, xdk, xdv)):
                        h_.copy_(d_, non_blocking=True)
                out_done[step_no % 2].record(s_out)
            stream.wait_stream(s_out)

        e2e_run(2)
        torch.cuda.synchronize()
        barrier()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(1, args.steps)
        with ClockSampler(local_rank) as e2e_clk:
            a.record(stream)
            e2e_run(n_e2e)
            b_.record(stream)
            torch.cuda.synchronize()
        if lsx.sync_status() != 0:
            raise RuntimeError("device status after the end-to-end steps")
        _, e2e_value = job_throughput(a.elapsed_time(b_), step_flops, n_e2e, world, dev)
        e2e = {"value": round(e2e_value, 2),
               "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": n_e2e,
               "copies": "pinned host memory; two copy streams, overlapped with the "
                         "neighbouring steps' compute",
               "clocks": e2e_clk.summary()}

    if rank != 0:
        return None

    pk = peaks()
    # dominant kernel by measured time; its algorithmic work per launch:
    # fwd_tc = the two forward GEMMs; bwd_fused_tc = all 5 backward GEMMs
    # (S^T, dP^T, dV, dK, dQ); in the deterministic mode bwd_dkdv_tc = S^T,
    # dP^T, dV, dK (4 of 5) and bwd_dq_tc = dQ (1 of 5; its S and dP are
    # recomputed).  Fractions are given against both measured peaks: the
    # sustained one (a long cuBLAS loop under the power cap, the reference for
    # kernels timed inside a long step) and the burst one.
    unit_gemm = f_fwd / 2.0
    algo = {"fwd_tc": 2 * unit_gemm, "bwd_fused_tc": 5 * unit_gemm,
            "bwd_dkdv_tc": 4 * unit_gemm, "bwd_dq_tc": 1 * unit_gemm}
    units = tile_pairs(w.B, w.Hq, w.N, w.causal)
    dom = max(ktimes.items(), key=lambda kv: kv[1][1]) if ktimes else None
    roofline = None
    kernels = {}
    for name, (cnt, tot) in ktimes.items():
        avg = tot / cnt
        ent = {"launches": cnt, "avg_ms": round(avg, 4), "share": round(tot / sum(t_[1] for t_ in ktimes.values()), 4)}
        if name in algo:
            ach = algo[name] / (avg / 1e3) / 1e12
            ent["achieved_tflops"] = round(ach, 1)
            ent["frac_of_peak"] = round(ach / pk["bf16_sustained"], 4)
            ent["frac_of_burst_peak"] = round(ach / pk["bf16"], 4)
            rec = recorded_traffic(name, units, w.D, w.causal) if name in KERNEL_SOURCES else None
            ent["dram_bytes_per_launch"] = round(rec["bytes"]) if rec else None
        kernels[name] = ent
    if dom is not None and dom[0] in algo:
        name, (cnt, tot) = dom
        rec = recorded_traffic(name, units, w.D, w.causal)
        traffic = args.traffic if args.traffic is not None else (round(rec["bytes"]) if rec else None)
        ach = algo[name] / (tot / cnt / 1e3) / 1e12
        roofline = {"kernel": name, "bound": "tensor", "achieved": round(ach, 1),
                    "peak": pk["bf16_sustained"], "unit": "TFLOP/s",
                    "frac": round(ach / pk["bf16_sustained"], 4), "traffic": traffic,
                    "peak_kind": f"{pk['source']} bf16 sustained (kernel timed inside a long step)",
                    "peak_burst": pk["bf16"], "frac_of_burst": round(ach / pk["bf16"], 4),
                    "peak_sustained_sm_mhz": pk.get("sustained_sm_mhz"),
                    "traffic_source": (rec["source"] + f" (ncu capture of {rec['captured_units']:.0f} "
                                       f"tile pairs, scaled to {units} by tile pairs)")
                    if rec and args.traffic is None else
                    ("--traffic" if args.traffic is not None else
                     "none for the current kernel source")}

    # SM idle fraction of the persistent kernels: one more (untimed) step
    # with the device-side schedule trace on
    schedule = traced(step, dev) if not args.no_trace else None

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(repeats=args.cpu_repeats)
        cpu["gpu_step_s"] = round(ms_max / args.steps / 1e3, 4)
    sec = None
    if not args.no_secondary:
        del q, k, v, d_o, o, lse, dq, dk, dv, ws, ws_f, x
        torch.cuda.empty_cache()
        sec = secondary(dev, pk)

    return {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1)*0.5 q/k/v, N(0,1) dO; one problem per rank)",
        "config": {"workload": workload, "B": w.B, "H": w.Hq, "N": w.N, "d": w.D,
                   "chunk_len": w.chunk, "causal": w.causal,
                   "deterministic_backward": bool(args.deterministic),
                   "flops_per_step": step_flops, "fwd_flops": f_fwd, "bwd_flops": f_bwd,
                   "l2": (f"inputs larger than L2 (q, k, v, dO {in_bytes / 2**30:.3g} GiB each; "
                          "no flush needed)" if 4 * in_bytes > L2_BYTES else
                          f"inputs of {4 * in_bytes / 2**20:.0f} MiB, within L2 (profiling case)"),
                   "pct_of_tensor_peak": round(100.0 * value / world / pk["bf16_sustained"], 2),
                   "pct_of_burst_tensor_peak": round(100.0 * value / world / pk["bf16"], 2)},
        "roofline": roofline, "kernels": kernels, "schedule": schedule, "secondary": sec,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": sum(c for c, _ in ktimes.values()),
        "clocks": clk.summary(),
    }


# ----------------------------------------------- bandwidth-bound rows
def secondary(dev, pk):
    """Rows of the path other than the headline, timed alone with CUDA events
    (median of 5 after 3 warm-ups; every input is larger than L2; the
    attention workloads also report their SM idle fractions from one more
    traced, untimed step):
      merge       attn_merge of two fp32 partials at the 128K row count
                  (B=1, H=32, N=131072, d=128): reads 2 x (O + LSE), writes 1
      tree_merge  attn_tree_merge of 8 fp32 partials at the 32K row count
      decode      attn_decode, B=8, Hq=32, Hkv=8, one query, 1,048,576-key
                  cache, chunks of 4096 (partials + tree merge); algorithmic
                  bytes = the K and V caches once + q + o
      causal_32k_ring, noncausal_64k_heavytail
                  chunked fwd+bwd of the other two attention workloads
                  (TFLOP/s against the sustained bf16 peak)
      decode_tree_1m_prefix
                  shared-prefix tree decode (prefix read once for the 8
                  branches) against plain decode over per-branch copies
      block_sparse_window_128k
                  block-sparse fwd+bwd at 128K with a sliding-window block
                  mask (only visible pairs credited)
      autograd_remat_32k
                  backward time through torch.autograd with the checkpoint
                  at the attention output vs at the layer input (re-run)
      split_rows_32k_h1
                  chunked forward of one head of 32K causal rows (64 query
                  pairs for 152 SMs): rows split into key pieces
                  merged by the LSE-weighted merge, against the unsplit
                  launch (a workspace with room for the V copy only); and
                  the chunked backward of one head of 16K causal rows (128
                  key-tile items): key columns split, partial dK / dV
                  summed, against the unsplit launch
    """
    import torch
    import long_sequence_exact_gb300 as lsx
    from long_sequence_exact_gb300.inputs import WORKLOADS, make_inputs, random_tensor

    def timed(fn, reps=5):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    out = {}
    peak = pk["hbm_gbs"]
    # pairwise merge
    shape = (1, 32, 131072, 128)
    oa = random_tensor(shape, 1, dtype=torch.float32, device=dev)
    ob = random_tensor(shape, 2, dtype=torch.float32, device=dev)
    la = random_tensor(shape[:3], 3, 5.0, dtype=torch.float32, device=dev)
    lb = random_tensor(shape[:3], 4, 5.0, dtype=torch.float32, device=dev)
    oo, lo = torch.empty_like(oa), torch.empty_like(la)
    ms = timed(lambda: lsx.merge(oa, la, ob, lb, out=oo, lse_out=lo))
    nbytes = 3 * (oa.numel() * 4 + la.numel() * 4)
    out["merge"] = {"gbs": round(nbytes / ms / 1e6, 1), "frac": round(nbytes / ms / 1e6 / peak, 4),
                    "ms": round(ms, 4), "bytes": nbytes}
    del oa, ob, la, lb, oo, lo
    # tree merge of 8 partials
    k = 8
    op = random_tensor((k, 1, 32, 32768, 128), 5, dtype=torch.float32, device=dev)
    lp = random_tensor((k, 1, 32, 32768), 6, 5.0, dtype=torch.float32, device=dev)
    to, tl = torch.empty(op.shape[1:], device=dev), torch.empty(lp.shape[1:], device=dev)
    ms = timed(lambda: lsx.tree_merge(op, lp, out=to, lse_out=tl))
    nbytes = (k + 1) * (to.numel() * 4 + tl.numel() * 4)
    out["tree_merge"] = {"gbs": round(nbytes / ms / 1e6, 1), "frac": round(nbytes / ms / 1e6 / peak, 4),
                         "ms": round(ms, 4), "bytes": nbytes, "k": k}
    del op, lp, to, tl
    # split-KV decode at 1M keys
    w = WORKLOADS["decode_gqa_1m"]
    x = make_inputs(w, device=dev, with_grad=False)
    q, kc, vc = x["q"], x["k"], x["v"]
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    ws = torch.empty(lsx.decode_workspace_size(q, kc, w.chunk), dtype=torch.uint8, device=dev)
    ms = timed(lambda: lsx.decode(q, kc, vc, w.chunk, out=o, lse=lse, workspace=ws))
    nbytes = kc.numel() * 2 + vc.numel() * 2 + q.numel() * 2 + o.numel() * 2 + lse.numel() * 4
    out["decode"] = {"gbs": round(nbytes / ms / 1e6, 1), "frac": round(nbytes / ms / 1e6 / peak, 4),
                     "ms": round(ms, 4), "bytes": nbytes,
                     "workload": "B=8 Hq=32 Hkv=8 N=1048576 d=128 chunk=4096"}
    del x, q, kc, vc, o, lse, ws
    torch.cuda.empty_cache()
    out["peak_gbs"] = peak
    out["peak_kind"] = f"{pk['source']} HBM copy bandwidth"
    # fwd+bwd throughput of the other attention workloads (same flop
    # convention: visible pairs only), against the sustained bf16 peak
    for name, causal in (("causal_32k_ring", True), ("noncausal_64k_heavytail", False)):
        w = WORKLOADS[name]
        x = make_inputs(w, device=dev)
        q, k, v, d_o = x["q"], x["k"], x["v"], x["d_o"]
        o, lse = lsx.chunked_fwd(q, k, v, w.chunk, causal=causal)
        grads = lsx.chunked_bwd(q, k, v, o, lse, d_o, w.chunk, causal=causal)

        def fwd_bwd():
            lsx.chunked_fwd(q, k, v, w.chunk, causal=causal, out=o, lse=lse)
            lsx.chunked_bwd(q, k, v, o, lse, d_o, w.chunk, causal=causal, dq=grads[0],
                            dk=grads[1], dv=grads[2])

        ms = timed(fwd_bwd)
        ff, fb = flops(w.B, w.Hq, w.N, w.D, causal)
        tf = (ff + fb) / (ms / 1e3) / 1e12
        out[name] = {"tflops": round(tf, 1), "frac": round(tf / pk["bf16_sustained"], 4),
                     "frac_of_burst": round(tf / pk["bf16"], 4),
                     "ms": round(ms, 3), "flops": ff + fb,
                     "schedule": traced(fwd_bwd, dev),
                     "workload": f"B={w.B} H={w.Hq} N={w.N} d={w.D} chunk={w.chunk} "
                                 f"{'causal' if causal else 'non-causal'}"}
        del x, q, k, v, d_o, o, lse, grads
        torch.cuda.empty_cache()
    out["tflops_peak"] = pk["bf16_sustained"]
    # shared-prefix tree decoding: 8 branches x (Hq=32, Hkv=8) sharing a
    # 1M-key prefix, each with its own 4096-key suffix; against plain decode
    # of every branch over its own copy of prefix + suffix
    nbr, hq_, hkv_, npre, nsuf = 8, 32, 8, 1 << 20, 4096
    q = random_tensor((nbr, hq_, 1, 128), 101, device=dev)
    pre_k = random_tensor((1, hkv_, npre, 128), 102, device=dev)
    pre_v = random_tensor((1, hkv_, npre, 128), 103, device=dev)
    sk = random_tensor((nbr, hkv_, nsuf, 128), 104, device=dev)
    sv = random_tensor((nbr, hkv_, nsuf, 128), 105, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    # chunks of 8192 keys: the prefix kernel's per-chunk start and merge of
    # its warps' states cost half as often as with 4096 (also reported)
    chunk_t = 8192
    ms_tree = timed(lambda: lsx.decode_tree(q, pre_k, pre_v, sk, sv, chunk_t, out=o, lse=lse))
    ms_tree_4096 = timed(lambda: lsx.decode_tree(q, pre_k, pre_v, sk, sv, 4096, out=o, lse=lse))
    tree_bytes = (pre_k.numel() + pre_v.numel() + sk.numel() + sv.numel()) * 2 + 2 * q.numel() * 2
    kc = torch.cat([pre_k.expand(nbr, -1, -1, -1), sk], dim=2)
    vc = torch.cat([pre_v.expand(nbr, -1, -1, -1), sv], dim=2)
    del pre_k, pre_v, sk, sv
    ms_flat = timed(lambda: lsx.decode(q, kc, vc, chunk_t, out=o, lse=lse))
    out["decode_tree_1m_prefix"] = {
        "gbs": round(tree_bytes / ms_tree / 1e6, 1),
        "frac": round(tree_bytes / ms_tree / 1e6 / peak, 4), "ms": round(ms_tree, 4),
        "bytes": tree_bytes, "ms_per_branch_copies": round(ms_flat, 4),
        "speedup": round(ms_flat / ms_tree, 2), "ms_chunk_4096": round(ms_tree_4096, 4),
        "workload": "8 branches, Hq=32, Hkv=8, shared 1,048,576-key prefix + 4096-key "
                    "suffix each, chunk 8192"}
    del q, kc, vc, o, lse
    torch.cuda.empty_cache()
    # block-sparse: causal sliding window of 32 blocks (4096 keys) at 128K
    w = WORKLOADS["causal_128k_balanced"]
    x = make_inputs(w, device=dev)
    q, k, v, d_o = x["q"], x["k"], x["v"], x["d_o"]
    nb = w.N // 128
    win = 32
    mask = torch.zeros((nb, nb), dtype=torch.uint8)
    for i in range(nb):
        mask[i, max(0, i - win + 1):i + 1] = 1
    mask = mask.to(dev)
    o, lse = lsx.block_sparse_fwd(q, k, v, mask, True)
    grads = lsx.block_sparse_bwd(q, k, v, o, lse, d_o, mask, True)

    def bs_step():
        lsx.block_sparse_fwd(q, k, v, mask, True, out=o, lse=lse)
        lsx.block_sparse_bwd(q, k, v, o, lse, d_o, mask, True, dq=grads[0], dk=grads[1],
                             dv=grads[2])

    ms = timed(bs_step)
    # visible pairs: full off-diagonal blocks plus causal diagonal blocks
    blocks = int(mask.sum().item())
    pairs = (blocks - nb) * 128 * 128 + nb * 128 * 129 // 2
    fl = 4.0 * w.B * w.Hq * pairs * w.D * 3.5
    tf = fl / (ms / 1e3) / 1e12
    out["block_sparse_window_128k"] = {
        "tflops": round(tf, 1), "frac": round(tf / pk["bf16_sustained"], 4), "ms": round(ms, 3),
        "flops": fl, "blocks_computed": blocks, "blocks_causal": nb * (nb + 1) // 2,
        "workload": "causal_128k_balanced with a 32-block (4096-key) sliding-window block mask"}
    del x, q, k, v, d_o, o, lse, grads, mask
    torch.cuda.empty_cache()
    # backward through torch.autograd with the checkpoint at the attention
    # output (O, LSE kept) against the layer-boundary form (forward re-run)
    w = WORKLOADS["causal_32k_ring"]
    x = make_inputs(w, device=dev)
    q, k, v = (x[n_].requires_grad_() for n_ in ("q", "k", "v"))
    d_o = x["d_o"]
    res = {}
    for mode in ("output", "inputs"):
        ts = []
        for it in range(8):
            o = lsx.chunked_attention(q, k, v, w.chunk, True, checkpoint=mode)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record()
            o.backward(d_o)
            b.record()
            torch.cuda.synchronize()
            if it >= 3:
                ts.append(a.elapsed_time(b))
            q.grad = k.grad = v.grad = None
            del o
        res[mode] = statistics.median(ts)
    out["autograd_remat_32k"] = {
        "bwd_ms_checkpoint_output": round(res["output"], 3),
        "bwd_ms_checkpoint_inputs": round(res["inputs"], 3),
        "speedup": round(res["inputs"] / res["output"], 3),
        "workload": "causal_32k_ring through lsx.chunked_attention (torch.autograd)"}
    del x, q, k, v, d_o
    torch.cuda.empty_cache()

    import ctypes
    from long_sequence_exact_gb300 import _lib
    n1 = 32768
    q1 = random_tensor((1, 1, n1, 128), 4242, 0.5, device=dev)
    k1 = random_tensor((1, 1, n1, 128), 4243, 0.5, device=dev)
    v1 = random_tensor((1, 1, n1, 128), 4244, 0.5, device=dev)
    lib = _lib.load()
    vq1, vk1 = _lib.view(q1), _lib.view(k1)
    full = lib.attn_chunked_fwd_workspace_size(ctypes.byref(vq1), ctypes.byref(vk1), 4096, 1)
    base = lib.attn_chunk_fwd_workspace_size(ctypes.byref(vq1), ctypes.byref(vk1))
    ws_full = torch.empty(int(full), dtype=torch.uint8, device=dev)
    ws_base = torch.empty(int(base), dtype=torch.uint8, device=dev)
    o1 = torch.empty_like(q1)
    l1 = torch.empty((1, 1, n1), dtype=torch.float32, device=dev)
    t_split = timed(lambda: lsx.chunked_fwd(q1, k1, v1, 4096, True, out=o1, lse=l1,
                                            workspace=ws_full))
    t_whole = timed(lambda: lsx.chunked_fwd(q1, k1, v1, 4096, True, out=o1, lse=l1,
                                            workspace=ws_base))
    f1, _ = flops(1, 1, n1, 128, True)
    out["split_rows_32k_h1"] = {
        "split": full > base,
        "ms_split": round(t_split, 3), "ms_unsplit": round(t_whole, 3),
        "speedup": round(t_whole / t_split, 3),
        "tflops_split": round(f1 / (t_split / 1e3) / 1e12, 1),
        "frac_split": round(f1 / (t_split / 1e3) / 1e12 / pk["bf16_sustained"], 4),
        "workload": "B=1 H=1 N=32768 d=128 causal, forward (chunked_fwd)"}
    del q1, k1, v1, o1, l1, ws_full, ws_base
    n2 = 16384
    q2 = random_tensor((1, 1, n2, 128), 4252, 0.5, device=dev)
    k2 = random_tensor((1, 1, n2, 128), 4253, 0.5, device=dev)
    v2 = random_tensor((1, 1, n2, 128), 4254, 0.5, device=dev)
    do2 = random_tensor((1, 1, n2, 128), 4255, 1.0, device=dev)
    o2, l2 = lsx.chunked_fwd(q2, k2, v2, 4096, True)
    vq2, vk2 = _lib.view(q2), _lib.view(k2)
    full2 = lib.attn_chunked_bwd_workspace_size(ctypes.byref(vq2), ctypes.byref(vk2), 4096, 1)
    base2 = lib.attn_chunk_bwd_workspace_size(ctypes.byref(vq2), ctypes.byref(vk2))
    wsb_full = torch.empty(int(full2), dtype=torch.uint8, device=dev)
    wsb_base = torch.empty(int(base2), dtype=torch.uint8, device=dev)
    g2 = (torch.empty_like(q2), torch.empty_like(k2), torch.empty_like(v2))
    tb_split = timed(lambda: lsx.chunked_bwd(q2, k2, v2, o2, l2, do2, 4096, True, dq=g2[0],
                                             dk=g2[1], dv=g2[2], workspace=wsb_full))
    tb_whole = timed(lambda: lsx.chunked_bwd(q2, k2, v2, o2, l2, do2, 4096, True, dq=g2[0],
                                             dk=g2[1], dv=g2[2], workspace=wsb_base))
    _, fb2 = flops(1, 1, n2, 128, True)
    out["split_cols_bwd_16k_h1"] = {
        "split": full2 > base2,
        "ms_split": round(tb_split, 3), "ms_unsplit": round(tb_whole, 3),
        "speedup": round(tb_whole / tb_split, 3),
        "tflops_split": round(fb2 / (tb_split / 1e3) / 1e12, 1),
        "workload": "B=1 H=1 N=16384 d=128 causal, backward (chunked_bwd)"}
    del q2, k2, v2, do2, o2, l2, g2, wsb_full, wsb_base
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------ CPU oracle
CPU_ROWS_PER_HEAD = 16   # seeded random query rows in every head ...
CPU_TAIL_ROWS = 256      # ... plus the last rows of head 0


def cpu_sample():
    """The bounded sample of the 128K workload that both CPU legs time: for
    each of the 32 heads, 16 seeded random query rows, plus the last 256 query
    rows of head 0 (the rows that see the most keys).  Each head's q, k, v, dO
    are drawn with their own seed at the workload's scale (N(0,1)*0.5 for q,
    k, v; N(0,1) for dO).  Returns [(rows, q, k, v, d_o) per head] as fp64
    arrays of the bf16 values and the FLOPs the sample stands for (visible
    pairs only, forward + 2.5x backward)."""
    import numpy as np
    import torch

    from long_sequence_exact_gb300.inputs import WORKLOADS, random_tensor

    w = WORKLOADS[WORKLOAD]
    rng = np.random.default_rng(w.seed)
    f = lambda t: t.double().numpy()  # noqa: E731
    heads, flops_ = [], 0.0
    for h in range(w.Hq):
        rows = np.sort(rng.choice(w.N, size=CPU_ROWS_PER_HEAD, replace=False))
        if h == 0:
            rows = np.union1d(rows, np.arange(w.N - CPU_TAIL_ROWS, w.N))
        base = w.seed * 1000 + 4 * h
        q, k, v = (f(random_tensor((1, 1, w.N, w.D), base + i, w.qk_amp, torch.bfloat16))
                   for i in range(3))
        d_o = f(random_tensor((1, 1, w.N, w.D), base + 3, 1.0, torch.bfloat16))
        heads.append((rows, q, k, v, d_o))
        flops_ += 4.0 * float(np.sum(rows + 1)) * w.D * 3.5
    return heads, flops_


def time_cpu_sample(sample):
    """Wall seconds of the fp64 oracle's forward + backward over the sample."""
    from oracle import attention as A
    heads, _ = sample
    t0 = time.perf_counter()
    for rows, q, k, v, d_o in heads:
        A.attn_fwd(q, k, v, 0, 0, True, rows=rows)
        A.attn_bwd(q, k, v, d_o, 0, 0, True, rows=rows)
    return time.perf_counter() - t0


def cpu_baseline(repeats=4, sample=None):
    """The fp64 oracle as it stands, on the host cores, timed on cpu_sample()
    `repeats` times.  Value in the metric's unit (TFLOP/s by the same visible-
    pair convention), with the labelled extrapolation of that rate to one full
    step of the 128K workload."""
    import torch
    cores = len(os.sched_getaffinity(0))
    torch.set_num_threads(cores)
    sample = sample or cpu_sample()
    dt = sum(time_cpu_sample(sample) for _ in range(repeats)) / repeats
    rate = sample[1] / dt
    f_fwd, f_bwd = flops(1, 32, 131072, 128, True)
    n_rows = sum(len(h[0]) for h in sample[0])
    return {"value": round(rate / 1e12, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"fp64 numpy oracle, fwd+bwd of {n_rows} query rows of the causal 128K "
                       f"workload ({CPU_ROWS_PER_HEAD} seeded random rows in each of the 32 heads "
                       f"+ the last {CPU_TAIL_ROWS} rows of head 0), {dt:.2f} s per pass, "
                       f"{repeats} passes"),
            "seconds": round(dt, 3),
            "extrapolated_full_step_s": round((f_fwd + f_bwd) / rate, 1),
            "extrapolation": "full 128K fwd+bwd FLOPs / the sample's rate (not run)"}


def run_reference(args, rank):
    if rank != 0:
        return None
    import torch
    cores = len(os.sched_getaffinity(0))
    torch.set_num_threads(cores)
    sample = cpu_sample()  # the same sample as the main arm's cpu_baseline leg
    for _ in range(args.warmup):
        time_cpu_sample(sample)
    ts = []
    for _ in range(args.steps):
        ts.append(time_cpu_sample(sample))
    total = sum(ts)
    value = sample[1] * len(ts) / total / 1e12
    f_fwd, f_bwd = flops(1, 32, 131072, 128, True)
    n_rows = sum(len(h[0]) for h in sample[0])
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "B": 1, "H": 32, "N": 131072,
                                        "d": 128, "chunk_len": 4096, "causal": True},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "kind": "oracle", "cores": cores,
                         "sample": (f"fp64 numpy oracle, fwd+bwd of {n_rows} query rows of the "
                                    f"causal 128K workload ({CPU_ROWS_PER_HEAD} seeded random rows "
                                    f"in each of the 32 heads + the last {CPU_TAIL_ROWS} rows of "
                                    "head 0) per step"),
                         "extrapolated_full_step_s": round((f_fwd + f_bwd) / (value * 1e12), 1)},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-repeats", type=int, default=4,
                    help="passes over the oracle's CPU sample (about 2.5 s each on 16 cores)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-trace", action="store_true",
                    help="skip the untimed step that records the SM idle fraction")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the merge / tree-merge / decode bandwidth rows")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the dominant kernel from an ncu capture")
    ap.add_argument("--n", type=int, default=None,
                    help="sequence length override (profiling captures on a smaller case)")
    ap.add_argument("--heads", type=int, default=None, help="head count override (profiling)")
    ap.add_argument("--workload", default=None,
                    choices=("causal_32k_ring", "causal_128k_balanced", "noncausal_64k_heavytail"),
                    help="another attention workload in place of the headline one (profiling)")
    ap.add_argument("--deterministic", action="store_true",
                    help="the bit-repeatable backward (dK/dV kernel + owner-computes dQ kernel) "
                         "in place of the fused one (profiling)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        out = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
