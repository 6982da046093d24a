#!/usr/bin/env python
"""Benchmark of LazyAttention's hot path on GB300 (one JSON line on rank 0).

A step is one pass of the whole hot path over one batch of the workload: write the query
tokens' keys/values into the position-free paged cache, the causal query prefill (keys rotated
by their document offset), then every decode step (write the new token, attend with Q rotated
at document boundaries).  The documents were written into the cache once beforehand: that is
the premise of the method (one cached copy per document, reused at any offset).

Default workload (the decode-bound configuration, the largest that fits one GPU): the 8B
attention shape (32/8/128, RoPE theta 5e5), 64 requests x 20 documents x 1600 tokens drawn from
a 500-document pool by Zipf alpha 2.1 in random order (32 000-token contexts), 128 decode steps,
16-token pages.  ``--sharing private`` (default) gives every (request, doc) its own pages so that
logical bytes equal the bytes that must come from HBM; ``shared`` keeps one physical copy per
document.  Inputs are seeded synthetic bf16 N(0,1).  The same JSON line carries the tensor-core
prefill timed on its own on the 70B shape (``--prefill-workload``, a dense contraction) with its
deferred-rotation overhead, and the small-batch RAG workload (``--extra``) as a sub-object.

Each step is captured once as a CUDA graph and replayed; L2 is flushed (512 MB write) between
timed steps, outside the step's own events.  Per-launch decode durations come from event
records inside the graph, on the launching stream.

``--impl reference`` times the CPU oracle (fp64 NumPy) on a bounded sample per step instead.
Multi-GPU (torchrun): replicas only -- every rank runs the full workload on its own GPU, no
collective on the data path; the value is the total over ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode HBM GB/s and prefill TFLOP/s (fraction of GB300 peak); tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD_TEXT = {
    "rag8b": "Llama-3.1-8B attention (32 q / 8 kv heads, D 128, RoPE theta 5e5, bf16); 16 requests "
             "x 10 docs x 200 tokens from a 200-doc pool by Zipf 1.1, shuffled; 32-token causal "
             "query prefill then 64 decode steps; 16-token pages",
    "decode32k": "8B attention shape; 64 requests x 20 docs x 1600 tokens (Zipf 2.1, 500-doc pool); "
                 "128 decode steps over 32 000-token contexts",
    "prefill70b": "Llama-3.1-70B attention (64/8/128); 8 requests x 20 docs x 512 tokens (Zipf 1.5) "
                  "+ 64-token causal query prefill",
    "mqa_alibi": "MQA 32/1/128 with ALiBi; 32 requests x 12 docs x 1000 tokens, 32-token prefill, "
                 "64 decode steps",
    "yarn8b": "8B shape with YaRN (s 8, L0 8192); 32 requests x 12 docs x 1000 tokens, 32-token "
              "prefill, 64 decode steps",
    "tiny": "1 request, 4/2 heads, D 64; docs of 48 + 80 tokens; 16-token prefill, 8 decode steps",
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="decode32k")
    p.add_argument("--prefill-workload", default="prefill70b",
                   help="workload of the separately timed tensor-core prefill ('none' to skip)")
    p.add_argument("--extra", default="rag8b", help="comma-separated workloads also timed (sub-objects)")
    p.add_argument("--overhead-reps", type=int, default=20, help="timed launches per overhead variant")
    p.add_argument("--sharing", choices=["private", "shared"], default="private")
    p.add_argument("--batch", type=int, default=None,
                   help="keep only the first requests of --workload (smaller cases for profiling)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="launch eagerly instead of graph replay")
    p.add_argument("--pos", default=None, help="override positional kind (e.g. none for the Delta=0 twin)")
    p.add_argument("--no-overhead", action="store_true", help="skip the deferred-rotation overhead runs")
    return p.parse_args()


# ------------------------------------------------------------------ distributed plumbing
class Dist:
    def __init__(self):
        import torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ clocks
class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 7:
                    try:
                        rows.append((float(parts[0]), float(parts[1]), parts[3:7]))
                    except ValueError:
                        pass
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, flags in rows for n, f in zip(names, flags) if f == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_hash(text: str) -> str:
    """sha256 (16 hex digits) of a C++/CUDA source with its comments and blank space removed:
    it changes when the code changes, not when a comment does."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [ln.strip() for ln in text.split("\n") if ln.strip()]
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def profiled_traffic(kernel_src: str, name: str):
    """Per-launch DRAM bytes recorded by an ncu capture in profiles/<name>, valid only while
    the kernel's code (comments aside) still hashes to the value recorded there."""
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    with open(os.path.join(ROOT, "position_agnostic_kv_gb300", "csrc", kernel_src)) as f:
        h = code_hash(f.read())
    text = open(path).read()
    m_h = re.search(r"code_sha256_16:\s*([0-9a-f]{16})", text)
    m_t = re.search(r"dram_bytes_per_launch_full:\s*([0-9.eE+]+)", text)
    if not m_h or not m_t or m_h.group(1) != h:
        return None
    return float(m_t.group(1))


def job_throughput(dist, tokens_per_step: int, step_ms: list) -> tuple:
    """Whole-job throughput of a replicas-only run: every rank processes `tokens_per_step` per
    step, and the job's step time is the slowest rank's mean (max over ranks)."""
    mean_ms = dist.max(sum(step_ms) / len(step_ms))
    return dist.world * tokens_per_step / (mean_ms / 1e3), mean_ms


# ------------------------------------------------------------------ our arm
def _prepare(w, dev, pos_kind=None):
    """Resident batch of workload `w`: documents written once (the method's premise), the
    step's inputs packed into one device buffer and its outputs into another, so that an
    end-to-end run moves them with one host->device and one device->host copy per step."""
    import torch
    from position_agnostic_kv_gb300.runner import PagedBatch
    pb = PagedBatch(w, device=dev, pos_kind=pos_kind)
    pb.fill_documents()
    torch.cuda.synchronize()
    in_blob, (pre, *decs) = pack_views([pb.upload_prefill() if pb.total_q else {}] +
                                       [pb.upload_decode(t) for t in range(w.n_decode)], dev)
    out_blob, outs = pack_views([{"o": torch.empty((max(pb.total_q, 1), w.Hq, w.D), dtype=torch.bfloat16)}] +
                                [{"o": torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16)}
                                 for _ in range(w.n_decode)], dev)
    return pb, (pre or None), decs, in_blob, out_blob, outs[0]["o"], [o["o"] for o in outs[1:]]


def measure_step(args, dist, lk, name, sharing, steps, warmup, clocks=None, e2e=False, overhead=True):
    """Time `steps` steps of workload `name` (each: the query tokens' KV write and prefill, then
    every decode step's KV write and decode), captured once as a CUDA graph and replayed, L2
    flushed before every timed step.  Returns the per-workload part of the JSON line."""
    import numpy as np
    import torch
    from workloads import make_workload

    dev = torch.device("cuda", dist.local_rank)
    w = make_workload(name, sharing=sharing, batch=args.batch if name == args.workload else None)
    pb, pre, decs, in_blob, out_blob, out_p, outs_d = _prepare(w, dev, args.pos)
    n_dec = w.n_decode
    stream = torch.cuda.Stream(device=dev)
    use_graph = not args.no_graph

    def mk():
        return torch.cuda.Event(enable_timing=True, external=True) if use_graph else \
            torch.cuda.Event(enable_timing=True)

    # Event pairs on the prefill and on every 8th decode launch: enough samples for the
    # per-launch times, few enough event nodes to leave the step's own time unchanged.
    ev_steps = list(range(0, n_dec, 8))
    ev_pre = (mk(), mk())
    ev_dec = {t: (mk(), mk()) for t in ev_steps}
    launches = 0

    def step():
        nonlocal launches
        launches = 0
        if pre is not None:
            lk.kv_write(pre["k"], pre["v"], pre["slot"], pre["lp"], pb.k_cache, pb.v_cache, pb.cfg,
                        stream=stream)
            ev_pre[0].record(stream)
            lk.attn_prefill(pre["q"], pb.cu_q, pb.q_start, pb.doc_blocks, pb.meta, pb.k_cache,
                            pb.v_cache, pb.cfg, out_p[: pb.total_q], pb.max_q, ws=pb.ws, stream=stream)
            ev_pre[1].record(stream)
            launches += 1 + launches_of("prefill", pb)
        for t in range(n_dec):
            d = decs[t]
            lk.kv_write(d["k"], d["v"], d["slot"], d["lp"], pb.k_cache, pb.v_cache, pb.cfg, stream=stream)
            if t in ev_dec:
                ev_dec[t][0].record(stream)
            lk.attn_decode(d["q"], d["seq_len"], pb.q_start, pb.doc_blocks, pb.meta, pb.k_cache,
                           pb.v_cache, pb.cfg, outs_d[t], ws=pb.ws, stream=stream)
            if t in ev_dec:
                ev_dec[t][1].record(stream)
            launches += 1 + launches_of("decode", pb)

    # warm-up (also sets kernel attributes before any capture)
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    graph = None
    if use_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                step()
            torch.cuda.synchronize()
        except Exception as e:  # graph capture unsupported here: launch eagerly
            print(f"[bench] graph capture failed ({e}); launching eagerly", file=sys.stderr)
            graph = None

    def run_step():
        with torch.cuda.stream(stream):
            if graph is not None:
                graph.replay()
            else:
                step()

    for _ in range(warmup):
        run_step()
    torch.cuda.synchronize()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    dec_ms, pre_ms, step_ms = [], [], []
    dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    wall0 = time.perf_counter()
    inner_ok = True
    for k in range(steps):
        with torch.cuda.stream(stream):
            flush.zero_()
            e0[k].record(stream)
            run_step()
            e1[k].record(stream)
        stream.synchronize()
        step_ms.append(e0[k].elapsed_time(e1[k]))
        if inner_ok:
            try:
                if pre is not None:
                    pre_ms.append(ev_pre[0].elapsed_time(ev_pre[1]))
                dec_ms.extend(a.elapsed_time(b) for a, b in ev_dec.values())
            except RuntimeError as e:
                print(f"[bench] in-graph event timing unavailable ({e})", file=sys.stderr)
                inner_ok = False
                pre_ms, dec_ms = [], []
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    dist.barrier()
    clk = clocks.stop() if clocks else None
    if not inner_ok:  # per-launch times from eager launches of the same step, L2 flushed
        for _ in range(min(steps, 10)):
            with torch.cuda.stream(stream):
                flush.zero_()
                step()
            stream.synchronize()
            pre_ms.append(ev_pre[0].elapsed_time(ev_pre[1]) if pre is not None else 0.0)
            dec_ms.extend(a.elapsed_time(b) for a, b in ev_dec.values())
    status = lk.device_status()
    if status:
        raise RuntimeError(f"device status {status:#x} after the timed region")

    tokens_per_step = pb.total_q + w.B * n_dec
    value, mean_ms = job_throughput(dist, tokens_per_step, step_ms)

    # algorithmic units (sizes only): decode bytes per launch, prefill flops per launch
    keys0 = pb.seq_len0_h.astype(np.int64)
    kv_row = w.Hkv * w.D * 2 * 2
    dec_bytes = []
    for t in range(n_dec):
        keys = keys0 + t + 1
        blocks = pb.doc_blocks_h.astype(np.int64) + (keys - 1 - pb.q_start_h) // 16 + 1
        dec_bytes.append(int(keys.sum()) * kv_row + 2 * w.B * w.Hq * w.D * 2 + int(blocks.sum()) * 8)
    avg_dec_bytes = statistics.mean(dec_bytes[t] for t in ev_steps) if ev_steps else 0.0
    avg_dec_ms = statistics.mean(dec_ms) if dec_ms else 0.0
    peaks, peak_kind = load_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    achieved_gbs = avg_dec_bytes / (avg_dec_ms / 1e3) / 1e9 if dec_ms else None
    pre_flops = prefill_flops(w, pb)
    # mean over the timed steps (single launches jitter in ~2 us steps; see rotation_overhead)
    pre_med = statistics.median(pre_ms) if pre_ms else None
    pre_mean = statistics.fmean(pre_ms) if pre_ms else None
    pre_tflops = pre_flops / (pre_mean / 1e3) / 1e12 if pre_mean else None
    bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))

    dec_total = avg_dec_ms * n_dec if dec_ms else 0.0
    if dec_total >= (pre_mean or 0.0):  # the dominant kernel of the step
        traffic = profiled_traffic("decode.cu", f"decode_{name}_{sharing}.md")
        roofline = {"kernel": "lazy_attn_decode (split-KV decode + lse merge)", "bound": "hbm",
                    "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved_gbs / hbm_peak, "peak_source": f"{peak_kind} hbm_gbs",
                    "traffic": traffic, "algorithmic_bytes_per_launch": avg_dec_bytes,
                    "avg_launch_us": avg_dec_ms * 1e3}
    else:
        traffic = profiled_traffic("prefill_tc.cu", f"prefill_{name}_{sharing}.md")
        roof = prefill_roof(pre_flops, prefill_bytes(w, pb), pre_mean * 1e3, peaks)
        if roof["bound"] == "tensor":
            roofline = {"kernel": "lazy_attn_prefill (tcgen05)", "bound": "tensor", "achieved": pre_tflops,
                        "peak": bf16_peak, "unit": "TFLOP/s", "frac": pre_tflops / bf16_peak,
                        "peak_source": f"{peak_kind} bf16_tflops (burst)", "traffic": traffic,
                        "algorithmic_flops_per_launch": pre_flops, "avg_launch_us": pre_mean * 1e3}
        else:
            roofline = {"kernel": "lazy_attn_prefill (tcgen05)", "bound": "hbm", "achieved": roof["hbm_gbs"],
                        "peak": hbm_peak, "unit": "GB/s", "frac": roof["frac_hbm_peak"],
                        "peak_source": f"{peak_kind} hbm_gbs", "traffic": traffic,
                        "algorithmic_bytes_per_launch": prefill_bytes(w, pb), "avg_launch_us": pre_mean * 1e3}
    res = {
        "value": value, "ms_per_step": mean_ms, "tokens_per_step": tokens_per_step,
        "workload": f"{name}: {WORKLOAD_TEXT[name]}" + (f" (first {w.B} requests)" if w.B != make_workload(
            name, sharing=sharing).B else ""), "sharing": sharing, "pos": args.pos or w.pos.kind,
        "global_batch": w.B * dist.world, "seq_len": int(keys0.max()) + n_dec,
        "launch": "CUDA graph per step" if graph is not None else "eager",
        "roofline": roofline,
        "decode": None if not n_dec else {
            "kernel": "lazy_attn_decode", "bytes_per_launch": avg_dec_bytes if dec_ms else None,
            "avg_launch_us": avg_dec_ms * 1e3 if dec_ms else None, "gbs": achieved_gbs,
            "timed_launches": f"decode steps {ev_steps} of every timed step (CUDA events in the graph)",
            "frac_hbm_peak": achieved_gbs / hbm_peak if achieved_gbs else None,
            "launches_per_step": n_dec},
        "step_prefill": None if pre is None else {
            "kernel": "lazy_attn_prefill", "flops_per_launch": pre_flops,
            "mean_us": pre_mean * 1e3 if pre_mean else None,
            "median_us": pre_med * 1e3 if pre_med else None, "tflops": pre_tflops,
            "frac_bf16_peak": pre_tflops / bf16_peak if pre_tflops else None,
            "hbm_bytes_per_launch": prefill_bytes(w, pb),
            "peak_source": f"{peak_kind} bf16_tflops (burst)",
            **(prefill_roof(pre_flops, prefill_bytes(w, pb), pre_mean * 1e3, peaks) if pre_mean else {})},
        "gpu_launches": launches * steps,
        "wall_s_timed_region": wall,
    }
    if clk is not None:
        res["clocks"] = clk
    if overhead and pb.cfg.kind in (lk.POS_ROPE, lk.POS_YARN):
        res["rotation_overhead"] = rotation_overhead(args, lk, pb, pre, decs, out_p, outs_d, stream, flush)
    if e2e:
        res["e2e"] = run_e2e(args, in_blob, out_blob, run_step, stream, dist, tokens_per_step)
    del graph
    return res


def prefill_flops(w, pb) -> int:
    """4 D Hq x (keys visible to each query row), summed: QK^T and PV, causal-exact."""
    flops = 0
    for b in range(w.B):
        L = int(w.q_len[b])
        flops += 4 * w.D * w.Hq * sum(int(pb.q_start_h[b]) + i + 1 for i in range(L))
    return flops


def prefill_bytes(w, pb) -> int:
    """Unique bytes a prefill launch must move: every visible key's K and V row once per KV head
    (Q rows and outputs included)."""
    keys = sum(int(pb.q_start_h[b]) + int(w.q_len[b]) for b in range(w.B) if w.q_len[b])
    return keys * w.Hkv * w.D * 2 * 2 + 2 * pb.total_q * w.Hq * w.D * 2


def prefill_roof(flops, nbytes, us, peaks):
    """Which roof bounds a prefill launch: its arithmetic intensity (FLOPs per unique HBM byte)
    against the ridge of the measured peaks (bf16 FLOP/s over copy bytes/s), and the launch's
    rate against the HBM roof (for short queries over long contexts the bytes, not the MMAs,
    set the floor)."""
    bf16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    intensity, ridge = flops / nbytes, bf16 * 1e12 / (hbm * 1e9)
    gbs = nbytes / (us / 1e6) / 1e9
    return {"bound": "tensor" if intensity > ridge else "hbm", "intensity_flop_per_byte": intensity,
            "ridge_flop_per_byte": ridge, "hbm_gbs": gbs, "frac_hbm_peak": gbs / hbm}


def prefill_probe(args, dist, lk, name, sharing):
    """The tensor-core prefill on its own workload (by default the 70B shape, whose prefill is
    a dense contraction): median of eager launches with L2 flushed before each, over the same
    resident caches as its Delta = 0 twin (the rotation_overhead runs)."""
    import torch
    from workloads import make_workload
    dev = torch.device("cuda", dist.local_rank)
    w = make_workload(name, sharing=sharing)
    pb, pre, _, _, _, out_p, _ = _prepare(w, dev, None)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        lk.kv_write(pre["k"], pre["v"], pre["slot"], pre["lp"], pb.k_cache, pb.v_cache, pb.cfg, stream=stream)
    stream.synchronize()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    ovh = rotation_overhead(args, lk, pb, pre, [], out_p, [], stream, flush)
    peaks, peak_kind = load_peaks()
    bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    flops = prefill_flops(w, pb)
    us = ovh["prefill"]["rot_us"]
    tflops = flops / (us / 1e6) / 1e12
    return {"workload": f"{name}: {WORKLOAD_TEXT[name]}", "sharing": sharing,
            "kernel": "lazy_attn_prefill (tcgen05)", "flops_per_launch": flops,
            "hbm_bytes_per_launch": prefill_bytes(w, pb), "mean_us": us,
            "median_us": ovh["prefill"]["median_us"]["rot"], "tflops": tflops,
            "frac_bf16_peak": tflops / bf16_peak, "peak": bf16_peak,
            "peak_source": f"{peak_kind} bf16_tflops (burst: the kernel is timed on its own)",
            **prefill_roof(flops, prefill_bytes(w, pb), us, peaks),
            "timing": "eager launches, L2 flushed before each, mean (same runs as rotation_overhead)",
            "traffic": profiled_traffic("prefill_tc.cu", f"prefill_{name}_{sharing}.md"),
            "rotation_overhead": ovh["prefill"] | {"method": ovh["method"],
                                                   **({"launch_errors": ovh["launch_errors"]}
                                                      if "launch_errors" in ovh else {})}}


def run_ours(args, dist):
    import torch
    import position_agnostic_kv_gb300 as lk

    torch.cuda.set_device(dist.local_rank)
    clocks = Clocks(dist.local_rank)
    main = measure_step(args, dist, lk, args.workload, args.sharing, args.steps, args.warmup, clocks=clocks,
                        e2e=not args.no_e2e, overhead=not args.no_overhead)
    res = {
        "metric": METRIC, "value": main["value"], "unit": "tokens/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16; Zipf-drawn documents)",
        "config": {"workload": main["workload"], "sharing": main["sharing"], "pos": main["pos"],
                   "global_batch": main["global_batch"], "seq_len": main["seq_len"],
                   "tokens_per_step": main["tokens_per_step"], "parallelism": f"replicas x{dist.world}",
                   "l2": "flushed between timed steps (512 MB write, outside the step events); "
                         "the K/V read per step also exceeds L2",
                   "launch": main["launch"]},
        "roofline": main["roofline"],
        "decode": main["decode"],
        "gpu_launches": main["gpu_launches"],
        "clocks": main.get("clocks"),
        "wall_s_timed_region": main["wall_s_timed_region"],
    }
    if main["step_prefill"] is not None:
        res["step_prefill"] = main["step_prefill"]
    ovh = {}
    if "rotation_overhead" in main:
        ovh = {k: v for k, v in main["rotation_overhead"].items()}
    if args.prefill_workload != "none":
        res["prefill"] = prefill_probe(args, dist, lk, args.prefill_workload, args.sharing)
        ovh["prefill_" + args.prefill_workload] = res["prefill"]["rotation_overhead"]
    if ovh:
        res["rotation_overhead"] = ovh
    extra = {}
    for name in [x for x in args.extra.split(",") if x and x not in ("none", args.workload)]:
        e = measure_step(args, dist, lk, name, args.sharing, min(args.steps, 20), args.warmup,
                         overhead=not args.no_overhead)
        extra[name] = {k: e[k] for k in ("value", "ms_per_step", "tokens_per_step", "workload", "decode",
                                         "step_prefill", "rotation_overhead", "roofline") if k in e}
    if extra:
        res["extra_workloads"] = extra
    if "e2e" in main:
        res["e2e"] = main["e2e"]
    return res


def rotation_overhead(args, lk, pb, pre, decs, out_p, outs_d, stream, flush):
    """Deferred-rotation cost: the same attention launches over the same caches with
    (rot) the workload's rotary kind, (delta0) the kernels built without any positional work
    (the Delta = 0 twin), and (same_delta) the rotary kernels with every block's Delta set to 0,
    so that no document boundary occurs.  Eager launches, L2 flushed before each; each time is
    the mean of the repetitions (a single launch takes one of a few values about 2 us apart,
    start-up jitter of the GPU, so a median snaps to one of them while the mean weighs them;
    the medians are reported too); overhead = t_rot / t_delta0 - 1."""
    import numpy as np
    import torch
    cfg_none = lk.pos_cfg_from("none", pb.D)
    meta0_h = pb.meta_h & ~np.uint64(0xFFFFFF << 16)  # Delta field cleared
    meta0 = torch.from_numpy(meta0_h.view(np.int64)).to(pb.meta.device)
    variants = {"rot": (pb.cfg, pb.meta), "delta0": (cfg_none, pb.meta), "same_delta": (pb.cfg, meta0)}
    reps = max(5, args.overhead_reps)
    dec_idx = list(range(0, len(decs), max(1, len(decs) // 8)))[:8]
    out = {}
    errors, statuses = {}, set()
    for phase in ("prefill", "decode"):
        if (phase == "prefill" and pre is None) or (phase == "decode" and not decs):
            continue
        med, mean = {}, {}
        for name, (cfg, meta) in variants.items():
            ts = []
            for r in range(reps + 2):
                for t in ([None] if phase == "prefill" else dec_idx):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    with torch.cuda.stream(stream):
                        flush.zero_()
                        e0.record(stream)
                        if phase == "prefill":
                            lk.attn_prefill(pre["q"], pb.cu_q, pb.q_start, pb.doc_blocks, meta, pb.k_cache,
                                            pb.v_cache, cfg, out_p[: pb.total_q], pb.max_q, ws=pb.ws, stream=stream)
                        else:
                            d = decs[t]
                            lk.attn_decode(d["q"], d["seq_len"], pb.q_start, pb.doc_blocks, meta, pb.k_cache,
                                           pb.v_cache, cfg, outs_d[t], ws=pb.ws, stream=stream)
                        e1.record(stream)
                    stream.synchronize()
                    status = lk.device_status(stream)
                    if status:  # a launch that reported an error is counted and not timed
                        errors[f"{phase}/{name}"] = errors.get(f"{phase}/{name}", 0) + 1
                        statuses.add(status)
                    elif r >= 2:
                        ts.append(e0.elapsed_time(e1) * 1e3)
            med[name] = statistics.median(ts) if ts else float("nan")
            mean[name] = statistics.fmean(ts) if ts else float("nan")
        out[phase] = {"rot_us": mean["rot"], "delta0_us": mean["delta0"], "same_delta_us": mean["same_delta"],
                      "overhead": mean["rot"] / mean["delta0"] - 1.0,
                      "boundary_share": (mean["rot"] - mean["same_delta"]) / mean["delta0"],
                      "median_us": {"rot": med["rot"], "delta0": med["delta0"], "same_delta": med["same_delta"]}}
    out["method"] = ("same caches and inputs; rot = rotary kind of the workload, delta0 = kernels "
                     "without positional work, same_delta = rotary kernels with every Delta = 0; "
                     f"eager launches, L2 flushed before each, mean of {reps} reps (medians alongside)"
                     + (f", decode steps {dec_idx}" if decs else ""))
    if errors:  # reported, not hidden: launches whose kernels set a device status bit
        out["launch_errors"] = {"count": errors, "status_bits": sorted(hex(x) for x in statuses)}
        print(f"[bench] overhead runs: launches reported device status {sorted(hex(x) for x in statuses)}: "
              f"{errors}", file=sys.stderr)
    return out


def launches_of(phase: str, pb) -> int:
    """Kernels one attention call launches: the attention kernel, plus the lse merge when the
    KV sequence is split (workspace needed)."""
    import position_agnostic_kv_gb300 as lk
    if phase == "decode":
        ws = lk.workspace_size(lk.PHASE_DECODE, pb.B, pb.B, pb.max_blocks, pb.Hq, pb.Hkv, pb.D)
    else:
        ws = lk.workspace_size(lk.PHASE_PREFILL, pb.total_q, pb.B, pb.max_blocks, pb.Hq, pb.Hkv, pb.D)
    return 1 + (1 if ws > 0 else 0)


def pack_views(dicts, dev):
    """One device buffer holding every tensor of `dicts` (each at a 256-byte aligned offset);
    returns the buffer and the same dicts with each tensor replaced by its view in it."""
    import torch
    offs, total = [], 0
    for d in dicts:
        o = {}
        for k, t in d.items():
            o[k] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        offs.append(o)
    blob = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
    views = []
    for d, o in zip(dicts, offs):
        v = {}
        for k, t in d.items():
            n = t.numel() * t.element_size()
            v[k] = blob[o[k]:o[k] + n].view(t.dtype).view(t.shape)
            v[k].copy_(t)
        views.append(v)
    return blob, views


def run_e2e(args, in_blob, out_blob, run_step, stream, dist, tokens_per_step):
    """Same step, but its inputs start in pinned host memory and its outputs return to pinned
    host memory: one host->device copy of the step's packed inputs (query tokens and every
    decode step's q, k, v, slots, positions, lengths), the step, one device->host copy of its
    packed outputs (prefill and every decode step's attention output), all timed."""
    import torch
    host_in = in_blob.cpu().pin_memory()
    host_out = torch.empty(out_blob.shape, dtype=out_blob.dtype).pin_memory()
    h2d, d2h = in_blob.numel() * in_blob.element_size(), out_blob.numel() * out_blob.element_size()
    times = []
    n = max(3, min(args.steps, 50))
    for k in range(n + 2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            in_blob.copy_(host_in, non_blocking=True)
            run_step()
            host_out.copy_(out_blob, non_blocking=True)
            e1.record(stream)
        stream.synchronize()
        if k >= 2:
            times.append(e0.elapsed_time(e1))
    if not torch.equal(host_out.view(-1)[:1024], out_blob.view(-1)[:1024].cpu()):
        raise RuntimeError("end-to-end outputs did not reach the host buffer")
    ms = dist.max(statistics.mean(times))
    return {"value": dist.world * tokens_per_step / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "steps": n, "api": "position_agnostic_kv_gb300 binding over liblazykv (C ABI); one packed "
                               "pinned host buffer each way per step"}


# ------------------------------------------------------------------ the oracle (CPU)
def oracle_sample(w, reqs, n_dec):
    """Prepare the oracle's caches for `reqs` (setup, untimed) and return a closure that runs
    one bounded sample of the step for them: KV write of their query tokens, their prefill rows,
    then n_dec decode steps."""
    import numpy as np
    import oracle
    shape = (w.num_pages, w.Hkv, oracle.PAGE, w.D)
    kc, vc = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    pos = w.pos.as_dict()
    for b in reqs:
        for i in w.req_inst[w.req_inst_off[b]:w.req_inst_off[b + 1]]:
            k, v = w.doc_kv(int(w.inst_doc[i]))
            slot, lp = w.inst_slots(int(i))
            oracle.kv_write(k, v, slot, lp, pos, kc, vc)
    _, meta, seq_len, q_start, doc_blocks = oracle.build_meta(
        w.req_inst_off, w.req_inst, w.inst_len, w.inst_page_off, w.inst_pages, w.q_len,
        w.q_page_off, w.q_pages, w.max_blocks)
    q, k, v, slot, lp = w.prefill_tokens()
    rows = np.concatenate([np.arange(w.cu_q[b], w.cu_q[b + 1]) for b in reqs]) if len(slot) else np.zeros(0, int)
    decs = [w.decode_tokens(t) for t in range(n_dec)]
    tokens = len(rows) + n_dec * len(reqs)

    def run():
        if len(rows):
            oracle.kv_write(k[rows], v[rows], slot[rows], lp[rows], pos, kc, vc)
            oracle.prefill(q, w.cu_q, q_start, doc_blocks, meta, kc, vc, pos, requests=reqs)
        for t, (qd, kd, vd, sd, lpd) in enumerate(decs):
            oracle.kv_write(kd[reqs], vd[reqs], sd[reqs], lpd[reqs], pos, kc, vc)
            oracle.decode(qd, seq_len + t + 1, q_start, doc_blocks, meta, kc, vc, pos, requests=reqs)
    return run, tokens


# Bounded oracle samples per workload: (requests, decode steps) for the CPU baseline of our
# line, and for one step of the reference arm.  One decode step of one decode32k request (32 000
# keys rotated and attended in fp64) takes about 0.6 s on 16 Arm cores.
ORACLE_SAMPLE = {"decode32k": ((8, 2), (2, 1)), "prefill70b": ((2, 0), (1, 0))}
DEFAULT_SAMPLE = ((8, 16), (1, 2))


def cpu_baseline(args):
    from workloads import make_workload
    w = make_workload(args.workload, sharing=args.sharing)
    (n_req, n_dec), _ = ORACLE_SAMPLE.get(args.workload, DEFAULT_SAMPLE)
    reqs = list(range(min(w.B, n_req)))
    n_dec = min(w.n_decode, n_dec)
    run, tokens = oracle_sample(w, reqs, n_dec)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    what = (f"their query prefill + {n_dec} decode steps" if w.q_len.sum() else f"{n_dec} decode step(s)")
    return {"value": tokens / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"{len(reqs)} requests of {args.workload}: {what} ({tokens} tokens, {dt:.1f} s, "
                      f"NumPy fp64, BLAS threads = all cores)"}


def run_reference(args, dist):
    """The oracle as the reference arm: each step = one bounded sample of the workload."""
    from workloads import make_workload
    w = make_workload(args.workload, sharing=args.sharing)
    _, (n_req, n_dec) = ORACLE_SAMPLE.get(args.workload, DEFAULT_SAMPLE)
    reqs = list(range(min(w.B, n_req)))
    n_dec = min(w.n_decode, n_dec)
    run, tokens = oracle_sample(w, reqs, n_dec)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    value = tokens / (ms / 1e3)
    cores = len(os.sched_getaffinity(0))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16; Zipf-drawn documents)",
            "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}",
                       "sharing": args.sharing, "sample_per_step": f"request 0: query prefill (if any) + {n_dec} decode steps"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"request 0 of {args.workload}: prefill (if any) + {n_dec} decode steps ({tokens} tokens) per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        class _D:  # no process group for the CPU arm
            world = int(os.environ.get("WORLD_SIZE", "1"))
        print(json.dumps(run_reference(args, _D())), flush=True)
        return
    dist = Dist()
    try:
        res = run_ours(args, dist)
        if dist.rank == 0:
            if dist.world == 1 and not args.no_cpu_baseline:
                res["cpu_baseline"] = cpu_baseline(args)
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
