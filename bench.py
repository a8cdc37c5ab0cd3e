"""Benchmark of the W8A8 INT8 attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  * prefill, Qwen3-8B shape: B1 Hq32 Hkv8 N4096 d128, bf16, causal, K-smoothing
    (K channel mean, per-row int8 quantisation of Q and K, int32 QK^T on the tensor
    cores, online softmax, bf16 P.V) -- the workload the metric is quoted on;
  * decode: split-KV over an int8 KV cache, B64 Hq32 Hkv8 d128, context lengths
    uniform on [1024, 8192] (q quantisation, split kernel, combine).
`value` is prefill TOPS (ops = 2 x 2 x d x causal pairs x heads, QK^T and P.V);
the decode KV GB/s sits in `decode`, and `paged_decode` repeats the decode over a
paged k8v8 cache (64-token pages in a seeded random order) in a loop of its own after
the timed steps, `decode_f16v` the decode with an fp16 V cache (int8 K), and
`prefill_chunk` the prefill's last 1024 positions as a query chunk (chunked prefill,
bottom-right causal), `prefill_w8a8` the prefill through attn_w8a8_fwd (scales per 32
positions, outlier-aware Q), and `decode_verify` the decode with 4 chained draft
queries per sequence (speculative verify).  Inputs are resident in HBM when the timed
region starts (the timed steps carry no per-launch instrumentation: per-kernel times
come from a separate traced pass); L2 is flushed before every step, outside the timed
events (a 256 MB
write, then a read of that buffer, so no dirty lines of the flush remain).  `e2e` repeats the prefill through the public API with pinned host
inputs copied in and the output copied back every step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the only reference this path has) on a
bounded sample of the same prefill workload.
"""
from __future__ import annotations

import argparse
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

PREFILL = "qwen3_8b"
DECODE = "decode"
L2_FLUSH_BYTES = 256 << 20
METRIC = "W8A8 attn prefill TOPS & decode KV GB/s (1xGB300, % of INT8-TC / HBM roofline)"


def prefill_ops(w) -> float:
    pairs = w.N * (w.N + 1) // 2 * w.Hq * w.B
    return 2.0 * 2.0 * w.d * pairs


CHUNK_Q = 1024   # query chunk of the chunked-prefill line: the last 1024 of the 4096 positions


def chunk_ops(w, nq) -> float:
    """QK^T + P.V ops of a causal query chunk of the last nq positions of N keys."""
    off = w.N - nq
    pairs = (nq * off + nq * (nq + 1) // 2) * w.Hq * w.B
    return 2.0 * 2.0 * w.d * pairs


def decode_bytes(w, lens) -> float:
    kv = float(np.sum(lens)) * w.Hkv * (2 * w.d + 2 * 4)
    return kv + w.B * w.Hq * w.d * 2 * 2


def decode_bytes_f16v(w, lens) -> float:
    """Algorithmic bytes of the fp16-V decode: int8 K codes + K scales + fp16 V, q and out."""
    kv = float(np.sum(lens)) * w.Hkv * (w.d + 4 + 2 * w.d)
    return kv + w.B * w.Hq * w.d * 2 * 2


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=p["hbm_gbs"], bf16_tflops=p["bf16_tflops"],
                    bf16_sustained=p.get("bf16_tflops_sustained", p["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ reference arm: the CPU oracle

def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    import workloads as W
    w = W.get(PREFILL)
    q, k, v = W.prefill_dense(w)
    qn, kn, vn = q.float().numpy(), k.float().numpy(), v.float().numpy()
    rows = [(0, h, i) for h in range(w.Hq) for i in range(w.N)]
    ops = 2.0 * 2.0 * w.d * sum(i + 1 for (_, _, i) in rows)
    times = []
    for it in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.attn_prefill(qn, kn, vn, causal=True, smooth_k=True, rows=rows)
        dt = time.perf_counter() - t0
        if it >= args.warmup:
            times.append(dt)
    sec = float(np.mean(times))
    tops = ops / sec / 1e12
    sample = f"the whole prefill workload, every query row of all {w.Hq} heads ({ops / 1e9:.1f} GOP per step)"
    line = {"impl": "reference", "metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{PREFILL} prefill sample (B1 Hq32 Hkv8 N4096 d128, causal, smooth_k)"},
            "cpu_baseline": {"value": tops, "unit": "TOPS", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": tops, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline_leg(w, qn, kn, vn):
    """The oracle as it stands on the prefill workload (every row; seconds of CPU work)."""
    import oracle
    rows = [(0, h, i) for h in range(w.Hq) for i in range(w.N)]
    ops = 2.0 * 2.0 * w.d * sum(i + 1 for (_, _, i) in rows)
    t0 = time.perf_counter()
    oracle.attn_prefill(qn, kn, vn, causal=True, smooth_k=True, rows=rows)
    sec = time.perf_counter() - t0
    return {"value": ops / sec / 1e12, "unit": "TOPS", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"the whole prefill workload, all {w.Hq} heads x {w.N} rows ({ops / 1e9:.1f} GOP), {sec:.1f} s"}


# ------------------------------------------------------------------ our arm

def run_ours(args, world, rank, local):
    import torch
    import workloads as W
    import w8a8_int8_flashattention_gb300 as sl8
    from w8a8_int8_flashattention_gb300 import build as sl8_build

    sl8_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()

    # ---- prefill inputs (HBM resident)
    wp = W.get(PREFILL)
    q, k, v = W.prefill_dense(wp)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ws = torch.empty(sl8.prefill_workspace_bytes(wp.B, wp.Hq, wp.Hkv, wp.N, wp.d), dtype=torch.uint8, device=dev)
    out = torch.empty_like(qd)

    # ---- decode inputs: fp32 cache values quantised into the int8 cache by the library
    wd = W.get(DECODE)
    if args.only in ("prefill", "w8a8"):
        wd = W.get(DECODE, B=1, extra={"lengths": [1024]})
    lens = W.seq_lengths(wd)
    kc = torch.zeros((wd.B, wd.Hkv, wd.lmax, wd.d), dtype=torch.int8, device=dev)
    vc = torch.zeros_like(kc)
    ks = torch.zeros((wd.B, wd.Hkv, wd.lmax), dtype=torch.float32, device=dev)
    vs = torch.zeros_like(ks)
    for b in range(wd.B):
        L = int(lens[b])
        for name, c, s in (("k", kc, ks), ("v", vc, vs)):
            vals = torch.from_numpy(W.decode_cache_values(wd, b, name)).to(dev)
            cc, sc = sl8.quant_rowwise(vals)
            c[b, :, :L], s[b, :, :L] = cc, sc
    qdec = W.decode_query(wd).to(dev)
    seq = torch.from_numpy(lens.astype(np.int32)).to(dev)
    S = sl8.decode_num_splits(wd.B, wd.Hkv, wd.lmax, wd.d, 0)
    o_part = torch.empty((wd.B, wd.Hq, S, wd.d), dtype=torch.float32, device=dev)
    l_part = torch.empty((wd.B, wd.Hq, S), dtype=torch.float32, device=dev)
    dout = torch.empty((wd.B, wd.Hq, wd.d), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)
    torch.cuda.synchronize(dev)
    st, site = sl8.last_device_status(dev)
    if st != sl8.SL8_OK:
        raise RuntimeError(f"device status {st} at {site} after set-up")

    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        # L2 flush outside the timed events: write a buffer twice the size of L2, then
        # read it, so that the step starts with none of its inputs in L2 and no dirty
        # lines left behind by the flush itself
        flush.zero_()
        flush_sink.copy_(flush.view(torch.int64).sum())
        if ev:
            ev[0].record(stream)
        if args.only == "w8a8":
            sl8.attn_w8a8_fwd(qd, kd, vd, causal=True, smooth_k=True, q_group=W8A8_GROUP, k_group=W8A8_GROUP,
                              q_outlier_ratio=W8A8_RATIO, workspace=ws, out=out)
        elif args.only != "decode":
            sl8.attn_int8_fwd(qd, kd, vd, causal=True, smooth_k=True, workspace=ws, out=out)
        if ev:
            ev[1].record(stream)
        if args.only not in ("prefill", "w8a8"):
            sl8.attn_int8_decode(qdec, kc, ks, vc, vs, seq, o_partial=o_part, lse_partial=l_part, out=dout)
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sl8.trace_enable(False)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            step(events[i])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    st, site = sl8.last_device_status(dev)
    if st != sl8.SL8_OK:
        raise RuntimeError(f"device status {st} at {site} during the timed steps")
    # Per-kernel durations and launch counts come from the same steps run again with every
    # launch bracketed by CUDA events.  Those events break the overlap of the
    # programmatically dependent launches, so they stay out of the timed steps above.
    trace_steps = min(args.steps, 100)
    sl8.trace_collect()
    sl8.trace_enable(True)
    for _ in range(trace_steps):
        step()
    torch.cuda.synchronize(dev)
    sl8.trace_enable(False)
    trace = sl8.trace_collect()

    pre_ms = sum(e[0].elapsed_time(e[1]) for e in events) / args.steps
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in events) / args.steps
    pre_ms = max_over_ranks(pre_ms, world)
    dec_ms = max_over_ranks(dec_ms, world)
    ops = prefill_ops(wp)
    dbytes = decode_bytes(wd, lens)
    tops = ops * world / (pre_ms * 1e-3) / 1e12
    gbs = dbytes * world / (dec_ms * 1e-3) / 1e9

    def kern(name):
        n, ms = trace.get(name, (0, 0.0))
        return n, (ms / n if n else float("nan"))

    n_attn, attn_ms = kern("prefill_attn")
    n_split, split_ms = kern("decode_split")
    attn_tflops = ops / (attn_ms * 1e-3) / 1e12
    split_gbs = dbytes / (split_ms * 1e-3) / 1e9
    launches = sum(n for n, _ in trace.values()) * args.steps // trace_steps  # launches in the timed steps
    traffic = load_traffic()
    if args.only != "all":
        if rank == 0:
            print(json.dumps({"only": args.only, "prefill_ms": pre_ms, "decode_ms": dec_ms,
                              "kernels": {n: {"launches": c, "ms_per_launch": ms / c}
                                          for n, (c, ms) in sorted(trace.items())}}), flush=True)
        return

    # ---- the same decode over a paged k8v8 cache
    pg_ms, pg_split_ms, pg_steps, pg_pages = measure_paged(sl8, W, wd, kc, ks, vc, vs, lens, qdec, seq, stream, flush,
                                                           flush_sink, args.steps, args.warmup, world)
    pg_gbs = dbytes * world / (pg_ms * 1e-3) / 1e9
    pg_split_gbs = dbytes / (pg_split_ms * 1e-3) / 1e9
    # ---- speculative verify: VERIFY_T chained drafts per sequence
    vf_ms, vf_steps = measure_verify(sl8, wd, kc, ks, vc, vs, lens, seq, stream, flush, flush_sink, args.steps,
                                     args.warmup, world)
    # ---- the prefill's last positions as a query chunk
    ch_ms, ch_attn_ms, ch_steps = measure_chunk(sl8, wp, qd, kd, vd, stream, flush, flush_sink, args.steps,
                                                args.warmup, world)
    ch_ops = chunk_ops(wp, CHUNK_Q)
    ch_tflops = ch_ops / (ch_attn_ms * 1e-3) / 1e12
    # ---- the same prefill with grouped ("per-warp") scales and outlier-aware Q
    w8_ms, w8_quant_ms, w8_attn_ms, w8_steps = measure_w8a8(sl8, wp, qd, kd, vd, stream, flush, flush_sink,
                                                            args.steps, args.warmup, world)
    w8_tflops = ops / (w8_attn_ms * 1e-3) / 1e12
    # ---- the same decode with an fp16 V cache
    fv_ms, fv_split_ms, fv_steps = measure_f16v(sl8, W, wd, kc, ks, lens, qdec, seq, stream, flush, flush_sink,
                                                args.steps, args.warmup, world)
    fv_bytes = decode_bytes_f16v(wd, lens)
    fv_gbs = fv_bytes * world / (fv_ms * 1e-3) / 1e9
    fv_split_gbs = fv_bytes / (fv_split_ms * 1e-3) / 1e9

    # ---- e2e: public API with pinned host buffers, H2D inputs + D2H output every step
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    qdh = W.decode_query(wd).pin_memory()
    doh = torch.empty((wd.B, wd.Hq, wd.d), dtype=torch.bfloat16).pin_memory()
    q2, k2, v2 = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    qdec2 = torch.empty_like(qdec)

    def e2e_step():
        q2.copy_(qh, non_blocking=True)
        k2.copy_(kh, non_blocking=True)
        v2.copy_(vh, non_blocking=True)
        sl8.attn_int8_fwd(q2, k2, v2, causal=True, smooth_k=True, workspace=ws, out=out)
        oh.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize(dev)
    e_steps = max(3, args.steps // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, world)
    h2d = (q.numel() + k.numel() + v.numel()) * 2
    d2h = out.numel() * 2

    if rank != 0:
        return
    cpu = cpu_baseline_leg(wp, q.float().numpy(), k.float().numpy(), v.float().numpy())
    line = {
        "metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": pre_ms + dec_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "i8 codes on bf16 tensor cores (exact int32 QK^T), bf16 P.V, f32 softmax",
        "data": "synthetic",
        "config": {"workload": "prefill B1 Hq32 Hkv8 N4096 d128 bf16 causal smooth_k (Qwen3-8B shape) + "
                               "decode B64 Hq32 Hkv8 d128 int8 KV, L~U[1024,8192]",
                   "prefill_ms": pre_ms, "decode_ms": dec_ms, "prefill_gops": ops / 1e9,
                   "decode_bytes": dbytes, "decode_splits": S,
                   "l2": "flushed before every step (256 MB write, then a read of it, outside the timed events)"},
        "decode": {"value": gbs, "unit": "GB/s", "ms": dec_ms,
                   "roofline": {"bound": "hbm", "achieved": split_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": split_gbs / peaks["hbm_gbs"],
                                "traffic": traffic.get("decode_split"), "kernel": "decode_split",
                                "peak_source": peaks["source"]}},
        "paged_decode": {"value": pg_gbs, "unit": "GB/s", "ms": pg_ms, "steps": pg_steps,
                         "config": f"the decode workload over a paged k8v8 cache, {PAGE_SIZE}-token pages in a "
                                   f"seeded random order ({pg_pages} pages), L2 flushed before every step",
                         "roofline": {"bound": "hbm", "achieved": pg_split_gbs, "peak": peaks["hbm_gbs"],
                                      "unit": "GB/s", "frac": pg_split_gbs / peaks["hbm_gbs"], "traffic": None,
                                      "kernel": "decode_split (paged)", "peak_source": peaks["source"]}},
        "decode_verify": {"value": dbytes * world / (vf_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": vf_ms,
                          "steps": vf_steps, "draft_tokens": VERIFY_T,
                          "config": f"the decode workload with {VERIFY_T} chained draft queries per sequence "
                                    "(speculative verify), split kernel + combine; GB/s counts the cache once, "
                                    f"the kernel reads it once per draft query ({VERIFY_T} times)"},
        "prefill_w8a8": {"value": ops * world / (w8_ms * 1e-3) / 1e12, "unit": "TOPS", "ms": w8_ms,
                         "steps": w8_steps, "quant_qk_ms": w8_quant_ms,
                         "config": f"the prefill workload through attn_w8a8_fwd: Q and K scales per {W8A8_GROUP} "
                                   f"positions, Q rows above {W8A8_RATIO} x their group's median maximum keep "
                                   "their own, L2 flushed before every step",
                         "roofline": {"bound": "tensor", "achieved": w8_tflops, "peak": peaks["bf16_tflops"],
                                      "unit": "TFLOP/s", "frac": w8_tflops / peaks["bf16_tflops"], "traffic": None,
                                      "kernel": "prefill_attn (w8a8)", "peak_source": peaks["source"]}},
        "prefill_chunk": {"value": ch_ops * world / (ch_ms * 1e-3) / 1e12, "unit": "TOPS", "ms": ch_ms,
                          "steps": ch_steps, "ops": ch_ops,
                          "config": f"the prefill workload's last {CHUNK_Q} positions as a query chunk against "
                                    f"all {wp.N} keys (bottom-right causal), quantisation included, L2 flushed "
                                    "before every step",
                          "roofline": {"bound": "tensor", "achieved": ch_tflops, "peak": peaks["bf16_tflops"],
                                       "unit": "TFLOP/s", "frac": ch_tflops / peaks["bf16_tflops"], "traffic": None,
                                       "kernel": "prefill_attn (chunk)", "peak_source": peaks["source"]}},
        "decode_f16v": {"value": fv_gbs, "unit": "GB/s", "ms": fv_ms, "steps": fv_steps, "bytes": fv_bytes,
                        "config": "the decode workload with int8 K and an fp16 V cache (attn_decode's fp16-V "
                                  "variant), L2 flushed before every step",
                        "roofline": {"bound": "hbm", "achieved": fv_split_gbs, "peak": peaks["hbm_gbs"],
                                     "unit": "GB/s", "frac": fv_split_gbs / peaks["hbm_gbs"], "traffic": None,
                                     "kernel": "decode_split (fp16 V)", "peak_source": peaks["source"]}},
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": attn_tflops / peaks["bf16_tflops"], "traffic": traffic.get("prefill_attn"),
                     "kernel": "prefill_attn", "launch_ms": attn_ms,
                     "peak_source": peaks["source"] + " bf16 burst (QK^T and P.V both run on the bf16 pipe)"},
        "kernels": {n: {"launches": c, "ms_per_launch": ms / c} for n, (c, ms) in sorted(trace.items())},
        "cpu_baseline": cpu,
        "e2e": {"value": ops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TOPS", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "wall_s_timed": t_wall,
    }
    print(json.dumps(line), flush=True)


def timed_then_traced(sl8, step, device, steps, warmup):
    """Run step(ev) warm-up times, then time up to 100 steps with events around each step
    only; then a short pass with every launch traced, for the per-kernel durations.
    Returns (steps timed, ms per step, trace)."""
    import torch
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(device)
    n = max(3, min(steps, 100))
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        step(events[i])
    torch.cuda.synchronize(device)
    ms = sum(e[0].elapsed_time(e[1]) for e in events) / n
    sl8.trace_collect()
    sl8.trace_enable(True)
    for _ in range(min(n, 20)):
        step()
    torch.cuda.synchronize(device)
    sl8.trace_enable(False)
    return n, ms, sl8.trace_collect()


PAGE_SIZE = 64


def measure_paged(sl8, W, wd, kc, ks, vc, vs, lens, qdec, seq, stream, flush, flush_sink, steps, warmup, world):
    """The same decode workload over a paged k8v8 cache (16-token pages in a seeded random
    order): the step is the paged split kernel plus the combine, L2 flushed before each."""
    import torch
    table, num_pages = W.page_table(wd, lens, PAGE_SIZE, max_blocks=wd.lmax // PAGE_SIZE)
    kp, ksp = W.paginate(kc, ks, table, lens, PAGE_SIZE, num_pages)
    vp, vsp = W.paginate(vc, vs, table, lens, PAGE_SIZE, num_pages)
    tab = torch.from_numpy(table).to(kc.device)
    S = sl8.decode_num_splits(wd.B, wd.Hkv, wd.lmax, wd.d, 0)
    o_part = torch.empty((wd.B, wd.Hq, S, wd.d), dtype=torch.float32, device=kc.device)
    l_part = torch.empty((wd.B, wd.Hq, S), dtype=torch.float32, device=kc.device)
    dout = torch.empty((wd.B, wd.Hq, wd.d), dtype=torch.bfloat16, device=kc.device)

    def step(ev=None):
        flush.zero_()
        flush_sink.copy_(flush.view(torch.int64).sum())
        if ev:
            ev[0].record(stream)
        sl8.attn_int8_paged_decode(qdec, kp, ksp, vp, vsp, tab, seq, o_partial=o_part, lse_partial=l_part, out=dout)
        if ev:
            ev[1].record(stream)

    n, ms, trace = timed_then_traced(sl8, step, kc.device, steps, warmup)
    st, site = sl8.last_device_status(kc.device)
    if st != sl8.SL8_OK:
        raise RuntimeError(f"device status {st} at {site} during the paged decode")
    ms = max_over_ranks(ms, world)
    c, split_ms = trace.get("decode_split", (0, 0.0))
    return ms, (split_ms / c if c else float("nan")), n, num_pages


def measure_f16v(sl8, W, wd, kc, ks, lens, qdec, seq, stream, flush, flush_sink, steps, warmup, world):
    """The same decode workload with its V cache kept in fp16 (the V values cast to fp16;
    K stays the int8 cache): split kernel plus combine, L2 flushed before each step."""
    import torch
    v16 = torch.zeros((wd.B, wd.Hkv, wd.lmax, wd.d), dtype=torch.float16, device=kc.device)
    for b in range(wd.B):
        L = int(lens[b])
        v16[b, :, :L] = torch.from_numpy(W.decode_cache_values(wd, b, "v")).to(kc.device).to(torch.float16)
    S = sl8.decode_num_splits(wd.B, wd.Hkv, wd.lmax, wd.d, 0)
    o_part = torch.empty((wd.B, wd.Hq, S, wd.d), dtype=torch.float32, device=kc.device)
    l_part = torch.empty((wd.B, wd.Hq, S), dtype=torch.float32, device=kc.device)
    dout = torch.empty((wd.B, wd.Hq, wd.d), dtype=torch.bfloat16, device=kc.device)

    def step(ev=None):
        flush.zero_()
        flush_sink.copy_(flush.view(torch.int64).sum())
        if ev:
            ev[0].record(stream)
        sl8.attn_int8_decode_f16v(qdec, kc, ks, v16, seq, o_partial=o_part, lse_partial=l_part, out=dout)
        if ev:
            ev[1].record(stream)

    n, ms, trace = timed_then_traced(sl8, step, kc.device, steps, warmup)
    st, site = sl8.last_device_status(kc.device)
    if st != sl8.SL8_OK:
        raise RuntimeError(f"device status {st} at {site} during the fp16-V decode")
    ms = max_over_ranks(ms, world)
    c, split_ms = trace.get("decode_split", (0, 0.0))
    del v16
    return ms, (split_ms / c if c else float("nan")), n


def measure_chunk(sl8, wp, qd, kd, vd, stream, flush, flush_sink, steps, warmup, world):
    """The prefill workload's last CHUNK_Q positions as a query chunk against all N keys
    (chunked prefill, bottom-right causal): quantisation and attention, L2 flushed before
    each step."""
    import torch
    qc = qd[:, :, wp.N - CHUNK_Q:].contiguous()
    ws = torch.empty(sl8.prefill_workspace_bytes(wp.B, wp.Hq, wp.Hkv, wp.N, wp.d), dtype=torch.uint8, device=qd.device)
    out = torch.empty_like(qc)

    def step(ev=None):
        flush.zero_()
        flush_sink.copy_(flush.view(torch.int64).sum())
        if ev:
            ev[0].record(stream)
        sl8.attn_int8_fwd_chunk(qc, kd, vd, causal=True, smooth_k=True, workspace=ws, out=out)
        if ev:
            ev[1].record(stream)

    n, ms, trace = timed_then_traced(sl8, step, qd.device, steps, warmup)
    st, site = sl8.last_device_status(qd.device)
    if st != sl8.SL8_OK:
        raise RuntimeError(f"device status {st} at {site} during the chunked prefill")
    ms = max_over_ranks(ms, world)
    c, attn_ms = trace.get("prefill_attn", (0, 0.0))
    return ms, (attn_ms / c if c else float("nan")), n


def measure_w8a8(sl8, wp, qd, kd, vd, stream, flush, flush_sink, steps, warmup, world):
    """The prefill workload through attn_w8a8_fwd (grouped scales, outlier-aware Q): the
    whole step, and the quantiser and attention kernels from the traced pass."""
    import torch
    ws = torch.empty(sl8.prefill_workspace_bytes(wp.B, wp.Hq, wp.Hkv, wp.N, wp.d), dtype=torch.uint8, device=qd.device)
    out = torch.empty_like(qd)

    def step(ev=None):
        flush.zero_()
        flush_sink.copy_(flush.view(torch.int64).sum())
        if ev:
            ev[0].record(stream)
        sl8.attn_w8a8_fwd(qd, kd, vd, causal=True, smooth_k=True, q_group=W8A8_GROUP, k_group=W8A8_GROUP,
                          q_outlier_ratio=W8A8_RATIO, workspace=ws, out=out)
        if ev:
            ev[1].record(stream)

    n, ms, trace = timed_then_traced(sl8, step, qd.device, steps, warmup)
    st, site = sl8.last_device_status(qd.device)
    if st != sl8.SL8_OK:
        raise RuntimeError(f"device status {st} at {site} during the w8a8 prefill")
    ms = max_over_ranks(ms, world)
    per = {}
    for name in ("quant_qk", "prefill_attn"):
        c, t = trace.get(name, (0, 0.0))
        per[name] = t / c if c else float("nan")
    return ms, per["quant_qk"], per["prefill_attn"], n


W8A8_GROUP = 32     # positions per shared scale in the w8a8 line (the rows of one softmax warp)
W8A8_RATIO = 4.0    # its Q outlier ratio

VERIFY_T = 4   # draft tokens per sequence of the verify line


def measure_verify(sl8, wd, kc, ks, vc, vs, lens, seq, stream, flush, flush_sink, steps, warmup, world):
    """Speculative verify on the decode workload: VERIFY_T chained draft queries per
    sequence (the cache's last VERIFY_T tokens are the drafts), split kernel plus combine,
    L2 flushed before each step."""
    import torch
    T = VERIFY_T
    g = torch.Generator(device="cpu").manual_seed(0x5EED0000 + 7)
    q = torch.randn((wd.B, T, wd.Hq, wd.d), generator=g).to(torch.bfloat16).to(kc.device)
    mask = torch.tensor([[(1 << (t + 1)) - 1 for t in range(T)]] * wd.B, dtype=torch.int32, device=kc.device)
    S = int(sl8.lib().sl8_attn_decode_verify_num_splits(wd.B, T, wd.Hq, wd.Hkv, wd.lmax, wd.d, 0))
    o_part = torch.empty((wd.B * T, wd.Hq, S, wd.d), dtype=torch.float32, device=kc.device)
    l_part = torch.empty((wd.B * T, wd.Hq, S), dtype=torch.float32, device=kc.device)
    out = torch.empty((wd.B, T, wd.Hq, wd.d), dtype=torch.bfloat16, device=kc.device)

    def step(ev=None):
        flush.zero_()
        flush_sink.copy_(flush.view(torch.int64).sum())
        if ev:
            ev[0].record(stream)
        sl8.attn_int8_decode_verify(q, kc, ks, vc, vs, seq, mask, o_partial=o_part, lse_partial=l_part, out=out)
        if ev:
            ev[1].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(kc.device)
    n = max(3, min(steps, 50))
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        step(events[i])
    torch.cuda.synchronize(kc.device)
    st, site = sl8.last_device_status(kc.device)
    if st != sl8.SL8_OK:
        raise RuntimeError(f"device status {st} at {site} during the verify")
    return max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in events) / n, world), n


def load_traffic():
    """DRAM bytes per launch (read + write) from the committed ncu summary, per kernel,
    only while the kernel's source file still has the hash the capture was taken on."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    out = {}
    if not os.path.exists(path):
        return out
    with open(path) as f:
        table = json.load(f)
    for name, ent in table.items():
        if not isinstance(ent, dict):
            continue
        src = os.path.join(ROOT, ent["source"])
        if os.path.exists(src) and hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] == ent["source_sha"]:
            out[name] = ent["bytes"]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--only", default="all", choices=["all", "prefill", "decode", "w8a8"],
                    help="time one half of the step only (profiling runs; w8a8: the prefill through "
                         "attn_w8a8_fwd); no e2e or CPU leg")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            if args.steps > 20:
                args.steps = 3  # each step is seconds of CPU work; keep the run within minutes
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
