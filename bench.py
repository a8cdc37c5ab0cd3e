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
`prefill_chunk` / `prefill_chunk_small` the prefill's last 1024 / 128 positions as a
query chunk (chunked prefill, bottom-right causal), `prefill_chunk_cache` the 1024-query
chunk onto an int8 cache of all positions, `prefill_w8a8` the prefill through
attn_w8a8_fwd (scales per 32 positions, outlier-aware Q), and `decode_verify` the
decode with 4 chained draft queries per sequence (speculative verify).  Inputs are
resident in HBM when the timed region starts (the timed steps carry no per-launch
instrumentation: per-kernel times come from a separate traced pass).  L2 is flushed
before the prefill and again before the decode of every step, outside the timed events
(a 256 MB write, then a read of that buffer, so no dirty lines of the flush or of the
prefill's outputs remain).  `e2e` repeats the prefill through the public API with
pinned host inputs copied in and the output copied back every step.

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
CHUNK_Q_SMALL = 128  # a short chunk (16 items for the SMs): the line on which keys are split across CTAs


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
    """SM clock and throttle-reason samples while the bench runs.

    Reads NVML directly (libnvidia-ml, read-only queries) every ``period`` seconds from a
    thread, so that even a timed region of a few milliseconds holds samples; falls back
    to ``nvidia-smi -lms 100`` where NVML cannot be loaded.  ``mark()`` brackets the timed
    region; ``summary()`` reports the samples inside it and, separately, every sample
    taken while the bench ran (the GPU under load)."""

    # NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period: float = 0.002):
        self.index = device_index
        self.period = period
        self.samples = []        # (t, sm_mhz, max_mhz, reasons set)
        self.window = None
        self.source = None
        self._stop = threading.Event()
        self._proc = None
        self._thread = None

    # ---- NVML
    def _nvml_handle(self):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.index)
        bus = getattr(props, "pci_bus_id", None)
        ok = False
        if bus is not None:
            dom, dev = getattr(props, "pci_domain_id", 0), getattr(props, "pci_device_id", 0)
            for fmt in ("%08X:%02X:%02X.0", "%04X:%02X:%02X.0"):
                if lib.nvmlDeviceGetHandleByPciBusId_v2((fmt % (dom, bus, dev)).encode(), ctypes.byref(h)) == 0:
                    ok = True
                    break
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons_fn

    def _nvml_loop(self, lib, h, reasons_fn):
        import ctypes
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.perf_counter()
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:        # NVML_CLOCK_SM
                lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
                reasons_fn(h, ctypes.byref(rs))
                names = {n for bit, n in self.REASONS.items() if rs.value & bit}
                self.samples.append((t, float(clk.value), float(mx.value), names))
            self._stop.wait(self.period)

    # ---- nvidia-smi fallback
    def _smi_loop(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            rs = {n for n, val in zip(names, parts[4:8]) if val.lower().startswith("active")}
            self.samples.append((time.perf_counter(), sm, mx, rs))

    def __enter__(self):
        try:
            lib, h, fn = self._nvml_handle()
            self._thread = threading.Thread(target=self._nvml_loop, args=(lib, h, fn), daemon=True)
            self.source = f"NVML every {self.period * 1e3:.0f} ms"
        except (OSError, AttributeError):
            try:
                self._proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                               "--format=csv,noheader,nounits", "-lms", "100"],
                                              stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self._thread = threading.Thread(target=self._smi_loop, daemon=True)
                self.source = "nvidia-smi -lms 100"
            except OSError:
                self._thread = None
        if self._thread:
            self._thread.start()
        return self

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread:
            self._thread.join(timeout=5)

    @staticmethod
    def _stats(samples):
        if not samples:
            return None, None, [], 0
        sm = [x[1] for x in samples]
        return (statistics.median(sm), max(x[2] for x in samples), sorted(set().union(*(x[3] for x in samples))),
                len(samples))

    def summary(self):
        timed = [x for x in self.samples if self.window and self.window[0] <= x[0] <= self.window[1]]
        sm, mx, reasons, n = self._stats(timed)
        asm, amx, areasons, an = self._stats(self.samples)
        return {"sm_mhz": sm, "sm_max_mhz": mx, "reasons": reasons, "samples": n,
                "run": {"sm_mhz": asm, "sm_max_mhz": amx, "reasons": areasons, "samples": an},
                "source": self.source,
                "note": "sm_mhz, reasons and samples: inside the timed steps; run: every sample while the bench ran"}


def dist_setup(args, backend=None):
    """Process group of a torchrun launch (none for one rank).  The backend is nccl when a
    GPU is visible, else gloo; ``backend`` or the SL8_DIST_BACKEND variable overrides it
    (the CPU test of this host logic forces gloo so it never touches a GPU)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = backend or os.environ.get("SL8_DIST_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def _reduce_device():
    import torch.distributed as dist
    return "cuda" if dist.get_backend() == "nccl" else "cpu"


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=_reduce_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ reference arm: the CPU oracle

WORKLOAD_DESC = ("prefill B1 Hq32 Hkv8 N4096 d128 bf16 causal smooth_k (Qwen3-8B shape) + "
                 "decode B64 Hq32 Hkv8 d128 int8 KV, L~U[1024,8192]")


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on the same workload as our arm.
    A step is the whole prefill (every query row of every head) plus the whole decode
    (every sequence and head over the int8 cache), run on the host cores."""
    if rank != 0:
        return
    import oracle
    import workloads as W
    w = W.get(PREFILL)
    q, k, v = W.prefill_dense(w)
    qn, kn, vn = q.float().numpy(), k.float().numpy(), v.float().numpy()
    rows = [(0, h, i) for h in range(w.Hq) for i in range(w.N)]
    ops = prefill_ops(w)
    # the decode cache, quantised by the oracle's own quantiser (set-up, not timed)
    wd = W.get(DECODE)
    lens = W.seq_lengths(wd)
    caches = {}
    for name in ("k", "v"):
        c = np.zeros((wd.B, wd.Hkv, wd.lmax, wd.d), np.int8)
        sc = np.zeros((wd.B, wd.Hkv, wd.lmax), np.float32)
        for b in range(wd.B):
            L = int(lens[b])
            c[b, :, :L], sc[b, :, :L] = oracle.quant_rowwise(W.decode_cache_values(wd, b, name))
        caches[name] = (c, sc)
    qdec = W.decode_query(wd).float().numpy()
    dbytes = decode_bytes(wd, lens)
    pre, dec = [], []
    for it in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.attn_prefill(qn, kn, vn, causal=True, smooth_k=True, rows=rows)
        t1 = time.perf_counter()
        oracle.attn_decode(qdec, caches["k"][0], caches["k"][1], caches["v"][0], caches["v"][1], lens)
        t2 = time.perf_counter()
        if it >= args.warmup:
            pre.append(t1 - t0)
            dec.append(t2 - t1)
    pre_s, dec_s = float(np.mean(pre)), float(np.mean(dec))
    tops = ops / pre_s / 1e12
    sample = (f"the whole workload every step: all {w.Hq} heads x {w.N} query rows of the prefill "
              f"({ops / 1e9:.1f} GOP) and all {wd.B} x {wd.Hq} decode rows")
    line = {"impl": "reference", "metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": (pre_s + dec_s) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC, "prefill_ms": pre_s * 1e3, "decode_ms": dec_s * 1e3},
            "decode": {"value": dbytes / dec_s / 1e9, "unit": "GB/s", "ms": dec_s * 1e3},
            "tokens_per_s": {"prefill": w.B * w.N / pre_s, "decode": wd.B / dec_s},
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
    if args.only in OTHER_PREFILL:
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        flush_sink = torch.empty((), dtype=torch.int64, device=dev)
        res = measure_prefill_config(sl8, W, args.only, dev, torch.cuda.current_stream(dev), flush, flush_sink,
                                     args.steps, args.warmup, world, peaks, rank=1)  # no CPU leg
        if rank == 0:
            print(json.dumps({"only": args.only, **res}), flush=True)
        return

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
    if args.only == "paged":
        pg_ms, pg_split_ms, pg_steps, pg_pages = measure_paged(sl8, W, wd, kc, ks, vc, vs, lens, qdec, seq, stream,
                                                               flush, flush_sink, args.steps, args.warmup, world)
        dbytes = decode_bytes(wd, lens)
        if rank == 0:
            print(json.dumps({"only": "paged", "ms": pg_ms, "split_ms": pg_split_ms, "pages": pg_pages,
                              "split_gbs": dbytes / (pg_split_ms * 1e-3) / 1e9,
                              "frac": dbytes / (pg_split_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}), flush=True)
        return

    def l2_flush():
        # outside the timed events: write a buffer twice the size of L2, then read it, so
        # that what follows starts with none of its inputs in L2 and no dirty lines (the
        # flush's own, or those the prefill's outputs left) to write back
        flush.zero_()
        flush_sink.copy_(flush.view(torch.int64).sum())

    def step(ev=None):
        l2_flush()
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
            l2_flush()
            if ev:
                ev[2].record(stream)
            sl8.attn_int8_decode(qdec, kc, ks, vc, vs, seq, o_partial=o_part, lse_partial=l_part, out=dout)
        elif ev:
            ev[2].record(stream)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sl8.trace_enable(False)
    barrier(world)
    torch.cuda.synchronize(dev)
    clk = ClockSampler(local).__enter__()
    time.sleep(0.01)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(events[i])
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    clk.mark(t0, t1)
    t_wall = t1 - t0
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
    dec_ms = sum(e[2].elapsed_time(e[3]) for e in events) / args.steps
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
        clk.__exit__(None, None, None)
        if rank == 0:
            print(json.dumps({"only": args.only, "prefill_ms": pre_ms, "decode_ms": dec_ms,
                              "kernels": {n: {"launches": c, "ms_per_launch": ms / c}
                                          for n, (c, ms) in sorted(trace.items())},
                              "clocks": clk.summary()}), flush=True)
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
    ch_ms, ch_attn_ms, ch_steps, ch_kernels = measure_chunk(sl8, wp, qd, kd, vd, stream, flush, flush_sink,
                                                            args.steps, args.warmup, world)
    ch_ops = chunk_ops(wp, CHUNK_Q)
    ch_tflops = ch_ops / (ch_attn_ms * 1e-3) / 1e12
    cs_ms, cs_attn_ms, cs_steps, cs_kernels = measure_chunk(sl8, wp, qd, kd, vd, stream, flush, flush_sink,
                                                            args.steps, args.warmup, world, nq=CHUNK_Q_SMALL)
    cs_ops = chunk_ops(wp, CHUNK_Q_SMALL)
    cs_tflops = cs_ops / (cs_attn_ms * 1e-3) / 1e12
    cc_ms, cc_attn_ms, cc_steps, cc_kernels = measure_chunk_cache(sl8, wp, qd, kd, vd, stream, flush, flush_sink,
                                                                  args.steps, args.warmup, world)
    cc_tflops = ch_ops / (cc_attn_ms * 1e-3) / 1e12
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

    # ---- the other prefill workloads: tiny latency case, Gemma3 shape at d = 256, ragged varlen
    others = {name: measure_prefill_config(sl8, W, name, dev, stream, flush, flush_sink, args.steps, args.warmup,
                                           world, peaks, rank)
              for name in OTHER_PREFILL}

    # ---- e2e: public API with pinned host buffers, H2D inputs + D2H output every step
    e2e_ms, h2d, d2h, e_steps = measure_e2e(sl8, q, k, v, ws, dev, stream, args.steps, args.warmup, world)

    clk.__exit__(None, None, None)
    if rank != 0:
        return
    cpu = cpu_baseline_leg(wp, q.float().numpy(), k.float().numpy(), v.float().numpy())
    line = {
        "metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": pre_ms + dec_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "i8 codes on bf16 tensor cores (exact int32 QK^T), bf16 P.V, f32 softmax",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC,
                   "prefill_ms": pre_ms, "decode_ms": dec_ms, "prefill_gops": ops / 1e9,
                   "decode_bytes": dbytes, "decode_splits": S,
                   "l2": "flushed before the prefill and again before the decode of every step (256 MB write, then a "
                         "read of it, outside the timed events)"},
        "tokens_per_s": {"prefill": wp.B * wp.N * world / (pre_ms * 1e-3),
                         "decode": wd.B * world / (dec_ms * 1e-3),
                         "note": "prefill: query tokens per second; decode: sequences advanced by one token per "
                                 "second (one query token each)"},
        "decode": {"value": gbs, "unit": "GB/s", "ms": dec_ms, "tokens_per_s": wd.B * world / (dec_ms * 1e-3),
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
                          "steps": ch_steps, "ops": ch_ops, "kernels_ms": ch_kernels,
                          "config": f"the prefill workload's last {CHUNK_Q} positions as a query chunk against "
                                    f"all {wp.N} keys (bottom-right causal), quantisation included, L2 flushed "
                                    "before every step",
                          "roofline": {"bound": "tensor", "achieved": ch_tflops, "peak": peaks["bf16_tflops"],
                                       "unit": "TFLOP/s", "frac": ch_tflops / peaks["bf16_tflops"], "traffic": None,
                                       "kernel": "prefill_attn (chunk)", "peak_source": peaks["source"]}},
        "prefill_chunk_cache": {"value": ch_ops * world / (cc_ms * 1e-3) / 1e12, "unit": "TOPS", "ms": cc_ms,
                                "steps": cc_steps, "ops": ch_ops, "kernels_ms": cc_kernels,
                                "config": f"the same {CHUNK_Q}-query chunk onto an int8 cache of all {wp.N} "
                                          "positions (the prefill's K and V quantised per token beforehand, "
                                          "outside the timed region): cache codes to the attention layout, Q "
                                          "quantisation and attention, L2 flushed before every step",
                                "roofline": {"bound": "tensor", "achieved": cc_tflops, "peak": peaks["bf16_tflops"],
                                             "unit": "TFLOP/s", "frac": cc_tflops / peaks["bf16_tflops"],
                                             "traffic": None, "kernel": "prefill_attn (chunk onto cache)",
                                             "peak_source": peaks["source"]}},
        "prefill_chunk_small": {"value": cs_ops * world / (cs_ms * 1e-3) / 1e12, "unit": "TOPS", "ms": cs_ms,
                                "steps": cs_steps, "ops": cs_ops, "kernels_ms": cs_kernels,
                                "config": f"the prefill workload's last {CHUNK_Q_SMALL} positions as a query chunk "
                                          f"against all {wp.N} keys: keys split across CTAs and merged "
                                          "(prefill_combine), quantisation of all keys included, L2 flushed "
                                          "before every step",
                                "roofline": {"bound": "tensor", "achieved": cs_tflops, "peak": peaks["bf16_tflops"],
                                             "unit": "TFLOP/s", "frac": cs_tflops / peaks["bf16_tflops"],
                                             "traffic": None, "kernel": "prefill_attn (split chunk)",
                                             "peak_source": peaks["source"]}},
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
        "prefill_configs": others,
        "kernels": {n: {"launches": c, "ms_per_launch": ms / c} for n, (c, ms) in sorted(trace.items())},
        "cpu_baseline": cpu,
        "e2e": {"value": ops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TOPS", "ms_per_step": e2e_ms,
                "steps": e_steps,
                "how": "sl8.attn_int8_fwd on device copies of pinned host q/k/v, output read back to pinned "
                       "host memory, every step; double-buffered: step i+1's H2D (own stream) and step i-1's D2H "
                       "(own stream) overlap step i's kernels; timed from the first H2D to the last D2H",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "wall_s_timed": t_wall,
    }
    print(json.dumps(line), flush=True)


OTHER_PREFILL = ("tiny", "gemma3_d256", "varlen")
OTHER_SAMPLE_STRIDE = {"tiny": 1, "gemma3_d256": 16, "varlen": 16}   # CPU baseline: every k-th query row


def _causal_ops(lens, Hq, d) -> float:
    return 2.0 * 2.0 * d * Hq * float(sum(int(L) * (int(L) + 1) // 2 for L in lens))


def measure_prefill_config(sl8, W, name, dev, stream, flush, flush_sink, steps, warmup, world, peaks, rank):
    """One more prefill workload (attn_int8_fwd, causal, K-smoothing): the step time with
    L2 flushed before each step, the attention kernel's roofline from the traced pass,
    tokens/s, and the oracle on a bounded sample of the same inputs (rank 0)."""
    import torch
    w = W.get(name)
    if w.kind == "varlen":
        q, k, v, cu = W.prefill_varlen(w)
        lens = [int(x) for x in np.diff(cu.numpy())]
        N = max(lens)
        cud = cu.to(dev)
        desc = (f"varlen causal prefill, {w.B} sequences, lengths U[{w.len_lo},{w.len_hi}] (seeded T = {sum(lens)}), "
                f"Hq{w.Hq} Hkv{w.Hkv} d{w.d} {w.dtype}, smooth_k")
    else:
        q, k, v = W.prefill_dense(w)
        lens = [w.N] * w.B
        N, cu, cud = w.N, None, None
        desc = f"causal prefill B{w.B} Hq{w.Hq} Hkv{w.Hkv} N{w.N} d{w.d} {w.dtype}, smooth_k={w.smooth_k}"
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ws = torch.empty(sl8.prefill_workspace_bytes(len(lens), w.Hq, w.Hkv, N, w.d, sum(lens) if cu is not None else 0),
                     dtype=torch.uint8, device=dev)
    out = torch.empty_like(qd)

    def step(ev=None):
        flush.zero_()
        flush_sink.copy_(flush.view(torch.int64).sum())
        if ev:
            ev[0].record(stream)
        sl8.attn_int8_fwd(qd, kd, vd, causal=True, smooth_k=w.smooth_k, cu_seqlens=cud,
                          max_seqlen=N if cud is not None else None, workspace=ws, out=out)
        if ev:
            ev[1].record(stream)

    n, ms, trace = timed_then_traced(sl8, step, dev, steps, warmup)
    st, site = sl8.last_device_status(dev)
    if st != sl8.SL8_OK:
        raise RuntimeError(f"device status {st} at {site} during the {name} prefill")
    ms = max_over_ranks(ms, world)
    ops = _causal_ops(lens, w.Hq, w.d)
    c, attn_ms = trace.get("prefill_attn", (0, 0.0))
    attn_ms = attn_ms / c if c else float("nan")
    tflops = ops / (attn_ms * 1e-3) / 1e12
    res = {"workload": desc, "value": ops * world / (ms * 1e-3) / 1e12, "unit": "TOPS", "ms": ms, "steps": n,
           "ops": ops, "tokens_per_s": sum(lens) * world / (ms * 1e-3),
           "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": tflops / peaks["bf16_tflops"], "traffic": load_traffic().get(f"prefill_attn:{name}"),
                        "kernel": "prefill_attn", "launch_ms": attn_ms,
                        "peak_source": peaks["source"] + " bf16 burst"},
           "kernels": {nm: {"launches": cc, "ms_per_launch": t / cc} for nm, (cc, t) in sorted(trace.items())},
           "l2": "flushed before every step"}
    del qd, kd, vd, ws, out
    if rank == 0:
        res["cpu_baseline"] = cpu_sample_leg(w, q, k, v, cu, lens, OTHER_SAMPLE_STRIDE[name])
    return res


def cpu_sample_leg(w, q, k, v, cu, lens, stride):
    """The oracle as it stands on every stride-th query row of every head (all of them at
    stride 1); the rate counts the causal (query, key) pairs of the rows it ran."""
    import oracle
    rows = [(s, h, i) for s, L in enumerate(lens) for h in range(w.Hq) for i in range(0, L, stride)]
    ops = 2.0 * 2.0 * w.d * float(sum(i + 1 for (_, _, i) in rows))
    qn, kn, vn = q.float().numpy(), k.float().numpy(), v.float().numpy()
    t0 = time.perf_counter()
    oracle.attn_prefill(qn, kn, vn, causal=True, smooth_k=w.smooth_k, rows=rows,
                        cu_seqlens=None if cu is None else cu.numpy())
    sec = time.perf_counter() - t0
    return {"value": ops / sec / 1e12, "unit": "TOPS", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"every {stride}. query row of all {w.Hq} heads ({len(rows)} rows, {ops / 1e9:.2f} GOP, "
                      f"quantisation of the whole input included), {sec:.2f} s"}


def measure_e2e(sl8, q, k, v, ws, dev, stream, steps, warmup, world):
    """The prefill end to end through the public API: every step copies its q, k, v from
    pinned host memory and reads its output back into pinned host memory.  The steps run
    as a pipeline over two device buffer sets: H2D on one stream, the library call on the
    compute stream, D2H on a third, ordered by events (step i+1's inputs land while step
    i computes and step i-1's output drains).  Returns (ms per step, H2D bytes per step,
    D2H bytes per step, steps timed)."""
    import torch
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    bufs = [tuple(torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (q, k, v)) for _ in range(2)]
    outs = [torch.empty(q.shape, dtype=q.dtype, device=dev) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
        ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
        h2d_done = [ev() for _ in range(n)]
        comp_done = [ev() for _ in range(n)]
        d2h_done = [ev() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(up)
        for i in range(n):
            qb, kb, vb = bufs[i % 2]
            if i >= 2:
                up.wait_event(comp_done[i - 2])      # step i-2 has finished reading this buffer set
            with torch.cuda.stream(up):
                qb.copy_(qh, non_blocking=True)
                kb.copy_(kh, non_blocking=True)
                vb.copy_(vh, non_blocking=True)
                h2d_done[i].record(up)
            stream.wait_event(h2d_done[i])
            if i >= 2:
                stream.wait_event(d2h_done[i - 2])   # step i-2's output has left this buffer
            sl8.attn_int8_fwd(qb, kb, vb, causal=True, smooth_k=True, workspace=ws, out=outs[i % 2])
            comp_done[i].record(stream)
            down.wait_event(comp_done[i])
            with torch.cuda.stream(down):
                oh.copy_(outs[i % 2], non_blocking=True)
                d2h_done[i].record(down)
        down.wait_event(d2h_done[n - 1])
        t1.record(down)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1) / n

    run(max(warmup, 3))
    n = max(8, steps)
    ms = max_over_ranks(run(n), world)
    return ms, (q.numel() + k.numel() + v.numel()) * q.element_size(), q.numel() * q.element_size(), n


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
    """The same decode workload over a paged k8v8 cache (PAGE_SIZE-token pages in a seeded random
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


def measure_chunk(sl8, wp, qd, kd, vd, stream, flush, flush_sink, steps, warmup, world, nq=CHUNK_Q):
    """The prefill workload's last nq positions as a query chunk against all N keys
    (chunked prefill, bottom-right causal): quantisation and attention, L2 flushed before
    each step."""
    import torch
    qc = qd[:, :, wp.N - nq:].contiguous()
    # the chunk workspace: room for the key-split partials the library uses on a small chunk
    ws = torch.empty(int(sl8.lib().sl8_attn_int8_fwd_chunk_workspace_size(wp.B, wp.Hq, wp.Hkv, nq, wp.N, wp.d)),
                     dtype=torch.uint8, device=qd.device)
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
    return ms, (attn_ms / c if c else float("nan")), n, {nm: t / cc for nm, (cc, t) in trace.items() if cc}


def measure_chunk_cache(sl8, wp, qd, kd, vd, stream, flush, flush_sink, steps, warmup, world, nq=CHUNK_Q):
    """The same query chunk onto an int8 cache holding all N positions: the prefill's K and
    V quantised per token once, before timing; each step converts the cache codes, quantises
    the chunk's queries and runs the attention, L2 flushed before each step."""
    import torch
    qc = qd[:, :, wp.N - nq:].contiguous()
    kc, ks = sl8.quant_rowwise(kd)
    vc, vs = sl8.quant_rowwise(vd)
    ws = torch.empty(int(sl8.lib().sl8_attn_int8_fwd_chunk_workspace_size(wp.B, wp.Hq, wp.Hkv, nq, wp.N, wp.d)),
                     dtype=torch.uint8, device=qd.device)
    out = torch.empty_like(qc)

    def step(ev=None):
        flush.zero_()
        flush_sink.copy_(flush.view(torch.int64).sum())
        if ev:
            ev[0].record(stream)
        sl8.attn_int8_fwd_chunk_cache(qc, kc, ks, vc, vs, Nk=wp.N, causal=True, workspace=ws, out=out)
        if ev:
            ev[1].record(stream)

    n, ms, trace = timed_then_traced(sl8, step, qd.device, steps, warmup)
    st, site = sl8.last_device_status(qd.device)
    if st != sl8.SL8_OK:
        raise RuntimeError(f"device status {st} at {site} during the chunk onto the int8 cache")
    ms = max_over_ranks(ms, world)
    c, attn_ms = trace.get("prefill_attn", (0, 0.0))
    return ms, (attn_ms / c if c else float("nan")), n, {nm: t / cc for nm, (cc, t) in trace.items() if cc}


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
    ap.add_argument("--only", default="all", choices=["all", "prefill", "decode", "paged", "w8a8", *OTHER_PREFILL],
                    help="time one part only (profiling runs): the prefill or decode half of the step, the "
                         "decode over the paged cache, the prefill through attn_w8a8_fwd, or one of the other "
                         "prefill workloads; no e2e or CPU leg")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            # each step is seconds of CPU work (the whole prefill and decode on the host cores):
            # at most 5 timed steps after one warm-up keep the run within a couple of minutes
            args.steps = max(1, min(args.steps, 5))
            args.warmup = 1
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
