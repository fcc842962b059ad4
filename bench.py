#!/usr/bin/env python3
"""Benchmark of the CSA2 hot path on one B300 (one JSON line on stdout).

Headline workload: hierarchical long-context decode, batch 1, context 1,048,576: a Full layer
scans every index key and builds the 2,048-block candidate pool, three Reindex layers rescore the
pool with their own FP8 indexer queries (Top-K 2048), two Reuse layers reuse the last indices;
all six layers run FP4 sparse attention with 64 heads.  One step = the whole layer sequence plus
the quantisation of the new token's KV row.  Metric: decode tokens/s, with the step's
algorithmic HBM bytes/s against 8 TB/s, and (`prefill`) chunked-prefill TFLOP/s on 4,096 new
tokens after a 262,144-token cached prefix.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-prefill]

--impl reference times the CPU oracle (single-threaded C, the definition of the path) on the same
workload and metric.  Multi-GPU: replicas only (every rank runs the full workload on its own GPU;
`value` sums the ranks); this path has no exchange step.
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

HEADLINE = "hier_decode_l1m"
HEADLINE_SWA = "hier_decode_l1m_swa128"
PREFILL = "prefill_t4096_p262144"
PREFILL_HIER = "prefill_hier_t4096_p262144"
METRIC = "sparse-attn decode tokens/s + HBM GB/s vs 8 TB/s at 1M ctx; prefill TFLOP/s"
HBM_TARGET_GBS = 8000.0
DECODE_CONFIGS = ("decode_b1_l4096_bf16idx", "decode_b8_l65536", "decode_ragged_b32")
# DRAM bytes (read + write) of one launch of the Full scan as csa2_index_block_max runs it, from
# one ncu capture (profiles/index_mma_scan_hier_decode_l1m.md); None when the kernel has changed
# since.
SCAN_TRAFFIC = 137_131_008
ROOT = os.path.dirname(os.path.abspath(__file__))


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class ClockSampler:
    """SM clock and throttle-reason samples with host timestamps, so the samples that fall
    inside the timed window can be picked out afterwards.  NVML is polled every ~0.5 ms (the
    timed window of a decode run lasts a few milliseconds); without NVML, nvidia-smi every 50 ms.
    Both only read the GPU's state."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    NVML_BITS = [("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40),
                 ("sw_thermal_slowdown", 0x20), ("sw_power_cap", 0x4)]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.nvml = None
        self.period = "50 ms"
        self.samples = []  # (host time, sm_mhz, sm_max_mhz, active reasons)
        self.running = False

    def _nvml_index(self):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if ids and all(x.isdigit() for x in ids) and self.index < len(ids):
            return int(ids[self.index])
        return self.index

    @staticmethod
    def _nvml_open(index):
        """Read-only NVML queries through the driver's library: (sm clock, max sm clock,
        active clock-event reason bits) as functions of nothing."""
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
            raise OSError("nvmlDeviceGetHandleByIndex")
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons

        def clock(fn):
            v = ctypes.c_uint()
            if fn(h, ctypes.c_int(1), ctypes.byref(v)) != 0:  # NVML_CLOCK_SM
                raise OSError("clock query")
            return float(v.value)

        def bits():
            v = ctypes.c_ulonglong()
            if reasons(h, ctypes.byref(v)) != 0:
                raise OSError("reason query")
            return int(v.value)
        return (lambda: clock(lib.nvmlDeviceGetClockInfo)), clock(lib.nvmlDeviceGetMaxClockInfo), bits

    def start(self):
        try:
            self.nvml = self._nvml_open(self._nvml_index())
            self.nvml[0]()
            self.nvml[2]()
            self.period = "0.5 ms"
            self.running = True
            self.t = threading.Thread(target=self._poll_nvml, daemon=True)
            self.t.start()
            return self
        except Exception:  # no NVML: nvidia-smi instead
            self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 5.0:  # wait for the first sample
                time.sleep(0.02)
        except OSError:
            self.proc = None
        return self

    def _poll_nvml(self):
        sm_fn, smax, bits_fn = self.nvml
        while self.running:
            try:
                sm = sm_fn()
                bits = bits_fn()
            except Exception:
                break
            act = [nm for nm, b in self.NVML_BITS if bits & b]
            self.samples.append((time.time(), sm, smax, act))
            time.sleep(0.0005)

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            act = [nm for nm, v in zip(self.NAMES, parts[4:8]) if v.lower().startswith("active")]
            self.samples.append((time.time(), sm, smax, act))

    def stop(self):
        if self.nvml:
            self.running = False
            self.t.join(timeout=2)
            return
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        where = "timed window"
        if not inside:  # window shorter than the sampling period: nearest samples around it
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            where = f"nearest to the timed window (window shorter than the {self.period} period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = sorted({r for s in inside for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": inside[0][2],
                "reasons": reasons, "samples": len(inside), "sampled": where,
                "source": "nvml" if self.nvml else "nvidia-smi"}


class L2Flush:
    """Empties L2 between timed steps: a 512 MB buffer (4x the 126 MB L2) is written and then
    read back, outside the timed region.  The read-back evicts the written lines, so no dirty
    line of the flush itself is left to be written back to HBM inside the next timed step."""
    WHAT = "flushed between timed steps (512 MB written, then read back)"

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.view = self.buf.view(torch.int32)

    def __call__(self):
        self.buf.zero_()
        self.view.max()


def slowest(seconds, world, device):
    """The job's time for a step every rank ran: the largest over ranks (all-reduce MAX; a no-op
    on one rank).  `device` is where the collective's tensor lives (CUDA for NCCL, CPU for gloo)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        seconds = float(t.item())
    return seconds


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------
def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist
    from fp4_kv_top_csa2_b300 import csa2, synth
    from fp4_kv_top_csa2_b300.step import Step

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks = _peaks()
    w = synth.WORKLOADS[HEADLINE]
    inp = synth.make_inputs(w)
    st = Step(inp, device=dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    clk = ClockSampler(dev.index).start()
    st.capture()  # the whole step as one CUDA graph (same C-ABI calls as Step.run)
    for _ in range(args.warmup):
        st.replay()
    torch.cuda.synchronize()
    launches_per_step = launches_of(st)
    launches0 = csa2.kernel_launches()

    # timed region: K graph replays, per-step events, L2 flushed between steps (outside events)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    tw0 = time.time()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        st.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    tw1 = time.time()
    # the clock record covers this timed window; the sampler's polling thread would otherwise
    # compete with the host-issued calls of the end-to-end timing below
    clk.stop()
    barrier()
    assert csa2.kernel_launches() == launches0  # replays enqueue no new host-side launches
    launches = launches_per_step * args.steps
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = slowest(sum(step_ms) / len(step_ms), world, dev)
    by = st.algorithmic_bytes()
    tokens_per_s = world * w.B / (ms / 1e3)
    step_gbs = by["total"] / (ms / 1e3) / 1e9

    # per-call device times: each call captured as its own graph, replayed with events
    parts = profile_calls(st, args.steps, flush)
    # The dominant kernel is the Full layer's scan (134 MB of the step's 145 MB of algorithmic
    # bytes).  Its own time: csa2_index_block_max (that scan alone, one launch) captured as its
    # own graph and replayed between events, L2 flushed before each replay.
    full = next(L for L in st.layers if L["mode"] == "full")
    scan_ms = time_graph(lambda s: st.block_max(full, st.bm, stream=s), args.steps, flush)
    dom_bytes = by["index_keys_full"]
    achieved = dom_bytes / (scan_ms / 1e3) / 1e9
    call_gbs = dom_bytes / (parts["full_index"] / 1e3) / 1e9
    # end to end through the C ABI with host buffers (direct calls, no graph), and with the graph
    e2e = run_e2e(st, args.steps, dev, world, graph=False)
    e2e_graph = run_e2e(st, args.steps, dev, world, graph=True)

    line = {
        "metric": METRIC, "value": round(tokens_per_s, 2), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp4-e2m1/e4m3 kv, fp8 indexer, bf16 attn (fp32 acc)",
        "data": "synthetic (seeded N(0,1) x log-uniform channel scales; no weights)",
        "config": {"workload": HEADLINE, "batch": w.B, "context": w.L[0], "heads": w.H,
                   "d_latent": 512, "indexer": f"{w.Hi}x{w.Di} e4m3", "topk": w.topk,
                   "pool": f"{w.n_pool_blocks}x8", "modes": list(w.modes),
                   "l2": L2Flush.WHAT, "parallelism": "replicas"},
        "hbm": {"algorithmic_bytes_per_step": by["total"], "gbs": round(step_gbs, 1),
                "frac_of_8tbs": round(step_gbs / HBM_TARGET_GBS, 4),
                "frac_of_measured": round(step_gbs / peaks["hbm_gbs"], 4), "bytes_by_part": by},
        "roofline": {"kernel": "index_mma_kernel<E4M3, SCAN> (Full scan, 1,048,576 keys)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "frac_of_8tbs": round(achieved / HBM_TARGET_GBS, 4),
                     "peak_source": peaks["source"] + " (burst copy)", "traffic": SCAN_TRAFFIC,
                     "ms_per_launch": round(scan_ms, 5), "algorithmic_bytes": dom_bytes,
                     "timed_as": "csa2_index_block_max alone, one CUDA graph per replay, L2 "
                                 "flushed before each",
                     "call": {"name": "csa2_index_score_topk_pool (scan + pool + Top-K)",
                              "ms": round(parts["full_index"], 5), "gbs": round(call_gbs, 1),
                              "frac": round(call_gbs / peaks["hbm_gbs"], 4)}},
        "breakdown_ms": {k: round(v, 5) for k, v in parts.items()},
        "timing": "step = one CUDA-graph replay of all calls; CUDA events on the launching stream",
        "e2e": e2e, "e2e_graph": e2e_graph, "gpu_launches": launches,
        "gpu_launches_per_step": launches_per_step, "wall_s_timed": round(wall, 4),
        "clocks": clk.summary(tw0, tw1),
    }
    del st
    torch.cuda.empty_cache()
    if args.configs and rank == 0:
        line["decode_configs"] = {name: run_decode_config(name, args, dev, peaks, flush)
                                  for name in DECODE_CONFIGS}
        # the headline step with every layer's local sliding window (128 FP8 local rows)
        line["hier_decode_swa"] = run_decode_config(HEADLINE_SWA, args, dev, peaks, flush)
        line["index_keys"] = run_index_keys(args, dev, peaks, flush)
        line["kv_quant"] = run_kv_quant(args, dev, peaks, flush)
    if args.prefill and rank == 0:
        line["prefill"] = run_prefill(args, dev, peaks)
        line["prefill_hier"] = run_prefill_hier(args, dev)
    if rank == 0 and args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, w, args.cpu_steps)
    return line


def launches_of(st):
    """Kernels one step launches (counted by the library while enqueuing one un-captured step)."""
    import torch
    from fp4_kv_top_csa2_b300 import csa2
    torch.cuda.synchronize()
    a = csa2.kernel_launches()
    st.run()
    torch.cuda.synchronize()
    return csa2.kernel_launches() - a


def profile_calls(st, steps, flush):
    """Device time of each C-ABI call of the step: every call is captured into its own CUDA graph
    and replayed `steps` times between CUDA events (L2 flushed before each replay)."""
    import torch
    from fp4_kv_top_csa2_b300 import csa2
    full = next(L for L in st.layers if L["mode"] == "full")
    reidx = next((L for L in st.layers if L["mode"] == "reindex"), None)
    calls = {
        "kv_quant": lambda s: st.quantize_new_rows(stream=s),
        # the step's first Full layer: with the candidate pool in the hierarchical decoder
        "full_index": ((lambda s: st.index_with_pool(full, stream=s)) if st.pool is not None
                       else (lambda s: st.index(full, stream=s))),
        "attention": lambda s: st.attend(full, full["idx"], stream=s),
    }
    if reidx is not None:
        calls["reindex_index"] = lambda s: st.index(reidx, cand=st.pool, stream=s)
    out = {}
    stream = torch.cuda.current_stream()
    for name, fn in calls.items():
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
                fn(side)
        stream.wait_stream(side)
        g.replay()
        torch.cuda.synchronize()
        tms = []
        for _ in range(steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            tms.append(a.elapsed_time(b))
        out[name] = sum(tms) / len(tms)
    return out


def time_graph(fn, steps, flush):
    """Mean device time (ms) of fn(stream) captured as one CUDA graph and replayed `steps`
    times between CUDA events on the launching stream, L2 flushed before each replay."""
    import torch
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
            fn(side)
    stream.wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    tms = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        tms.append(a.elapsed_time(b))
    return sum(tms) / len(tms)


def run_decode_config(name, args, dev, peaks, flush):
    """One of the non-hierarchical decode workloads: its whole step (new rows' quantisation,
    Full selection, attention) as one CUDA graph, timed like the headline step."""
    import torch
    from fp4_kv_top_csa2_b300 import synth
    from fp4_kv_top_csa2_b300.step import Step
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w)
    st = Step(inp, device=dev)
    st.drop_source_rows()
    inp["kv_bf16"] = None
    launches = launches_of(st)
    st.capture()
    for _ in range(args.warmup):
        st.replay()
    stream = torch.cuda.current_stream()
    tms = []
    for _ in range(args.steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        st.replay()
        b.record(stream)
        torch.cuda.synchronize()
        tms.append(a.elapsed_time(b))
    ms = sum(tms) / len(tms)
    by = st.algorithmic_bytes()
    gbs = by["total"] / (ms / 1e3) / 1e9
    out = {"batch": w.B, "context": (list(inp["lengths"]) if w.ragged else w.L[0]),
           "context_total": int(sum(inp["lengths"])), "heads": w.H,
           "indexer": f"{w.Hi}x{w.Di} {'bf16' if w.idx_dtype == 0 else 'e4m3'}", "topk": w.topk,
           "ms_per_step": round(ms, 5), "tokens_per_s": round(w.B / (ms / 1e3), 1),
           "algorithmic_bytes_per_step": by["total"], "gbs": round(gbs, 1),
           "frac_of_8tbs": round(gbs / HBM_TARGET_GBS, 4),
           "frac_of_measured": round(gbs / peaks["hbm_gbs"], 4), "gpu_launches_per_step": launches,
           "l2": L2Flush.WHAT}
    if w.ragged:
        out["context"] = f"{min(inp['lengths'])}..{max(inp['lengths'])} (ragged, {w.B} sequences)"
    if w.n_win:
        out["local_window"] = w.n_win
        out["modes"] = list(w.modes)
    del st
    torch.cuda.empty_cache()
    return out


def run_index_keys(args, dev, peaks, flush, n_rows=1 << 20):
    """Index keys derived from a 1,048,576-row FP4 cache (the cache build of the 1M-context
    workload): 2 * 128 * 512 FLOP per row on the tensor cores, 288 B read and 132 B written."""
    import torch
    from fp4_kv_top_csa2_b300 import csa2
    g = torch.Generator(device=dev).manual_seed(0)
    codes = torch.randint(0, 256, (n_rows, 256), dtype=torch.uint8, device=dev, generator=g)
    sf = torch.randint(0x28, 0x48, (n_rows, 32), dtype=torch.uint8, device=dev, generator=g)
    W = (torch.randn(128, 512, device=dev, generator=g) / 16).to(torch.bfloat16)
    keys = torch.empty((n_rows, 128), dtype=torch.uint8, device=dev)
    ks = torch.empty(n_rows, dtype=torch.float32, device=dev)
    ms = time_graph(lambda s: csa2.csa2_index_keys_from_kv(codes, sf, W, keys, ks, stream=s),
                    args.steps, flush)
    flops = 2.0 * 128 * 512 * n_rows
    by = n_rows * (288 + 128 + 4)
    tf = flops / (ms / 1e3) / 1e12
    return {"rows": n_rows, "ms": round(ms, 4), "rows_per_s": round(n_rows / (ms / 1e3), 1),
            "tflops": round(tf, 1), "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
            "gbs": round(by / (ms / 1e3) / 1e9, 1),
            "frac_of_hbm": round(by / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)}


def run_kv_quant(args, dev, peaks, flush, n_rows=1 << 20):
    """FP4 quantisation of 1,048,576 bf16 rows (the 1M-context cache build): 1,024 B read and
    256 + 32 B written per row.  Rows drawn with a per-channel spread of two decades."""
    import torch
    from fp4_kv_top_csa2_b300 import csa2
    g = torch.Generator(device=dev).manual_seed(0)
    sigma = 10.0 ** (torch.rand(512, device=dev, generator=g) * 2 - 1)
    x = (torch.randn(n_rows, 512, device=dev, generator=g) * sigma).to(torch.bfloat16)
    codes = torch.empty((n_rows, 256), dtype=torch.uint8, device=dev)
    sf = torch.empty((n_rows, 32), dtype=torch.uint8, device=dev)
    ms = time_graph(lambda s: csa2.csa2_kv_quant_fp4(x, codes, sf, stream=s), args.steps, flush)
    by = n_rows * (1024 + 256 + 32)
    gbs = by / (ms / 1e3) / 1e9
    return {"rows": n_rows, "ms": round(ms, 4), "gbs": round(gbs, 1),
            "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}


def run_e2e(st, steps, dev, world=1, graph=False):
    """Same step through the C ABI, inputs copied from pinned host memory each step and the
    attention outputs read back, all inside the timed region.  The step's per-token inputs
    (new rows, every layer's queries and weights) sit in one device arena and its outputs in
    another; Step.run(io=...) copies them layer by layer on two copy streams, overlapped with
    the computation (layer i's inputs cross while earlier layers compute, its output leaves
    once its attention is done).  graph=True replays that whole step, copies included, as one
    captured graph instead of issuing the calls one by one.  With several ranks the job's rate
    is the tokens of all ranks over the slowest rank's time."""
    import torch
    host_in = st.in_arena.buf.cpu().pin_memory()
    host_out = torch.empty_like(st.out_arena.buf, device="cpu").pin_memory()
    h2d = host_in.numel()
    d2h = host_out.numel()
    io = (host_in, host_out)
    g = st.capture(io=io) if graph else None

    def one():
        if graph:
            g.replay()
        else:
            st.run(io=io)

    one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    dt = slowest((time.perf_counter() - t0) / steps, world, dev)
    return {"value": round(world * st.w.B / dt, 2), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(dt * 1e3, 4),
            "path": "graph replay" if graph else "direct C-ABI calls"}


def run_prefill(args, dev, peaks):
    import torch
    from fp4_kv_top_csa2_b300 import csa2, synth
    from fp4_kv_top_csa2_b300.step import Step
    w = synth.WORKLOADS[PREFILL]
    inp = synth.make_inputs(w)
    st = Step(inp, device=dev)
    stream = torch.cuda.current_stream()
    L = st.layers[0]
    for _ in range(max(1, args.warmup // 2)):
        st.run()
    torch.cuda.synchronize()
    ti, ta, tq, tf = [], [], [], []
    for _ in range(args.prefill_steps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        e[0].record(stream)
        st.quantize_new_rows()
        e[1].record(stream)
        st.index(L)
        e[2].record(stream)
        st.attend(L, L["idx"])
        e[3].record(stream)
        csa2.csa2_sparse_attn_prefill_fp4pv(L["q_attn"], st.q_seq, st.codes, st.sf, st.cu_ctx,
                                            L["idx"], st.scale, L["out"], L["lse"])
        e[4].record(stream)
        torch.cuda.synchronize()
        tf.append(e[3].elapsed_time(e[4]))
        tq.append(e[0].elapsed_time(e[1]))
        ti.append(e[1].elapsed_time(e[2]))
        ta.append(e[2].elapsed_time(e[3]))
    P0 = w.L[0]
    pairs = sum(P0 + i + 1 for i in range(w.T))
    f_idx = 2.0 * pairs * w.Hi * w.Di
    f_attn = 4.0 * w.T * w.topk * w.H * 512
    mi, ma, mq, mf = (statistics.median(x) for x in (ti, ta, tq, tf))
    bf16 = peaks["bf16_tflops"]
    p_fp8 = 2.0 * bf16  # nominal dense fp8 / bf16 ratio 4.5 / 2.25
    p_fp4 = 6.0 * bf16  # nominal dense fp4 / bf16 ratio 13.5 / 2.25
    # Attention's FLOP-weighted peak if QK^T ran as block-scaled FP4 and PV as f16 (half the
    # FLOPs each): 1 / (0.5 / P_fp4 + 0.5 / P_f16).
    p_mixed = 1.0 / (0.5 / p_fp4 + 0.5 / bf16)
    ta_fl = f_attn / (ma / 1e3) / 1e12
    ti_fl = f_idx / (mi / 1e3) / 1e12
    src = peaks["source"]
    return {"workload": PREFILL, "tokens": w.T, "cached": P0, "topk": w.topk, "heads": w.H,
            "ms_indexer": round(mi, 4), "ms_attention": round(ma, 4), "ms_kv_quant": round(mq, 4),
            "indexer_tflops": round(ti_fl, 2), "attention_tflops": round(ta_fl, 2),
            "tokens_per_s": round(w.T / ((mi + ma + mq) / 1e3), 1),
            "flops_indexer": f_idx, "flops_attention": f_attn,
            "attention_fp4pv": {"ms": round(mf, 4),
                                "tflops": round(f_attn / (mf / 1e3) / 1e12, 2),
                                "what": "csa2_sparse_attn_prefill_fp4pv: P and V re-quantised to "
                                        "block-scaled FP4 along the slots (two passes: S^T, then "
                                        "S^T and PV)"},
            "roofline": {
                "kernel": "csa2_sparse_attn_prefill (FP4 query quantisation + attn_prefill_kernel)",
                "bound": "tensor", "achieved": round(ta_fl, 1), "peak": bf16, "unit": "TFLOP/s",
                "frac": round(ta_fl / bf16, 4),
                "peak_source": f"{src} bf16 burst; the contraction runs as tcgen05 kind::f16, "
                               "whose dense rate equals bf16's",
                "frac_of_mixed_fp4_f16_peak": round(ta_fl / p_mixed, 4),
                "mixed_peak": round(p_mixed, 1),
                "mixed_peak_source": f"{src} bf16 burst x 6 for QK^T (nominal fp4 / bf16 13.5 / "
                                     "2.25) and x 1 for PV, weighted by their equal FLOPs",
                "traffic": None},
            "indexer_roofline": {
                "kernel": "csa2_index_score_topk (index_multi_kernel scan + block and position "
                          "Top-K)",
                "bound": "tensor", "achieved": round(ti_fl, 1), "peak": round(p_fp8, 1),
                "unit": "TFLOP/s", "frac": round(ti_fl / p_fp8, 4),
                "peak_source": f"{src} bf16 burst x 2 (nominal fp8 / bf16 4.5 / 2.25)",
                "traffic": None}}


def run_prefill_hier(args, dev):
    """Chunked prefill through the hierarchical indexer (a candidate pool per query token, three
    Reindex layers, two Reuse layers, six sparse attentions): each call kind and the whole step,
    timed with CUDA events on the launching stream."""
    import torch
    from fp4_kv_top_csa2_b300 import synth
    from fp4_kv_top_csa2_b300.step import Step
    w = synth.WORKLOADS[PREFILL_HIER]
    inp = synth.make_inputs(w)
    st = Step(inp, device=dev)
    st.drop_source_rows()
    inp["kv_bf16"] = None
    stream = torch.cuda.current_stream()
    full = st.layers[0]
    reidx = next(L for L in st.layers if L["mode"] == "reindex")
    calls = {"step": lambda: st.run(),
             "full_index_with_pool": lambda: st.index_with_pool(full),
             "reindex_index": lambda: st.index(reidx, cand=st.pool),
             "attention": lambda: st.attend(full, full["idx"])}
    st.run()
    torch.cuda.synchronize()
    ms = {}
    for name, fn in calls.items():
        ts = []
        for _ in range(args.prefill_steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms[name] = round(statistics.median(ts), 4)
    out = {"workload": PREFILL_HIER, "tokens": w.T, "cached": w.L[0], "topk": w.topk,
           "pool": f"{w.n_pool_blocks}x8 per query token", "modes": list(w.modes),
           "ms_per_step": ms["step"], "tokens_per_s": round(w.T / (ms["step"] / 1e3), 1),
           "ms_by_call": {k: v for k, v in ms.items() if k != "step"},
           "reindex_tflops": round(2.0 * w.T * w.n_pool_blocks * 8 * w.Hi * w.Di /
                                   (ms["reindex_index"] / 1e3) / 1e12, 2)}
    del st
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------------------------------------
# the oracle (CPU): reference arm and cpu_baseline
# ------------------------------------------------------------------------------------------------
def oracle_step(inp, w):
    """One decode step of the headline workload, executed by the CPU oracle.  The oracle gathers
    FP4 rows by quantising the selected bf16 rows on demand (bit-identical to the cache)."""
    import numpy as np
    import oracle
    from fp4_kv_top_csa2_b300.synth import new_token_rows, to_numpy_bits
    kv = inp["_np_kv"]
    cu = inp["cu_ctx"].numpy()
    k_idx = inp["_np_k"]
    q_seq, q_vis = inp["q_seq"].numpy(), inp["q_vis"].numpy()
    oracle.kv_quant_fp4(kv[new_token_rows(inp).numpy()])
    pool = None
    last = None
    scale = 1.0 / np.sqrt(512)
    for L in inp["layers"]:
        if L["mode"] == "full":
            r = oracle.index_score_topk(to_numpy_bits(L["q_idx"]), w.idx_dtype, L["w"].numpy(),
                                        k_idx, cu, q_seq, q_vis, w.topk)
            last = np.stack([r[n]["idx"] for n in range(len(q_seq))])
            if w.kind == "hier" and pool is None:
                pool = np.stack([oracle.candidate_pool(r[n]["bm"], w.n_pool_blocks)
                                 for n in range(len(q_seq))])
        elif L["mode"] == "reindex":
            r = oracle.index_score_topk(to_numpy_bits(L["q_idx"]), w.idx_dtype, L["w"].numpy(),
                                        k_idx, cu, q_seq, q_vis, w.topk, cand_blocks=pool)
            last = np.stack([r[n]["idx"] for n in range(len(q_seq))])
        qa = to_numpy_bits(L["q_attn"])
        for b in range(len(q_seq)):
            sel = last[b][last[b] >= 0]
            rows = kv[cu[b] + sel]
            c, s = oracle.kv_quant_fp4(rows)
            oracle.sparse_attn(oracle.bf16_to_double(qa[b]), c, s, np.arange(len(sel), dtype=np.int32),
                               scale)


def cpu_baseline(inp, w, steps):
    from fp4_kv_top_csa2_b300.synth import to_numpy_bits
    inp["_np_kv"] = to_numpy_bits(inp["kv_bf16"])
    inp["_np_k"] = to_numpy_bits(inp["k_idx"])
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(inp, w)
    dt = (time.perf_counter() - t0) / steps
    return {"value": round(w.B / dt, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{steps} full decode step(s) of {HEADLINE} on 1 host core "
                      f"(of {os.cpu_count()}), {dt:.2f} s/step"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from fp4_kv_top_csa2_b300 import synth
    from fp4_kv_top_csa2_b300.synth import to_numpy_bits
    w = synth.WORKLOADS[HEADLINE]
    inp = synth.make_inputs(w)
    inp["_np_kv"] = to_numpy_bits(inp["kv_bf16"])
    inp["_np_k"] = to_numpy_bits(inp["k_idx"])
    for _ in range(args.warmup):
        oracle_step(inp, w)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(inp, w)
    dt = (time.perf_counter() - t0) / args.steps
    v = round(w.B / dt, 4)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": HEADLINE, "batch": w.B, "context": w.L[0], "heads": w.H,
                       "topk": w.topk, "pool": f"{w.n_pool_blocks}x8", "modes": list(w.modes)},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} full decode steps of {HEADLINE}, 1 core"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def profile_step(name, steps, prefill_tokens=0, block_max_only=False):
    """A short run for profiler captures: build one workload's step (optionally a prefill with
    fewer new tokens), run it `steps` times, print one JSON line.  The bf16 source rows are dropped
    once the cache is quantised, so the device holds only what the step reads.  block_max_only:
    run the Full layer's scan alone (csa2_index_block_max, the kernel the headline roofline
    times) instead of the step."""
    import torch
    from fp4_kv_top_csa2_b300 import synth
    from fp4_kv_top_csa2_b300.step import Step
    w = synth.WORKLOADS[name]
    if prefill_tokens and w.kind == "prefill":
        w = synth.scaled(w, T=prefill_tokens)
    st = Step(synth.make_inputs(w), device="cuda")
    st.drop_source_rows()
    full = next(L for L in st.layers if L["mode"] == "full")
    for _ in range(steps):
        if block_max_only:
            st.block_max(full, st.bm)
        else:
            st.run()
    torch.cuda.synchronize()
    return {"profile_step": name, "steps": steps, "T": w.T,
            "device_bytes": torch.cuda.memory_allocated()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-prefill", dest="prefill", action="store_false")
    ap.add_argument("--prefill-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip timing the three non-hierarchical decode workloads")
    ap.add_argument("--cpu-steps", type=int, default=2)
    ap.add_argument("--profile-step", default=None,
                    help="run only this workload's step (--steps times) for a profiler capture")
    ap.add_argument("--prefill-tokens", type=int, default=0,
                    help="with --profile-step on the prefill workload: new tokens per step")
    ap.add_argument("--block-max-only", action="store_true",
                    help="with --profile-step: run the Full layer's scan alone")
    args = ap.parse_args()
    if args.profile_step:
        sys.path.insert(0, ROOT)
        print(json.dumps(profile_step(args.profile_step, args.steps, args.prefill_tokens,
                                      args.block_max_only)), flush=True)
        return
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # N replicas, one process per GPU, launched the way the multi-GPU contract runs them
        import socket
        with socket.socket() as so:
            so.bind(("127.0.0.1", 0))
            port = so.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
               "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
        os.execv(sys.executable, cmd)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    sys.path.insert(0, ROOT)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.init_process_group("nccl")
    line = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
