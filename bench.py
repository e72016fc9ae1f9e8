#!/usr/bin/env python
"""Benchmark of the affine group-quantized GEMV / GEMM hot path on B300.

Default workload (one "step"): a Qwen3-0.6B-shaped Q4 (group 64) decode pass
at M = 1 -- 28 layers of q 1024->2048, k/v 1024->1024, o 2048->1024, gate/up
1024->3072, down 3072->1024, each with its own weights and its own fp16 x,
plus an lm_head 1024->151936: 197 dequant-GEMVs, 335,241,216 bytes of packed
codes + fp16 scales/biases, run as the library's decode pass object (one
batched launch, recorded once as a CUDA graph and replayed per step).
Weights are synthetic (seeded N(0, 0.02), min/max-quantized); they exceed the
126 MB L2, so no flush is needed between steps.

Metric: weight GB/s (codes + scales + biases per pass / pass time), the
BaseRT pages' decode-bandwidth view (the bytes read per token fall with the
bit width).  The same run also times the Llama-3.2-3B-shaped prefill
GEMM pass (M = 128 and 512, TFLOP/s, key "prefill") and the Qwen3-30B-A3B-
shaped MoE layer (M = 1 and 128, key "moe"), the small-batch decode pass
(key "small_batch") and the decode step as 113 dependent stages through the
pass object (key "dependent_pass"); --legs selects them.

``--impl reference`` times the fp64 CPU oracle on bounded samples of the same
workload (the only other code path of this workload).  Under torchrun each
rank runs an independent replica (the path does not shard); rank 0 prints one
JSON line.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dequant_gemv_gemm_bt_b300 import synth  # noqa: E402

METRIC = "Q4 dequant-GEMV decode weight GB/s vs HBM peak; prefill qGEMM TFLOP/s"
GROUP = 64

# Qwen3-0.6B-shaped decode pass: (N, K) per projection in a layer, 28 layers, + lm_head.
QWEN06_LAYER = [("q", 2048, 1024), ("k", 1024, 1024), ("v", 1024, 1024), ("o", 1024, 2048),
                ("gate", 3072, 1024), ("up", 3072, 1024), ("down", 1024, 3072)]
QWEN06_LAYERS = 28
QWEN06_LM_HEAD = ("lm_head", 151936, 1024)
# Llama-3.2-3B-shaped prefill pass.
LLAMA3B_LAYER = [("q", 3072, 3072), ("k", 1024, 3072), ("v", 1024, 3072), ("o", 3072, 3072),
                 ("gate", 8192, 3072), ("up", 8192, 3072), ("down", 3072, 8192)]
LLAMA3B_LAYERS = 28
# Llama-3.2-1B-shaped decode pass, swept over bit widths.
LLAMA1B_LAYER = [("q", 2048, 2048), ("k", 512, 2048), ("v", 512, 2048), ("o", 2048, 2048),
                 ("gate", 8192, 2048), ("up", 8192, 2048), ("down", 2048, 8192)]
LLAMA1B_LAYERS = 16
SWEEP_BITS = (2, 3, 4, 6, 8)


def weight_bytes(n: int, k: int, bits: int) -> int:
    return n * k * bits // 8 + 4 * n * (k // GROUP)


def decode_pass_shapes():
    shapes = []
    for layer in range(QWEN06_LAYERS):
        for name, n, k in QWEN06_LAYER:
            shapes.append((f"L{layer}.{name}", n, k))
    shapes.append(QWEN06_LM_HEAD)
    return shapes


def sweep_pass_shapes():
    return [(f"L{l}.{name}", n, k) for l in range(LLAMA1B_LAYERS) for name, n, k in LLAMA1B_LAYER]


def prefill_pass_shapes():
    return [(f"L{l}.{name}", n, k) for l in range(LLAMA3B_LAYERS) for name, n, k in LLAMA3B_LAYER]


def gen_weights(tag, shapes, bits, threads=16):
    """Seeded packed weights for every (name, N, K), generated on host threads."""
    import concurrent.futures as cf

    def one(item):
        name, n, k = item
        return synth.make_qweight(synth.rng_for(tag, name, "w"), n, k, bits)
    with cf.ThreadPoolExecutor(threads) as ex:
        return list(ex.map(one, shapes))


def gen_x(tag, shapes, m, dtype):
    return [synth.draw_activations(synth.rng_for(tag, name, "x"), m, k, dtype) for name, n, k in shapes]


# ------------------------------------------------------------------ helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def source_digest(patterns):
    """Digest of the code in the matching files: comments and blank lines do not count."""
    h = hashlib.sha256()
    for pat in patterns:
        for f in sorted(glob.glob(os.path.join(ROOT, pat))):
            text = re.sub(r"/\*.*?\*/", "", open(f).read(), flags=re.S)
            for line in text.splitlines():
                code = re.sub(r"//.*", "", line).rstrip()
                if code.strip():
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profile_traffic(summary_file, digest):
    """Per-launch DRAM bytes from a committed ncu summary (profiles/<name>.json:
    {"kernel_source_digest": ..., "traffic_bytes_per_launch": ...}), if it was
    taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", summary_file)
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
        if d.get("kernel_source_digest") != digest:
            return None
        return float(d["traffic_bytes_per_launch"])
    except (ValueError, KeyError, TypeError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-i", str(self.gpu),
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        return max([d.get("num_threads", 1) for d in info if d.get("user_api") == "blas"] or [1])
    except Exception:
        return 1


def host_cores():
    """os.cpu_count() and the cores this process may run on."""
    try:
        aff = len(os.sched_getaffinity(0))
    except AttributeError:
        aff = os.cpu_count() or 1
    return os.cpu_count() or 1, aff


# ------------------------------------------------------------------ oracle leg
LM_HEAD_SLICE = 8192   # rows of the lm_head a worker computes per visit (bounded memory per worker)


def _oracle_worker(tag, shapes, indices, budget_s, warmup_s, ready, start, results):
    """One host core: its share of the pass's projections (generated here, untimed),
    `warmup_s` of untimed oracle work, then the fp64 oracle over them in pass
    order until the budget is spent."""
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    import oracle.bt_oracle as O
    try:
        from threadpoolctl import threadpool_limits
        threadpool_limits(1)
    except Exception:
        pass
    work = []
    for i in indices:
        name, n, k = shapes[i]
        qw = synth.make_qweight(synth.rng_for(tag, name, "w"), n, k, 4)
        x = O.decode_f16(synth.draw_activations(synth.rng_for(tag, name, "x"), 1, k, "f16")[0])
        work.append((qw, x))
    def one(j):
        qw, x = work[j % len(work)]
        rows = np.arange(0, min(qw.n, LM_HEAD_SLICE)) if qw.n > LM_HEAD_SLICE else None
        O.qgemv(qw.codes, qw.scales, qw.biases, qw.bits, x, rows=rows)
        return weight_bytes(qw.n if rows is None else len(rows), qw.k, qw.bits)

    tw = time.perf_counter()
    j = 0
    while work and time.perf_counter() - tw < warmup_s:
        one(j)
        j += 1
    ready.put(1)
    start.wait()
    t0 = time.perf_counter()
    done, count = 0, 0
    while work:
        done += one(j)
        count += 1
        j += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    results.put((done, count, time.perf_counter() - t0))


def oracle_rate(tag, shapes, budget_s: float, procs: int = 0, warmup_s: float = 0.0):
    """The fp64 oracle on the host's cores: `procs` spawned workers (default: every
    core in this process's affinity set), each running its share of the pass's
    projections for about `budget_s`.  Returns (GB/s of weight bytes, bytes,
    projections, workers).  Workers are spawned (not forked), so this may run
    after CUDA is initialised."""
    import multiprocessing as mp
    procs = min(procs or min(host_cores()[1], 64), len(shapes))
    ctx = mp.get_context("spawn")
    ready, results, start = ctx.Queue(), ctx.Queue(), ctx.Event()
    order = list(range(len(shapes)))
    ps = [ctx.Process(target=_oracle_worker,
                      args=(tag, shapes, order[w::procs], budget_s, warmup_s, ready, start, results))
          for w in range(procs)]
    for p in ps:
        p.start()
    for _ in ps:
        ready.get()
    t0 = time.perf_counter()
    start.set()
    got = [results.get() for _ in ps]
    wall = time.perf_counter() - t0
    for p in ps:
        p.join()
    done = sum(g[0] for g in got)
    count = sum(g[1] for g in got)
    return done / wall / 1e9, done, count, procs


# ------------------------------------------------------------------ GPU legs
def gemv_kernel_name(bt, bits):
    """The kernel the library plans for the decode pass's one batched launch."""
    p, _ = bt.bt_plan_gemv_batch(bits, [(n, k) for _, n, k in decode_pass_shapes()])
    kind = {0: "qgemv_kernel (CUDA cores", 1: "qgemv_mma_kernel (tensor pipe, diagonal consumer",
            2: "qgemv_mma_kernel (tensor pipe, four-column consumer"}[p["tensor_pipe"]]
    return kind + "; batched, mixed K; 1 launch per pass)"


def build_decode_pass(torch, bt, weights, xs16, dev):
    bufs = []
    for qw, x16 in zip(weights, xs16):
        c = torch.from_numpy(qw.codes.view(np.int32)).to(dev)
        s = torch.from_numpy(qw.scales.view(np.float16)).to(dev)
        b = torch.from_numpy(qw.biases.view(np.float16)).to(dev)
        x = torch.from_numpy(x16[0].view(np.int16)).to(dev).view(torch.float16)
        y = torch.empty(qw.n, dtype=torch.float32, device=dev)
        bufs.append((c, s, b, x, y, qw.bits))
    return bufs


class EagerReplay:
    """Stands in for a captured graph: replay() issues the same launches directly on the stream."""

    def __init__(self, torch, fn, stream):
        self.torch, self.fn, self.stream = torch, fn, stream

    def replay(self):
        with self.torch.cuda.stream(self.stream):
            self.fn()


EAGER = False   # set by --eager: no graph capture (for profilers that cannot follow graph replays)


def capture(torch, fn, stream):
    if EAGER:
        return EagerReplay(torch, fn, stream)
    with torch.cuda.stream(stream):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


def max_over_ranks(torch, dist, seconds, device):
    """The slowest rank's timed seconds (every rank gets it); `seconds` itself on one GPU."""
    if dist is None:
        return seconds
    tt = torch.tensor([seconds], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return tt.item()


def whole_job_rate(units_per_step, steps, world, seconds):
    """Units all ranks processed per second, each of `world` replicas doing `units_per_step`."""
    return units_per_step * steps * world / seconds


def timed(torch, dist, stream, fn, steps, warmup, gpu_index):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index) as clk:
        ev0.record(stream)
        for _ in range(steps):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    return ms / 1e3, clk.summary()


def pack_rows(ws):
    """Concatenate packed weights along N (row-major layout: row slices stay contiguous)."""
    return synth.QuantWeight(np.concatenate([w.codes for w in ws]), np.concatenate([w.scales for w in ws]),
                             np.concatenate([w.biases for w in ws]), ws[0].bits, sum(w.n for w in ws), ws[0].k)


def to_dev_w(torch, qw, dev):
    return (torch.from_numpy(qw.codes.view(np.int32)).to(dev), torch.from_numpy(qw.scales.view(np.float16)).to(dev),
            torch.from_numpy(qw.biases.view(np.float16)).to(dev))


def run_prefill(torch, bt, dev, stream, steps, warmup, gpu_index, peaks):
    """Llama-3.2-3B-shaped prefill pass, Q4, bf16 X and Y, M = 128 and 512.

    Per layer the weights are stored as the runtime would keep them: q|k|v
    concatenated (N = 5120) and gate|up concatenated (N = 16384), plus o and
    down.  The "fused" pass runs 4 GEMMs per layer (q, k, v share X; gate, up
    share X); the "unfused" pass runs the 7 projections separately on row
    slices of the same weights.  FLOPs are identical: 2*M*sum(N*K).
    """
    bits = 4
    shapes = prefill_pass_shapes()
    t0 = time.time()
    ws = gen_weights("prefill-pass", shapes, bits)
    gen_s = time.time() - t0
    per_layer = len(LLAMA3B_LAYER)
    layers = []
    for l in range(LLAMA3B_LAYERS):
        q, k, v, o, g, u, d = ws[l * per_layer:(l + 1) * per_layer]
        layers.append({"qkv": to_dev_w(torch, pack_rows([q, k, v]), dev), "o": to_dev_w(torch, o, dev),
                       "gu": to_dev_w(torch, pack_rows([g, u]), dev), "down": to_dev_w(torch, d, dev)})
    del ws
    flops_per_token = 2 * sum(n * k for _, n, k in shapes)
    wbytes = sum(weight_bytes(n, k, bits) for _, n, k in shapes)
    out = {"workload": "Llama-3.2-3B-shaped prefill pass: 28 layers x (q 3072->3072, k/v 3072->1024, o 3072->3072, "
                       "gate/up 3072->8192, down 8192->3072), Q4 g64, bf16 X/Y, fp32 accumulate",
           "weight_bytes_per_pass": wbytes, "weight_gen_s": round(gen_s, 1)}
    sustained = float(peaks.get("bf16_tflops_sustained", 1400.0))
    burst = float(peaks.get("bf16_tflops", 1800.0))
    for m in (128, 512):
        xs = [torch.randn(m, 3072, device=dev).bfloat16() for _ in range(3)]
        xd = torch.randn(m, 8192, device=dev).bfloat16()
        y_qkv = torch.empty(m, 5120, device=dev, dtype=torch.bfloat16)
        y_o = torch.empty(m, 3072, device=dev, dtype=torch.bfloat16)
        y_gu = torch.empty(m, 16384, device=dev, dtype=torch.bfloat16)
        y_d = torch.empty(m, 3072, device=dev, dtype=torch.bfloat16)

        def fused():
            for L in layers:
                bt.bt_qgemm(*L["qkv"], bits, xs[0], y_qkv)
                bt.bt_qgemm(*L["o"], bits, xs[1], y_o)
                bt.bt_qgemm(*L["gu"], bits, xs[2], y_gu)
                bt.bt_qgemm(*L["down"], bits, xd, y_d)

        ys = {nm: torch.empty(m, n, device=dev, dtype=torch.bfloat16) for nm, n, _ in LLAMA3B_LAYER}
        rows = {"q": ("qkv", 0, 3072), "k": ("qkv", 3072, 4096), "v": ("qkv", 4096, 5120),
                "gate": ("gu", 0, 8192), "up": ("gu", 8192, 16384)}

        def unfused():
            for L in layers:
                for nm, n, kk in LLAMA3B_LAYER:
                    if nm in rows:
                        key, a, b = rows[nm]
                        c, sc, bi = L[key]
                        w = (c[a:b], sc[a:b], bi[a:b])
                    else:
                        w = L["o" if nm == "o" else "down"]
                    x = xd if nm == "down" else xs[0 if nm in ("q", "k", "v") else (1 if nm == "o" else 2)]
                    bt.bt_qgemm(*w, bits, x, ys[nm])

        res = {}
        for tag, fn, launches in (("fused", fused, 4 * LLAMA3B_LAYERS), ("unfused", unfused, 7 * LLAMA3B_LAYERS)):
            g = capture(torch, fn, stream)
            n_steps = max(3, min(steps, 50))
            with torch.cuda.stream(stream):
                t, clk = timed(torch, None, stream, lambda: g.replay(), n_steps, max(3, min(warmup, 5)), gpu_index)
            tfl = flops_per_token * m * n_steps / t / 1e12
            res[tag] = {"tflops": round(tfl, 1), "ms_per_pass": round(t / n_steps * 1e3, 3), "launches_per_pass": launches,
                        "frac_of_sustained_bf16": round(tfl / sustained, 4), "frac_of_burst_bf16": round(tfl / burst, 4),
                        "clocks": clk}
            del g
        out[f"M{m}"] = res
    if bt.bt_last_device_error() != bt.BT_OK:
        raise RuntimeError("device error in the prefill leg")
    return out


def run_c1(torch, bt, dev, stream, steps, warmup, gpu_index, hbm):
    """The single Q4 GEMV (N=2048, K=1024, fp16 x, fp32 y; 1,179,648 weight bytes),
    timed twice: as-is (the same weights every launch, so they stay in the 126 MB
    L2 and the launch is latency-bound), and rotating over enough distinct
    device copies of the weights to exceed 2x L2, so each launch reads HBM.
    Each is a CUDA graph of back-to-back bt_qgemv launches with PDL."""
    n, k, bits = 2048, 1024, 4
    per = weight_bytes(n, k, bits)
    qw = synth.make_qweight(synth.rng_for("c1", "w"), n, k, bits)
    x16 = synth.draw_activations(synth.rng_for("c1", "x"), 1, k, "f16")
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    copies = -(-2 * l2 // per) + 8
    base = to_dev_w(torch, qw, dev)
    ws = [tuple(t.clone() for t in base) for _ in range(copies)]
    x = torch.from_numpy(x16[0].view(np.int16)).to(dev).view(torch.float16)
    y = torch.empty(n, dtype=torch.float32, device=dev)
    bt.bt_set_option(bt.BT_OPT_PDL, 1)
    bt.bt_set_option(bt.BT_OPT_CONST_WEIGHTS, 1)
    out = {"workload": "single Q4 GEMV N=2048 K=1024 g64, fp16 x, fp32 y", "bytes_per_gemv": per,
           "rotated_copies": copies, "rotated_bytes": copies * per, "l2_bytes": l2}
    for tag, seq in (("as_is", [base] * copies), ("rotated", ws)):
        g = capture(torch, lambda seq=seq: [bt.bt_qgemv(c, s, b, bits, x, y) for c, s, b in seq], stream)
        n_steps = max(3, min(steps, 50))
        with torch.cuda.stream(stream):
            t, clk = timed(torch, None, stream, lambda: g.replay(), n_steps, max(3, min(warmup, 5)), gpu_index)
        launches = n_steps * len(seq)
        gbs = per * launches / t / 1e9
        out[tag] = {"us_per_gemv": round(t / launches * 1e6, 3), "gbs": round(gbs, 1),
                    "frac_of_hbm": round(gbs / hbm, 4), "launches_per_graph": len(seq), "clocks": clk}
        del g
    del ws
    if bt.bt_last_device_error() != bt.BT_OK:
        raise RuntimeError("device error in the single-GEMV leg")
    return out


def run_sweep(torch, bt, dev, stream, steps, warmup, gpu_index, hbm):
    """Llama-3.2-1B-shaped decode pass (16 layers x 7 projections, fp16 x, fp32 y) at
    Q2/Q3/Q4/Q6/Q8: one mixed-K bt_qgemv_batched launch per pass (K = 2048 and 8192),
    captured in a CUDA graph with PDL; weight GB/s per bit width."""
    shapes = sweep_pass_shapes()
    bt.bt_set_option(bt.BT_OPT_PDL, 1)
    bt.bt_set_option(bt.BT_OPT_CONST_WEIGHTS, 1)
    xs16 = gen_x("sweep-pass", shapes, 1, "f16")
    out = {"workload": "Llama-3.2-1B-shaped decode pass: 16 layers x (q/o 2048->2048, k/v 2048->512, "
                       "gate/up 2048->8192, down 8192->2048), g64, fp16 x, fp32 y; 1 batched launch per pass"}
    n_steps = max(3, min(steps, 200))
    for bits in SWEEP_BITS:
        t0 = time.time()
        ws = gen_weights("sweep-pass", shapes, bits)
        gen_s = time.time() - t0
        pass_bytes = sum(weight_bytes(n, k, bits) for _, n, k in shapes)
        bufs = build_decode_pass(torch, bt, ws, xs16, dev)
        del ws
        groups = [[b[:5] for b in bufs]]   # one mixed-K launch (K = 2048 and 8192)

        def run_pass():
            for g in groups:
                bt.bt_qgemv_batched(g, bits)
        g = capture(torch, run_pass, stream)
        with torch.cuda.stream(stream):
            t, clk = timed(torch, None, stream, lambda: g.replay(), n_steps, max(3, min(warmup, 5)), gpu_index)
        gbs = pass_bytes * n_steps / t / 1e9
        out[f"Q{bits}"] = {"gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4),
                           "us_per_pass": round(t / n_steps * 1e6, 2), "bytes_per_pass": pass_bytes,
                           "launches_per_pass": len(groups), "weight_gen_s": round(gen_s, 1), "clocks": clk}
        del g, bufs, groups
        torch.cuda.synchronize()
    if bt.bt_last_device_error() != bt.BT_OK:
        raise RuntimeError("device error in the bit-width sweep leg")
    return out


def run_small(torch, bt, dev, stream, steps, warmup, gpu_index, hbm):
    """Qwen3-0.6B-shaped decode pass with M = 2..16 tokens per step (small-batch
    decode), Q4 g64, fp16 x, fp32 y.  Per layer the weights are stored as the
    runtime keeps them: q|k|v (N=4096, K=1024), o (1024, 2048), gate|up (6144,
    1024), down (1024, 3072); plus the lm_head (151936, 1024): 113 bt_qgemm
    products per pass, in one CUDA graph with PDL.  Each weight crosses HBM once
    per pass for all M tokens, so GB/s counts the packed bytes of the pass.
    "batched" is one bt_qgemm_batched call per pass (one launch of the
    small-token tensor-pipe kernel for M <= 16); "per_product" is one bt_qgemm
    launch per product (the library's path); "cuda_core_tile" forces the
    fp32-FMA tile the small-token kernel replaces."""
    bits = 4
    layer = [("qkv", 4096, 1024), ("o", 1024, 2048), ("gu", 6144, 1024), ("down", 1024, 3072)]
    shapes = [(f"L{l}.{nm}", n, k) for l in range(QWEN06_LAYERS) for nm, n, k in layer] + [QWEN06_LM_HEAD]
    t0 = time.time()
    ws = [to_dev_w(torch, w, dev) for w in gen_weights("small-pass", shapes, bits)]
    gen_s = time.time() - t0
    wbytes = sum(weight_bytes(n, k, bits) for _, n, k in shapes)
    out = {"workload": "Qwen3-0.6B-shaped decode pass at M tokens: 28 layers x (q|k|v 1024->4096, o 2048->1024, "
                       "gate|up 1024->6144, down 3072->1024) + lm_head 1024->151936, Q4 g64, fp16 x, fp32 y",
           "bytes_per_pass": wbytes, "products_per_pass": len(shapes), "weight_gen_s": round(gen_s, 1)}
    n_steps = max(3, min(steps, 100))
    for m in (2, 4, 8, 16):
        xs = {k: torch.randn(m, k, device=dev).half() for k in (1024, 2048, 3072)}
        ys = [torch.empty(m, n, device=dev, dtype=torch.float32) for _, n, _ in shapes]
        res = {"path": bt.bt_plan_gemm(bits, m, 4096, 1024, x_dtype=torch.float16)["path"]}
        probs = [(c, s, b, xs[k], y) for (c, s, b), (_, _, k), y in zip(ws, shapes, ys)]
        for tag, path in (("batched", None), ("per_product", 0), ("cuda_core_tile", 1)):
            bt.bt_set_option(bt.BT_OPT_GEMM_PATH, path or 0)
            try:
                if path is None:
                    g = capture(torch, lambda: bt.bt_qgemm_batched(probs, bits), stream)
                else:
                    g = capture(torch, lambda: [bt.bt_qgemm(c, s, b, bits, x, y) for c, s, b, x, y in probs], stream)
            finally:
                bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)
            with torch.cuda.stream(stream):
                t, clk = timed(torch, None, stream, lambda: g.replay(), n_steps, max(3, min(warmup, 5)), gpu_index)
            t /= n_steps
            gbs = wbytes / t / 1e9
            res[tag] = {"gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4), "us_per_pass": round(t * 1e6, 2),
                        "tokens_per_s": round(m / t, 1), "clocks": clk}
            del g
        out[f"M{m}"] = res
    if bt.bt_last_device_error() != bt.BT_OK:
        raise RuntimeError("device error in the small-batch leg")
    return out


def run_chain(torch, bt, bufs, dev, stream, steps, warmup, gpu_index, hbm, pass_bytes):
    """The decode leg's Qwen3-0.6B-shaped weights as a DEPENDENT decode step: per
    layer the stages [q, k, v] (read the hidden state), [o] (reads q's output),
    [gate, up] (read o's output) and [down] (reads gate's output; its output is
    the next layer's hidden state), then [lm_head]: 113 stages in order, each
    stage's fp16 output the next one's x (the products alone, with no attention,
    norm or activation between them).  "pass": bt_pass_run, the library's CUDA
    graph recorded with PDL and the constant-weights prefetch; "pass_no_pdl":
    the same recorded without PDL; "eager": one bt_qgemm_batched call per stage
    from Python, no graph (host-bound)."""
    bits = 4
    per_layer = len(QWEN06_LAYER)
    out = {"workload": "Qwen3-0.6B-shaped decode step as 113 dependent stages (28 layers x [q,k,v] [o] "
                       "[gate,up] [down] + [lm_head]), Q4 g64, fp16 x and y", "stages": 28 * 4 + 1,
           "bytes_per_pass": pass_bytes}
    n_steps = max(3, min(steps, 50))
    for m in (1, 4):
        h = torch.randn(m, 1024, device=dev).half()
        stages = []
        for layer in range(QWEN06_LAYERS):
            w = bufs[layer * per_layer:(layer + 1) * per_layer]
            ys = [torch.empty(m, qw[4].numel(), dtype=torch.float16, device=dev) for qw in w]
            q, k, v, o, gate, up, down = [(c, s_, b) for c, s_, b, *_ in w]
            yq, yk, yv, yo, yg, yu, yd = ys
            stages += [[(*q, h, yq), (*k, h, yk), (*v, h, yv)], [(*o, yq, yo)], [(*gate, yo, yg), (*up, yo, yu)],
                       [(*down, yg, yd)]]
            h = yd
        lm = bufs[-1]
        stages.append([(lm[0], lm[1], lm[2], h, torch.empty(m, lm[4].numel(), dtype=torch.float16, device=dev))])
        res = {"launches_per_pass": len(stages)}
        for tag, pdl in (("pass", 1), ("pass_no_pdl", 0)):
            bt.bt_set_option(bt.BT_OPT_PDL, pdl)
            bt.bt_set_option(bt.BT_OPT_CONST_WEIGHTS, pdl)
            try:
                dp = bt.bt_pass_create(stages, bits)
                with torch.cuda.stream(stream):
                    dp.run(stream)   # first run: direct launches, then the recording
                torch.cuda.synchronize()
            finally:
                bt.bt_set_option(bt.BT_OPT_PDL, 1)
                bt.bt_set_option(bt.BT_OPT_CONST_WEIGHTS, 1)
            with torch.cuda.stream(stream):
                t, clk = timed(torch, None, stream, lambda: dp.run(stream), n_steps, max(3, min(warmup, 5)), gpu_index)
            t /= n_steps
            gbs = pass_bytes / t / 1e9
            res[tag] = {"us_per_pass": round(t * 1e6, 2), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4),
                        "clocks": clk}
            dp.close()

        def eager():
            for st in stages:
                bt.bt_qgemm_batched(st, bits, stream=stream)
        with torch.cuda.stream(stream):
            t, _ = timed(torch, None, stream, eager, 5, 3, gpu_index)
        t /= 5
        res["eager"] = {"us_per_pass": round(t * 1e6, 2), "gbs": round(pass_bytes / t / 1e9, 1)}
        out[f"M{m}"] = res
    if bt.bt_last_device_error() != bt.BT_OK:
        raise RuntimeError("device error in the dependent-stage leg")
    return out


def interleave_rows(a, b):
    """Two [N, .] arrays -> [2N, .] with a's row i at 2i and b's at 2i+1 (gate/up pairs)."""
    return np.stack([a, b], axis=1).reshape(2 * a.shape[0], *a.shape[1:])


def run_moe(torch, bt, dev, stream, steps, warmup, gpu_index, hbm):
    """Qwen3-30B-A3B-shaped expert layer, Q4, at M = 1 (decode) and M = 128 (prefill).

    Fused layer (the timed one):
      M = 1:   bt_moe_qgemv_pairs (gate|up with the SwiGLU epilogue, experts read from
               the top-k ids, no sort) -> bt_moe_down_combine (down products with the
               gate-weighted combine in the store): 2 launches;
      M = 128: bt_moe_route -> bt_moe_qgemm_swiglu (grouped gate|up + SwiGLU) ->
               bt_moe_qgemm (grouped down) -> bt_moe_combine: 4 launches.
    The unfused layer (route, gate|up, SwiGLU, down, combine: 5 launches) is timed
    beside it.  Each timed step uses a fresh routing draw (cycled from 16 seeded
    draws) and L2 is flushed between steps (a 256 MB write outside the timed
    events), so expert weights come from HBM.  GB/s counts the packed bytes of the
    experts the step's routing touches.
    """
    bits, E, H, I, top_k = 4, 128, 2048, 768, 8
    t0 = time.time()
    g_w = gen_weights("moe-layer-gate", [(f"e{e}", I, H) for e in range(E)], bits)
    u_w = gen_weights("moe-layer-up", [(f"e{e}", I, H) for e in range(E)], bits)
    dn_w = gen_weights("moe-layer-down", [(f"e{e}", H, I) for e in range(E)], bits)
    gen_s = time.time() - t0

    def stack(arrs):
        return torch.from_numpy(np.stack(arrs)).to(dev)

    def dev_w(ws_codes, ws_s, ws_b):
        return (stack(ws_codes).view(torch.int32), stack(ws_s).view(torch.float16), stack(ws_b).view(torch.float16))
    # gate|up stored interleaved for the fused epilogue, concatenated for the unfused layer
    GUI = dev_w([interleave_rows(g.codes, u.codes) for g, u in zip(g_w, u_w)],
                [interleave_rows(g.scales, u.scales) for g, u in zip(g_w, u_w)],
                [interleave_rows(g.biases, u.biases) for g, u in zip(g_w, u_w)])
    GUC = dev_w([np.concatenate([g.codes, u.codes]) for g, u in zip(g_w, u_w)],
                [np.concatenate([g.scales, u.scales]) for g, u in zip(g_w, u_w)],
                [np.concatenate([g.biases, u.biases]) for g, u in zip(g_w, u_w)])
    DN = dev_w([w.codes for w in dn_w], [w.scales for w in dn_w], [w.biases for w in dn_w])
    per_expert = 2 * weight_bytes(I, H, bits) + weight_bytes(H, I, bits)
    del g_w, u_w, dn_w
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    out = {"workload": "Qwen3-30B-A3B-shaped MoE layer: hidden 2048, 128 experts, gate/up 2048->768, down "
                       "768->2048, top-8, Q4 g64", "weight_gen_s": round(gen_s, 1)}
    for tokens in (1, 128):
        xdt = torch.float16 if tokens == 1 else torch.bfloat16
        draws = []
        for i in range(16):
            r = synth.rng_for("moe-layer", tokens, i)
            ids, gates = synth.draw_routing(r, tokens, E, top_k)
            x = torch.randn(tokens, H, device=dev).to(xdt)
            ids_t = torch.from_numpy(ids).to(dev)
            gates_t = torch.from_numpy(gates).to(dev)
            touched = len(set(ids.reshape(-1).tolist()))
            bufs = dict(off=torch.empty(E + 1, dtype=torch.int32, device=dev),
                        pidx=torch.empty(tokens * top_k, dtype=torch.int32, device=dev),
                        prow=torch.empty(tokens * top_k, dtype=torch.int32, device=dev),
                        rowi=torch.empty(tokens * top_k, dtype=torch.int32, device=dev),
                        ygu=torch.empty(tokens * top_k, 2 * I, device=dev, dtype=xdt),
                        h=torch.empty(tokens * top_k, I, device=dev, dtype=xdt),
                        yd=torch.empty(tokens * top_k, H, device=dev, dtype=xdt),
                        out=torch.empty(tokens, H, device=dev, dtype=torch.float32))
            draws.append((ids_t, gates_t, x, bufs, touched))

        def fused(d):
            ids_t, gates_t, x, b, _ = d
            if tokens == 1:
                bt.bt_moe_qgemv_pairs(*GUI, bits, ids_t, x, b["h"], swiglu=True)
                bt.bt_moe_down_combine(*DN, bits, ids_t, gates_t, b["h"], b["out"])
            else:
                bt.bt_moe_route(ids_t, E, b["off"], b["pidx"], b["prow"], b["rowi"])
                bt.bt_moe_qgemm_swiglu(*GUI, bits, b["off"], x, b["h"], x_row_index=b["rowi"])
                bt.bt_moe_qgemm(*DN, bits, b["off"], b["h"], b["yd"])
                bt.bt_moe_combine(b["yd"], gates_t, b["prow"], top_k, b["out"])

        def unfused(d):
            ids_t, gates_t, x, b, _ = d
            bt.bt_moe_route(ids_t, E, b["off"], b["pidx"], b["prow"], b["rowi"])
            bt.bt_moe_qgemm(*GUC, bits, b["off"], x, b["ygu"], x_row_index=b["rowi"])
            bt.bt_swiglu(b["ygu"], b["h"])
            bt.bt_moe_qgemm(*DN, bits, b["off"], b["h"], b["yd"])
            bt.bt_moe_combine(b["yd"], gates_t, b["prow"], top_k, b["out"])

        res = {}
        for tag, fn, launches in (("fused", fused, 2 if tokens == 1 else 4), ("unfused", unfused, 5)):
            graphs = [capture(torch, lambda d=d: fn(d), stream) for d in draws]
            n_steps = max(3, min(steps, 100))
            times = []
            touched_bytes = 0
            with torch.cuda.stream(stream):
                for i in range(max(3, min(warmup, 5))):
                    graphs[i % len(graphs)].replay()
                torch.cuda.synchronize()
                # events made up front and no host wait inside the loop: the host
                # stays ahead of the device, so no submission gap lands between
                # the events (each step's flush keeps the device busy meanwhile)
                ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(n_steps)]
                with ClockSampler(gpu_index) as clk:
                    for i in range(n_steps):
                        flush.fill_(float(i))
                        ev[i][0].record(stream)
                        graphs[i % len(graphs)].replay()
                        ev[i][1].record(stream)
                        touched_bytes += draws[i % len(draws)][4] * per_expert
                    torch.cuda.synchronize()
                times = [e0.elapsed_time(e1) / 1e3 for e0, e1 in ev]
            t = sum(times)
            gbs = touched_bytes / t / 1e9
            flops = 2 * tokens * top_k * (2 * I * H + H * I)
            res[tag] = {"us_per_layer": round(t / n_steps * 1e6, 2),
                        "us_per_layer_median": round(float(np.median(times)) * 1e6, 2), "weight_gbs": round(gbs, 1),
                        "frac_of_hbm": round(gbs / hbm, 4), "tflops": round(flops * n_steps / t / 1e12, 3),
                        "experts_touched_mean": round(touched_bytes / n_steps / per_expert, 2),
                        "launches_per_layer": launches, "clocks": clk.summary()}
            del graphs
        out[f"M{tokens}"] = res
    if bt.bt_last_device_error() != bt.BT_OK:
        raise RuntimeError("device error in the MoE leg")
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--legs", default="decode,c1,sweep,prefill,moe,small,chain",
                    help="comma list of legs to run: decode (headline), c1 (single GEMV), sweep (bit widths), "
                         "prefill, moe, small (M = 2..16 decode pass), chain (dependent-stage pass; needs decode)")
    ap.add_argument("--no-compare", action="store_true",
                    help="skip the side measurement of the pass as 197 single-GEMV launches")
    ap.add_argument("--eager", action="store_true",
                    help="launch directly instead of replaying CUDA graphs (profiling runs only: the times then "
                         "include host launch overhead)")
    args = ap.parse_args()
    global EAGER
    EAGER = args.eager
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    shapes = decode_pass_shapes()
    bits = 4
    pass_bytes = sum(weight_bytes(n, k, bits) for _, n, k in shapes)
    config = {"workload": "Qwen3-0.6B-shaped decode pass, M=1: 28 layers x 7 projections + lm_head 1024->151936",
              "execution": "1 batched GEMV launch per pass (197 problems, mixed K) in the library's decode pass "
                           "object: bt_pass_create once, then bt_pass_run per step (a CUDA graph with PDL)",
              "bits": bits, "group_size": GROUP, "gemvs_per_pass": len(shapes), "weight_bytes_per_pass": pass_bytes,
              "x_dtype": "f16", "y_dtype": "f32",
              "l2": "inputs exceed L2 (335 MB of packed weights per pass vs 126 MB L2); no flush",
              "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}

    if args.eager:
        config["execution"] = "eager launches (--eager profiling run; times include host launch overhead)"

    if args.impl == "reference":
        if rank != 0:
            return 0
        # the oracle on every host core; the run is K bounded samples back to back
        # (each ~per_step seconds of work per core) after W untimed ones
        per_step = max(0.005, min(2.0, 90.0 / (args.steps + args.warmup)))
        val, tot, done, procs = oracle_rate("decode-pass", shapes, per_step * args.steps,
                                            warmup_s=per_step * args.warmup)
        el = tot / (val * 1e9)
        ncpu, naff = host_cores()
        sample = (f"{done} projections of the pass on {procs} spawned workers, one BLAS thread each "
                  f"(lm_head sliced to {LM_HEAD_SLICE} rows); {args.steps} steps of ~{per_step:.3f} s")
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": procs, "kind": "oracle",
                             "sample": sample, "host_cpu_count": ncpu, "affinity_cores": naff, "blas_threads": 1},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return 0

    legs = set(args.legs.split(","))
    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from dequant_gemv_gemm_bt_b300 import bt

    if "decode" not in legs:   # other legs only (profiling); no headline value
        stream = torch.cuda.Stream(device=dev)
        peaks, _ = measured_peaks()
        out = {"metric": METRIC, "value": None, "unit": "GB/s", "legs": sorted(legs)}
        if "c1" in legs:
            out["c1"] = run_c1(torch, bt, dev, stream, args.steps, args.warmup, local_rank, float(peaks["hbm_gbs"]))
        if "sweep" in legs:
            out["sweep"] = run_sweep(torch, bt, dev, stream, args.steps, args.warmup, local_rank,
                                     float(peaks["hbm_gbs"]))
        if "prefill" in legs:
            out["prefill"] = run_prefill(torch, bt, dev, stream, args.steps, args.warmup, local_rank, peaks)
        if "moe" in legs:
            out["moe"] = run_moe(torch, bt, dev, stream, args.steps, args.warmup, local_rank, float(peaks["hbm_gbs"]))
        if "small" in legs:
            out["small_batch"] = run_small(torch, bt, dev, stream, args.steps, args.warmup, local_rank,
                                           float(peaks["hbm_gbs"]))
        if rank == 0:
            print(json.dumps(out))
        return 0

    # CPU baseline first (rank 0, single GPU only), before any GPU work: the
    # oracle on every host core (spawned workers, one BLAS thread each)
    cpu_baseline = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        rate, nbytes, cnt, procs = oracle_rate("decode-pass", shapes, args.cpu_budget)
        ncpu, naff = host_cores()
        cpu_baseline = {"value": round(rate, 4), "unit": "GB/s", "cores": procs, "kind": "oracle",
                        "host_cpu_count": ncpu, "affinity_cores": naff, "blas_threads": 1,
                        "sample": f"{cnt} projections of the pass ({nbytes/1e6:.1f} MB of packed weights, lm_head "
                                  f"sliced to {LM_HEAD_SLICE} rows), fp64 numpy, {procs} spawned workers, "
                                  f"~{args.cpu_budget:.0f} s"}
    weights = gen_weights("decode-pass", shapes, bits)
    xs16 = gen_x("decode-pass", shapes, 1, "f16")

    bufs = build_decode_pass(torch, bt, weights, xs16, dev)
    del weights
    bt.bt_set_option(bt.BT_OPT_PDL, 1)
    bt.bt_set_option(bt.BT_OPT_CONST_WEIGHTS, 1)

    # The pass's projections are independent (each has its own x), so the whole
    # pass is one stage: one mixed-K batched launch (K = 1024, 2048, 3072), in
    # pass order, planned once by bt_pass_create and replayed by the library as
    # a CUDA graph (bt_pass_run).
    groups = [[(c, s, b, x, y) for c, s, b, x, y, _ in bufs]]

    def run_pass():
        for g in groups:
            bt.bt_qgemv_batched(g, bits)

    def as_rows(g):
        return [(c, s, b, x.view(1, -1), y.view(1, -1)) for c, s, b, x, y in g]

    def run_pass_single():
        for c, s, b, x, y, nb in bufs:
            bt.bt_qgemv(c, s, b, nb, x, y)

    stream = torch.cuda.Stream(device=dev)
    if EAGER:
        graph = capture(torch, run_pass, stream)
        replay = graph.replay
    else:
        dpass = bt.bt_pass_create([as_rows(g) for g in groups], bits)
        with torch.cuda.stream(stream):
            dpass.run(stream)   # the first run launches directly and records the graph
        torch.cuda.synchronize()

        def replay():
            dpass.run(stream)
    graph_single = None if args.no_compare else capture(torch, run_pass_single, stream)
    if bt.bt_last_device_error() != bt.BT_OK:
        raise RuntimeError("device error during capture")

    with torch.cuda.stream(stream):
        t_pass, clocks = timed(torch, dist, stream, replay, args.steps, args.warmup, local_rank)
        if graph_single is not None:
            t_single, _ = timed(torch, None, stream, lambda: graph_single.replay(), max(3, args.steps // 4), 3,
                                local_rank)
    single_gbs = pass_bytes * max(3, args.steps // 4) / t_single / 1e9 if graph_single is not None else None
    t_pass = max_over_ranks(torch, dist, t_pass, dev)
    if bt.bt_last_device_error() != bt.BT_OK:
        raise RuntimeError("device error during the timed region")
    sec_per_step = t_pass / args.steps
    value = whole_job_rate(pass_bytes, args.steps, world, t_pass) / 1e9

    # lm_head alone (the largest single GEMV), for context
    lm = bufs[-1]
    lm_bytes = weight_bytes(QWEN06_LM_HEAD[1], QWEN06_LM_HEAD[2], bits)
    g_lm = capture(torch, lambda: [bt.bt_qgemv(lm[0], lm[1], lm[2], lm[5], lm[3], lm[4]) for _ in range(20)], stream)
    with torch.cuda.stream(stream):
        t_lm, _ = timed(torch, None, stream, lambda: g_lm.replay(), 20, 3, local_rank)
    lm_gbs = lm_bytes * 20 * 20 / t_lm / 1e9

    # end to end through the public API: H2D of the pass's activations from pinned
    # host memory, the pass, D2H of every output, each step
    x_host = torch.cat([x for _, _, _, x, _, _ in bufs]).cpu().pin_memory()
    y_total = sum(y.numel() for *_, y, _ in bufs)
    y_host = torch.empty(y_total, dtype=torch.float32).pin_memory()
    x_dev_views, off = [], 0
    x_all = torch.empty_like(x_host, device=dev)
    for c, s, b, x, y, nb in bufs:
        x_dev_views.append(x_all[off:off + x.numel()])
        off += x.numel()
    y_all = torch.empty(y_total, dtype=torch.float32, device=dev)
    y_views, off = [], 0
    for *_, y, _ in bufs:
        y_views.append(y_all[off:off + y.numel()])
        off += y.numel()

    e2e_groups = [[(bufs[i][0], bufs[i][1], bufs[i][2], x_dev_views[i], y_views[i]) for i in range(len(bufs))]]

    def run_pass_e2e():
        for g in e2e_groups:
            bt.bt_qgemv_batched(g, bits)
    if EAGER:
        e2e_run = capture(torch, run_pass_e2e, stream).replay
    else:
        e2e_pass = bt.bt_pass_create([as_rows(g) for g in e2e_groups], bits)
        with torch.cuda.stream(stream):
            e2e_pass.run(stream)
        torch.cuda.synchronize()

        def e2e_run():
            e2e_pass.run(stream)

    def e2e_step():
        x_all.copy_(x_host, non_blocking=True)
        e2e_run()
        y_host.copy_(y_all, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 200))
    with torch.cuda.stream(stream):
        t_e2e, _ = timed(torch, dist, stream, e2e_step, e2e_steps, 3, local_rank)
    t_e2e = max_over_ranks(torch, dist, t_e2e, dev)
    e2e_val = whole_job_rate(pass_bytes, e2e_steps, world, t_e2e) / 1e9

    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    launches = len(groups)
    achieved = (pass_bytes / launches) / (sec_per_step / launches) / 1e9
    digest = source_digest(["dequant_gemv_gemm_bt_b300/csrc/qgemv*", "dequant_gemv_gemm_bt_b300/csrc/bt_common.cuh"])
    traffic = profile_traffic("qgemv_decode_pass.json", digest)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sec_per_step * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u4 codes, f16 x, f32 accumulate",
        "data": "synthetic (seeded N(0,0.02) weights, min/max Q4 g64; x ~ N(0,1) fp16)",
        "config": config,
        "roofline": {"bound": "hbm", "kernel": gemv_kernel_name(bt, bits),
                     "achieved": round(achieved, 2), "peak": hbm, "peak_kind": f"{peak_kind} HBM copy GB/s",
                     "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": traffic, "kernel_source_digest": digest},
        "cpu_baseline": cpu_baseline,
        "clocks": clocks,
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": int(x_host.numel() * 2),
                "d2h_bytes_per_step": int(y_total * 4),
                "how": "per step: pinned H2D of all 197 activation vectors, the pass (bt_pass_run: the "
                       "library's CUDA graph of 1 batched GEMV launch), D2H of all outputs"},
        "gpu_launches": launches * args.steps,
        "per_gemv_graph": {"gbs": round(single_gbs, 2) if single_gbs else None, "launches_per_pass": len(bufs),
                           "how": "the same pass as 197 bt_qgemv launches in one CUDA graph with PDL"},
        "lm_head_gemv": {"gbs": round(lm_gbs, 1), "frac_of_hbm": round(lm_gbs / hbm, 4),
                         "shape": "N=151936 K=1024 Q4", "bytes": lm_bytes},
    }
    if "c1" in legs:
        out["c1"] = run_c1(torch, bt, dev, stream, args.steps, args.warmup, local_rank, hbm)
    if "sweep" in legs:
        out["sweep"] = run_sweep(torch, bt, dev, stream, args.steps, args.warmup, local_rank, hbm)
    if "prefill" in legs:
        out["prefill"] = run_prefill(torch, bt, dev, stream, args.steps, args.warmup, local_rank, peaks)
    if "moe" in legs:
        out["moe"] = run_moe(torch, bt, dev, stream, args.steps, args.warmup, local_rank, hbm)
    if "small" in legs:
        out["small_batch"] = run_small(torch, bt, dev, stream, args.steps, args.warmup, local_rank, hbm)
    if "chain" in legs:
        out["dependent_pass"] = run_chain(torch, bt, bufs, dev, stream, args.steps, args.warmup, local_rank, hbm,
                                          pass_bytes)
    if rank == 0:
        print(json.dumps(out))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
