"""Benchmark: W4/W8 lm_head logits (+ top-8, + exact rescoring) on one GB300.

One step = one pass of the hot path over the 151936 x 1024 W4-g64 head
("Fused WNA16 GEMM for tied quantized lm_head logits", Perf evals table):
for each M in (1, 32, 256), wql_logits with top-8 candidates followed by
wql_topk_rescore of those candidates from the fp16 reference rows.
Quantisation (load time) is timed once, outside the steps.

Timing: each step is a CUDA-graph replay of its calls (captured once per
phase of the copy rotation), bracketed by CUDA events on the launching
stream, so the host's per-call launch work is not on the device timeline.
Every call reads one of four copies of the quantised weight in turn, so the
copy it reads was not touched by the three calls before it (3 x 83 MB > the
129 MB L2): weights always come from HBM.  `value` is the algorithmic bytes
of the step (packed weight + scales + X + logits written + top-K + rescored
rows) over the summed device time.  `e2e` runs the same step as eager calls
of the public API with X copied in from pinned host memory and the outputs
copied back every step.  `--gpus N`
under torchrun runs N independent replicas (the head is replicated, not
sharded) and reports the units of all ranks over the slowest rank's time.

The same line carries a `configs` block: every head of the metric at each
token count it is quoted at -- the 50304 x 512 W4-g64 head (L2-resident),
the 151936 x 1024 W4-g64 and W8-g128 heads at M = 1/32/256, the 248320 x
5120 int4-g128 MSE head at M = 1..5 and 16, and the int8 per-row head with
top-8 rescoring and its greedy-token agreement counts -- each call's median
and 10th-percentile device time over 120 calls, with its own clock record;
and `roofline_decode_m1`, the decode kernel alone at M = 1 with top-K off.

`--impl reference` times the CPU oracle (the slow binary64 C restatement) on
a bounded row sample of the same workload and prints the same JSON line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import math
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

N_VOCAB, K_HIDDEN, GROUP, TOPK = 151936, 1024, 64, 8
MS = (1, 32, 256)
WORKLOAD = "lm_head 151936x1024 W4-g64 RTN fp16-scale, X fp16 at M=1/32/256, top-8 + rescore"
METRIC = "HBM GB/s and us/call of W4/W8 lm_head logits at M=1/32/256 (% of roofline)"
N_COPIES = 4          # rotating weight copies: inputs larger than L2 between reuses


# ---------------------------------------------------------------------------
# byte / flop accounting (what the method itself must move)
# ---------------------------------------------------------------------------

def logits_bytes(m: int, n: int, k: int, bits: int, group: int, out_bytes: int = 2,
                 x_bytes: int = 2, scale_bytes: int = 2, topk: int = 0) -> int:
    """Packed weight + scale table + X read + logits written (+ top-K out)."""
    g = k if group == 0 else group
    w = n * k * bits // 8
    s = n * (k // g) * scale_bytes
    return w + s + m * k * x_bytes + m * n * out_bytes + m * topk * 8


def rescore_bytes(m: int, k: int, topk: int, w_bytes: int = 2, x_bytes: int = 2) -> int:
    """The K reference rows read per token row (+ x, + values written back)."""
    return m * topk * k * w_bytes + m * k * x_bytes + m * topk * (8 + 2)


def step_bytes(ms=MS) -> int:
    return sum(logits_bytes(m, N_VOCAB, K_HIDDEN, 4, GROUP, topk=TOPK) +
               rescore_bytes(m, K_HIDDEN, TOPK) for m in ms)


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_src_hash(names) -> str:
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "weight_only_quantized_wql_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, src_hash: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    this exact kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        if line.startswith("#") or "=" not in line:
            continue
        kv = dict(tok.split("=", 1) for tok in line.split())
        if kv.get("kernel") == kernel and kv.get("workload") == workload and \
                kv.get("src") == src_hash:
            return int(kv["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"wql_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, rank: int, world: int, local_rank: int) -> dict | None:
    import torch
    import weight_only_quantized_wql_gb300 as wql

    MS = tuple(args.ms)   # noqa: N806  (token counts timed in this run)
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wql.load()
    stream = torch.cuda.current_stream(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    w = torch.randn(N_VOCAB, K_HIDDEN, generator=gen, device=dev).mul_(0.02)
    w_ref = w.half()
    xs = {}
    for m in MS:
        g2 = torch.Generator(device=dev)
        g2.manual_seed(1000 + m)
        xs[m] = torch.randn(m, K_HIDDEN, generator=g2, device=dev).half()
    # load-time quantisation, timed once
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    qw = wql.wql_quantize(w, 4, GROUP, torch.float16, wql.CLIP_RTN)
    e1.record(stream)
    torch.cuda.synchronize()
    quant_ms = e0.elapsed_time(e1)
    del w
    # the weights are written once, before any timed call: static (the decode
    # kernel may start copying them before the preceding kernel ends)
    qw.static = True
    copies = [qw] + [wql.QuantizedWeight(qw.qweight.clone(), qw.scales.clone(), qw.bits,
                                         qw.group, qw.n, qw.k, static=True)
                     for _ in range(N_COPIES - 1)]
    ws = wql.Workspace(dev)
    outs = {m: torch.empty(m, N_VOCAB, dtype=torch.float16, device=dev) for m in MS}
    idx = {m: torch.empty(m, TOPK, dtype=torch.int32, device=dev) for m in MS}
    val = {m: torch.empty(m, TOPK, dtype=torch.float32, device=dev) for m in MS}
    counter = [0]

    def call(m):
        c = copies[counter[0] % N_COPIES]
        counter[0] += 1
        wql.wql_logits(xs[m], c, topk=TOPK, workspace=ws, out=outs[m], topk_idx=idx[m],
                       topk_val=val[m])

    def rescore(m):
        wql.wql_topk_rescore(xs[m], w_ref, idx[m], val[m], outs[m])

    def one_step():
        for m in MS:
            call(m)
            rescore(m)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # Warm-up, eager: sizes the workspace and loads every kernel before capture.
    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()

    # The device-timed step is a CUDA graph replay: one graph per phase of the
    # weight-copy rotation, so replay s reads exactly the copies an eager step
    # s would.  The host's per-call launch work (ctypes marshalling, tensor-map
    # encoding) then stays off the device timeline; the e2e leg below keeps it.
    cap = torch.cuda.Stream(dev)
    nph = N_COPIES // math.gcd(N_COPIES, len(MS))     # steps until the rotation repeats

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                fn()
        stream.wait_stream(cap)
        return g

    graphs = []
    n0 = wql.wql_launch_count()
    for ph in range(nph):
        counter[0] = ph * len(MS)
        graphs.append(capture(one_step))
    launches_per_step = (wql.wql_launch_count() - n0) // nph
    for i in range(max(args.warmup, nph)):
        graphs[i % nph].replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local_rank)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_wall0 = time.perf_counter()
    for st in range(args.steps):
        evs[st][0].record(stream)
        graphs[st % nph].replay()
        evs[st][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    launches = launches_per_step * args.steps
    barrier()
    clk = clocks.stop()
    step_us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    dev_s = sum(step_us) * 1e-6

    # ---- per-call breakdown: graphs of R calls of one kind, rotating copies ----
    R = 20

    def time_graph(g, reps=3):
        g.replay()
        torch.cuda.synchronize()
        per = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            per.append(a.elapsed_time(b) * 1e3 / R)
        return sorted(per)

    def logits_calls(m, topk):
        def fn():
            for r in range(R):
                if topk:
                    wql.wql_logits(xs[m], copies[r % N_COPIES], topk=topk, workspace=ws,
                                   out=outs[m], topk_idx=idx[m], topk_val=val[m])
                else:
                    wql.wql_logits(xs[m], copies[r % N_COPIES], topk=0, workspace=ws,
                                   out=outs[m])
        return fn

    def rescore_calls(m):
        def fn():
            for _ in range(R):
                rescore(m)
        return fn

    logit_us = {m: time_graph(capture(logits_calls(m, TOPK))) for m in MS}
    resc_us = {m: time_graph(capture(rescore_calls(m))) for m in MS}

    # the same calls on one weight copy only: after the first call the 83 MB
    # head stays in the 129 MB L2 (L2-resident, not HBM; context only)
    def hot_calls(m):
        def fn():
            for _ in range(R):
                wql.wql_logits(xs[m], copies[0], topk=TOPK, workspace=ws, out=outs[m],
                               topk_idx=idx[m], topk_val=val[m])
        return fn

    hot_us = {m: time_graph(capture(hot_calls(m))) for m in MS}

    # ---- end to end: pinned host X in, logits + top-K out, every call ----
    hx = {m: xs[m].cpu().pin_memory() for m in MS}
    hout = {m: torch.empty(m, N_VOCAB, dtype=torch.float16).pin_memory() for m in MS}
    hidx = {m: torch.empty(m, TOPK, dtype=torch.int32).pin_memory() for m in MS}
    hval = {m: torch.empty(m, TOPK, dtype=torch.float32).pin_memory() for m in MS}
    dx = {m: torch.empty_like(xs[m]) for m in MS}
    h2d = sum(hx[m].numel() * 2 for m in MS)
    d2h = sum(hout[m].numel() * 2 + hidx[m].numel() * 4 + hval[m].numel() * 4 for m in MS)
    e2e_events = []
    for it in range(args.warmup + args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for m in MS:
            dx[m].copy_(hx[m], non_blocking=True)
            c = copies[counter[0] % N_COPIES]
            counter[0] += 1
            wql.wql_logits(dx[m], c, topk=TOPK, workspace=ws, out=outs[m], topk_idx=idx[m],
                           topk_val=val[m])
            wql.wql_topk_rescore(dx[m], w_ref, idx[m], val[m], outs[m])
            hout[m].copy_(outs[m], non_blocking=True)
            hidx[m].copy_(idx[m], non_blocking=True)
            hval[m].copy_(val[m], non_blocking=True)
        b.record(stream)
        if it >= args.warmup:
            e2e_events.append((a, b))
    torch.cuda.synchronize()
    e2e_us = [a.elapsed_time(b) * 1e3 for a, b in e2e_events]
    assert ws.error_word() == 0, "a kernel's bounded wait timed out"

    # ---- the dominant kernel alone: the logits call with the largest share
    # of device time, with top-K off, which is one launch of its logits kernel
    # per call (decode_kernel for M <= 16, tc_logits_kernel above) ----
    dom_m = max(MS, key=lambda m: statistics.median(logit_us[m]))
    n0 = wql.wql_launch_count()
    g_dom = capture(logits_calls(dom_m, 0))
    assert wql.wql_launch_count() - n0 == R, "one launch per call expected"
    kern_us = time_graph(g_dom, reps=max(3, args.steps // 4))

    # ---- reduce over ranks: the slowest rank's times ----
    dev_s, e2e_s, t_wall = aggregate_over_ranks([dev_s, sum(e2e_us) * 1e-6, t_wall], world,
                                                device=dev)
    if rank != 0:
        return None

    pk = peaks()
    configs = None if args.no_configs else run_configs(dev, stream, pk)
    value = job_throughput_gbs(step_bytes(MS), args.steps, world, dev_s)
    med = {m: statistics.median(logit_us[m]) for m in MS}   # each entry: mean of R calls
    calls = {}
    for m in MS:
        b = logits_bytes(m, N_VOCAB, K_HIDDEN, 4, GROUP, topk=TOPK)
        fl = 2.0 * m * N_VOCAB * K_HIDDEN
        gbs = b / (med[m] * 1e-6) / 1e9
        tfl = fl / (med[m] * 1e-6) / 1e12
        calls[f"M{m}"] = {
            "us_median": round(med[m], 2),
            "us_min": round(min(logit_us[m]), 2),
            "GBps": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 3),
            "TFLOPs": round(tfl, 2), "frac_tensor": round(tfl / pk["bf16_tflops"], 4),
            "rescore_us": round(statistics.median(resc_us[m]), 2),
            "us_l2_resident": round(statistics.median(hot_us[m]), 2)}
    # dominant kernel, timed alone above (mean launch duration)
    dom_us = statistics.median(kern_us)
    dom_flops = 2.0 * dom_m * N_VOCAB * K_HIDDEN
    dom_bytes = logits_bytes(dom_m, N_VOCAB, K_HIDDEN, 4, GROUP, topk=0)
    kern = "tc_logits_kernel" if dom_m > 16 else "decode_kernel"
    src = kernel_src_hash(["tc_gemm.cu", "wql_common.cuh", "sm100.cuh"] if dom_m > 16 else
                          ["decode_impl.cuh", "decode.cu", "wql_common.cuh", "sm100.cuh"])
    traffic = recorded_traffic(kern, f"M{dom_m}", src)
    if dom_flops / dom_bytes > 286 and dom_m > 16:
        achieved = dom_flops / (dom_us * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2),
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / pk["bf16_tflops"], 4), "traffic": traffic,
                "kernel": kern, "call": f"M={dom_m}, top-K off", "launch_us": round(dom_us, 2),
                "peak_note": f"{pk['source']} bf16 burst; fp16 dense rate is the same"}
        if pk.get("bf16_tflops_sustained"):
            roof["frac_of_sustained"] = round(achieved / pk["bf16_tflops_sustained"], 4)
    else:
        achieved = dom_bytes / (dom_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": traffic,
                "kernel": kern, "call": f"M={dom_m}, top-K off", "launch_us": round(dom_us, 2),
                "peak_note": f"{pk['source']} copy"}
    # the decode kernel at M = 1 with top-K off: one launch per call, so the
    # per-call time of the W4 head is that kernel's launch duration
    roof_m1 = None
    if configs is not None:
        c = configs["C2"]["calls"]["M1_top0"]
        src_d = kernel_src_hash(["decode_impl.cuh", "decode.cu", "wql_common.cuh", "sm100.cuh"])
        roof_m1 = {"bound": "hbm", "achieved": c["GBps"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                   "frac": round(c["GBps"] / pk["hbm_gbs"], 4),
                   "frac_of_spec": round(c["GBps"] / SPEC_HBM_GBS, 4),
                   "traffic": recorded_traffic("decode_kernel", "M1", src_d),
                   "kernel": "decode_kernel", "call": "151936x1024 W4-g64, M=1, top-K off",
                   "launch_us_median": c["us_median"], "launch_us_p10": c["us_p10"],
                   "algorithmic_bytes": c["bytes"],
                   "peak_note": f"{pk['source']} copy; spec {SPEC_HBM_GBS:.0f} GB/s"}
    return {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dev_s / args.steps * 1e3 / 1.0, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4 x f16 products, f32 accumulate", "data": "synthetic",
        "config": {"workload": WORKLOAD, "n": N_VOCAB, "k": K_HIDDEN, "group": GROUP,
                   "ms": list(MS), "topk": TOPK, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {N_COPIES} rotating weight copies "
                         f"({N_COPIES * 83} MB), each call reads a copy untouched for 3 calls",
                   "step_bytes": step_bytes(MS),
                   "timing": "device: CUDA-graph replay of each step (one graph per phase of "
                             "the copy rotation), events around each replay; calls and "
                             "roofline: graphs of 20 calls; e2e: eager public-API calls"},
        "calls": calls, "quantize_ms": round(quant_ms, 3),
        "roofline": roof,
        "roofline_decode_m1": roof_m1,
        "configs": configs,
        "cpu_baseline": None,
        "e2e": {"value": round(job_throughput_gbs(step_bytes(MS), args.steps, world, e2e_s), 1),
                "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "wall_s_timed": round(t_wall, 4),
        "clocks": clk,
    }


# ---------------------------------------------------------------------------
# Every workload of the metric: per-call times of each head and token count
# ---------------------------------------------------------------------------

SPEC_HBM_GBS = 8000.0     # GB300 HBM3e nominal rate (context beside the measured copy rate)


def call_stats(per_call_us: list[float]) -> dict:
    """Median and 10th percentile of the per-call samples."""
    v = sorted(per_call_us)
    p10 = v[max(0, int(math.floor(0.1 * (len(v) - 1))))]
    return {"us_median": round(statistics.median(v), 2), "us_p10": round(p10, 2)}


def run_configs(dev, stream, pk: dict, calls_per_sample: int = 12, samples: int = 10) -> dict:
    """Each head of the metric at each token count it is quoted at: device
    time per wql_logits call (top-K off and top-8), as CUDA-graph replays of
    `calls_per_sample` consecutive calls that rotate over weight copies, so
    every call but the small head's reads its weights from HBM.  Each sample
    is one replay's mean per call; `samples` replays give median and p10
    over samples x calls_per_sample calls."""
    import torch
    import weight_only_quantized_wql_gb300 as wql
    from weight_only_quantized_wql_gb300 import synth

    R = calls_per_sample
    cap = torch.cuda.Stream(dev)
    ws = wql.Workspace(dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                fn()
        stream.wait_stream(cap)
        return g

    def time_calls(x, copies, topk, n):
        out = torch.empty(x.shape[0], n, dtype=x.dtype, device=dev)
        idx = torch.empty(x.shape[0], max(topk, 1), dtype=torch.int32, device=dev)
        val = torch.empty(x.shape[0], max(topk, 1), dtype=torch.float32, device=dev)

        def fn():
            for r in range(R):
                c = copies[r % len(copies)]
                if topk:
                    wql.wql_logits(x, c, topk=topk, workspace=ws, out=out, topk_idx=idx,
                                   topk_val=val)
                else:
                    wql.wql_logits(x, c, topk=0, workspace=ws, out=out)
        fn()
        torch.cuda.synchronize()
        g = capture(fn)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        per = []
        for _ in range(samples):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            per.append(a.elapsed_time(b) * 1e3 / R)
        del g
        return per

    def entry(wl, m, topk, copies, x, bits, group, wbytes):
        st = call_stats(time_calls(x, copies, topk, wl.n))
        # the weight as stored (codes, scales, zero points) + X + logits + top-K
        b = wbytes + m * wl.k * 2 + m * wl.n * 2 + m * topk * 8
        gbs = b / (st["us_median"] * 1e-6) / 1e9
        e = dict(st, n_calls=R * samples, bytes=b, GBps=round(gbs, 1),
                 frac_hbm=round(gbs / pk["hbm_gbs"], 3),
                 frac_hbm_spec=round(gbs / SPEC_HBM_GBS, 3))
        if m >= 32:
            tfl = 2.0 * m * wl.n * wl.k / (st["us_median"] * 1e-6) / 1e12
            e.update(TFLOPs=round(tfl, 1), frac_tensor=round(tfl / pk["bf16_tflops"], 3))
        return e

    def make_head(wl, ncopies, fmt, bits, group, clip):
        w = synth.weight(wl.n, wl.k, wl.w_dtype, seed=wl.w_seed, device=dev)
        sdt = torch.float16 if wl.scale_dtype == synth.F16 else torch.bfloat16
        wql.wql_quantize(w[:256], bits, group, sdt, clip, fmt=fmt)   # load the kernel
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        qw = wql.wql_quantize(w, bits, group, sdt, clip, fmt=fmt)
        b.record(stream)
        torch.cuda.synchronize()
        qms = a.elapsed_time(b)
        qw.static = True          # written once, before any timed call
        copies = [qw] + [wql.QuantizedWeight(
            qw.qweight.clone(), qw.scales.clone(), qw.bits, qw.group, qw.n, qw.k, qw.fmt,
            qw.zeros.clone() if qw.zeros is not None else None, True)
            for _ in range(ncopies - 1)]
        return w, copies, qms

    def head_block(key, ncopies, topks, label, fmt=wql.FMT_SYM, bits=None, group=None,
                   ms=None):
        wl = synth.WORKLOADS[key]
        bits = wl.bits if bits is None else bits
        group = wl.group if group is None else group
        clip = wl.clip if fmt == wql.FMT_SYM else wql.CLIP_RTN
        w, copies, qms = make_head(wl, ncopies, fmt, bits, group, clip)
        del w
        wbytes = copies[0].nbytes()
        blk = {"workload": key, "n": wl.n, "k": wl.k, "bits": bits,
               "group": group or "row", "clip": "mse" if clip else "rtn",
               "format": {wql.FMT_SYM: "symmetric", wql.FMT_E4M3: "fp8 e4m3",
                          wql.FMT_ASYM: "int4 with zero points"}[fmt],
               "weight_copies": ncopies, "weight_bytes": wbytes, "quantize_ms": round(qms, 2),
               "l2": label, "calls": {}}
        for m in (wl.ms if ms is None else ms):
            x = synth.activations(m, wl.k, wl.x_dtype, seed=1000 + m, device=dev)
            for topk in topks(m):
                blk["calls"][f"M{m}_top{topk}"] = entry(wl, m, topk, copies, x, bits, group,
                                                        wbytes)
        del copies
        torch.cuda.empty_cache()
        return blk

    hbm = "inputs larger than L2: rotating weight copies, each call reads a copy that " \
          "the call before it did not"
    res = {"timing": f"CUDA-graph replays of {R} consecutive calls; each sample one replay's "
                     f"mean per call; median and p10 over {samples} samples "
                     f"({R * samples} calls)",
           "peak_hbm_gbs": pk["hbm_gbs"], "spec_hbm_gbs": SPEC_HBM_GBS}
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    res["C1"] = head_block("pr_fixture_50304x512_w4g64", 1, lambda m: (0, 8),
                           "L2-resident: the 12.9 MB head stays in the 129 MB L2 between calls")
    res["C2"] = head_block("qwen_151936x1024_w4g64", 4, lambda m: (0, 8), hbm)
    res["C3"] = head_block("qwen_151936x1024_w8g128", 2, lambda m: (0, 8), hbm)
    res["C5"] = head_block("head_248320x5120_w4g128_mse", 2,
                           lambda m: (0, 8) if m == 1 else (8,), hbm)
    res["C5_fp8"] = head_block("head_248320x5120_w4g128_mse", 2, lambda m: (0, 8), hbm,
                               fmt=wql.FMT_E4M3, bits=8, group=0, ms=(1, 16))
    res["C2_asym"] = head_block("qwen_151936x1024_w4g64", 4, lambda m: (0, 8), hbm,
                                fmt=wql.FMT_ASYM, bits=4, group=128, ms=(1, 16))
    res["C4"] = argmax_study(dev)
    res["clocks"] = clocks.stop()
    return res


# ---------------------------------------------------------------------------
# Argmax study: int8 per-row head, M = 1 rows, top-8 rescoring
# ---------------------------------------------------------------------------

def run_argmax_study(args) -> dict:
    import torch
    return argmax_study(torch.device("cuda", 0))


def argmax_study(dev) -> dict:
    """The 151936 x 2048 int8 per-row head with an fp16 reference weight
    ("Fused WNA16 GEMM for tied quantized lm_head logits", reviewer comment
    items 1-2): 4096 seeded rows, each an M = 1 wql_logits call with top-8
    followed by wql_topk_rescore from the fp16 rows.  Reports how often the
    greedy token agrees with the fp16 reference -- the argmax of x . W_fp16
    computed with exact products and fp32 accumulation (torch matmul of the
    widened operands) -- for the int8 logits alone and after rescoring, the
    rows whose reference top-1/top-2 margin is below 2^-10 * sum|x w| (near
    ties no weight precision decides), and the device time per call.  The
    pages' own agreement rates come from captured decode states that are not
    available here; synthetic rows have no comparable argmax structure."""
    import torch
    import weight_only_quantized_wql_gb300 as wql
    from weight_only_quantized_wql_gb300 import synth

    wl = synth.WORKLOADS["qwen_151936x2048_w8row_rescore"]
    torch.cuda.set_device(dev)
    wql.load()
    stream = torch.cuda.current_stream(dev)
    w_ref = synth.weight(wl.n, wl.k, wl.w_dtype, seed=wl.w_seed, device=dev)    # fp16
    qw = wql.wql_quantize(w_ref, wl.bits, wl.group, torch.float16, wl.clip)
    qw.static = True              # written once, before any timed call
    xs = synth.activations(wl.rows, wl.k, wl.x_dtype, seed=wl.x_seed, device=dev)
    # fp16 reference: exact products, fp32 accumulation; the near-tie scale
    # sum|x w| from the absolute values
    ref_top = torch.empty(wl.rows, 2, dtype=torch.int64, device=dev)
    near = torch.empty(wl.rows, dtype=torch.bool, device=dev)
    wf = w_ref.float()
    for r0 in range(0, wl.rows, 256):
        xf = xs[r0:r0 + 256].float()
        lg = xf @ wf.t()
        v2, i2 = lg.topk(2, dim=1)
        ref_top[r0:r0 + 256] = i2
        absw = (xf.abs() @ wf.abs().t()).gather(1, i2[:, :1]).squeeze(1)
        near[r0:r0 + 256] = (v2[:, 0] - v2[:, 1]) < absw * 2.0 ** -10
        del lg
    del wf
    B = 16                                    # rows per captured graph replay
    xbuf = torch.empty(B, wl.k, dtype=torch.float16, device=dev)
    lbuf = torch.empty(B, wl.n, dtype=torch.float16, device=dev)
    ibuf = torch.empty(B, wl.rescore_k, dtype=torch.int32, device=dev)
    vbuf = torch.empty(B, wl.rescore_k, dtype=torch.float32, device=dev)
    ws = wql.Workspace(dev)

    def rows_fn(rescore):
        def fn():
            for i in range(B):
                wql.wql_logits(xbuf[i:i + 1], qw, topk=wl.rescore_k, workspace=ws,
                               out=lbuf[i:i + 1], topk_idx=ibuf[i:i + 1],
                               topk_val=vbuf[i:i + 1])
                if rescore:
                    wql.wql_topk_rescore(xbuf[i:i + 1], w_ref, ibuf[i:i + 1],
                                         vbuf[i:i + 1], lbuf[i:i + 1])
        return fn

    xbuf.copy_(xs[:B])
    for _ in range(3):
        rows_fn(True)()
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(dev)
    graphs = {}
    for resc in (False, True):
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                rows_fn(resc)()
        stream.wait_stream(cap)
        graphs[resc] = g
    top1 = {False: torch.empty(wl.rows, dtype=torch.int64, device=dev),
            True: torch.empty(wl.rows, dtype=torch.int64, device=dev)}
    dev_us = {False: 0.0, True: 0.0}
    for resc in (False, True):
        for r0 in range(0, wl.rows, B):
            xbuf.copy_(xs[r0:r0 + B])
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graphs[resc].replay()
            b.record(stream)
            # the greedy token of each row: the top candidate of the int8
            # logits (fp32 values), or after rescoring the argmax over the
            # whole scattered row
            top1[resc][r0:r0 + B] = (lbuf.float().argmax(dim=1) if resc
                                     else ibuf[:, 0].long())
            torch.cuda.synchronize()
            dev_us[resc] += a.elapsed_time(b) * 1e3
    assert ws.error_word() == 0, "a kernel's bounded wait timed out"
    ref1 = ref_top[:, 0]
    agree = {resc: int((top1[resc] == ref1).sum()) for resc in (False, True)}
    n_near = int(near.sum())
    far = ~near
    agree_far = {resc: int(((top1[resc] == ref1) & far).sum()) for resc in (False, True)}
    per_call = dev_us[False] / wl.rows
    per_pair = dev_us[True] / wl.rows
    b_logits = logits_bytes(1, wl.n, wl.k, 8, 0, topk=wl.rescore_k)
    b_pair = b_logits + rescore_bytes(1, wl.k, wl.rescore_k)
    pk = peaks()
    return {
        "study": "argmax agreement, int8 per-row lm_head 151936x2048 + top-8 rescore from "
                 "fp16 rows, 4096 seeded M=1 rows",
        "data": "synthetic",
        "rows": wl.rows,
        "agree_int8": agree[False], "agree_rescored": agree[True],
        "agree_int8_frac": round(agree[False] / wl.rows, 5),
        "agree_rescored_frac": round(agree[True] / wl.rows, 5),
        "near_tie_rows": n_near,
        "agree_int8_excl_near_ties": agree_far[False],
        "agree_rescored_excl_near_ties": agree_far[True],
        "rows_excl_near_ties": wl.rows - n_near,
        "us_per_call_logits_top8": round(per_call, 2),
        "GBps_logits_top8": round(b_logits / (per_call * 1e-6) / 1e9, 1),
        "frac_hbm_logits_top8": round(b_logits / (per_call * 1e-6) / 1e9 / pk["hbm_gbs"], 3),
        "us_per_call_with_rescore": round(per_pair, 2),
        "GBps_with_rescore": round(b_pair / (per_pair * 1e-6) / 1e9, 1),
        "timing": "device: CUDA-graph replays of 16 consecutive rows (one call pair per "
                  "row), events around each replay",
        "reference": "argmax of x . W_fp16 with exact products and fp32 accumulation",
    }


def run_embed_study(args) -> dict:
    """Tied-embedding gather from the 151936 x 1024 W4-g64 head ("Fused
    WNA16 GEMM for tied quantized lm_head logits", Purpose): t seeded token
    ids -> [t, 1024] fp16 rows.  Bytes per call: the ids, each id's packed
    row and scale row, and the fp16 output; CUDA-graph replays of 20 calls,
    events around each replay."""
    import torch
    import weight_only_quantized_wql_gb300 as wql

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wql.load()
    stream = torch.cuda.current_stream(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    w = torch.randn(N_VOCAB, K_HIDDEN, generator=gen, device=dev).mul_(0.02)
    qw = wql.wql_quantize(w, 4, GROUP, torch.float16, wql.CLIP_RTN)
    del w
    R = 20
    pk = peaks()
    res = {"study": "tied-embedding gather, lm_head 151936x1024 W4-g64 fp16 scales -> fp16 "
                    "rows", "data": "synthetic", "calls": {}}
    cap = torch.cuda.Stream(dev)
    for t in (4096, 65536):
        ids = torch.randint(0, N_VOCAB, (t,), generator=gen, device=dev, dtype=torch.int32)
        out = torch.empty(t, K_HIDDEN, dtype=torch.float16, device=dev)
        for _ in range(3):
            wql.wql_embed_gather(ids, qw, out=out)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for _ in range(R):
                    wql.wql_embed_gather(ids, qw, out=out)
        stream.wait_stream(cap)
        g.replay()
        torch.cuda.synchronize()
        per = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            per.append(a.elapsed_time(b) * 1e3 / R)
        us = statistics.median(per)
        nbytes = t * (4 + K_HIDDEN // 2 + (K_HIDDEN // GROUP) * 2 + K_HIDDEN * 2)
        gbs = nbytes / (us * 1e-6) / 1e9
        res["calls"][f"T{t}"] = {"us_median": round(us, 2), "bytes": nbytes,
                                 "GBps": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 3)}
    res["timing"] = "device: CUDA-graph replays of 20 calls, events around each replay"
    res["note"] = ("4096 ids move 10.7 MB, which L2 absorbs; 65536 ids move 171 MB (the "
                   "output alone exceeds L2)")
    return res


# ---------------------------------------------------------------------------
# CPU oracle arm (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

def oracle_sample_step(rows: int, nthreads: int, state: dict) -> tuple[float, int]:
    """One oracle step on the first `rows` vocab rows: logits at M=1/32/256,
    top-8 over the sampled rows, exact rescoring of the candidates.
    Returns (seconds, algorithmic bytes of the sampled work)."""
    import numpy as np
    import oracle
    if "qw" not in state:
        import torch
        from weight_only_quantized_wql_gb300 import synth
        w = synth.weight(rows, K_HIDDEN, synth.F32, seed=0)
        state["w_ref"] = w.half().numpy()
        state["qw"], state["s"] = oracle.quantize_packed(w.numpy(), oracle.F32, 4, GROUP,
                                                         oracle.F16, 0, nthreads=nthreads)
        state["x"] = {m: synth.activations(m, K_HIDDEN, synth.F16, seed=1000 + m).numpy()
                      for m in MS}
        del torch
    t0 = time.perf_counter()
    nbytes = 0
    for m in MS:
        out, _ = oracle.logits(state["x"][m], oracle.F16, state["qw"], 4, state["s"], oracle.F16,
                               GROUP, rows, K_HIDDEN, nthreads=nthreads)
        idx, _ = oracle.topk(out, TOPK)
        oracle.rescore(state["x"][m], oracle.F16, state["w_ref"], oracle.F16, idx)
        nbytes += logits_bytes(m, rows, K_HIDDEN, 4, GROUP, topk=TOPK) + \
            rescore_bytes(m, K_HIDDEN, TOPK)
    return time.perf_counter() - t0, nbytes


def cpu_rows_for_budget(nthreads: int, seconds: float, state_probe: dict) -> int:
    """Size the oracle sample so one step takes about `seconds` of CPU time."""
    probe = 512
    dt, _ = oracle_sample_step(probe, nthreads, state_probe)
    rows = int(probe * seconds / max(dt, 1e-6))
    return max(probe, min(N_VOCAB, rows // 16 * 16))


def cpu_baseline(nthreads: int, seconds: float = 12.0) -> dict:
    rows = cpu_rows_for_budget(nthreads, seconds, {})
    dt, nbytes = oracle_sample_step(rows, nthreads, {})
    # the same oracle on one host thread, on a smaller sample (context)
    rows1 = cpu_rows_for_budget(1, 3.0, {})
    dt1, nbytes1 = oracle_sample_step(rows1, 1, {})
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"first {rows} of {N_VOCAB} vocab rows, M=1/32/256 logits + top-8 + "
                      f"rescore, binary64 C, {nthreads} threads, {dt:.1f} s",
            "single_thread": {"value": round(nbytes1 / dt1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"first {rows1} vocab rows, 1 thread, {dt1:.1f} s"}}


def run_reference(args) -> dict:
    nthreads = os.cpu_count() or 1
    budget = max(1.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    rows = cpu_rows_for_budget(nthreads, budget, {})
    state = {}
    for _ in range(args.warmup):
        oracle_sample_step(rows, nthreads, state)
    tot_s, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, nb = oracle_sample_step(rows, nthreads, state)
        tot_s += dt
        tot_b += nb
    value = tot_b / tot_s / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "n": N_VOCAB, "k": K_HIDDEN, "group": GROUP,
                   "ms": list(MS), "topk": TOPK, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthreads,
                         "kind": "oracle",
                         "sample": f"first {rows} of {N_VOCAB} vocab rows per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------

def aggregate_over_ranks(local: list[float], world: int, device=None) -> list[float]:
    """Every rank's timings reduced to the slowest rank's (MAX) across the
    process group: a tensor on `device` (CUDA under NCCL, CPU under gloo)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(local, dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput_gbs(step_bytes_: int, steps: int, world: int, slowest_s: float) -> float:
    """Whole-job GB/s: the bytes all replicas moved over the slowest rank's
    time (each rank runs the same step on its own copy of the head)."""
    return step_bytes_ * steps * world / slowest_s / 1e9


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload block (all five heads at each token count)")
    ap.add_argument("--study", choices=["argmax", "embed"], default=None,
                    help="argmax: the int8 per-row head's greedy-token agreement study; "
                         "embed: the tied-embedding gather (each a separate JSON line, "
                         "not the bench line)")
    ap.add_argument("--ms", type=int, nargs="+", default=list(MS),
                    help="token counts M timed per step (default: 1 32 256); a subset "
                         "is for profiling one call, not a bench line")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.study is not None:
        if rank == 0:
            fn = run_argmax_study if args.study == "argmax" else run_embed_study
            print(json.dumps(fn(args)), flush=True)
        return 0

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(os.cpu_count() or 1)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
