#!/usr/bin/env python3
"""Benchmark of the Hadamard-folded 1-bit GEMV (decode tokens/s and weight GB/s).

One step = one bitlin_forward call: M tokens through one folded one-bit
matrix (default: the ffn_gate shape, M=1, K=5120, N=17408).  Consecutive steps
cycle through R distinct copies of the matrix whose total size is at least
four times the L2 cache, so every step streams its weights from HBM.  Steps
are replayed from CUDA graphs; the timed region is bracketed by a barrier and
a device synchronize, timed with CUDA events on the launching stream, and the
max over ranks is reported.

--impl reference times the CPU oracle (the plain f64 definition) on the
host's cores instead, in row chunks sized so the whole run ends within a few
minutes; its tokens/s counts the fraction of a token each chunk completes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode tokens/s and weight GB/s (% of HBM peak), 1-bit WHT GEMV K=5120 N=17408"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ffn_gate")
    ap.add_argument("--op", choices=["gemv", "mlp", "embed", "lmhead"], default="gemv",
                    help="gemv: one folded product per step (the headline); mlp: the MLP block "
                         "(gate+up 5120x34816, SiLU, down 17408x5120) per step; embed: M embedding "
                         "lookups with the inverse rotation in a 248,320 x 5120 table per step; lmhead: "
                         "the 248,320 x 5120 vocabulary product and the argmax per step")
    ap.add_argument("--M", type=int, default=None)
    ap.add_argument("--path", choices=["auto", "decode", "prefill", "exact"], default="auto",
                    help="force the library's path (bitlin_set_path) instead of its choice by M")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0)
    ap.add_argument("--e2e-steps", type=int, default=20000)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--copies", type=int, default=0,
                    help="distinct weight copies to cycle (default: enough for 4x the L2 size)")
    return ap.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def traffic_record(kernel: str, workload: str, M: int | None = None):
    """Per-launch DRAM bytes from a committed ncu summary, if it still matches the kernel source.
    A record taken at this token count ("kernel:workload:M") is preferred to one for the
    workload at any token count ("kernel:workload")."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = (rec.get(f"{kernel}:{workload}:{M}") if M is not None else None) or rec.get(f"{kernel}:{workload}")
    if not entry:
        return None
    src = os.path.join(ROOT, "hadamard_rotated_binary_gb300", "csrc", entry["source"])
    try:
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    return entry["bytes_per_launch"] if digest == entry["sha256"] else None


def max_over_ranks(v: float, pg, device) -> float:
    """The largest of every rank's v (the slowest rank's time), on every rank; v itself at N = 1."""
    if pg is None:
        return v
    import torch

    t = torch.tensor([v], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def roofline(w: synth.Workload, s_per_step: float, peaks: dict, peak_kind: str, path: int,
             kernels: int) -> dict:
    """Roofline of the dominant kernel of a call on `path` (the library's BITLIN_PATH_*, from
    bitlin_plan: 1 decode, 2 bf16 tensor path, 3 exact tensor path) launching `kernels` kernels.
    Decode: HBM-bound, algorithmic bytes per call over the step time (one GEMV per step; with
    kernels = 2 the step also holds the small split-K sum, which the GEMV overlaps through
    programmatic dependent launch, so the fraction is a lower bound).  Tensor paths: the tcgen05
    GEMM (one launch, or two when its tiles past the last full wave of SMs run as a split-K launch
    of their own), 2*M*N*K bf16 MMA flops per call (the exact path multiplies three bf16 digit
    columns per token, 3x that) over the step time, which also holds the small rotation kernel,
    so the fraction is a lower bound; peak = the measured burst bf16 GEMM rate (the timed loop
    lasts milliseconds); traffic = DRAM bytes of the call's GEMM launches together."""
    if path == 1:
        kernel = "bitlin_decode_gemv" + (" + bitlin_decode_reduce" if kernels == 2 else "")
        achieved = w.algorithmic_bytes() / s_per_step / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_kind": peak_kind, "kernel": kernel,
                "bytes_per_launch": w.algorithmic_bytes(), "traffic": traffic_record(kernel, w.name, w.M)}
    kernel = "bitlin_tc_gemm"
    digits = 3 if path == 3 else 1
    flops = 2.0 * w.M * digits * w.N * w.K
    achieved = flops / s_per_step / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"], "peak_kind": peak_kind, "kernel": kernel,
            "flops_per_launch": flops, "traffic": traffic_record(kernel, w.name, w.M)}


def cpu_model() -> str:
    """The host CPU's model string (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.processor() or platform.machine()


def timed_calls(fn, seconds: float, min_calls: int = 1):
    """Call fn() until `seconds` have passed (at least min_calls times): (calls, seconds)."""
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds and n >= min_calls:
            return n, el


def oracle_rates(fn, tokens_per_call: float, seconds: float) -> dict:
    """The oracle call fn, as it stands, on every host core for about `seconds` and on one
    thread for about a third of that: tokens/s, cores, both times per call, the CPU model."""
    import oracle

    cores = oracle.max_threads()
    n, el = timed_calls(fn, seconds)
    oracle.set_threads(1)
    try:
        n1, el1 = timed_calls(fn, seconds / 3)
    finally:
        oracle.set_threads(cores)
    return {"value": n * tokens_per_call / el, "cores": cores, "calls": n, "seconds": el,
            "ms_per_call_all_cores": 1e3 * el / n, "ms_per_call_one_thread": 1e3 * el1 / n1,
            "one_thread_tokens_per_s": n1 * tokens_per_call / el1, "cpu_model": cpu_model()}


def cpu_baseline(w: synth.Workload, inputs, seconds: float):
    """The oracle, as it stands, on the host cores: on every core for about `seconds`, and on
    one thread for a third of that.  A call covers every output row when a whole call takes
    at most a quarter of `seconds` on all cores; otherwise the leading rows that take about a
    twentieth (tokens/s then counts the fraction of each token's rows a call computes)."""
    import oracle

    oracle.build()
    bits, scales, signs, x = inputs
    probe = np.arange(min(64, w.N))
    t0 = time.perf_counter()
    oracle.forward(bits, scales, signs, w.perm, x, probe)
    est = (time.perf_counter() - t0) * w.N / probe.size
    rows = w.N if est <= seconds / 4 else max(1, min(w.N, int(w.N * seconds / 20 / est)))
    sel = None if rows == w.N else np.arange(rows)
    r = oracle_rates(lambda: oracle.forward(bits, scales, signs, w.perm, x, sel), w.M * rows / w.N, seconds)
    what = "whole oracle calls" if rows == w.N else f"oracle calls on the first {rows} of {w.N} output rows"
    return {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
            "cpu_model": r["cpu_model"], "ms_per_call_all_cores": r["ms_per_call_all_cores"],
            "ms_per_call_one_thread": r["ms_per_call_one_thread"],
            "one_thread_value": r["one_thread_tokens_per_s"],
            "sample": f"{r['calls']} {what} (M={w.M}, K={w.K}, N={w.N}) in {r['seconds']:.1f} s "
                      f"on {r['cores']} threads, then the same calls on one thread; f64, OpenMP over output rows"}


def run_reference(args, w: synth.Workload):
    """Reference arm: the CPU oracle on this workload, in bounded row chunks."""
    import oracle

    oracle.build()
    bits, scales, signs, x = synth.make_inputs(w)
    # Calibrate: one rotation and one chunk of 256 rows.
    t0 = time.perf_counter()
    xt = oracle.rotate(x, signs, w.perm)
    t_rot = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.product(bits, scales, xt, np.arange(min(256, w.N)))
    t_row = (time.perf_counter() - t0) / min(256, w.N)
    total_steps = args.steps + args.warmup
    per_step = args.ref_seconds / max(total_steps, 1)
    # rows per step so that rows * t_row plus the rotation's share fits per_step
    rows = int(max(1, min(w.N, per_step / max(t_row, 1e-9))))
    while rows > 1 and rows * t_row + t_rot * rows / w.N > per_step:
        rows = max(1, rows // 2)
    # A step computes `rows` output rows of the current token; the token's
    # rotation is computed at its first chunk and reused by the rest of it.
    chunks_per_token = (w.N + rows - 1) // rows
    state = {"i": 0, "xt": None}

    def step():
        c = state["i"] % chunks_per_token
        if c == 0 or state["xt"] is None:
            state["xt"] = oracle.rotate(x, signs, w.perm)
        lo = c * rows
        r = np.arange(lo, min(w.N, lo + rows))
        oracle.product(bits, scales, state["xt"], r)
        state["i"] += 1
        return r.size

    for _ in range(args.warmup):
        step()
    state["i"] = 0
    done = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        done += step()
    el = time.perf_counter() - t0
    tokens = w.M * done / w.N
    value = tokens / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64: Bernoulli(0.5) bits, U[0.005,0.03] fp16 scales, +-1 signs, N(0,1) x)",
        "config": {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "perm": w.perm,
                   "rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{args.steps} steps of {rows} output rows each (rotation once per token)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


MLP_METRIC = "MLP block tokens/s and weight GB/s (1-bit WHT-folded gate+up 5120x34816, SiLU, down 17408x5120)"
EMBED_METRIC = "embedding lookups/s with the inverse rotation (1-bit WHT-folded table 248320x5120)"
LMHEAD_METRIC = "LM head tokens/s and weight GB/s (1-bit WHT-folded 248320x5120 product + argmax)"


def flush_l2(dev, l2_bytes: int, stream):
    """Overwrite a buffer twice the L2 size on `stream`, so that nothing a warm-up left in L2
    is still there when the timed region starts."""
    import torch

    with torch.cuda.stream(stream):
        buf = torch.empty(2 * l2_bytes // 4 + 1, dtype=torch.float32, device=dev)
        buf.zero_()
    stream.synchronize()
    del buf


# Device-side delay before the first timed event (cycles of the SM clock, about 1 ms): the
# stream is then busy while the host enqueues the event and the graph replays, so the timed
# region holds device work only, not the host's launch latency.
HOLD_CYCLES = 2_000_000


def run_timed(replays, stream, pg, dev, gpu_index: int, lead=None):
    """The timed region: a barrier and a device synchronize, a device-side hold, the untimed
    lead-in graph `lead` (calls on weight copies the timed region reaches last, so none of the
    first timed calls' inputs is in L2), an event, `replays` (graphs, each already replayed
    once), an event, a device synchronize and a barrier.  nvidia-smi samples the clocks
    throughout.  Returns (ms over ranks, clocks)."""
    import torch

    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        torch.cuda._sleep(HOLD_CYCLES)
        if lead is not None:
            lead.replay()
        ev0.record(stream)
        for g in replays:
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    return max_over_ranks(ev0.elapsed_time(ev1), pg, dev), clocks


def capture_lead(step, stream, cycle: int, steps: int):
    """A graph of the calls that end the cycle of `cycle` distinct inputs (the last
    min(20, cycle // 2, cycle - steps) of them when the timed steps do not reach them, else
    the last min(20, cycle // 2)), replayed once here: the untimed lead-in of the timed
    region.  Returns None when the cycle is too short for one."""
    import torch

    n = min(20, cycle // 2, cycle - steps) if steps < cycle else min(20, cycle // 2)
    if n < 1:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(cycle - n, cycle):
                step(i)
        g.replay()
    stream.synchronize()
    return g


def capture_steps(step, stream, steps: int, chunk: int):
    """CUDA graphs of `chunk` consecutive calls (as many as fit in `steps`) and one of the
    remainder; every graph is replayed once before it is returned, so that the timed
    region never holds a graph's first launch (its upload).  Returns the replay list whose
    calls add up to exactly `steps`."""
    import torch

    def capture(n, first):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(first, first + n):
                    step(i)
        return g

    full, rem = divmod(steps, chunk)
    g_chunk = capture(chunk, 0) if full else None
    g_rem = capture(rem, full * chunk) if rem else None
    with torch.cuda.stream(stream):
        for g in (g_chunk, g_rem):
            if g is not None:
                g.replay()
    stream.synchronize()
    return [g_chunk] * full + ([g_rem] if g_rem is not None else [])


def timed_graph(step, stream, steps: int, warmup: int, pg, dev, cycle: int, chunk: int = 256):
    """Warm up, capture `step` calls in CUDA graphs (each replayed once) and the lead-in,
    flush L2, replay exactly `steps` calls in the timed region (run_timed).  step(i) uses
    input i % cycle.  Returns (ms, clocks)."""
    import torch

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
    stream.synchronize()
    replays = capture_steps(step, stream, steps, min(chunk, max(1, steps)))
    lead = capture_lead(step, stream, cycle, steps)
    flush_l2(dev, torch.cuda.get_device_properties(dev).L2_cache_size, stream)
    return run_timed(replays, stream, pg, dev, torch.cuda.current_device(), lead)


def run_op(args, ws, rank, local, pg):
    """--op mlp / --op embed: the NEXT operations on the same kernels, one JSON line."""
    import torch

    import hadamard_rotated_binary_gb300 as hrb
    from hadamard_rotated_binary_gb300 import build as hbuild

    hbuild.build()
    dev = torch.device("cuda", local)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    M = args.M or 1
    stream = torch.cuda.Stream(device=dev)
    peaks, peak_kind = measured_peaks()
    if args.op == "mlp":
        wgu, wdn = synth.workload("gate_up", M), synth.workload("ffn_down", M)
        gu_in, dn_in = synth.make_inputs(wgu), synth.make_inputs(wdn)
        wbytes = wgu.weight_bytes() + wdn.weight_bytes()
        R = args.copies if args.copies else max(2, -(-4 * l2 // wbytes))

        def dev_layer(inp):
            b, sc, sg, _ = inp
            return hrb.BitLinear(torch.from_numpy(b.view(np.int32)).to(dev),
                                 torch.from_numpy(sc.view(np.int16)).to(dev), torch.from_numpy(sg).to(dev), 0)

        pairs = [(dev_layer(gu_in), dev_layer(dn_in)) for _ in range(R)]
        x = gu_in[3]
        xd = torch.from_numpy(x).to(dev)
        yd = torch.empty((M, wdn.N), dtype=torch.float32, device=dev)

        def step(i):
            hrb.mlp_forward(pairs[i % R][0], pairs[i % R][1], xd, out=yd, stream=stream)

        ms, clocks = timed_graph(step, stream, args.steps, max(args.warmup, R), pg, dev, R)
        s_step = ms / 1e3 / args.steps
        algo = wbytes + 4 * M * wgu.K + 4 * M * wdn.N + 4 * (wgu.K + wdn.K)
        flops = 2.0 * M * (wgu.N * wgu.K + wdn.N * wdn.K)
        (pgu, kgu), (pdn, kdn) = pairs[0][0].plan(M), pairs[0][1].plan(M)
        kernels = kgu + kdn
        if pgu == pdn == hrb.PATH_DECODE:
            roof = {"bound": "hbm", "achieved": algo / s_step / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "kernel": "bitlin_decode_gemv (x2)" + " + bitlin_decode_reduce" * (kernels - 2),
                    "bytes_per_launch": algo}
        else:
            digits = 3 if M < 64 else 1
            roof = {"bound": "tensor", "achieved": digits * flops / s_step / 1e12, "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "kernel": "bitlin_tc_gemm (x2)", "flops_per_launch": digits * flops}
        roof.update({"frac": roof["achieved"] / roof["peak"], "peak_kind": peak_kind, "traffic": None})
        metric, config = MLP_METRIC, {"workload": "mlp_block", "M": M, "hidden": wgu.K, "ffn": wdn.K,
                                      "weight_copies": R, "weight_set_bytes": R * wbytes,
                                      "l2": f"inputs larger than L2: {R} distinct weight pairs cycled"}
        launches = kernels
        wgb = wbytes / s_step / 1e9

        def e2e_call(xh, yh):
            xd.copy_(xh, non_blocking=True)
            hrb.mlp_forward(pairs[0][0], pairs[0][1], xd, out=yd)
            yh.copy_(yd, non_blocking=True)
            torch.cuda.current_stream().synchronize()

        h2d, d2h, out_shape = 4 * M * wgu.K, 4 * M * wdn.N, (M, wdn.N)

        def cpu_call():
            import oracle

            oracle.build()
            return lambda: oracle.mlp(gu_in[:3] + (0,), dn_in[:3] + (0,), x)
    elif args.op == "lmhead":
        N, K = 248320, 5120
        seed = 0xB1711A00 + 12
        bits = synth.random_bits(seed, N, K)
        scales = synth.random_scales(seed, N, K, 0.005, 0.03)
        signs = synth.random_signs(seed, K)
        tb = torch.from_numpy(bits.view(np.int32)).to(dev)
        ts = torch.from_numpy(scales.view(np.int16)).to(dev)
        tg = torch.from_numpy(signs).to(dev)
        wbytes = N * K // 8 + 2 * N * (K // 128)
        R = args.copies if args.copies else max(2, -(-4 * l2 // wbytes))
        heads = [hrb.BitLinear(tb, ts, tg, 0) for _ in range(R)]
        del tb, ts, tg
        x = synth.random_x(seed, M, K)
        xd = torch.from_numpy(x).to(dev)
        lg = torch.empty((M, N), dtype=torch.float32, device=dev)
        idd = torch.empty((M,), dtype=torch.int32, device=dev)

        def step(i):
            heads[i % R].argmax(xd, logits=lg, ids=idd, stream=stream)

        ms, clocks = timed_graph(step, stream, args.steps, max(args.warmup, R), pg, dev, R)
        s_step = ms / 1e3 / args.steps
        algo = wbytes + 4 * M * K + 4 * M * N + 4 * K + 4 * M
        hpath, hk = heads[0].plan(M)
        # One token through cluster split-K (one kernel): the pick is fused into the product's finish.
        fused = hpath == hrb.PATH_DECODE and hk == 1
        if hpath == hrb.PATH_DECODE:
            roof = {"bound": "hbm", "achieved": algo / s_step / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "kernel": ("bitlin_decode_gemv (argmax fused)" if fused else
                               "bitlin_decode_gemv" + " + bitlin_decode_reduce" * (hk - 1) + " + bitlin_argmax_rows"),
                    "bytes_per_launch": algo}
        else:
            digits = 3 if M < 64 else 1
            flops = 2.0 * M * digits * N * K
            roof = {"bound": "tensor", "achieved": flops / s_step / 1e12, "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "kernel": "bitlin_tc_gemm + bitlin_argmax_rows", "flops_per_launch": flops}
        roof.update({"frac": roof["achieved"] / roof["peak"], "peak_kind": peak_kind,
                     "traffic": traffic_record(roof["kernel"], "lm_head", M)})
        metric, config = LMHEAD_METRIC, {"workload": "lm_head", "M": M, "N": N, "K": K, "weight_copies": R,
                                         "weight_set_bytes": R * wbytes,
                                         "l2": f"inputs larger than L2: {R} distinct copies cycled"}
        launches, wgb = hk + (0 if fused else 1), wbytes / s_step / 1e9

        def e2e_call(xh, yh):
            xd.copy_(xh, non_blocking=True)
            heads[0].argmax(xd, logits=lg, ids=idd)
            yh.copy_(idd, non_blocking=True)
            torch.cuda.current_stream().synchronize()

        h2d, d2h = 4 * M * K, 4 * M

        def cpu_call():
            import oracle

            oracle.build()
            return lambda: np.argmax(oracle.forward(bits, scales, signs, 0, x), axis=1)
    else:
        N, K = 248320, 5120
        seed = 0xB1711A00 + 12
        bits = synth.random_bits(seed, N, K)
        scales = synth.random_scales(seed, N, K, 0.005, 0.03)
        signs = synth.random_signs(seed, K)
        layer = hrb.BitLinear(torch.from_numpy(bits.view(np.int32)).to(dev),
                              torch.from_numpy(scales.view(np.int16)).to(dev), torch.from_numpy(signs).to(dev), 0)
        nsets = 64
        ids = (synth.stream(seed, 5, nsets * M) % np.uint64(N)).astype(np.int32).reshape(nsets, M)
        idd = torch.from_numpy(ids).to(dev)
        yd = torch.empty((M, K), dtype=torch.float32, device=dev)

        def step(i):
            layer.embed(idd[i % nsets], out=yd, stream=stream)

        ms, clocks = timed_graph(step, stream, args.steps, max(args.warmup, 3), pg, dev, nsets)
        s_step = ms / 1e3 / args.steps
        row = K // 8 + 2 * (K // 128)
        algo = M * (row + 4 + 4 * K) + 4 * K
        roof = {"bound": "hbm", "achieved": algo / s_step / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "kernel": "bitlin_embed_rows", "bytes_per_launch": algo}
        roof.update({"frac": roof["achieved"] / roof["peak"], "peak_kind": peak_kind,
                     "traffic": traffic_record("bitlin_embed_rows", "embed", M)})
        metric, config = EMBED_METRIC, {"workload": "embed", "M": M, "N": N, "K": K,
                                        "l2": f"table of {N * row / 1e6:.0f} MB > L2; {nsets} id sets of random rows"}
        launches, wgb = 1, M * row / s_step / 1e9
        x = ids[0]

        def e2e_call(xh, yh):
            idd[0].copy_(xh, non_blocking=True)
            layer.embed(idd[0], out=yd)
            yh.copy_(yd, non_blocking=True)
            torch.cuda.current_stream().synchronize()

        h2d, d2h, out_shape = 4 * M, 4 * M * K, (M, K)

        def cpu_call():
            import oracle

            oracle.build()
            return lambda: oracle.embed(bits, scales, signs, ids[0])

    # end to end through the Python API: pinned host input -> device, call, device -> pinned host
    xh = torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    if args.op == "lmhead":
        yh = torch.empty((M,), dtype=torch.int32).pin_memory()
    else:
        yh = torch.empty(out_shape, dtype=torch.float32).pin_memory()
    e2e_steps = min(args.steps, args.e2e_steps)
    for _ in range(3):
        e2e_call(xh, yh)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_call(xh, yh)
    e2e_s = max_over_ranks(time.perf_counter() - t0, pg, dev)
    if rank != 0:
        return
    line = {
        "metric": metric, "value": ws * M / s_step, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded SplitMix64: Bernoulli(0.5) bits, U[0.005,0.03] fp16 scales, +-1 signs, N(0,1) x)",
        "config": config, "weight_gbs": wgb, "roofline": roof, "gpu_launches": args.steps * launches,
        "clocks": clocks,
        "e2e": {"value": ws * M * e2e_steps / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "api": "python binding, pinned host buffers"},
    }
    if not args.no_cpu_baseline:
        r = oracle_rates(cpu_call(), M, args.cpu_seconds)
        line["cpu_baseline"] = {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                                "cpu_model": r["cpu_model"], "ms_per_call_all_cores": r["ms_per_call_all_cores"],
                                "ms_per_call_one_thread": r["ms_per_call_one_thread"],
                                "one_thread_value": r["one_thread_tokens_per_s"],
                                "sample": f"{r['calls']} whole oracle calls in {r['seconds']:.1f} s on "
                                          f"{r['cores']} threads, then whole calls on one thread; f64"}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, local = dist_env()
    w = synth.workload(args.workload, args.M)

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w)
        return

    import torch

    torch.cuda.set_device(local)
    pg = None
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    if args.op != "gemv":
        run_op(args, ws, rank, local, pg)
        if pg:
            pg.destroy_process_group()
        return

    import hadamard_rotated_binary_gb300 as hrb
    from hadamard_rotated_binary_gb300 import build as hbuild

    hbuild.build()
    dev = torch.device("cuda", local)
    inputs = synth.make_inputs(w)
    bits, scales, signs, x = inputs
    tb = torch.from_numpy(bits.view(np.int32)).to(dev)
    ts = torch.from_numpy(scales.view(np.int16)).to(dev)
    tg = torch.from_numpy(signs).to(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    wbytes = w.weight_bytes()
    R = args.copies if args.copies else max(2, -(-4 * l2 // wbytes))
    layers = [hrb.BitLinear(tb, ts, tg, w.perm) for _ in range(R)]
    del tb, ts, tg
    forced = {"auto": hrb.PATH_AUTO, "decode": hrb.PATH_DECODE, "prefill": hrb.PATH_PREFILL,
              "exact": hrb.PATH_TC_EXACT}[args.path]
    for layer in layers:
        layer.set_path(forced)
    xd = torch.from_numpy(x).to(dev)
    yd = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)

    stream = torch.cuda.Stream(device=dev)
    # Warm-up (also allocates every handle's scratch before capture).
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, R)):
            layers[i % R](xd, out=yd, stream=stream)
    stream.synchronize()

    # Graphs of whole cycles through the R copies; step i uses copy i % R, so a call
    # re-reads a copy only after R - 1 others (R * the matrix size >= 4x L2).
    def step(i):
        layers[i % R](xd, out=yd, stream=stream)

    replays = capture_steps(step, stream, args.steps, R * max(1, 256 // R))
    lead = capture_lead(step, stream, R, args.steps)
    flush_l2(dev, l2, stream)
    ms, clocks = run_timed(replays, stream, pg, dev, local, lead)
    assert layers[0].get_error() == 0

    # End to end through the host-buffer entry point (pinned host memory).
    e2e_steps = min(args.steps, args.e2e_steps)
    xh = torch.from_numpy(x).pin_memory().numpy()
    yh = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory().numpy()
    for i in range(min(R, 50)):
        layers[i % R].forward_host(xh, yh, stream=stream)
    if pg:
        pg.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        layers[i % R].forward_host(xh, yh, stream=stream)
    e2e_s = max_over_ranks(time.perf_counter() - t0, pg, dev)

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return

    peaks, peak_kind = measured_peaks()
    s_per_step = ms / 1e3 / args.steps
    path, kernels = layers[0].plan(w.M)
    tokens_per_s = ws * w.M / s_per_step
    algo_bytes = w.algorithmic_bytes()
    achieved = algo_bytes / s_per_step / 1e9
    line = {
        "metric": METRIC,
        "value": tokens_per_s,
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if path == hrb.PATH_DECODE else "bf16",
        "data": "synthetic (seeded SplitMix64: Bernoulli(0.5) bits, U[0.005,0.03] fp16 scales, +-1 signs, N(0,1) x)",
        "config": {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "perm": w.perm, "path": args.path,
                   "kernel_path": {1: "decode GEMV (f32)", 2: "tcgen05, bf16 activations",
                                   3: "tcgen05, three exact bf16 digits, f32 accumulation"}[path],
                   "weight_copies": R, "weight_set_bytes": R * wbytes,
                   "l2": f"inputs larger than L2: {R} distinct weight copies ({R * wbytes / 1e6:.0f} MB) cycled; "
                         f"L2 flushed before the timed region",
                   "timing": "CUDA events on the launching stream around graph replays that were each replayed "
                             "once before; the stream is held by a device-side delay while the host enqueues them, "
                             "then an untimed lead-in of calls on the copies the timed region reaches last",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "weight_gbs": w.weight_bytes() / s_per_step / 1e9,
        "hbm_frac_of_8tbs": achieved / 8000.0,
        "roofline": roofline(w, s_per_step, peaks, peak_kind, path, kernels),
        "gpu_launches": args.steps * kernels,  # the library's own count per call (bitlin_plan)
        "clocks": clocks,
        "e2e": {"value": ws * w.M * e2e_steps / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": 4 * w.M * w.K, "d2h_bytes_per_step": 4 * w.M * w.N,
                "steps": e2e_steps, "api": "bitlin_forward_host"},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inputs, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    for layer in layers:
        layer.close()
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
