"""Throughput of the weight-quantized linear layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--reps R] [--workload NAME] [--impl reference]

One step is one call of the layer (qgemm_run) on the workload's synthetic inputs. The headline
workload is the largest of the five: W4A8, M=2048, K=4096, N=14336 (per-channel INT4 weights,
bf16 activations quantized per row to INT8, exact int32 sums, bf16 output), reported in TFLOPS =
2*M*K*N / t (the benchmark page's convention, "MNN GemmSpeed 基准测试实战" «测量流程»). The same
JSON line carries a per_config object with the other workloads: the Int4-Block64 small case
(M=4, K=256, N=512, f32), the decode GEMV (M=1, K=4096, N=11008), Int8-Block0 at K=N=4096 for
M in {1, 2, 4, 8, 16}, the Int4-Block64 prefill (M=1024, K=N=4096) and the fp16 GEMM beside W4A8;
HBM-bound (M <= 16) workloads are reported in weight-stream GB/s (the layer's algorithmic bytes:
packed weights, {offset, scale} table, activations in, output out), the others in TFLOPS.

Timing: weights are packed once (offline, as on the page), then copied into enough rotating
copies (with the activations when M > 16) to exceed the L2 cache 3x, so every call streams from
HBM. W warm-up calls, then K calls captured in one CUDA graph; the graph is replayed R times, each
replay between CUDA events on the launching stream with a barrier and synchronize on both sides
(max over ranks); the per-call time is the median replay / K (the minimum is reported beside it).
The decode kernels are timed with and without programmatic dependent launch. GPU clocks are
sampled with nvidia-smi during the headline's timed replays.

--impl reference times the CPU oracle (float64 plain loops, the test suite's reference) on
this host's cores on a bounded sample of the same workload; it is a deliberately slow
baseline, not a target.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from weight_quantized_gemm_gb300 import synth  # noqa: E402

METRIC = "qGEMM TFLOPS (2*M*K*N/s) and weight-stream HBM GB/s, % of roofline"
HEADLINE_WORKLOAD = "w4a8_m2048_k4096_n14336"
DTYPE_NAME = {0: "f32", 1: "f16", 2: "bf16"}


# ---------------------------------------------------------------- workload accounting
def algorithmic_bytes(w: synth.Workload, bias: bool = False, residual: bool = False) -> int:
    """Bytes one call must move: packed weights + table + activations in + output out (+ the
    fused epilogue's bias and residual reads)."""
    esz = {0: 4, 1: 2, 2: 2}
    extra = (w.N * 4 if bias else 0) + (w.M * w.N * esz[w.c_dtype] if residual else 0)
    if w.mode == synth.MODE_FLOAT:
        wb = w.K * w.N * esz[w.a_dtype]
        tb = 0
    else:
        wb = w.K * w.N * (4 if w.mode in (synth.MODE_INT4, synth.MODE_W4A8) else 8) // 8
        blk = w.K if w.block == 0 else w.block
        tb = w.N * (w.K // blk) * 8
    return wb + tb + w.M * w.K * esz[w.a_dtype] + w.M * w.N * esz[w.c_dtype] + extra


def bound_of(w: synth.Workload) -> str:
    return "hbm" if w.M <= 16 else "tensor"


# source files of each workload's dominant kernel: a recorded DRAM-traffic figure is used only
# while these files are unchanged since the capture
KERNEL_SOURCES = {
    "decode": ["decode_stream.cuh", "decode_kernel.cuh", "decode_int4.cu", "decode_int8.cu", "decode_float.cu",
               "epilogue.cuh", "ptx.cuh", "internal.h"],
    "prefill": ["prefill_kernel.cuh", "prefill.cu", "prefill_codes.cu", "epilogue.cuh", "ptx.cuh", "internal.h"],
    "f32": ["decode.cu", "epilogue.cuh", "internal.h"],
}


def kernel_of(w: synth.Workload) -> str:
    if w.a_dtype == synth.F32 and w.mode != synth.MODE_W4A8:
        return "f32"      # the exact CUDA-core kernel
    return "decode" if (w.M <= 16 and w.mode != synth.MODE_W4A8) else "prefill"


def src_hash(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_quantized_gemm_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:12]


def measured_traffic(w: synth.Workload):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary
    (profiles/traffic.txt: workload M K N kernel source-hash bytes), if it was taken on this
    shape and this source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    kern = kernel_of(w)
    cur = src_hash(kern)
    key = [w.name, str(w.M), str(w.K), str(w.N), kern, cur]
    for ln in open(path):
        parts = ln.split()
        if len(parts) >= 7 and not ln.startswith("#") and parts[:6] == key:
            return int(float(parts[6]))
    return None


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- the oracle arm
def oracle_step_fn(w: synth.Workload, A, W):
    """Returns (callable running one bounded oracle sample, units of work per call, description)."""
    import oracle
    if w.mode == synth.MODE_FLOAT:
        Bt = oracle.values(oracle.pack_float(W, w.a_dtype), w.a_dtype)
        A64 = oracle.values(A, w.a_dtype)
        rows = max(1, min(w.M, int(2e8 // (w.K * w.N))))
        return (lambda: oracle.gemm(A64[:rows], Bt)), rows, f"float GEMM of {rows} row(s) of A"
    qmax = oracle.QMAX[w.mode]
    blk = w.K if w.block == 0 else w.block
    q, T = oracle.quantize(W, blk, qmax)       # offline step, not timed
    A64 = oracle.values(A, w.a_dtype)
    if w.mode == synth.MODE_W4A8:
        rows = max(1, min(w.M, int(4e8 // (w.K * w.N))))
        A32 = A64[:rows].astype(np.float32)

        def run():
            qa, s, rs = oracle.act_quant(A32)
            if blk != w.K:
                return oracle.w4a8_block_out(qa, s, q, T, blk)
            return oracle.w4a8_out(oracle.w4a8_acc(qa, q), s, rs, T)
        return run, rows, f"W4A8 on {rows} row(s) of A"
    rows = max(1, min(w.M, int(4e8 // (w.K * w.N))))

    def run():
        return oracle.gemm(A64[:rows], oracle.dequant(q, T, blk))
    return run, rows, f"dequant + float64 GEMM of {rows} row(s) of A"


def run_reference(args, w: synth.Workload) -> dict:
    import oracle
    threads = len(os.sched_getaffinity(0))
    oracle.set_threads(threads)
    A = synth.make_activations(w)
    W = synth.make_weights(w)
    fn, rows, desc = oracle_step_fn(w, A, W)
    for _ in range(max(1, min(args.warmup, 1))):
        fn()
    steps = max(1, args.steps)
    budget = getattr(args, "cpu_seconds", 60.0)
    t0 = time.perf_counter()
    done = 0
    while done < steps:
        fn()
        done += 1
        if time.perf_counter() - t0 > budget:    # bound the CPU arm's run time
            break
    dt = (time.perf_counter() - t0) / done
    frac = rows / w.M
    bytes_per = algorithmic_bytes(w) * frac
    value = bytes_per / dt / 1e9
    return {"value": value, "unit": "GB/s", "ms_per_step": dt * 1e3, "steps": done, "cores": oracle.set_threads(0),
            "sample": f"{desc} of {w.name} per step ({frac:.3g} of the layer), {done} step(s)",
            "tflops": 2.0 * rows * w.K * w.N / dt / 1e12}


# ---------------------------------------------------------------- the GPU arm
def max_over_ranks(ms: float, dist, device) -> float:
    """The timed region as the slowest rank saw it; every rank gets the same value."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_step: float, step_s: float, world: int) -> float:
    """Whole-job throughput: every rank runs the same per-step work (replicas, weak scaling)."""
    return units_per_step / step_s * world


def to_torch(arr: np.ndarray, code: int, device):
    import torch
    if code == synth.BF16:
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.to(device)


ACTS = {"none": 0, "relu": 1, "silu": 2, "gelu_tanh": 3}


class Layer:
    """One workload on the GPU: packed weights in enough rotating copies (and, for M > 16,
    activations) to exceed the L2 cache 3x, so that every call streams from HBM."""

    def __init__(self, w: synth.Workload, device, stream, bias=False, residual=False, act="none"):
        import torch

        import weight_quantized_gemm_gb300 as qg
        self.w, self.device, self.stream = w, device, stream
        self.qg, self.lib = qg, qg.load()
        tdt = {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}
        K, N, M = w.K, w.N, w.M
        with torch.cuda.stream(stream):
            A = to_torch(synth.make_activations(w), w.a_dtype, device)
            Wd = torch.from_numpy(synth.make_weights(w)).to(device)
            self.pb = qg.qgemm_packed_bytes(K, N, w.mode, w.w_dtype if w.mode == 0 else 0)
            self.tb = qg.qgemm_table_bytes(K, N, w.mode, w.block)
            Bp0 = torch.empty(self.pb, dtype=torch.uint8, device=device)
            T0 = torch.empty(max(self.tb // 4, 4), dtype=torch.float32, device=device)
            qg.qgemm_pack(Wd, K, N, w.mode, w.block, w.a_dtype if w.mode == 0 else 0, Bp0,
                          T0 if self.tb else None, stream=stream)
            del Wd
            self.l2 = torch.cuda.get_device_properties(device).L2_cache_size
            a_bytes = A.numel() * A.element_size() if M > 16 else 0
            self.copy_bytes = self.pb + self.tb
            self.copies = max(2, -(-3 * self.l2 // max(self.copy_bytes + a_bytes, 1)))
            self.Bps = [Bp0] + [Bp0.clone() for _ in range(self.copies - 1)]
            self.Ts = [T0] + [T0.clone() for _ in range(self.copies - 1)]
            self.As = [A] + ([A.clone() for _ in range(self.copies - 1)] if M > 16 else [])
            self.C = torch.empty((M, N), dtype=tdt[w.c_dtype], device=device)
            self.wsb = qg.qgemm_workspace_bytes(M, K, N, w.mode, w.block, w.a_dtype, w.c_dtype)
            self.ws = torch.empty(max(self.wsb, 16), dtype=torch.uint8, device=device)
            self.bias = (torch.from_numpy(synth.normal64(N, 11, stream=4, std=0.5).astype(np.float32)).to(device)
                         if bias else None)
            self.res = (to_torch(synth.encode(synth.normal64(M * N, 12, stream=5).reshape(M, N), w.c_dtype),
                                 w.c_dtype, device) if residual else None)
            # the activation pass alone (W4A8): same rows, codes written as int8
            if w.mode == synth.MODE_W4A8:
                self.qa = torch.empty((M, K), dtype=torch.int8, device=device)
                self.asc = torch.empty(M, dtype=torch.float32, device=device)
                self.rsum = torch.empty(M, dtype=torch.int32, device=device)
        stream.synchronize()
        self.act = ACTS[act]
        self.fused = self.bias is not None or self.res is not None or self.act != 0

    def launches_per_call(self, decode_max_m: int) -> int:
        """This library's kernels per call: W4A8 = activation quantization + GEMM; otherwise one
        launch per 16-row decode launch (or one tensor-core launch), plus the split-K reduction."""
        w = self.w
        if w.mode == synth.MODE_W4A8:
            return 2
        decode_path = w.a_dtype != synth.F32 and w.M <= decode_max_m
        return (-(-w.M // 16) if decode_path else 1) * (2 if self.wsb > 0 else 1)

    def call(self, i: int):
        w, lib, s_ptr = self.w, self.lib, self.stream.cuda_stream
        A, Bp = self.As[i % len(self.As)].data_ptr(), self.Bps[i % self.copies].data_ptr()
        T = self.Ts[i % self.copies].data_ptr() if self.tb else None
        if self.fused:
            rc = lib.qgemm_run_fused(w.M, w.K, w.N, w.mode, w.block, A, w.a_dtype, Bp, T,
                                     None if self.bias is None else self.bias.data_ptr(), self.act,
                                     None if self.res is None else self.res.data_ptr(), self.C.data_ptr(), w.c_dtype,
                                     self.ws.data_ptr(), self.wsb, s_ptr)
        else:
            rc = lib.qgemm_run(w.M, w.K, w.N, w.mode, w.block, A, w.a_dtype, Bp, T, self.C.data_ptr(), w.c_dtype,
                               self.ws.data_ptr(), self.wsb, s_ptr)
        if rc != 0:
            raise self.qg.QgemmError(rc, "qgemm_run")

    def act_quant_call(self, i: int):
        w = self.w
        rc = self.lib.qgemm_act_quant(w.M, w.K, self.As[i % len(self.As)].data_ptr(), w.a_dtype, self.qa.data_ptr(),
                                      self.asc.data_ptr(), self.rsum.data_ptr(), self.stream.cuda_stream)
        if rc != 0:
            raise self.qg.QgemmError(rc, "qgemm_act_quant")

    def graph(self, fn, calls: int, overlap: int):
        import torch
        self.qg.qgemm_set_option(self.qg.OPT_LAUNCH_OVERLAP, overlap)
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(calls):
                    fn(i)
        finally:
            self.qg.qgemm_set_option(self.qg.OPT_LAUNCH_OVERLAP, 0)
        return g


def time_graph(g, stream, reps: int, dist, device) -> list[float]:
    """Milliseconds of each of `reps` replays of graph g, each replay bracketed by a barrier and a
    synchronize on both sides and timed with CUDA events on the launching stream (max over
    ranks). One untimed replay first keeps the graph's own first-launch cost out."""
    import torch
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    out = []
    for _ in range(reps):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):     # replay() launches on the current stream
            start.record(stream)
            g.replay()
            end.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        out.append(max_over_ranks(start.elapsed_time(end), dist, device))
    return out


def per_call(ms_list: list[float], calls: int) -> dict:
    return {"median_ms": statistics.median(ms_list) / calls, "min_ms": min(ms_list) / calls}


def roofline_of(w: synth.Workload, call_ms: float, peaks: dict, alg: int, kernel_ms: float | None = None) -> dict:
    bound = bound_of(w)
    t = (kernel_ms if kernel_ms is not None else call_ms) / 1e3
    if bound == "hbm":
        achieved, peak, unit, src = alg / t / 1e9, peaks["hbm_gbs"], "GB/s", "hbm_gbs"
    else:
        achieved, peak, unit, src = w.flops / t / 1e12, peaks["bf16_tflops"], "TFLOP/s", "bf16_tflops"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "peak_source": f"{peaks['source']} ({src})", "traffic": measured_traffic(w), "algorithmic_bytes": alg,
            "kernel": kernel_of(w)}


def metric_value(w: synth.Workload, step_s: float, alg: int, world: int = 1) -> tuple[float, str]:
    if bound_of(w) == "hbm":
        return job_rate(alg, step_s, world) / 1e9, "GB/s"
    return job_rate(w.flops, step_s, world) / 1e12, "TFLOP/s"


def calls_for(layer: Layer, min_ms: float = 1.0, cap: int = 4000) -> int:
    """Calls per graph so that one replay lasts at least min_ms (from a short eager estimate)."""
    import torch
    for i in range(3):
        layer.call(i)
    s = layer.stream
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s)
    for i in range(10):
        layer.call(i)
    end.record(s)
    s.synchronize()
    est = max(start.elapsed_time(end) / 10, 1e-3)
    return int(min(cap, max(20, -(-min_ms // est))))


def bench_entry(w: synth.Workload, device, stream, peaks: dict, reps: int, dist, decode_max_m: int,
                cpu_seconds: float, rank: int) -> dict:
    """One per-config line: median / min per-call time over `reps` replays of a graph of calls
    lasting >= 1 ms, with and without launch overlap for the decode kernels, its roofline and
    the oracle timed on a bounded sample."""
    layer = Layer(w, device, stream)
    calls = calls_for(layer)
    alg = algorithmic_bytes(w)
    modes = (1, 0) if kernel_of(w) == "decode" else (0,)
    out = {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "mode": synth.MODE_NAMES[w.mode],
           "a_dtype": DTYPE_NAME[w.a_dtype], "c_dtype": DTYPE_NAME[w.c_dtype], "calls_per_replay": calls,
           "replays": reps}
    for mode in modes:
        g = layer.graph(layer.call, calls, mode)
        t = per_call(time_graph(g, stream, reps, dist, device), calls)
        del g
        value, unit = metric_value(w, t["median_ms"] / 1e3, alg)
        key = "" if mode == modes[0] else "_no_overlap"
        out["ms_per_step" + key] = t["median_ms"]
        out["ms_per_step_min" + key] = t["min_ms"]
        out["value" + key] = value
        out["unit"] = unit
        if mode == modes[0]:
            out["launch_overlap"] = bool(mode)
            out["roofline"] = roofline_of(w, t["median_ms"], peaks, alg)
            out["tflops"] = w.flops / (t["median_ms"] / 1e3) / 1e12
            out["gbs"] = alg / (t["median_ms"] / 1e3) / 1e9
    if rank == 0 and cpu_seconds > 0:
        ref = run_reference(argparse.Namespace(steps=10 ** 6, warmup=1, cpu_seconds=cpu_seconds), w)
        out["cpu_baseline"] = {"value": ref["value"] if bound_of(w) == "hbm" else ref["tflops"],
                               "unit": "GB/s" if bound_of(w) == "hbm" else "TFLOP/s", "cores": ref["cores"],
                               "kind": "oracle", "sample": ref["sample"]}
    del layer
    return out


def bench_fused_pair(device, stream, reps: int, dist) -> dict:
    """Two chained W4A8 layers of a 7B-class FFN, M=2048: the headline up-projection 4096 -> 14336,
    then the down-projection 14336 -> 4096. Plain: the second layer quantizes its activations
    itself (qgemm_run; rows of 14336 are longer than its register cache, so part of each row is
    read twice); fused: the first layer's epilogue hands its row maxima to a one-read pass that
    writes the codes (qgemm_run_fused_quant) and the second layer starts from them
    (qgemm_run_w4a8_codes). Median per pair over `reps` replays."""
    import torch

    import weight_quantized_gemm_gb300 as qg
    lib = qg.load()
    w1 = synth.WORKLOADS["w4a8_m2048_k4096_n14336"]
    w2 = synth.Workload("pair_down", 2048, 14336, 4096, synth.MODE_W4A8, 0, synth.BF16, synth.BF16, 0, 3)
    l1, l2 = Layer(w1, device, stream), Layer(w2, device, stream)
    M, K1, N1, N2 = w1.M, w1.K, w1.N, w2.N
    C1 = torch.empty((M, N1), dtype=torch.bfloat16, device=device)
    qa = torch.empty((M, N1), dtype=torch.float16, device=device)
    asc = torch.empty(M, dtype=torch.float32, device=device)
    rs = torch.empty(M, dtype=torch.int32, device=device)
    fq = qg.qgemm_fused_quant_workspace_bytes(M, K1, N1, 3, 0, synth.BF16, synth.BF16)
    ws1 = torch.empty(max(fq, l1.wsb, 16), dtype=torch.uint8, device=device)
    wsc = qg.qgemm_w4a8_codes_workspace_bytes(M, N1, N2, 0)
    ws2 = torch.empty(max(wsc, 16), dtype=torch.uint8, device=device)
    s_ptr = stream.cuda_stream

    def check(rc, what):
        if rc != 0:
            raise qg.QgemmError(rc, what)

    def plain(i):
        check(lib.qgemm_run(M, K1, N1, 3, 0, l1.As[i % len(l1.As)].data_ptr(), synth.BF16,
                            l1.Bps[i % l1.copies].data_ptr(), l1.Ts[i % l1.copies].data_ptr(), C1.data_ptr(),
                            synth.BF16, ws1.data_ptr(), l1.wsb, s_ptr), "layer 1")
        check(lib.qgemm_run(M, N1, N2, 3, 0, C1.data_ptr(), synth.BF16, l2.Bps[i % l2.copies].data_ptr(),
                            l2.Ts[i % l2.copies].data_ptr(), l2.C.data_ptr(), synth.BF16, l2.ws.data_ptr(), l2.wsb,
                            s_ptr), "layer 2")

    def fused(i):
        check(lib.qgemm_run_fused_quant(M, K1, N1, 3, 0, l1.As[i % len(l1.As)].data_ptr(), synth.BF16,
                                        l1.Bps[i % l1.copies].data_ptr(), l1.Ts[i % l1.copies].data_ptr(), None, 0,
                                        None, C1.data_ptr(), synth.BF16, qa.data_ptr(), asc.data_ptr(), rs.data_ptr(),
                                        ws1.data_ptr(), fq, s_ptr), "layer 1 (fused)")
        check(lib.qgemm_run_w4a8_codes(M, N1, N2, 0, qa.data_ptr(), asc.data_ptr(), rs.data_ptr(),
                                       l2.Bps[i % l2.copies].data_ptr(), l2.Ts[i % l2.copies].data_ptr(), None, 0,
                                       None, l2.C.data_ptr(), synth.BF16, ws2.data_ptr(), wsc, s_ptr),
              "layer 2 (codes)")

    out = {"layers": "W4A8 M=2048: K=4096 -> N=14336, then K=14336 -> N=4096", "pairs_per_replay": 10}
    with torch.cuda.stream(stream):
        for i in range(3):
            plain(i)
            fused(i)
    stream.synchronize()
    for name, fn in (("plain", plain), ("fused", fused)):
        g = l1.graph(fn, 10, 0)
        out[name + "_ms_per_pair"] = per_call(time_graph(g, stream, reps, dist, device), 10)["median_ms"]
        del g
    out["saved_ms_per_pair"] = out["plain_ms_per_pair"] - out["fused_ms_per_pair"]
    return out


def run_headline(args, w: synth.Workload, device, stream, peaks: dict, dist, world: int) -> dict:
    """The headline workload: K calls in one CUDA graph, replayed `reps` times (median and min
    per call), clocks sampled during the timed replays, the end-to-end rate through the public
    binding with host buffers, and (W4A8) the activation pass timed alone."""
    import torch
    layer = Layer(w, device, stream, bias=args.bias, residual=args.residual, act=args.act)
    decode = kernel_of(w) == "decode"
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            layer.call(i)
    stream.synchronize()
    graphs = {m: layer.graph(layer.call, args.steps, m) for m in ((1, 0) if decode else (0,))}
    main_mode = 1 if decode else 0
    res = {}
    if decode:
        res["plain"] = per_call(time_graph(graphs[0], stream, args.reps, dist, device), args.steps)
    with ClockSampler(device.index if device.index is not None else 0) as clk:
        t_wall = time.perf_counter()
        res["main"] = per_call(time_graph(graphs[main_mode], stream, args.reps, dist, device), args.steps)
        t_wall = time.perf_counter() - t_wall
        if t_wall < 1.0:    # keep the sampler running long enough to see the load (replays are identical)
            with torch.cuda.stream(stream):
                for _ in range(min(int(1.0 / max(t_wall / args.reps, 1e-5)), 5000)):
                    graphs[main_mode].replay()
            stream.synchronize()
    res["clocks"] = clk.summary()
    if w.mode == synth.MODE_W4A8:
        g = layer.graph(layer.act_quant_call, args.steps, 0)
        res["act_quant"] = per_call(time_graph(g, stream, args.reps, dist, device), args.steps)
        del g
    del graphs

    # end to end through the public binding with host buffers: H2D of A, the call, D2H of C, per step
    qg = layer.qg
    A, C = layer.As[0], layer.C
    A_host = A.cpu().pin_memory()
    C_host = torch.empty(C.shape, dtype=C.dtype).pin_memory()
    e2e_steps = max(1, min(args.steps, 300))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            A.copy_(A_host, non_blocking=True)
            qg.qgemm_run(w.M, w.K, w.N, w.mode, w.block, A, w.a_dtype, layer.Bps[i % layer.copies],
                         layer.Ts[i % layer.copies] if layer.tb else None, C, w.c_dtype,
                         layer.ws if layer.wsb else None, layer.wsb, stream=stream)
            C_host.copy_(C, non_blocking=True)
            stream.synchronize()
    res["e2e_s"] = (time.perf_counter() - t0) / e2e_steps
    res.update(copies=layer.copies, copy_bytes=layer.copy_bytes, l2=layer.l2,
               launches_per_call=layer.launches_per_call(args.decode_max_m or 16),
               h2d=A.numel() * A.element_size(), d2h=C.numel() * C.element_size())
    return res


def profile_calls(w: synth.Workload, calls: int) -> dict:
    """Pack the workload's weights and run `calls` plain (eager, non-overlapped) layer calls."""
    import torch

    import weight_quantized_gemm_gb300 as qg
    device = torch.device("cuda", torch.cuda.current_device())
    A = to_torch(synth.make_activations(w), w.a_dtype, device)
    Wd = torch.from_numpy(synth.make_weights(w)).to(device)
    pb = qg.qgemm_packed_bytes(w.K, w.N, w.mode, w.a_dtype if w.mode == 0 else 0)
    tb = qg.qgemm_table_bytes(w.K, w.N, w.mode, w.block)
    Bp = torch.empty(pb, dtype=torch.uint8, device=device)
    T = torch.empty(max(tb // 4, 4), dtype=torch.float32, device=device)
    qg.qgemm_pack(Wd, w.K, w.N, w.mode, w.block, w.a_dtype if w.mode == 0 else 0, Bp, T if tb else None)
    tdt = {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}
    C = torch.empty((w.M, w.N), dtype=tdt[w.c_dtype], device=device)
    wsb = qg.qgemm_workspace_bytes(w.M, w.K, w.N, w.mode, w.block, w.a_dtype, w.c_dtype)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=device)
    for _ in range(calls):
        qg.qgemm_run(w.M, w.K, w.N, w.mode, w.block, A, w.a_dtype, Bp, T if tb else None, C, w.c_dtype, ws, wsb)
    torch.cuda.synchronize()
    return {"workload": w.name, "M": w.M, "calls": calls, "status": qg.qgemm_status()}


# the workloads measured beside the headline (one GPU each, the same JSON line)
PER_CONFIG = [
    ("int4_b64_m4_k256_n512_f32", None),
    ("int4_b64_decode_m1_k4096_n11008_bf16", None),
    *[("int8_b0_k4096_n4096_f16", m) for m in synth.INT8_M_SWEEP],
    ("int4_b64_prefill_m1024_k4096_n4096", None),
    ("float_f16_m2048_k4096_n14336", None),
]


def main():
    import dataclasses
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20, help="calls per timed CUDA graph (the K of the contract)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--reps", type=int, default=25, help="timed replays of the graph (the median is reported)")
    ap.add_argument("--workload", default=HEADLINE_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--per-config", choices=["auto", "on", "off"], default="auto",
                    help="also measure the other workloads into a per_config object (auto: with the headline)")
    ap.add_argument("--m", type=int, default=0, help="override the workload's M (e.g. the Int8-Block0 M sweep)")
    ap.add_argument("--k", type=int, default=0, help="override the workload's K (e.g. the MNN shape grid)")
    ap.add_argument("--n", type=int, default=0, help="override the workload's N (e.g. the MNN shape grid)")
    ap.add_argument("--block", type=int, default=-1,
                    help="override the workload's K-block of the {offset, scale} table (0: per channel)")
    ap.add_argument("--a-dtype", default="", choices=["", "f16", "bf16", "f32"],
                    help="override the workload's activation dtype")
    ap.add_argument("--decode-max-m", type=int, default=0,
                    help="QGEMM_OPT_DECODE_MAX_M for the run (the decode / tensor-core crossover)")
    ap.add_argument("--no-split-k", action="store_true",
                    help="QGEMM_OPT_SPLIT_K = 0: the tensor-core kernel never splits K")
    ap.add_argument("--act", default="none", choices=sorted(ACTS),
                    help="fused epilogue activation (qgemm_run_fused)")
    ap.add_argument("--bias", action="store_true", help="fused epilogue: add a float32 bias [N]")
    ap.add_argument("--residual", action="store_true", help="fused epilogue: add a residual [M][N]")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle budget of the headline's cpu_baseline")
    ap.add_argument("--print-src-hash", action="store_true", help="print the dominant kernel's source hash and exit")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="pack, run this many plain calls of the layer, print a status line and exit "
                         "(a small fixed command to run under a profiler; no timing)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.reps < 1:
        ap.error("--reps must be >= 1")
    w = synth.WORKLOADS[args.workload]
    if args.a_dtype:
        w = dataclasses.replace(w, a_dtype={"f16": synth.F16, "bf16": synth.BF16, "f32": synth.F32}[args.a_dtype])
    if args.block >= 0:
        w = dataclasses.replace(w, block=args.block)
    if args.m or args.k or args.n:
        w = dataclasses.replace(w, M=args.m or w.M, K=args.k or w.K, N=args.n or w.N)
    fused = args.bias or args.residual or args.act != "none"
    headline_default = (args.workload == HEADLINE_WORKLOAD and not (args.m or args.k or args.n or args.a_dtype)
                        and args.block < 0 and not fused)
    per_config = args.per_config == "on" or (args.per_config == "auto" and headline_default)

    if args.print_src_hash:
        print(kernel_of(w), src_hash(kernel_of(w)))
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    peaks = load_peaks()
    config = {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "mode": synth.MODE_NAMES[w.mode],
              "block": w.block if w.block else w.K, "a_dtype": DTYPE_NAME[w.a_dtype],
              "c_dtype": DTYPE_NAME[w.c_dtype]}
    if fused:
        config["epilogue"] = {"bias": args.bias, "act": args.act, "residual": args.residual}
    bound = bound_of(w)
    unit = "GB/s" if bound == "hbm" else "TFLOP/s"
    dtype = "s8" if w.mode == synth.MODE_W4A8 else DTYPE_NAME[w.a_dtype]

    if args.impl == "reference":
        if rank != 0:
            return
        r = run_reference(args, w)
        value = r["value"] if bound == "hbm" else r["tflops"]
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
                "steps": r["steps"], "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config, "tflops": r["tflops"],
                "cpu_baseline": {"value": value, "unit": unit, "cores": r["cores"], "kind": "oracle",
                                 "sample": r["sample"]},
                "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if args.profile_calls:
        print(json.dumps(profile_calls(w, args.profile_calls)))
        return
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist_mod.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = dist_mod
    import weight_quantized_gemm_gb300 as qg
    if args.decode_max_m:
        qg.qgemm_set_option(qg.OPT_DECODE_MAX_M, args.decode_max_m)
    if args.no_split_k:
        qg.qgemm_set_option(qg.OPT_SPLIT_K, 0)
    device = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream(device)

    r = run_headline(args, w, device, stream, peaks, dist, world)
    step_s = r["main"]["median_ms"] / 1e3
    alg = algorithmic_bytes(w, args.bias, args.residual)
    value, _ = metric_value(w, step_s, alg, world)
    # the dominant kernel's time: W4A8 calls are the activation pass plus the GEMM; the GEMM's
    # share is the call time less the activation pass timed alone in its own graph
    kernel_ms = None
    if w.mode == synth.MODE_W4A8:
        kernel_ms = r["main"]["median_ms"] - r["act_quant"]["median_ms"]
    roof = roofline_of(w, r["main"]["median_ms"], peaks, alg, kernel_ms)
    if kernel_ms is not None:
        roof["kernel"] = "prefill (W4A8 GEMM; time = call - activation pass alone)"
        whole = roofline_of(w, r["main"]["median_ms"], peaks, alg)
        roof["whole_call"] = {"achieved": whole["achieved"], "frac": whole["frac"],
                              "ms": r["main"]["median_ms"]}
    line = {
        "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic (seeded SplitMix64/Box-Muller inputs of the workload's shape)",
        "config": config,
        "setup": {"parallelism": f"replicas x{world}",
                  "l2": f"{r['copies']} rotating copies of the weights ({r['copy_bytes'] / 1e6:.1f} MB)"
                        f"{' and activations' if w.M > 16 else ''} (> 3x the {r['l2'] / 1e6:.0f} MB L2)",
                  "timing": f"CUDA graph of {args.steps} back-to-back calls, {args.reps} timed replays "
                            f"(CUDA events, barrier + synchronize around each); ms_per_step = median replay / "
                            f"{args.steps}",
                  "launch_overlap": ("QGEMM_OPT_LAUNCH_OVERLAP=1 (programmatic dependent launch); "
                                     "value_no_overlap without it") if kernel_of(w) == "decode" else "n/a",
                  "dtype": ("int8 activation codes x 4-bit weight codes, exact int32 sums (f16 tensor "
                            "cores, every partial sum an exact integer)") if w.mode == synth.MODE_W4A8 else
                           f"{DTYPE_NAME[w.a_dtype]} activations, float32 accumulation"},
        "ms_per_step_min": r["main"]["min_ms"],
        "tflops": w.flops / step_s / 1e12 * world, "gbs": alg / step_s / 1e9 * world,
        "roofline": roof, "clocks": r["clocks"],
        "gpu_launches": args.steps * r["launches_per_call"] * args.reps,
        "gpu_launches_per_step": r["launches_per_call"],
        "e2e": {"value": metric_value(w, r["e2e_s"], alg, world)[0], "unit": unit, "ms_per_step": r["e2e_s"] * 1e3,
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
    }
    if "plain" in r:
        line["ms_per_step_no_overlap"] = r["plain"]["median_ms"]
        line["value_no_overlap"] = metric_value(w, r["plain"]["median_ms"] / 1e3, alg, world)[0]
    if "act_quant" in r:
        line["act_quant_ms_per_step"] = r["act_quant"]["median_ms"]
    if rank == 0 and not args.no_cpu_baseline:
        ra = argparse.Namespace(steps=10 ** 6, warmup=1, cpu_seconds=args.cpu_seconds)
        ref = run_reference(ra, w)
        line["cpu_baseline"] = {"value": ref["value"] if bound == "hbm" else ref["tflops"], "unit": unit,
                                "cores": ref["cores"], "kind": "oracle", "sample": ref["sample"]}
    if per_config:
        entries = {}
        for name, m in PER_CONFIG:
            pw = synth.WORKLOADS[name]
            if m is not None:
                pw = dataclasses.replace(pw, M=m)
            key = name if m is None else f"{name}_m{m}"
            entries[key] = bench_entry(pw, device, stream, peaks, args.reps, dist, args.decode_max_m or 16,
                                       0.0 if args.no_cpu_baseline else 3.0, rank)
            torch.cuda.empty_cache()
        entries["fused_act_quant_pair"] = bench_fused_pair(device, stream, args.reps, dist)
        line["per_config"] = entries
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
