"""Throughput of the weight-quantized linear layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step is one call of the layer (qgemm_run) on the workload's synthetic inputs. The
default workload is the decode GEMV of a 7B-class FFN up-projection: Int4-Block64 weights,
M=1, K=4096, N=11008, bf16 activations and output. Its metric is the weight-stream
bandwidth (the layer's algorithmic bytes: packed weights, {offset, scale} table,
activations in, output out) and, beside it, TFLOPS = 2*M*K*N / t (the benchmark page's
convention, "MNN GemmSpeed 基准测试实战" «测量流程»).

Timing: weights are packed once (offline, as on the page), then copied into enough
rotating copies to exceed the L2 cache about 3x, so every call streams its weights from HBM.
W warm-up calls, then exactly K calls captured in one CUDA graph and replayed between CUDA
events on the launching stream, with a barrier and synchronize on both sides; the time is
the max over ranks. GPU clocks are sampled with nvidia-smi during the timed region.

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
DEFAULT_WORKLOAD = "int4_b64_decode_m1_k4096_n11008_bf16"
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
}


def kernel_of(w: synth.Workload) -> str:
    return "decode" if (w.M <= 16 and w.mode != synth.MODE_W4A8 and w.a_dtype != synth.F32) else "prefill"


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


def run_gpu(args, w: synth.Workload, rank: int, world: int, dist) -> dict:
    import torch

    import weight_quantized_gemm_gb300 as qg
    if args.decode_max_m:
        qg.qgemm_set_option(qg.OPT_DECODE_MAX_M, args.decode_max_m)
    if args.no_split_k:
        qg.qgemm_set_option(qg.OPT_SPLIT_K, 0)
    device = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream(device)
    tdt = {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}
    A_np = synth.make_activations(w)
    W_np = synth.make_weights(w)
    K, N, M = w.K, w.N, w.M
    with torch.cuda.stream(stream):
        A = to_torch(A_np, w.a_dtype, device)
        Wd = torch.from_numpy(W_np).to(device)
        pb = qg.qgemm_packed_bytes(K, N, w.mode, w.w_dtype if w.mode == 0 else 0)
        tb = qg.qgemm_table_bytes(K, N, w.mode, w.block)
        Bp0 = torch.empty(pb, dtype=torch.uint8, device=device)
        T0 = torch.empty(max(tb // 4, 4), dtype=torch.float32, device=device)
        qg.qgemm_pack(Wd, K, N, w.mode, w.block, w.a_dtype if w.mode == 0 else 0, Bp0, T0 if tb else None,
                      stream=stream)
        del Wd
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        copy_bytes = pb + tb
        a_bytes = A.numel() * A.element_size() if M > 16 else 0
        copies = max(2, -(-3 * l2 // max(copy_bytes + a_bytes, 1)))
        Bps = [Bp0] + [Bp0.clone() for _ in range(copies - 1)]
        Ts = [T0] + [T0.clone() for _ in range(copies - 1)]
        # for M > 16 the activations are large too: rotate them with the weights
        As = [A] + ([A.clone() for _ in range(copies - 1)] if M > 16 else [])
        C = torch.empty((M, N), dtype=tdt[w.c_dtype], device=device)
        wsb = qg.qgemm_workspace_bytes(M, K, N, w.mode, w.block, w.a_dtype, w.c_dtype)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=device)
        # the fused epilogue's inputs (qgemm_run_fused), when asked for
        bias = (torch.from_numpy(synth.normal64(N, 11, stream=4, std=0.5).astype(np.float32)).to(device)
                if args.bias else None)
        res = (to_torch(synth.encode(synth.normal64(M * N, 12, stream=5).reshape(M, N), w.c_dtype), w.c_dtype, device)
               if args.residual else None)
    stream.synchronize()
    s_ptr = stream.cuda_stream
    lib = qg.load()
    act = ACTS[args.act]
    fused = bias is not None or res is not None or act != 0

    def call(i):
        if fused:
            rc = lib.qgemm_run_fused(M, K, N, w.mode, w.block, As[i % len(As)].data_ptr(), w.a_dtype,
                                     Bps[i % copies].data_ptr(), Ts[i % copies].data_ptr() if tb else None,
                                     None if bias is None else bias.data_ptr(), act,
                                     None if res is None else res.data_ptr(), C.data_ptr(), w.c_dtype,
                                     ws.data_ptr(), wsb, s_ptr)
        else:
            rc = lib.qgemm_run(M, K, N, w.mode, w.block, As[i % len(As)].data_ptr(), w.a_dtype,
                               Bps[i % copies].data_ptr(), Ts[i % copies].data_ptr() if tb else None, C.data_ptr(),
                               w.c_dtype, ws.data_ptr(), wsb, s_ptr)
        if rc != 0:
            raise qg.QgemmError(rc, "qgemm_run")

    # kernels per call: W4A8 = activation quantization + GEMM; otherwise one GEMM launch per
    # 16-row decode launch (or one tensor-core launch), plus the split-K reduction when the call
    # splits K (its workspace holds the partial sums)
    if w.mode == synth.MODE_W4A8:
        launches_per_call = 2
    else:
        decode_path = w.a_dtype != synth.F32 and M <= (args.decode_max_m or 16)
        launches_per_call = (-(-M // 16) if decode_path else 1) * (2 if wsb > 0 else 1)
    # warm-up (eager), then one CUDA graph of exactly K calls per launch mode: plain stream
    # order, and with QGEMM_OPT_LAUNCH_OVERLAP (each decode call may start while the previous
    # one finishes; it prefetches weights and waits for the previous kernel before A and C).
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(i)
    stream.synchronize()
    graphs = {}
    for mode in (0, 1):
        qg.qgemm_set_option(qg.OPT_LAUNCH_OVERLAP, mode)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(args.steps):
                call(i)
        graphs[mode] = g
    qg.qgemm_set_option(qg.OPT_LAUNCH_OVERLAP, 0)
    stream.synchronize()

    def timed(g):
        g.replay()          # one untimed replay: the graph's own first-launch cost stays out
        stream.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            start.record(stream)
            g.replay()
            end.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        return max_over_ranks(start.elapsed_time(end), dist, device)

    ms_plain = timed(graphs[0])
    with ClockSampler(device.index if device.index is not None else 0) as clk:
        t_wall = time.perf_counter()
        ms = timed(graphs[1])
        t_wall = time.perf_counter() - t_wall
        if t_wall < 1.0:    # keep the sampler running long enough to see the load (replays are identical)
            with torch.cuda.stream(stream):
                for _ in range(min(int(1.0 / max(t_wall, 1e-4)), 2000)):
                    graphs[1].replay()
            stream.synchronize()
    clocks = clk.summary()

    # end to end through the public API with host buffers: H2D of A, the call, D2H of C, per step
    A_host = A.cpu().pin_memory()
    C_host = torch.empty(C.shape, dtype=C.dtype).pin_memory()
    e2e_steps = max(1, min(args.steps, 300))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            A.copy_(A_host, non_blocking=True)
            qg.qgemm_run(M, K, N, w.mode, w.block, A, w.a_dtype, Bps[i % copies], Ts[i % copies] if tb else None, C,
                         w.c_dtype, ws if wsb else None, wsb, stream=stream)
            C_host.copy_(C, non_blocking=True)
            stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    return {"ms": ms, "ms_plain": ms_plain, "clocks": clocks, "copies": copies, "copy_bytes": copy_bytes, "l2": l2,
            "launches_per_call": launches_per_call, "e2e_s": e2e_s,
            "h2d": A.numel() * A.element_size(), "d2h": C.numel() * C.element_size()}


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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
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
    ap.add_argument("--print-src-hash", action="store_true", help="print the dominant kernel's source hash and exit")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="pack, run this many plain calls of the layer, print a status line and exit "
                         "(a small fixed command to run under a profiler; no timing)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    import dataclasses
    w = synth.WORKLOADS[args.workload]
    if args.a_dtype:
        w = dataclasses.replace(w, a_dtype={"f16": synth.F16, "bf16": synth.BF16, "f32": synth.F32}[args.a_dtype])
    if args.block >= 0:
        w = dataclasses.replace(w, block=args.block)
    if args.m or args.k or args.n:
        w = dataclasses.replace(w, M=args.m or w.M, K=args.k or w.K, N=args.n or w.N)

    if args.print_src_hash:
        print(kernel_of(w), src_hash(kernel_of(w)))
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    peaks = load_peaks()
    base_config = {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "mode": synth.MODE_NAMES[w.mode],
                   "block": w.block if w.block else w.K, "a_dtype": DTYPE_NAME[w.a_dtype],
                   "c_dtype": DTYPE_NAME[w.c_dtype]}
    if args.bias or args.residual or args.act != "none":
        base_config["epilogue"] = {"bias": args.bias, "act": args.act, "residual": args.residual}

    if args.impl == "reference":
        if rank != 0:
            return
        r = run_reference(args, w)
        line = {"impl": "reference", "metric": METRIC, "value": r["value"], "unit": r["unit"], "n_gpus": args.gpus,
                "steps": r["steps"], "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": base_config, "tflops": r["tflops"],
                "cpu_baseline": {"value": r["value"], "unit": r["unit"], "cores": r["cores"], "kind": "oracle",
                                 "sample": r["sample"]},
                "e2e": {"value": r["value"], "unit": r["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
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
    r = run_gpu(args, w, rank, world, dist)
    step_s = r["ms"] / 1e3 / args.steps
    alg = algorithmic_bytes(w, args.bias, args.residual)
    gbs = job_rate(alg, step_s, world) / 1e9
    tflops = job_rate(w.flops, step_s, world) / 1e12
    bound = bound_of(w)
    if bound == "hbm":
        achieved, peak, unit = alg / step_s / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = w.flops / step_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    line = {
        "metric": METRIC, "value": gbs if bound == "hbm" else tflops, "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[w.a_dtype],
        "data": "synthetic (seeded SplitMix64/Box-Muller inputs of the workload's shape)",
        "config": dict(base_config, parallelism=f"replicas x{world}",
                       l2=f"{r['copies']} rotating copies of the weights ({r['copy_bytes'] / 1e6:.1f} MB)"
                          f"{' and activations' if w.M > 16 else ''} (> 3x the {r['l2'] / 1e6:.0f} MB L2)",
                       timing=f"CUDA graph of {args.steps} back-to-back calls, CUDA events",
                       launch_overlap="QGEMM_OPT_LAUNCH_OVERLAP=1 (programmatic dependent launch)"),
        "tflops": tflops, "gbs": gbs,
        "ms_per_step_no_overlap": r["ms_plain"] / args.steps,
        "value_no_overlap": (job_rate(alg, r["ms_plain"] / 1e3 / args.steps, world) / 1e9) if bound == "hbm"
        else (job_rate(w.flops, r["ms_plain"] / 1e3 / args.steps, world) / 1e12),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                     "peak_source": f"{peaks['source']} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops'})",
                     "traffic": measured_traffic(w), "algorithmic_bytes": alg,
                     "kernel": kernel_of(w)},
        "clocks": r["clocks"], "gpu_launches": args.steps * r["launches_per_call"],
        "e2e": {"value": (alg / r["e2e_s"] / 1e9) if bound == "hbm" else (w.flops / r["e2e_s"] / 1e12),
                "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "ms_per_step": r["e2e_s"] * 1e3,
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
    }
    if rank == 0 and not args.no_cpu_baseline:
        ra = argparse.Namespace(steps=10 ** 6, warmup=1, cpu_seconds=10.0)
        ref = run_reference(ra, w)
        line["cpu_baseline"] = {"value": ref["value"], "unit": ref["unit"], "cores": ref["cores"], "kind": "oracle",
                                "sample": ref["sample"]}
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
