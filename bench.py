#!/usr/bin/env python3
"""Benchmark of the FP32 GEMM library on GB300: one JSON line on stdout.

A step is one call of the library on the workload's synthetic inputs, already
resident in HBM (default workload: M = N = K = 4096, alpha = 1, beta = 0,
row-major, A and B uniform[-1, 1) from seed 2).  The L2 is flushed between
timed steps by a 256 MiB memset outside the step's event pair.  The call is
fgemm_sgemm_staged with the launch-time model's staging choice and a workspace
allocated once beforehand (``--entry plain``: the plain entry points, no workspace);
its copies of the operands stored with k contiguous are part of every timed step.

Reported, besides the contract keys:
  roofline      the GEMM kernel against the CUDA-core FP32 peak
                (SMs x 128 FMA/clk x 2 FLOP x 2070 MHz), "bound": "alu"
  e2e           the same metric with pinned host buffers: H2D of A, B, the call,
                D2H of C, every step
  cpu_baseline  the FP64 oracle timed on this host's cores on a bounded sample
                of the same problem (whole rows of C)
  clocks        nvidia-smi samples taken during the timed region
  secondary     (default run) the fused FC layer against the plain GEMM of its shape,
                256^3 back to back in a CUDA graph, 1024^3 with alpha and beta

``--impl reference`` times the FP64 oracle instead (the only reference
implementation this project has), each step a bounded sample of the workload.

Under torchrun (WORLD_SIZE > 1) every rank runs its own copy of the workload
(weak scaling, no data-path collective); the step time is the max over ranks
and ``value`` counts the work of all ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from dense_fp32_gemm_sm_gb300 import workloads  # noqa: E402

METRIC = "FP32 GEMM TFLOP/s (2*M*N*K/s) at 4096^3; fraction of GB300 FP32 peak"
UNIT = "TFLOP/s"
FMA_PER_CLK_PER_SM = 128  # FP32 lanes per SM
STATED_SM_MHZ = 2070.0  # maximum SM clock of GB300
L2_FLUSH_BYTES = 256 << 20
# Best FP32 kernel of GPU架构下的矩阵乘法深入优化 at 4096^3 ("5. warp tiling + double
# buffer", V100S-PCIE-32GB): 10642 GFLOPS.  Other hardware: context only.
PAGES_4096_TFLOPS = 10.642
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("fgemm", "reference"), default="fgemm")
    ap.add_argument("--workload", choices=workloads.WORKLOADS, default="square4096")
    ap.add_argument("--entry", choices=("staged", "plain"), default="staged",
                    help="FP32 calls through fgemm_sgemm_staged (the model decides whether to "
                         "copy k-contiguous operands k-major into a workspace first) or the "
                         "plain entry points")
    ap.add_argument("--config", type=int, default=-1,
                    help="explicit kernel configuration id (default: the library's choice)")
    ap.add_argument("--e2e-steps", type=int, default=100,
                    help="pipelined end-to-end steps timed (the first inputs and the last "
                         "result are not overlapped; more steps amortise them)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the fused-vs-unfused FC layer timing added to the default run")
    ap.add_argument("--math", choices=("fp32", "tf32", "3xtf32"), default="fp32",
                    help="arithmetic: FP32 CUDA cores (the metric) or the tcgen05 tensor-core path")
    ap.add_argument("--splitk", type=int, default=0,
                    help="S > 1: split-K GEMM into S slices with a workspace (single problems)")
    ap.add_argument("--epilogue", choices=("workload", "none"), default="workload",
                    help="'none' drops the workload's bias/ReLU (plain sgemm at the same shape)")
    ap.add_argument("--graph-calls", type=int, default=None,
                    help="N > 0: also time N back-to-back library calls captured in one CUDA "
                         "graph (warm L2, no host launch cost): the per-call latency of small "
                         "shapes (default: 200 for square256, 0 otherwise)")
    ap.add_argument("--cpu-baseline-table", action="store_true",
                    help="no GPU: time the FP64 oracle on every workload on one host core and on "
                         "all of them (bounded samples), one JSON line each")
    return ap.parse_args(argv)


KERNEL_SOURCES = {
    "simt": ("simt_gemm.cuh", "simt_launch.cuh", "inst_nn.cu", "inst_nt.cu", "inst_tn.cu",
             "inst_tt.cu"),
    "stage": ("stage.cu",),
    "tcgen05": ("tc_gemm.cuh", "tc_gemm.cu"),
}


def _code_only(text: str) -> str:
    """C/CUDA source without comments and with whitespace collapsed (the sources'
    string literals hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(family: str) -> str:
    """Short hash of one kernel family's CUDA code (comments and layout ignored), or of
    several joined by '+' (a staged call: "simt+stage"); profile summaries record the
    hash of the code they measured."""
    m = hashlib.sha256()
    for name in [n for f in family.split("+") for n in KERNEL_SOURCES[f]]:
        m.update(name.encode())
        with open(os.path.join(ROOT, "dense_fp32_gemm_sm_gb300", "csrc", name), encoding="utf-8") as fh:
            m.update(_code_only(fh.read()).encode())
    return m.hexdigest()[:16]


def build_info():
    """nvcc version and the flags the library was compiled with."""
    from dense_fp32_gemm_sm_gb300 import _build
    try:
        out = subprocess.run([_build.nvcc(), "--version"], capture_output=True, text=True,
                             timeout=30).stdout
        lines = [l for l in out.splitlines() if "release" in l]
        version = lines[0].strip() if lines else "unknown"
    except (OSError, subprocess.SubprocessError):
        version = "unknown"
    flags = [f for f in _build.ARCH + _build.NVCC_FLAGS if not f.startswith("-I")]
    return {"nvcc": version, "flags": " ".join(flags)}


def recorded_traffic(config_name: str, workload: str):
    """DRAM bytes per launch from profiles/<config>_<workload>.md, if measured on these sources."""
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (config_name, workload))
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path, encoding="utf-8") as f:
        for line in f:
            key, sep, val = line.strip().partition(":")
            if sep and key in ("source_sha256", "traffic_bytes_per_launch"):
                fields[key] = val.strip()
    family = config_name.split("_")[0]
    if family not in KERNEL_SOURCES:
        return None
    if "_staged_" in config_name:
        family += "+stage"
    if (fields.get("source_sha256") != kernel_source_hash(family)
            or "traffic_bytes_per_launch" not in fields):
        return None
    return int(fields["traffic_bytes_per_launch"])


# ---- distributed plumbing (one process per GPU, replicas) -----------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world):
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def aggregate(units: float, seconds: float, world: int, device=None):
    """Sum of the ranks' units and max of their times (a no-op for one process)."""
    if world <= 1:
        return units, seconds
    t = torch.tensor([units, seconds], dtype=torch.float64, device=device)
    s = t.clone()
    torch.distributed.all_reduce(s, op=torch.distributed.ReduceOp.SUM)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(s[0]), float(t[1])


# ---- clocks -------------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples every 50 ms while the timed region runs."""

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.gpu_index, self.enabled = gpu_index, enabled
        self.proc, self.path = None, None

    def __enter__(self):
        if self.enabled:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + SMI_FIELDS,
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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

    def summary(self):
        if not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        busy = [v for v in sm if mx and v > 0.5 * max(mx)] or sm
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# ---- the library arm ----------------------------------------------------------------------

def tensor_peak_tflops(math: str):
    """Dense TF32 tensor peak derived from the measured BF16 peak (MEASURED_PEAKS.json,
    burst) times the nominal TF32/BF16 ratio 1.1/2.25; 3xTF32 does three TF32 products
    per FP32 product, so its FP32-equivalent peak is a third of that."""
    bf16, src = 1900.0, "fallback 1.9 PFLOP/s bf16"
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            bf16, src = float(json.load(f)["bf16_tflops"]), "measured bf16 burst"
    tf32 = bf16 * 1.1 / 2.25
    div = 3.0 if math == "3xtf32" else 1.0
    return tf32 / div, "%s %.1f TFLOP/s x 1.1/2.25 (nominal TF32/BF16)%s" % (
        src, bf16, " / 3 products" if div == 3.0 else "")


def calibrate_tf32_tflops(dev, n: int = 8192, reps: int = 5):
    """Calibration of the dense TF32 tensor rate on this GPU (never a product path):
    the vendor library's TF32 GEMM (torch.matmul with TF32 allowed) on one n^3 problem,
    best of `reps` calls after warm-up, CUDA events.  Returns TFLOP/s."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        g = torch.Generator(device=dev).manual_seed(0)
        a = torch.rand((n, n), device=dev, generator=g)
        b = torch.rand((n, n), device=dev, generator=g)
        c = torch.empty((n, n), device=dev)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) / 1e3
            best = t if best is None else min(best, t)
        del a, b, c
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / best / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def small_secondary(fg, dev, stream, graph_calls: int = 200, calls: int = 20):
    """The small workloads beside the headline: 256^3 as the device time per call of
    `graph_calls` calls captured back to back in one CUDA graph (warm L2, no host launch
    cost), and 1024^3 with alpha = 1.5, beta = 0.5 as the median of `calls` single calls
    with L2 flushed (C restored from C0 outside the timed events)."""
    out = {}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sh = stream.cuda_stream
    w = workloads.make("square256")
    dA, dB, dC = w.A.to(dev), w.B.to(dev), torch.empty((w.M, w.N), device=dev)

    def call256():
        fg.sgemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta, dC, w.ldc,
                 stream=sh)

    with torch.cuda.stream(stream):
        call256()  # one-time setup outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(graph_calls):
            call256()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        graph.replay()
        torch.cuda.synchronize()
        g0.record(stream)
        graph.replay()
        g1.record(stream)
    torch.cuda.synchronize()
    per = g0.elapsed_time(g1) / 1e3 / graph_calls
    out["square256_back_to_back"] = {"workload": describe(w), "calls": graph_calls,
                                     "us_per_call": round(per * 1e6, 3),
                                     "tflops": round(w.flops / per / 1e12, 3),
                                     "l2": "warm (calls back to back in one CUDA graph)"}
    del graph
    w = workloads.make("square1024")
    dA, dB = w.A.to(dev), w.B.to(dev)
    dC0, dC = w.C0.to(dev), torch.empty((w.M, w.N), device=dev)
    times = []
    with torch.cuda.stream(stream):
        for i in range(calls + 3):
            flush.zero_()
            dC.copy_(dC0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fg.sgemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta, dC, w.ldc,
                     stream=sh)
            e1.record(stream)
            e1.synchronize()
            if i >= 3:
                times.append(e0.elapsed_time(e1) / 1e3)
    t = statistics.median(times)
    out["square1024_alpha_beta"] = {"workload": describe(w), "calls": calls,
                                    "us_per_call": round(t * 1e6, 2),
                                    "tflops": round(w.flops / t / 1e12, 3),
                                    "l2": "flushed before every call"}
    del flush
    torch.cuda.empty_cache()
    return out


def fc_secondary(fg, dev, stream, calls: int = 3, clocks: bool = True, entry: str = "staged"):
    """The fully-connected layer (X 8192 x 4096, W 4096 x 11008, bias, ReLU) fused in the
    GEMM epilogue against the plain GEMM of the same shape: `calls` timed calls each
    (one warm-up call, L2 flushed before every call, CUDA events on the stream), and
    the fused/unfused throughput ratio.  Both through the same entry point as the
    headline (`entry`)."""
    w = workloads.make("fc8192x4096x11008")
    dA, dB, dbias = w.A.to(dev), w.B.to(dev), w.bias.to(dev)
    dC = torch.empty((w.M, w.N), device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sh = stream.cuda_stream
    ws, need = staged_workspace(fg, w, dev) if entry == "staged" else (None, 0)

    def call(bias, relu):
        if entry == "staged":
            fg.sgemm_staged(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, 0, dB, w.ldb, 0,
                            w.beta, dC, w.ldc, 0, 1, bias, relu, fg.STAGE_AUTO, ws, need,
                            stream=sh)
        elif bias is not None or relu:
            fg.sgemm_bias_relu(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta,
                               dC, w.ldc, bias, relu, stream=sh)
        else:
            fg.sgemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta, dC, w.ldc,
                     stream=sh)

    def fused():
        call(dbias, True)

    def plain():
        call(None, False)

    out = {}
    sampler = ClockSampler(dev.index or 0, enabled=clocks)
    with sampler, torch.cuda.stream(stream):
        for name, fn in (("fused_bias_relu", fused), ("plain_gemm", plain)):
            fn()
            times = []
            for _ in range(calls):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1) / 1e3)
            t = statistics.median(times)
            out[name] = {"tflops": round(w.flops / t / 1e12, 3), "ms": round(t * 1e3, 4)}
    del dA, dB, dbias, dC, flush, ws
    torch.cuda.empty_cache()
    res = {"workload": describe(w), "calls_each": calls, "entry": entry,
           "l2": "flushed before every call",
           "fused_over_unfused": round(out["fused_bias_relu"]["tflops"] /
                                       out["plain_gemm"]["tflops"], 4), **out}
    clk = sampler.summary()
    if clk is not None:
        res["clocks"] = clk
    return res


def stated_peak_tflops(device) -> tuple:
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    return sms * FMA_PER_CLK_PER_SM * 2 * STATED_SM_MHZ * 1e6 / 1e12, sms


MATHS = {"fp32": 0, "tf32": 1, "3xtf32": 2}


def _launch(fg, w, cfg, dA, dB, dC, dbias, stream, math="fp32", splitk=None, staged=None):
    """One step: the library call of the workload (the bench's unit of work).
    staged: (workspace, bytes) to call fgemm_sgemm_staged with the model's choice."""
    nb = max(1, w.batch)
    sA = w.M * w.K if w.batch else 0
    sB = w.N * w.K if w.batch else 0
    sC = w.M * w.N if w.batch else 0
    if staged is not None and splitk is None and math == "fp32" and cfg < 0:
        ws, need = staged
        fg.sgemm_staged(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, sA, dB, w.ldb, sB, w.beta,
                        dC, w.ldc, sC, nb, dbias, w.relu, fg.STAGE_AUTO, ws, need, stream=stream)
    elif splitk is not None:
        splits, ws, need = splitk
        fg.sgemm_splitk(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta, dC,
                        w.ldc, dbias, w.relu, splits, ws, need, stream=stream)
    elif math != "fp32":
        fg.gemm_math(MATHS[math], w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, sA, dB, w.ldb, sB,
                     w.beta, dC, w.ldc, sC, nb, dbias, w.relu, stream=stream)
    elif cfg >= 0:
        fg.gemm_explicit(cfg, w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, sA, dB, w.ldb, sB,
                         w.beta, dC, w.ldc, sC, nb, dbias, w.relu, stream=stream)
    elif w.batch:
        fg.sgemm_strided_batched(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, sA, dB, w.ldb, sB,
                                 w.beta, dC, w.ldc, sC, w.batch, stream=stream)
    elif w.bias is not None or w.relu:
        fg.sgemm_bias_relu(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta, dC,
                           w.ldc, dbias, w.relu, stream=stream)
    else:
        fg.sgemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta, dC, w.ldc,
                 stream=stream)


def cpu_baseline(w, seconds: float, threads=None):
    """FP64 oracle on whole rows of C (all columns), sized to take about `seconds`, on
    `threads` host threads (default: all)."""
    import oracle
    threads = threads or oracle.default_threads()
    A = w.A.numpy().reshape(-1) if not w.batch else w.A[0].numpy().reshape(-1)
    B = w.B.numpy().reshape(-1) if not w.batch else w.B[0].numpy().reshape(-1)
    C0 = None if w.C0 is None else w.C0.numpy().reshape(-1)

    def timed(rows):
        t0 = time.perf_counter()
        oracle.gemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, A, w.lda, B, w.ldb, w.beta, C0, w.ldc,
                    bias=w.bias, relu=w.relu, rows=rows, threads=threads, want_mag=False)
        return time.perf_counter() - t0

    probe = min(w.M, max(threads, 8))
    t_probe = timed(list(range(probe)))
    n = int(min(w.M, max(probe, seconds / max(t_probe, 1e-9) * probe)))
    n = max(threads, (n // threads) * threads) if n >= threads else n
    t = timed(list(range(n)))
    flops = 2.0 * n * w.N * w.K
    return {"value": flops / t / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "%d of %d rows of C (all %d columns)%s, FP64 oracle, %.1f s" % (
                n, w.M, w.N, " of problem 0 of %d" % w.batch if w.batch else "", t)}


def run_fgemm(args, rank, world, local_rank):
    import dense_fp32_gemm_sm_gb300 as fg
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device; the library has no CPU path")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fg.library()
    w = workloads.make(args.workload)
    if args.epilogue == "none":
        w.bias, w.relu = None, False
    stream = torch.cuda.Stream(dev)
    sh = stream.cuda_stream

    dA, dB = w.A.to(dev), w.B.to(dev)
    dbias = w.bias.to(dev) if w.bias is not None else None
    c_shape = (max(1, w.batch), w.M, w.N) if w.batch else (w.M, w.N)
    dC = torch.zeros(c_shape, device=dev)
    dC0 = w.C0.to(dev) if w.C0 is not None else None
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    splitk = None
    if args.splitk > 1:
        if w.batch:
            raise SystemExit("bench.py: --splitk takes single problems")
        need = fg.splitk_workspace_size(w.M, w.N, w.K, args.splitk)
        splitk = (args.splitk, torch.empty(need // 4, device=dev), need)
    staged = staged_workspace(fg, w, dev) if args.entry == "staged" else None
    torch.cuda.synchronize()

    def step():
        if dC0 is not None:  # beta != 0: restore C so every step computes the same thing
            dC.copy_(dC0)
        _launch(fg, w, args.config, dA, dB, dC, dbias, sh, args.math, splitk, staged)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local_rank, enabled=not args.no_clocks)
    barrier(world)
    torch.cuda.synchronize()
    with sampler, torch.cuda.stream(stream):
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()  # evict A, B, C from L2 (outside the event pair)
            if dC0 is not None:
                dC.copy_(dC0)
            starts[i].record(stream)
            _launch(fg, w, args.config, dA, dB, dC, dbias, sh, args.math, splitk, staged)
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier(world)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    local_s = sum(step_ms) / 1e3
    total_flops, max_s = aggregate(w.flops * args.steps, local_s, world,
                                   dev if world > 1 else None)
    value = total_flops / max_s / 1e12
    kernel_ms = statistics.mean(step_ms)
    peak, sms = stated_peak_tflops(dev)
    achieved = w.flops / (kernel_ms / 1e3) / 1e12

    # End to end: every step copies its inputs from pinned host memory to the device,
    # runs the library call and reads its result back into pinned host memory.  The
    # steps are pipelined as a user would: three streams (host->device copies, the
    # GEMM, device->host copies) and two device buffer sets, so the copies of one step
    # overlap the GEMM of its neighbours.  The timed region runs from the first copy
    # of the first timed step to the end of the last result read.
    hA, hB = w.A.pin_memory(), w.B.pin_memory()
    hC = [torch.empty(c_shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    hC0 = w.C0.pin_memory() if w.C0 is not None else None
    h2d = hA.numel() * 4 + hB.numel() * 4 + (hC0.numel() * 4 if hC0 is not None else 0)
    d2h = hC[0].numel() * 4
    sets = [(dA, dB, dC), (torch.empty_like(dA), torch.empty_like(dB), torch.empty_like(dC))]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for it in range(args.e2e_steps + 2):
        b = it % 2
        xA, xB, xC = sets[b]
        if it >= 2:  # buffers of step it-2: its result must have been read back
            h2d_s.wait_event(ev_out[b])
        if it == 2:
            e_start.record(h2d_s)
        with torch.cuda.stream(h2d_s):
            xA.copy_(hA, non_blocking=True)
            xB.copy_(hB, non_blocking=True)
            if hC0 is not None:
                xC.copy_(hC0, non_blocking=True)
        ev_in[b].record(h2d_s)
        stream.wait_event(ev_in[b])
        with torch.cuda.stream(stream):
            _launch(fg, w, args.config, xA, xB, xC, dbias, sh, args.math, splitk, staged)
        ev_done[b].record(stream)
        d2h_s.wait_event(ev_done[b])
        with torch.cuda.stream(d2h_s):
            hC[b].copy_(xC, non_blocking=True)
        ev_out[b].record(d2h_s)
    e_end.record(d2h_s)
    torch.cuda.synchronize()
    e2e_s = e_start.elapsed_time(e_end) / 1e3 / args.e2e_steps
    e2e_flops, e2e_max = aggregate(w.flops, e2e_s, world, dev if world > 1 else None)

    back_to_back = None
    if args.graph_calls is None:
        args.graph_calls = 200 if args.workload == "square256" else 0
    if args.graph_calls > 0:
        # N calls back to back in one CUDA graph: no host launch cost and no L2 flush in
        # between, so this is the device time per call of a user's captured sequence.
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            step()  # every one-time setup happens before the capture
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(args.graph_calls):
                _launch(fg, w, args.config, dA, dB, dC, dbias, sh, args.math, splitk, staged)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            graph.replay()
            torch.cuda.synchronize()
            g0.record(stream)
            graph.replay()
            g1.record(stream)
        torch.cuda.synchronize()
        per_call = g0.elapsed_time(g1) / 1e3 / args.graph_calls
        back_to_back = {"calls": args.graph_calls, "us_per_call": round(per_call * 1e6, 3),
                        "value": round(w.flops / per_call / 1e12, 4), "unit": UNIT,
                        "l2": "warm (calls back to back in one CUDA graph)"}

    def launches(config, M, N, K, batch, ta=w.ta, tb=w.tb):
        """Kernel launches of one library call with this configuration (None: select),
        as the library counts them (fgemm_launch_count)."""
        if config is None or config < 0:
            config = fg.select_config(ta, tb, M, N, K, batch, True, sms)
        name = fg.config_name(config)
        kk = K if w.alpha != 0 else 0
        return name, fg.launch_count(config, ta, tb, M, N, kk, batch, True, sms)

    stage_mask = 0
    if staged is not None and args.config < 0 and splitk is None and args.math == "fp32":
        stage_mask = fg.staged_choice(w.ta, w.tb, w.M, w.N, w.K, max(1, w.batch), False, False,
                                      True, True, sms)
    if stage_mask:
        # the copies (one launch per staged operand and 65535 problems), then the GEMM
        # in the layout they leave
        nb = max(1, w.batch)
        kernel_name, n_batch_launches = launches(
            None, w.M, w.N, w.K, nb, 1 if stage_mask & 1 else w.ta, 0 if stage_mask & 2 else w.tb)
        n_batch_launches += bin(stage_mask).count("1") * (-(-nb // 65535))
        kernel_name += {1: "_staged_a", 2: "_staged_b", 3: "_staged_ab"}[stage_mask]
    else:
        kernel_name, n_batch_launches = launches(args.config, w.M, w.N, w.K, max(1, w.batch))
    if splitk is not None:
        # partial GEMMs: the slices of equal depth as one strided batch, the shorter last
        # slice as a second call; then the reduction kernel
        Ks = -(-(-(-w.K // args.splitk)) // 32) * 32
        S = -(-w.K // Ks)
        Klast = w.K - (S - 1) * Ks
        full = S if Klast == Ks else S - 1
        parts = []
        n_batch_launches = 1
        if full > 0:
            name, n = launches(None, w.M, w.N, Ks, full)
            parts.append(name)
            n_batch_launches += n
        if full < S:
            name, n = launches(None, w.M, w.N, Klast, 1)
            parts.append(name)
            n_batch_launches += n
        kernel_name = "splitk%d(%s)" % (args.splitk, "+".join(parts))
    # The tensor-core kernels take every layout of these (16-byte aligned) workloads;
    # TF32 runs 128 x 256 MMAs when one operand is stored K-major, 3xTF32 128 x 128.
    tensor_path = args.math != "fp32"
    if tensor_path:
        wide = args.math == "tf32" and (w.ta == 0 or w.tb == 1)
        kernel_name = "tcgen05_%s_mma128x%d" % (args.math, 256 if wide else 128)
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_s * 1e3 /
                                                                          args.steps, 5),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (round(value / PAGES_4096_TFLOPS, 3)
                        if args.workload == "square4096" else None),
        "dtype": {"fp32": "f32", "tf32": "tf32 (fp32 accumulate)",
                  "3xtf32": "3xtf32 (tf32 hi/lo split, fp32 accumulate)"}[args.math]
        if tensor_path else "f32", "data": "synthetic",
        "config": {"workload": describe(w), "kernel_config": kernel_name,
                   "entry": entry_text(args, staged, stage_mask),
                   "l2": "flushed between steps (256 MiB memset outside the timed event pair)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "gpu_launches": args.steps * n_batch_launches,
        "roofline": {"bound": "alu", "achieved": round(achieved, 4), "peak": round(peak, 3),
                     "unit": UNIT, "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic(kernel_name, args.workload),
                     "peak_source": "derived: %d SMs x %d FP32 FMA/clk x 2 FLOP x %.0f MHz" % (
                         sms, FMA_PER_CLK_PER_SM, STATED_SM_MHZ)},
        "e2e": {"value": round(e2e_flops / e2e_max / 1e12, 4), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "wall_s_timed_region": round(wall, 3),
        "step_ms": {"median": round(statistics.median(step_ms), 5), "min": round(min(step_ms), 5),
                    "max": round(max(step_ms), 5)},
        "build": build_info(),
    }
    gemm_name = re.sub(r"_staged_(a|b|ab)$", "", kernel_name)
    copies = bin(stage_mask).count("1") * (-(-max(1, w.batch) // 65535))
    if gemm_name.endswith(("_split", "_ksplit", "_kchain")) and not tensor_path:
        line["roofline"]["kernels"] = (
            "%slaunches of simt_gemm_kernel (whole tiles, then the last wave's tiles as %s), "
            "timed together as one call" % (
                "the k-major copy of %s (stage_transpose_kernel), then " % (
                    {1: "A", 2: "B", 3: "A and B"}[stage_mask]) if stage_mask else "",
                "k-slice clusters" if gemm_name.endswith("_ksplit")
                else "%d chained k-slice launches" % (n_batch_launches - copies - 1)
                if gemm_name.endswith("_kchain") else "quarter tiles"))
    elif stage_mask and not tensor_path:
        line["roofline"]["kernels"] = (
            "the k-major copy of %s (stage_transpose_kernel), then simt_gemm_kernel, timed "
            "together as one call" % {1: "A", 2: "B", 3: "A and B"}[stage_mask])
    # Algorithmic HBM bytes per step (A and B read, C written, C read when beta != 0,
    # the bias) over the step time: the bandwidth side of the roofline, which matters
    # for the skinny shapes (the QK^T batch writes 2 GiB).
    alg_bytes = 4 * (w.M * w.K + w.K * w.N + w.M * w.N) * max(1, w.batch)
    if w.beta != 0:
        alg_bytes += 4 * w.M * w.N * max(1, w.batch)
    if w.bias is not None:
        alg_bytes += 4 * w.N
    line["bandwidth"] = {"algorithmic_bytes_per_step": alg_bytes,
                         "gb_s": round(alg_bytes / (kernel_ms / 1e3) / 1e9, 1)}
    if back_to_back is not None:
        line["back_to_back"] = back_to_back
    if tensor_path:
        derived, dsrc = tensor_peak_tflops(args.math)
        cal = calibrate_tf32_tflops(dev)
        div = 3.0 if args.math == "3xtf32" else 1.0
        tpeak = cal / div
        line["roofline"] = {"bound": "tensor", "achieved": round(achieved, 4),
                            "peak": round(tpeak, 2), "unit": UNIT,
                            "frac": round(achieved / tpeak, 4),
                            "traffic": recorded_traffic(kernel_name, args.workload),
                            "peak_source": "calibrated on this GPU: vendor TF32 GEMM (torch.matmul, "
                                           "TF32 allowed) 8192^3, best of 5 = %.1f TFLOP/s%s" % (
                                               cal, " / 3 products" if div == 3.0 else ""),
                            "peak_derived": round(derived, 2), "peak_derived_source": dsrc,
                            "frac_of_derived": round(achieved / derived, 4)}
    clk = sampler.summary()
    if clk is not None:
        line["clocks"] = clk
        if clk.get("sm_mhz") and not tensor_path:
            line["roofline"]["frac_at_measured_clock"] = round(
                achieved / (peak * clk["sm_mhz"] / STATED_SM_MHZ), 4)
    if (rank == 0 and not args.no_secondary and args.workload == "square4096"
            and not tensor_path and args.config < 0 and splitk is None):
        # the fused-epilogue target: FC layer fused against the plain GEMM of its shape
        line["secondary"] = {"fc_fused_vs_unfused": fc_secondary(
            fg, dev, stream, clocks=not args.no_clocks, entry=args.entry),
            **small_secondary(fg, dev, stream)}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    return line


def staged_workspace(fg, w, dev):
    """(workspace tensor, bytes) for fgemm_sgemm_staged on this workload, allocated once."""
    need = fg.staged_workspace_size(w.ta, w.tb, w.M, w.N, w.K, max(1, w.batch))
    return torch.empty(max(1, need // 4), dtype=torch.float32, device=dev), need


def entry_text(args, staged, stage_mask):
    if args.math != "fp32":
        return "fgemm_gemm_math"
    if args.splitk > 1:
        return "fgemm_sgemm_splitk"
    if args.config >= 0:
        return "fgemm_gemm_explicit"
    if staged is None:
        return "plain (fgemm_sgemm / _bias_relu / _strided_batched)"
    what = {0: "no copy (the model keeps the operands as stored)", 1: "A copied k-major",
            2: "B copied k-major", 3: "A and B copied k-major"}[stage_mask]
    return "fgemm_sgemm_staged, the model's choice: %s; workspace %.0f MiB allocated once" % (
        what, staged[1] / 2**20)


def describe(w):
    """One-line description of a workload (name, shape, scalars, epilogue, seed)."""
    s = "%s: M=%d N=%d K=%d alpha=%g beta=%g op(A)=%s op(B)=%s" % (
        w.name, w.M, w.N, w.K, w.alpha, w.beta, "T" if w.ta else "N", "T" if w.tb else "N")
    if w.batch:
        s += " batch=%d" % w.batch
    if w.bias is not None:
        s += " +bias"
    if w.relu:
        s += " +ReLU"
    return s + ", seed %d" % w.seed


# ---- the reference arm: the FP64 oracle on host cores ------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    w = workloads.make(args.workload)
    threads = oracle.default_threads()
    A = (w.A[0] if w.batch else w.A).numpy().reshape(-1)
    B = (w.B[0] if w.batch else w.B).numpy().reshape(-1)
    C0 = None if w.C0 is None else w.C0.numpy().reshape(-1)
    # each step: whole rows of C, sized so the whole run stays within a few minutes
    budget_s = 120.0
    per_step = budget_s / max(1, args.steps + args.warmup)
    t0 = time.perf_counter()
    oracle.gemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, A, w.lda, B, w.ldb, w.beta, C0, w.ldc,
                bias=w.bias, relu=w.relu, rows=list(range(min(w.M, threads))), threads=threads,
                want_mag=False)
    t_row = (time.perf_counter() - t0) / min(w.M, threads)
    rows = int(max(1, min(w.M, per_step / max(t_row, 1e-9))))
    rows = min(w.M, max(threads, rows - rows % threads))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.gemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, A, w.lda, B, w.ldb, w.beta, C0, w.ldc,
                    bias=w.bias, relu=w.relu, rows=list(range(rows)), threads=threads,
                    want_mag=False)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    flops = 2.0 * rows * w.N * w.K
    value = flops * len(times) / sum(times) / 1e12
    sample = "%d of %d rows of C (all %d columns) per step, FP64 oracle" % (rows, w.M, w.N)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sum(times) / len(times) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(w), "sample": sample},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def cpu_baseline_table(args):
    """The oracle beside the GPU numbers, per workload: one core and every core."""
    import oracle
    for name in workloads.WORKLOADS:
        w = workloads.make(name)
        for threads in (1, oracle.default_threads()):
            r = cpu_baseline(w, args.cpu_seconds, threads)
            print(json.dumps({"workload": describe(w), "cpu_baseline": r}), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_baseline_table:
        cpu_baseline_table(args)
        return
    rank, world, local_rank = dist_env()
    if args.gpus != world and world > 1:
        print("bench.py: --gpus %d but WORLD_SIZE %d" % (args.gpus, world), file=sys.stderr)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        dist_init(world)
        line = run_fgemm(args, rank, world, local_rank)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
