#!/usr/bin/env python
"""Benchmark of the TwELL activation-sparse feed-forward hot path on one GB300.

One step = the whole hot path over one batch of the training workload
(M=16384 tokens, d_model=4096, d_ff=16384, ReLU, bias -2.33 -> ~99 % of the
hidden activations zero, TwELL tiles of 128 rows, dy ~ N(0,1), L1 coefficient
1e-4 on h):

    twell_ffn_fwd    tcgen05 up-projection, TwELL built in its epilogue (a1-a3),
                     then y = TwELL x W_down (a4)
    twell_ffn_bwd    dpre, dx, column lists, dW_up, dW_down, db             (a6-a9)

Inputs are resident in HBM when the timed region starts; L2 is flushed (a
512 MB write, then a 512 MB read so that what stays in L2 is clean) between
timed steps. Every stage is timed with CUDA events on the stream it runs on.
Prints one JSON line (rank 0). Besides the headline it reports, on the same
GPU: the forward alone on the inference workload (4096 x 2048 x 8192), the
same layer computed densely with this build's tcgen05 GEMMs (forward and
backward), the gated decode batches, the sparsity/skew sweep, energy per
token, peak memory, and the oracle on the host cores.

--impl reference times the CPU oracle (plain C, fp64) on the host cores on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synthetic as syn  # noqa: E402

METRIC = "sparse-FFN tokens/s fwd & fwd+bwd at 99% sparsity; % of HBM/tensor roofline"
UNIT = "tokens/s"
CONFIG_NAME = "training"
STAGE_CAP = 32
WORKLOAD = ("training step: M=16384 tokens, d_model=4096, d_ff=16384, bf16, ReLU, bias=-2.33 (~99% sparse), "
            "dy~N(0,1); fwd + bwd (y, dx, dW_up, dW_down, db) with L1 coefficient 1e-4 on h, TwELL tile=128 rows, "
            "fp32 accumulation")
L1 = 1e-4
FLUSH_BYTES = 512 << 20
# The pages' own end-to-end numbers (H100, trained 0.5B-2B models): context, not the target.
PAGES_CONTEXT = {
    "inference_throughput_vs_dense": 1.205, "training_throughput_vs_dense": 1.219,
    "energy_per_token_vs_dense": 0.83, "peak_memory_vs_dense": "<0.76",
    "hardware": "NVIDIA H100", "scope": "end-to-end language models (0.5B-2B parameters, >99% FFN sparsity)",
    "source": "Sparser, Faster, Lighter Transformer Language Models - Resumo Tecnico, 4 Resultados",
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sust=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    sm_max_mhz=float(p.get("sm_max_mhz", 2070.0)), src="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, sm_max_mhz=2070.0, src="fallback")


# ------------------------------------------------------------- clock sampler --

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle --

def oracle_step(inp: syn.FFNInputs, S: int):
    """The oracle's fwd + bwd on the first S tokens of the workload (same weights)."""
    import oracle
    rows = np.arange(S, dtype=np.int32)
    fw = oracle.ffn_fwd_rows(inp.x, inp.W_up, None, inp.b, inp.W_down, inp.M, inp.d, inp.F, rows=rows)
    X = oracle.bf16_to_f64(inp.x[:S])
    DY = oracle.bf16_to_f64(inp.dy[:S])
    H = oracle.bf16_to_f64(fw["h"])
    Wu = oracle.bf16_to_f64(inp.W_up)
    Wd = oracle.bf16_to_f64(inp.W_down)
    oracle.ffn_bwd_rows(X, Wu, Wd, H, DY, L1)
    oracle.ffn_bwd_cols(X, Wu, Wd, H, DY, L1)


def _omp_set_threads(n: int) -> None:
    """Sets the OpenMP thread count of this process (the oracle's parallel loops)."""
    for name in ("libgomp.so.1", "libgomp.so"):
        try:
            ctypes.CDLL(name).omp_set_num_threads(int(n))
            return
        except OSError:
            continue


def oracle_rate(inp: syn.FFNInputs, budget_s: float, one_core_s: float = 6.0):
    """Tokens/s of the oracle on a sample of the workload sized to take about budget_s:
    the first S tokens (S from an 8-token probe, at most the whole batch), repeated
    until budget_s has passed; then the same on one core for about one_core_s."""
    import oracle
    oracle.build()
    cores = oracle.num_threads()
    S0 = 8
    t0 = time.perf_counter()
    oracle_step(inp, S0)
    t_probe = time.perf_counter() - t0
    S = int(max(1, min(inp.M, S0 * budget_s / 2 / max(t_probe, 1e-3))))
    done, t0 = 0, time.perf_counter()
    while True:
        oracle_step(inp, S)
        done += S
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    one = None
    if one_core_s > 0:
        _omp_set_threads(1)
        try:
            if oracle.num_threads() == 1:
                S1 = 2
                n1, t1 = 0, time.perf_counter()
                while True:
                    oracle_step(inp, S1)
                    n1 += S1
                    d1 = time.perf_counter() - t1
                    if d1 >= one_core_s:
                        break
                one = {"value": n1 / d1, "tokens": n1, "seconds": d1}
        finally:
            _omp_set_threads(cores)
    return done / dt, S, dt, cores, done, one


def max_over_ranks(value: float, world: int) -> float:
    """The largest of the ranks' values: the job's step time is its slowest
    replica's. Collective over the initialised process group when world > 1."""
    if world <= 1:
        return value
    on_gpu = torch.distributed.get_backend() == "nccl"
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_replica: int, world: int, ms_step: float) -> float:
    """Tokens per second of the whole job: every replica processes its own batch."""
    return world * tokens_per_replica / (ms_step / 1000.0)


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = syn.config_inputs(CONFIG_NAME, with_dy=True)
    total_budget = 150.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    # size the per-step sample from an 8-token probe
    t0 = time.perf_counter()
    oracle_step(inp, 8)
    t_probe = time.perf_counter() - t0
    S = int(max(1, min(inp.M, 8 * per_step / max(t_probe, 1e-3))))
    for _ in range(args.warmup):
        oracle_step(inp, S)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(inp, S)
        times.append(time.perf_counter() - t0)
    ms = 1000.0 * statistics.mean(times)
    value = S / (ms / 1000.0)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded splitmix64/Box-Muller)",
        "config": {"workload": WORKLOAD, "sample_tokens_per_step": S},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"first {S} tokens of the workload per step, same weights (fwd + bwd)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- GPU path ----

def dev16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


class Layer:
    """Device buffers of one workload and the three stages of a step."""

    def __init__(self, inp: syn.FFNInputs, l1: float, cap: int | None = None, sparse: bool = True):
        import activation_sparse_transformer_tcgen05_gb300 as tw
        self.tw = tw
        self.inp = inp
        self.l1 = l1
        M, d, F, T = inp.M, inp.d, inp.F, inp.T
        self.x, self.Wu, self.Wd = dev16(inp.x), dev16(inp.W_up), dev16(inp.W_down)
        self.dy = dev16(inp.dy) if inp.dy is not None else None
        self.b = torch.from_numpy(inp.b).cuda()
        self.st = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.ws_b = None
        if not sparse:  # inputs only (the dense layer brings its own buffers)
            return
        # slot capacity: M x 256 is ~1.3x the widest 128-row tile at 1 % density
        # on these shapes (a tile wider than that reports a capacity error)
        self.cap = cap if cap is not None else M * min(F, 256)
        self.buf = tw.TwellBuffers(M, F, T, self.cap)
        self.y = torch.empty(M, d, dtype=torch.int16, device="cuda")
        # epilogue staging of 32 entries per (row, 256-column block): ~13x the
        # mean count at 1 % density (the full 256 would be as large as an fp32 h)
        self.ws_f = torch.empty(tw.twell_fwd_workspace_bytes(M, d, F, T, self.cap, STAGE_CAP), dtype=torch.uint8,
                                device="cuda")

    def alloc_bwd(self):
        tw, inp = self.tw, self.inp
        M, d, F, T = inp.M, inp.d, inp.F, inp.T
        self.ws_b = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_BWD, M, d, F, T, self.cap), dtype=torch.uint8,
                                device="cuda")
        self.dx = torch.empty(M, d, dtype=torch.int16, device="cuda")
        self.dWu = torch.empty(F, d, dtype=torch.float32, device="cuda")
        self.dWd = torch.empty(F, d, dtype=torch.float32, device="cuda")
        self.db = torch.empty(F, dtype=torch.float32, device="cuda")

    def fwd(self):
        self.tw.twell_ffn_fwd(self.x, self.Wu, None, self.b, self.Wd, self.inp.T, self.buf, self.y, self.ws_f,
                              self.st)

    def bwd(self):
        self.tw.twell_ffn_bwd(self.x, self.Wu, self.Wd, self.buf, self.dy, self.l1, self.dx, self.dWu, self.dWd,
                              self.db, self.ws_b, self.st)

    def check(self, where: str):
        code = self.tw.twell_check(self.st)
        if code != 0:
            raise RuntimeError(f"{where}: device status {code}: {self.tw.twell_status_string(code)}")


class DenseLayer:
    """The same layer computed densely with this build's tcgen05 GEMMs (forward and backward)."""

    def __init__(self, L: Layer):
        tw, inp = L.tw, L.inp
        M, d, F = inp.M, inp.d, inp.F
        self.L, self.tw = L, tw
        self.h = torch.empty(M, F, dtype=torch.int16, device="cuda")
        self.y = torch.empty(M, d, dtype=torch.int16, device="cuda")
        self.ws = None

    def alloc_bwd(self):
        inp = self.L.inp
        M, d, F = inp.M, inp.d, inp.F
        self.ws = torch.empty(self.tw.twell_dense_bwd_workspace_bytes(M, d, F), dtype=torch.uint8, device="cuda")
        self.dx = torch.empty(M, d, dtype=torch.int16, device="cuda")
        self.dWu = torch.empty(F, d, dtype=torch.float32, device="cuda")
        self.dWd = torch.empty(F, d, dtype=torch.float32, device="cuda")
        self.db = torch.empty(F, dtype=torch.float32, device="cuda")

    def fwd(self):
        L = self.L
        self.tw.twell_dense_ffn_fwd(L.x, L.Wu, L.b, L.Wd, self.h, self.y, L.st)

    def bwd(self):
        L = self.L
        self.tw.twell_dense_ffn_bwd(L.x, L.Wu, L.Wd, self.h, L.dy, L.l1, self.dx, self.dWu, self.dWd, self.db,
                                    self.ws, L.st)

    def free(self):
        for k in ("h", "y", "ws", "dx", "dWu", "dWd", "db"):
            if hasattr(self, k):
                setattr(self, k, None)


SITES = {1: "up_gemm", 2: "spmm_down", 3: "sddmm", 4: "dx", 5: "csc", 6: "wgrad"}
# Call sites whose kernels run on the library's side stream, concurrently with
# another site's: their event time spans that overlap, so they never count as
# the dominant kernel.
CONCURRENT_SITES = {5: "sddmm"}


# ------------------------------------------------------------------ probes --

PROBE_SRC = os.path.join(ROOT, "probes.cu")
PROBE_LIB = os.path.join(ROOT, "_build", "libprobes.so")


def build_probes() -> str:
    """Compiles probes.cu (FMA and gather ceilings of this benchmark) for sm_103a."""
    if os.path.exists(PROBE_LIB) and os.path.getmtime(PROBE_LIB) >= os.path.getmtime(PROBE_SRC):
        return PROBE_LIB
    os.makedirs(os.path.dirname(PROBE_LIB), exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = PROBE_LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
                           "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared", "-o", tmp, PROBE_SRC])
    os.replace(tmp, PROBE_LIB)
    return PROBE_LIB


_probes = None


def load_probes():
    global _probes
    if _probes is None:
        lib = ctypes.CDLL(build_probes())
        P, I = ctypes.c_void_p, ctypes.c_int
        lib.probe_fma.restype = I
        lib.probe_fma.argtypes = [I, I, I, P, P]
        lib.probe_gather.restype = I
        lib.probe_gather.argtypes = [I, P, I, I, P, I, I, P, P, P]
        _probes = lib
    return _probes


def fma_peak(stream, sm_count: int):
    """Measured FP32 FMA rate (TFLOP/s), best of 5: fmaf and the mixed bf16 x bf16 + fp32 form."""
    lib = load_probes()
    sink = torch.empty(sm_count * 8 * 256, dtype=torch.float32, device="cuda")
    blocks, iters = sm_count * 8, 4096
    out = {}
    for mode, name in ((0, "fp32_fma"), (1, "bf16_mixed_fma")):
        best = 0.0
        for rep in range(6):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if lib.probe_fma(mode, blocks, iters, ctypes.c_void_p(sink.data_ptr()),
                             ctypes.c_void_p(stream.cuda_stream)) != 0:
                raise RuntimeError("probe_fma failed")
            b.record(stream)
            torch.cuda.synchronize()
            if rep:
                flops = 2.0 * 8 * 16 * iters * blocks * 256
                best = max(best, flops / (a.elapsed_time(b) * 1e-3) / 1e12)
        out[name] = best
    return out


def gather_ceiling(W, nnz_per_row: int, reps: int = 6):
    """Measured rate (TB/s) at which stretches of random rows of W (L2-resident)
    reach the SMs: 128-bit loads with 4 or 8 in flight per lane in row order,
    bulk copies into shared memory with 3 or 6 batches in flight per warp, and
    128-bit loads in the down-projection's column-group-major order (two
    256-column chunks per lane); best of `reps` each after warm-up. The
    ceiling is the fastest form."""
    lib = load_probes()
    F, d = W.shape
    rows = 4096
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    idx = torch.randint(0, F, (rows, nnz_per_row), dtype=torch.int32, device="cuda", generator=g)
    sink = torch.empty(rows * ((d + 255) // 256), dtype=torch.float32, device="cuda")  # >= rows * ceil(d/512)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    out = {}
    for mode, name in ((0, "ldg4"), (1, "ldg8"), (2, "bulk3"), (3, "bulk6"), (4, "ldg_cols")):
        def call():
            rc = lib.probe_gather(mode, ctypes.c_void_p(W.data_ptr()), F, d, ctypes.c_void_p(idx.data_ptr()), rows,
                                  nnz_per_row, ctypes.c_void_p(sink.data_ptr()), ctypes.c_void_p(st.data_ptr()),
                                  ctypes.c_void_p(stream.cuda_stream))
            if rc != 0:
                raise RuntimeError(f"probe_gather mode {mode} failed ({rc})")
        for _ in range(3):
            call()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        if int(st.item()) != 0:
            raise RuntimeError("probe_gather: a bounded wait gave up")
        best = min(a.elapsed_time(b) for a, b in ts) * 1e-3
        out[name] = rows * nnz_per_row * d * 2 / best / 1e12
    out["best"] = max(out.values())
    return out


class PowerSampler:
    """nvidia-smi board power samples (50 ms) with their timestamps."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=timestamp,power.draw", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        """[(unix time, watts)]"""
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        samples = []
        for line in out.strip().splitlines():
            parts = [q.strip() for q in line.split(",")]
            if len(parts) < 2:
                continue
            try:
                t = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                samples.append((t + frac, float(parts[1])))
            except ValueError:
                continue
        return samples


def energy_leg(tw, local_rank: int, runs: dict, tokens: int, seconds: float = 2.0):
    """Energy per token of back-to-back calls of each callable in `runs`
    (board power from nvidia-smi, averaged over the samples inside the loop)."""
    out = {}
    stream = torch.cuda.current_stream()
    for name, fn in runs.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(5):
            fn()
        b2.record(stream)
        torch.cuda.synchronize()
        per = a.elapsed_time(b2) / 5 / 1000.0
        n = max(10, int(seconds / per))
        ps = PowerSampler(local_rank)
        ps.start()
        time.sleep(0.5)
        t0 = time.time()
        a.record(stream)
        for _ in range(n):
            fn()
        b2.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        samples = [w for t, w in ps.stop() if t0 + 0.1 <= t <= t1]
        if not samples:
            out[name] = None
            continue
        s_run = a.elapsed_time(b2) / 1000.0
        watts = statistics.mean(samples)
        out[name] = {"watts": watts, "ms_per_call": s_run / n * 1000.0, "mJ_per_call": watts * s_run / n * 1000.0,
                     "uJ_per_token": watts * s_run / (n * tokens) * 1e6, "samples": len(samples), "calls": n}
    return out


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
# each call site's kernel, from one ncu capture per (workload, site), with the
# SHA-256 of the source file it was built from: once that file changes the
# figure no longer describes the kernel and the site reports traffic null.
NCU_TRAFFIC = {
    # training workload, from the ncu summary of that step under profiles/; a call site's
    # figure is the sum over its launches (site 3: the slices and the combine,
    # which also scatters the column lists; site 6: the dW_down and the dW_up
    # gathers)
    ("training", 1): ("twell_gemm.cu", "787b72d9dc15eecd18efb32473080d26db82d17f855a5870c857c92fb2f102f9", 813.3e6),
    ("training", 2): ("twell_sparse.cu", "42b071ee146ebaf6a8b4676ead682fa924bb798e16a0309fe3a524371086b17d", 311.1e6),
    ("training", 3): ("twell_sparse.cu", "42b071ee146ebaf6a8b4676ead682fa924bb798e16a0309fe3a524371086b17d", 511.2e6),
    ("training", 4): ("twell_sparse.cu", "42b071ee146ebaf6a8b4676ead682fa924bb798e16a0309fe3a524371086b17d", 356.3e6),
    ("training", 6): ("twell_sparse.cu", "42b071ee146ebaf6a8b4676ead682fa924bb798e16a0309fe3a524371086b17d", 935.1e6),
}


# The sources a kernel's code comes from: its translation unit and the
# library headers it includes, hashed together in this order.
KERNEL_SOURCES = {
    "twell_gemm.cu": ("common.cuh", "launch.h", "twell_gemm.cu"),
    "twell_sparse.cu": ("common.cuh", "launch.h", "sparse_common.cuh", "twell_sparse.cu"),
}


def source_digest(unit: str):
    """SHA-256 over the bytes of a translation unit's sources (None if one is missing)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[unit]:
        try:
            with open(os.path.join(ROOT, "activation_sparse_transformer_tcgen05_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        except OSError:
            return None
    return h.hexdigest()


def ncu_traffic(site: int, workload: str):
    """The committed ncu DRAM traffic of a call site, or None once its kernels'
    sources differ from the ones the counters were taken on."""
    ent = NCU_TRAFFIC.get((workload, site))
    if ent is None:
        return None
    return ent[2] if source_digest(ent[0]) == ent[1] else None


# Rows of d bf16 each sparse kernel pulls through L2 per stored entry:
# down-projection and SDDMM a W_down row, dx a W_up row, weight gradients an x
# row and a dy row.
GATHER_ROWS = {2: 1, 3: 1, 4: 1, 6: 2}


def site_work(site: int, inp, slots: int, nnz: int):
    """(flops, compulsory bytes) of one launch of a call site: every input read
    once, every output written once (the roofline's algorithmic work)."""
    M, d, F = inp.M, inp.d, inp.F
    if site == 1:  # up GEMM + TwELL epilogue: x, W_up in; staged entries out
        return 2.0 * M * d * F, M * d * 2 + F * d * 2 + nnz * 4 + F * 4
    if site == 2:  # y = TwELL W_down
        return 2.0 * nnz * d, F * d * 2 + slots * 6 + M * d * 2
    if site == 3:  # dpre on the stored slots, then each entry's row, h, dpre into the column lists
        return 2.0 * nnz * d, M * d * 2 + F * d * 2 + slots * (4 + 2) + slots * 4 + nnz * 10
    if site == 4:  # dx = dpre W_up
        return 2.0 * nnz * d, F * d * 2 + slots * 8 + M * d * 2
    if site == 5:  # column lists: masks, counts, pointers (TwELL indices only)
        rb = (M + 63) // 64
        return 0.0, slots * 4 + M * 4 + rb * F * (8 + 4) * 2 + F * 8
    if site == 6:  # dW_up, dW_down, db from the column lists
        return 4.0 * nnz * d, 2 * M * d * 2 + nnz * 10 + 2 * F * d * 4 + F * 4
    raise ValueError(site)


def kernel_roofline(site: int, us: float, inp, slots: int, nnz: int, peaks, ceil: dict, workload: str):
    """Roofline of one call site. tensor-bound: FLOPs at the bf16 peak. CUDA-core
    gathers: the slower of compulsory bytes at the HBM peak and FLOPs at the
    measured FP32 FMA peak ("alu"), plus the HBM-only fraction the north-star
    target is stated in, the most that fraction can be when the FMAs run at
    peak, and the gathered bytes against the measured gather ceiling."""
    s = us * 1e-6
    flops, byts = site_work(site, inp, slots, nnz)
    hbm = peaks["hbm"] * 1e9
    if site == 1:
        a = flops / s / 1e12
        return {"bound": "tensor", "achieved": a, "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": a / peaks["bf16"], "traffic": ncu_traffic(site, workload),
                "algorithmic": f"{flops / 1e9:.1f} GFLOP (2 M d_model d_ff)", "hbm_frac": byts / s / hbm}
    if site == 5:
        a = byts / s / 1e9
        return {"bound": "hbm", "achieved": a, "peak": peaks["hbm"], "unit": "GB/s", "frac": a / peaks["hbm"],
                "traffic": None, "algorithmic": f"{byts / 1e6:.1f} MB"}
    fma = ceil["fma_tflops"] * 1e12
    t_roof = max(byts / hbm, flops / fma)
    a = flops / s / 1e12
    out = {"bound": "alu", "achieved": a, "peak": ceil["fma_tflops"], "unit": "TFLOP/s", "frac": a / ceil["fma_tflops"],
           "traffic": ncu_traffic(site, workload),
           "algorithmic": f"{flops / 1e9:.2f} GFLOP of fp32 FMAs on the stored entries; {byts / 1e6:.0f} MB compulsory",
           "roofline_frac": t_roof / s,
           "hbm_frac": byts / s / hbm,
           "hbm_frac_at_fma_peak": min(1.0, (byts / hbm) / (flops / fma))}
    if site in GATHER_ROWS and ceil.get("gather_tbs"):
        by = GATHER_ROWS[site] * nnz * inp.d * 2
        out["l2_gather"] = {"bytes": by, "achieved_TBs": by / s / 1e12, "ceiling_TBs": ceil["gather_tbs"],
                            "frac": by / s / 1e12 / ceil["gather_tbs"]}
    return out


def stage_roofline(name, ms, inp, slots, nnz, peaks):
    M, d, F = inp.M, inp.d, inp.F
    s = ms / 1000.0
    if name == "ffn_fwd":
        flops = 2.0 * M * d * F
        a = flops / s / 1e12
        return {"bound": "tensor", "achieved": a, "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": a / peaks["bf16"],
                "algorithmic": f"{flops / 1e9:.1f} GFLOP (2 M d_model d_ff, the up GEMM; the gather's "
                               f"{2.0 * nnz * d / 1e9:.1f} GFLOP not counted)"}
    else:
        # compulsory: x, dy, W_up, W_down, TwELL read once; dx, dW_up, dW_down, db written once
        by = 2 * M * d * 2 + 2 * F * d * 2 + slots * 6 + M * d * 2 + 2 * F * d * 4 + F * 4
    a = by / s / 1e9
    return {"bound": "hbm", "achieved": a, "peak": peaks["hbm"], "unit": "GB/s", "frac": a / peaks["hbm"],
            "algorithmic": f"{by / 1e6:.1f} MB compulsory"}


def call_roofline(sites, ms_call: float, inp, slots: int, nnz: int, peaks, ceil: dict):
    """Roofline fraction of one library call: the sum over its kernels of
    max(compulsory bytes / HBM peak, FLOPs / pipe peak) over the measured call
    time (bf16 tensor peak for the GEMM, the measured FP32 FMA rate for the
    CUDA-core kernels). "attainable" adds each gather's L2-to-SM bytes at the
    measured gather ceiling as a third bound."""
    hbm, fma, bf16 = peaks["hbm"] * 1e9, ceil["fma_tflops"] * 1e12, peaks["bf16"] * 1e12
    t_roof = t_att = 0.0
    parts = {}
    for site in sites:
        flops, byts = site_work(site, inp, slots, nnz)
        t = max(byts / hbm, flops / (bf16 if site == 1 else fma))
        g = GATHER_ROWS.get(site, 0) * nnz * inp.d * 2 / (ceil["gather_tbs"] * 1e12)
        t_roof += t
        t_att += max(t, g)
        parts[SITES[site]] = {"roofline_us": t * 1e6, "attainable_us": max(t, g) * 1e6}
    s = ms_call / 1000.0
    return {"frac": t_roof / s, "roofline_ms": t_roof * 1e3, "attainable_frac": t_att / s,
            "attainable_ms": t_att * 1e3, "ms": ms_call, "kernels": parts,
            "rule": "sum over kernels of max(bytes / HBM, FLOPs / pipe peak) / call time; attainable adds "
                    "gathered bytes / measured L2-to-SM gather ceiling"}


class L2Flush:
    """Evicts L2 between timed steps: writes a buffer larger than L2 (129 MB),
    then reads another one, so that the lines left behind are clean. (Writing
    alone leaves L2 full of dirty lines whose write-back would be charged to
    the first kernel of the next step, which a real preceding layer, mostly
    reading weights, does not do.)"""

    def __init__(self, nbytes: int):
        self.w = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(nbytes // 4, dtype=torch.int32, device="cuda")

    def fill_(self, v: int):
        self.w.fill_(v)
        self.sink = torch.amax(self.r)


def decode_leg(tw, peaks, flush, stream, reps: int = 30, batches=(1, 8, 64)):
    """Gated decode forward (M = 1, 8, 64 tokens, d_model 4096, d_ff 14336, ~99.5 % sparse):
    time of one twell_ffn_fwd call with L2 flushed before it, and its HBM roofline
    (algorithmic bytes: W_gate once, the union of active W_up and W_down rows once, x, y)."""
    out = {}
    for name in (f"decode{m}" for m in batches):
        inp = syn.config_inputs(name)
        M, d, F, T = inp.M, inp.d, inp.F, inp.T
        x, Wu, Wg, Wd = dev16(inp.x), dev16(inp.W_up), dev16(inp.W_gate), dev16(inp.W_down)
        b = torch.from_numpy(inp.b).cuda()
        cap = M * F
        buf = tw.TwellBuffers(M, F, T, cap)
        y = torch.empty(M, d, dtype=torch.int16, device="cuda")
        ws = torch.empty(tw.twell_workspace_bytes(tw.OP_GATED_FWD, M, d, F, T, cap), dtype=torch.uint8,
                         device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        evs = []
        for i in range(reps + 3):
            flush.fill_(i & 0xff)
            a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            tw.twell_ffn_fwd(x, Wu, Wg, b, Wd, T, buf, y, ws, st)
            b2.record(stream)
            if i >= 3:
                evs.append((a, b2))
        torch.cuda.synchronize()
        if tw.twell_check(st) != 0:
            raise RuntimeError(f"{name}: device status {tw.twell_check(st)}")
        us = statistics.median(a.elapsed_time(b2) for a, b2 in evs) * 1000.0
        # the same call replayed from a CUDA graph (how a decode loop would issue it)
        us_graph = None
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                tw.twell_ffn_fwd(x, Wu, Wg, b, Wd, T, buf, y, ws, st)
            gevs = []
            for i in range(reps + 3):
                flush.fill_(i & 0xff)
                a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                b2.record(stream)
                if i >= 3:
                    gevs.append((a, b2))
            torch.cuda.synchronize()
            if tw.twell_check(st) != 0:
                raise RuntimeError(f"{name}: device status {tw.twell_check(st)} (graph)")
            us_graph = statistics.median(a.elapsed_time(b2) for a, b2 in gevs) * 1000.0
            del g
        except RuntimeError as exc:
            if "device status" in str(exc):
                raise
            us_graph = None
        n = buf.slots()
        idx = buf.idx[:n].cpu().numpy()
        union = int(len(np.unique(idx[idx >= 0])))
        byts = F * d * 2 + 2 * union * d * 2 + 2 * M * d * 2 + F * 4
        gbs = byts / (us * 1e-6) / 1e9
        out[name] = {"us": us, "us_graph": us_graph, "tokens_per_s": M / (us * 1e-6), "active_units_union": union,
                     "algorithmic_MB": byts / 1e6, "achieved_GBs": gbs, "hbm_frac": gbs / peaks["hbm"],
                     "dense_gated_roofline_us": 3 * F * d * 2 / (peaks["hbm"] * 1e9) * 1e6}
        del x, Wu, Wg, Wd, buf, ws
    return out


# ELL capacity of the hybrid format as a fraction of d_ff: a row is cheaper
# dense than gathered once nnz * 2 d bytes at the gather rate (~18.6 TB/s)
# exceed 2 F d FLOP at the dense GEMM's rate (~1.65 PFLOP/s), i.e. above
# ~1.1 % of d_ff.
HYBRID_C_FRAC = 0.0125


def down_variants(tw, buf, Wd, y, st, flush, stream, reps: int = 5):
    """The down-projection of one TwELL two ways, L2 flushed before each call:
    the row gather on the CUDA cores (twell_spmm_down) and the tensor-core
    product over 128-token group unions (twell_spmm_down_tc, both its kernels)."""
    ws = torch.empty(tw.twell_spmm_down_tc_workspace_bytes(buf.M, buf.F, buf.cap_slots), dtype=torch.uint8,
                     device="cuda")

    def timed(fn):
        evs = []
        for i in range(reps + 2):
            flush.fill_(i & 0xff)
            a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b2.record(stream)
            if i >= 2:
                evs.append((a, b2))
        torch.cuda.synchronize()
        code = tw.twell_check(st)
        if code != 0:
            raise RuntimeError(f"down variants: device status {code}: {tw.twell_status_string(code)}")
        return statistics.median(a.elapsed_time(b2) for a, b2 in evs) * 1000.0

    rows_us = timed(lambda: tw.twell_spmm_down(buf, Wd, y, st))
    tc_us = timed(lambda: tw.twell_spmm_down_tc(buf, Wd, y, ws, st))
    a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    b2.record(stream)
    build = []
    for i in range(3):
        flush.fill_(i & 0xff)
        tw.twell_set_kernel_timer(tw.twell.SITE_UNION_BUILD, a, b2)
        tw.twell_spmm_down_tc(buf, Wd, y, ws, st)
        tw.twell_set_kernel_timer(0)
        torch.cuda.synchronize()
        build.append(a.elapsed_time(b2) * 1000.0)
    return {"rows_us": rows_us, "union_tc_us": tc_us, "union_build_us": statistics.median(build),
            "rows_over_union_tc": rows_us / tc_us}


def timed_ms(fn, flush, stream, st, tw, n: int = 5, warm: int = 2):
    """Median time (ms) of fn(), L2 flushed before each call."""
    evs = []
    for i in range(n + warm):
        flush.fill_(i & 0xff)
        a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b2.record(stream)
        if i >= warm:
            evs.append((a, b2))
    torch.cuda.synchronize()
    code = tw.twell_check(st)
    if code != 0:
        raise RuntimeError(f"device status {code}: {tw.twell_status_string(code)}")
    return statistics.median(a.elapsed_time(b2) for a, b2 in evs)


SWEEP_NAMES = ("sweep90", "sweep99", "sweep999", "sweep90s", "sweep99s", "sweep999s")


def hybrid_leg(tw, flush, stream, reps: int = 5):
    """The sparsity/skew sweep (8192 tokens, d_model 4096, d_ff 16384, x rows
    scaled by LogNormal(0, 1); biases for 90 / 99 / 99.9 % sparsity, nominal and
    skew-corrected): forward and fwd + bwd time and memory of plain TwELL, of
    the hybrid ELL + dense-overflow format (C = 1.25 % of d_ff), and of the
    dense layer (this build's tcgen05 GEMMs, forward and backward measured)."""
    inp = syn.config_inputs("sweep90", with_dy=True)  # the six differ only in the bias
    M, d, F, T = inp.M, inp.d, inp.F, inp.T
    x, Wu, Wd, dy = dev16(inp.x), dev16(inp.W_up), dev16(inp.W_down), dev16(inp.dy)
    WdT = Wd.view(F, d).t().contiguous()
    WuT = Wu.view(F, d).t().contiguous()
    C = round(HYBRID_C_FRAC * F)
    l1 = 1e-4
    y = torch.empty(M, d, dtype=torch.int16, device="cuda")
    dx = torch.empty(M, d, dtype=torch.int16, device="cuda")
    dWu = torch.empty(F, d, dtype=torch.float32, device="cuda")
    dWd = torch.empty(F, d, dtype=torch.float32, device="cuda")
    db = torch.empty(F, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def timed(fn, n=reps):
        return timed_ms(fn, flush, stream, st, tw, n=n)

    # the dense layer does not depend on the sparsity: one measurement per bias
    # only differs in the ReLU mask (its GEMMs do the same work)
    out = {"C": C, "workload": "M=8192, d_model=4096, d_ff=16384, T=128, x rows x LogNormal(0,1), l1=1e-4",
           "targets": {n: syn.SWEEP_TARGETS[n] for n in SWEEP_NAMES}}
    for name in SWEEP_NAMES:
        b = torch.full((F,), float(syn.CONFIGS[name]["bias"]), dtype=torch.float32, device="cuda")
        buf = tw.TwellBuffers(M, F, T, M * F)
        ws = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_FWD, M, d, F, T, M * F), dtype=torch.uint8,
                         device="cuda")
        ms_tw = timed(lambda: tw.twell_ffn_fwd(x, Wu, None, b, Wd, T, buf, y, ws, st))
        slots, nnz = buf.slots(), int(buf.nnz.sum().item())
        del ws
        down = down_variants(tw, buf, Wd, y, st, flush, stream)
        wsb = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_BWD, M, d, F, T, M * F), dtype=torch.uint8,
                          device="cuda")
        ms_tw_b = timed(lambda: tw.twell_ffn_bwd(x, Wu, Wd, buf, dy, l1, dx, dWu, dWd, db, wsb, st), n=2)
        del buf, wsb
        hb = tw.TwellBuffers(M, F, T, M * C)
        ov = tw.TwellOverflow(F, C, M)
        wsh = torch.empty(tw.twell_workspace_bytes(tw.OP_HYBRID_FWD, M, d, F, T, 0), dtype=torch.uint8,
                          device="cuda")
        ms_h = timed(lambda: tw.twell_hybrid_ffn_fwd(x, Wu, b, Wd, WdT, T, hb, ov, y, wsh, st))
        n_ov, ell_slots = int(ov.n_rows.item()), hb.slots()
        del wsh
        wshb = torch.empty(tw.twell_hybrid_bwd_workspace_bytes(M, d, F, T, hb.cap_slots, M), dtype=torch.uint8,
                           device="cuda")
        ms_h_b = timed(lambda: tw.twell_hybrid_ffn_bwd(x, Wu, Wd, WuT, hb, ov, dy, l1, dx, dWu, dWd, db, wshb, st))
        del hb, ov, wshb
        hd = torch.empty(M, F, dtype=torch.int16, device="cuda")
        wsd = torch.empty(tw.twell_dense_bwd_workspace_bytes(M, d, F), dtype=torch.uint8, device="cuda")
        ms_d = timed(lambda: tw.twell_dense_ffn_fwd(x, Wu, b, Wd, hd, y, st))
        ms_d_b = timed(lambda: tw.twell_dense_ffn_bwd(x, Wu, Wd, hd, dy, l1, dx, dWu, dWd, db, wsd, st))
        del hd, wsd
        best = min(ms_tw + ms_tw_b, ms_h + ms_h_b)
        out[name] = {"bias": syn.CONFIGS[name]["bias"], "density": nnz / (M * F), "padding_ratio": slots / max(nnz, 1),
                     "twell_ms": ms_tw, "hybrid_ms": ms_h, "dense_ms": ms_d,
                     "twell_bwd_ms": ms_tw_b, "hybrid_bwd_ms": ms_h_b, "dense_bwd_ms": ms_d_b,
                     "twell_step_ms": ms_tw + ms_tw_b, "hybrid_step_ms": ms_h + ms_h_b, "dense_step_ms": ms_d + ms_d_b,
                     "best_sparse_step_vs_dense_step": (ms_d + ms_d_b) / best,
                     "twell_MB": slots * 6 / 1e6, "hybrid_MB": (ell_slots * 6 + n_ov * F * 2) / 1e6,
                     "dense_h_MB": M * F * 2 / 1e6,
                     "overflow_rows": n_ov, "hybrid_vs_twell": ms_tw / ms_h, "hybrid_vs_dense": ms_d / ms_h,
                     "hybrid_step_vs_twell_step": (ms_tw + ms_tw_b) / (ms_h + ms_h_b),
                     "down_projection": down}
    return out


def inference_leg(tw, flush, stream, peaks, reps: int = 20):
    """The inference workload's forward (4096 tokens, d_model 2048, d_ff 8192,
    ~99 % sparse, TwELL tile 128): twell_ffn_fwd against this build's dense
    tcgen05 forward, L2 flushed before each call."""
    inp = syn.config_inputs("inference")
    L = Layer(inp, 0.0)
    D = DenseLayer(L)
    ms = timed_ms(L.fwd, flush, stream, L.st, tw, n=reps)
    ms_d = timed_ms(D.fwd, flush, stream, L.st, tw, n=reps)
    nnz = int(L.buf.nnz.sum().item())
    up_flops = 2.0 * inp.M * inp.d * inp.F
    out = {"workload": "M=4096, d_model=2048, d_ff=8192, T=128, bias=-2.33, forward only",
           "tokens_per_s": inp.M / (ms / 1000.0), "ms": ms, "density": nnz / (inp.M * inp.F),
           "dense_tcgen05_fwd_ms": ms_d, "dense_tokens_per_s": inp.M / (ms_d / 1000.0),
           "sparse_vs_dense": ms_d / ms,
           "up_gemm_tensor_frac_if_alone": None}
    del L, D
    return out, up_flops


def training_memory_leg(tw, inp, l1: float):
    """Peak device memory (torch.cuda.max_memory_allocated) of one training
    step, sparse against dense, each in a fresh scope: the resident inputs and
    weights (x, dy, W_up, W_down, b), then everything the step allocates (the
    TwELL sized for the workload, the forward's and backward's workspaces,
    y, dx and the fp32 weight gradients; for the dense layer the dense h, its
    backward's workspace and the same outputs)."""
    out = {}
    for kind in ("twell", "dense"):
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        L = Layer(inp, l1, sparse=False)
        resident = torch.cuda.memory_allocated() - base
        if kind == "twell":
            M, d, F, T = inp.M, inp.d, inp.F, inp.T
            L.cap = M * min(F, 256)
            L.buf = tw.TwellBuffers(M, F, T, L.cap)
            L.y = torch.empty(M, d, dtype=torch.int16, device="cuda")
            L.ws_f = torch.empty(tw.twell_fwd_workspace_bytes(M, d, F, T, L.cap, STAGE_CAP), dtype=torch.uint8,
                                 device="cuda")
            L.fwd()
            torch.cuda.synchronize()
            L.ws_f = None  # the forward's staging is transient
            L.alloc_bwd()
            L.bwd()
        else:
            D = DenseLayer(L)
            D.fwd()
            D.alloc_bwd()
            D.bwd()
        torch.cuda.synchronize()
        L.check(f"memory leg ({kind})")
        peak = torch.cuda.max_memory_allocated() - base
        out[kind] = {"peak_MB": peak / 1e6, "resident_inputs_MB": resident / 1e6,
                     "step_MB": (peak - resident) / 1e6}
        del L
        if kind == "dense":
            del D
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    out["twell_over_dense_peak"] = out["twell"]["peak_MB"] / out["dense"]["peak_MB"]
    out["twell_over_dense_step"] = out["twell"]["step_MB"] / out["dense"]["step_MB"]
    return out


EXTRA_LEGS = ("e2e", "dense", "crossover", "inference", "energy", "memory", "down", "decode", "hybrid")

# Biases of the training workload's shape at higher sparsity (no row skew):
# Phi^-1 of the target density.
CROSSOVER_BIASES = {"99.0": -2.3263, "99.5": -2.5758, "99.9": -3.0902}


def crossover_leg(tw, L: "Layer", flush, stream, dense_step_ms, reps: int = 5):
    """The training step on the training workload's inputs at 99 / 99.5 /
    99.9 % nominal sparsity (only the bias changes), against the dense step
    (whose work does not depend on the bias): where the sparse path overtakes
    the dense layer on this GPU."""
    out = {}
    b0 = L.b
    try:
        for name, bias in CROSSOVER_BIASES.items():
            L.b = torch.full_like(b0, bias)
            ms = timed_ms(lambda: (L.fwd(), L.bwd()), flush, stream, L.st, tw, n=reps)
            nnz = int(L.buf.nnz.sum().item())
            out[name] = {"bias": bias, "density": nnz / (L.inp.M * L.inp.F), "step_ms": ms,
                         "tokens_per_s": L.inp.M / (ms / 1000.0)}
            if dense_step_ms:
                out[name]["sparse_vs_dense"] = dense_step_ms / ms
    finally:
        L.b = b0
    return out


def dominant_site(site_us: dict) -> int:
    """The call site with the longest time among those that run alone."""
    return max((k for k in site_us if k not in CONCURRENT_SITES), key=site_us.get)


def leg_on(args, name: str) -> bool:
    if args.no_extras:
        return False
    return args.legs == "all" or name in args.legs.split(",")


def e2e_leg(tw, L: Layer, inp, flush, stream, steps: int, world: int):
    """The step through the public API (twell_ffn_fwd + twell_ffn_bwd) with host
    buffers, as a training loop runs it: every step copies its x and dy in from
    pinned host memory and its y and dx out, inside the timed region. The
    copies run on two copy streams beside the compute stream, double-buffered
    on the device: step i+1's inputs come in while step i computes, and step
    i's y goes out during its backward and its dx during step i+1. The time is
    that of the whole loop, from the first input copy to the last output copy,
    divided by the steps (no L2 flush: x, dy and the weights are 134 MB each,
    more than L2)."""
    xh = torch.from_numpy(np.ascontiguousarray(inp.x).view(np.int16)).pin_memory()
    dyh = torch.from_numpy(np.ascontiguousarray(inp.dy).view(np.int16)).pin_memory()
    yh = torch.empty(inp.M, inp.d, dtype=torch.int16).pin_memory()
    dxh = torch.empty(inp.M, inp.d, dtype=torch.int16).pin_memory()
    X = [L.x, torch.empty_like(L.x)]
    DY = [L.dy, torch.empty_like(L.dy)]
    Y = [L.y, torch.empty_like(L.y)]
    DX = [L.dx, torch.empty_like(L.dx)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def ev(s):
        e = torch.cuda.Event()
        e.record(s)
        return e

    def loop(n: int) -> float:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        h2d.wait_event(ev(stream))
        with torch.cuda.stream(h2d):
            X[0].copy_(xh, non_blocking=True)
            DY[0].copy_(dyh, non_blocking=True)
        inputs_in = ev(h2d)
        bwd_done, y_out, dx_out = [], [], []
        for i in range(n):
            b = i % 2
            stream.wait_event(inputs_in)
            if i >= 2:
                stream.wait_event(y_out[i - 2])  # Y[b] has reached the host
            tw.twell_ffn_fwd(X[b], L.Wu, None, L.b, L.Wd, inp.T, L.buf, Y[b], L.ws_f, L.st)
            fwd_done = ev(stream)
            if i >= 2:
                stream.wait_event(dx_out[i - 2])  # DX[b] has reached the host
            tw.twell_ffn_bwd(X[b], L.Wu, L.Wd, L.buf, DY[b], L.l1, DX[b], L.dWu, L.dWd, L.db, L.ws_b, L.st)
            bwd_done.append(ev(stream))
            if i + 1 < n:
                # the other buffers were last read by step i-1's backward
                if i >= 1:
                    h2d.wait_event(bwd_done[i - 1])
                with torch.cuda.stream(h2d):
                    X[1 - b].copy_(xh, non_blocking=True)
                    DY[1 - b].copy_(dyh, non_blocking=True)
                inputs_in = ev(h2d)
            d2h.wait_event(fwd_done)
            with torch.cuda.stream(d2h):
                yh.copy_(Y[b], non_blocking=True)
            y_out.append(ev(d2h))
            d2h.wait_event(bwd_done[i])
            with torch.cuda.stream(d2h):
                dxh.copy_(DX[b], non_blocking=True)
            dx_out.append(ev(d2h))
        stream.wait_event(dx_out[-1])
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    loop(2)
    L.check("e2e warm-up")
    n = max(4, min(steps, 30))
    ms = loop(n) / n
    L.check("e2e")
    del X[1], DY[1], Y[1], DX[1]
    return {"value": world * inp.M / (ms / 1000.0), "unit": UNIT,
            "h2d_bytes_per_step": int(xh.numel() * 2 + dyh.numel() * 2),
            "d2h_bytes_per_step": int(yh.numel() * 2 + dxh.numel() * 2), "ms_per_step": ms,
            "steps": n, "api": "twell_ffn_fwd + twell_ffn_bwd",
            "copies": "x, dy in and y, dx out every step on two copy streams, double-buffered beside the compute"}


def run_ours(args, rank: int, world: int, local_rank: int):
    import activation_sparse_transformer_tcgen05_gb300 as tw
    from activation_sparse_transformer_tcgen05_gb300 import build as tbuild
    tbuild.build()
    torch.cuda.set_device(local_rank)
    peaks = _peaks()
    inp = syn.config_inputs(CONFIG_NAME, with_dy=True)
    L = Layer(inp, L1)
    L.alloc_bwd()
    flush = L2Flush(FLUSH_BYTES)
    stream = torch.cuda.current_stream()

    def step(evs):
        evs[0].record(stream)
        L.fwd()
        evs[1].record(stream)
        L.bwd()
        evs[2].record(stream)

    for i in range(args.warmup):
        flush.fill_(i & 0xff)
        step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    L.check("warm-up")
    slots = L.buf.slots()
    nnz = int(L.buf.nnz.sum().item())

    # per-kernel calibration: every call site timed with the library's event hook
    site_us = {}
    for site in SITES:
        evs = []
        for i in range(4):
            a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            b2.record(stream)
            tw.twell_set_kernel_timer(site, a, b2)
            flush.fill_(i & 0xff)
            step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
            evs.append((a, b2))
        tw.twell_set_kernel_timer(0)
        torch.cuda.synchronize()
        site_us[site] = statistics.mean(a.elapsed_time(b2) for a, b2 in evs[1:]) * 1000.0
    dom_site = dominant_site(site_us)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b2 in kev:
        a.record(stream)
        b2.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.2)
    launches0 = tw.twell_kernel_launches()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_((i + 7) & 0xff)
        tw.twell_set_kernel_timer(dom_site, kev[i][0], kev[i][1])
        step(events[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    tw.twell_set_kernel_timer(0)
    launches = tw.twell_kernel_launches() - launches0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    L.check("timed steps")

    fwd = [e[0].elapsed_time(e[1]) for e in events]
    bwd = [e[1].elapsed_time(e[2]) for e in events]
    ms = {"ffn_fwd": statistics.mean(fwd), "ffn_bwd": statistics.mean(bwd)}
    ms_step = max_over_ranks(sum(ms.values()), world)
    value = whole_job_rate(inp.M, world, ms_step)
    ms_fwd = ms["ffn_fwd"]

    # ---- measured ceilings of the CUDA-core kernels (probes.cu, same run)
    sms = tw.twell_device_sm_count()
    fma = fma_peak(stream, sms)
    gath = gather_ceiling(L.Wd.view(inp.F, inp.d), max(1, round(nnz / inp.M)))
    ceil = {"fma_tflops": fma["bf16_mixed_fma"], "gather_tbs": gath["best"]}

    stages = {k: dict(ms=v, **stage_roofline(k, v, inp, slots, nnz, peaks)) for k, v in ms.items()}
    dom_us = statistics.mean(a.elapsed_time(b2) for a, b2 in kev) * 1000.0
    full = kernel_roofline(dom_site, dom_us, inp, slots, nnz, peaks, ceil, CONFIG_NAME)
    roof = {k: full[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    roof["kernel"] = SITES[dom_site]
    roof["us_per_launch"] = dom_us
    roof["algorithmic"] = full["algorithmic"]
    roof["peak_source"] = ("measured (MEASURED_PEAKS.json)" if roof["bound"] != "alu" else
                           "measured in this run: probes.cu FP32 FMA probe (fma.rn.f32.bf16, the kernels' form)")
    for k in ("roofline_frac", "hbm_frac", "hbm_frac_at_fma_peak", "l2_gather"):
        if k in full:
            roof[k] = full[k]
    kernels = {}
    for k, v in site_us.items():
        kr = kernel_roofline(k, v, inp, slots, nnz, peaks, ceil, CONFIG_NAME)
        kernels[SITES[k]] = dict(us=v, **{q: r for q, r in kr.items() if q != "algorithmic"})
        if k in CONCURRENT_SITES:
            kernels[SITES[k]]["concurrent_with"] = CONCURRENT_SITES[k]

    e2e = e2e_leg(tw, L, inp, flush, stream, args.steps, world) if leg_on(args, "e2e") else None

    # ---- the same step computed densely with this build's tcgen05 GEMMs
    dense = None
    D = None
    if leg_on(args, "dense"):
        D = DenseLayer(L)
        D.alloc_bwd()
        d_f = timed_ms(D.fwd, flush, stream, L.st, tw, n=8)
        d_b = timed_ms(D.bwd, flush, stream, L.st, tw, n=8)
        gemm_flops = 2.0 * inp.M * inp.d * inp.F
        dense = {"fwd_ms": d_f, "bwd_ms": d_b, "step_ms": d_f + d_b,
                 "tokens_per_s": world * inp.M / ((d_f + d_b) / 1000.0),
                 "tensor_frac_of_bf16_sustained": 6 * gemm_flops / ((d_f + d_b) / 1000.0) / 1e12 / peaks["bf16_sust"],
                 "sparse_step_vs_dense_step": (d_f + d_b) / ms_step,
                 "sparse_fwd_vs_dense_fwd": d_f / ms_fwd}

    crossover = None
    if leg_on(args, "crossover"):
        crossover = crossover_leg(tw, L, flush, stream, dense["step_ms"] if dense else None)

    energy = None
    if leg_on(args, "energy"):
        runs = {"twell_step": lambda: (L.fwd(), L.bwd())}
        if D is not None:
            runs["dense_step"] = lambda: (D.fwd(), D.bwd())
        energy = energy_leg(tw, local_rank, runs, inp.M)
        if energy.get("twell_step") and energy.get("dense_step"):
            energy["twell_over_dense_per_token"] = (energy["twell_step"]["uJ_per_token"] /
                                                    energy["dense_step"]["uJ_per_token"])
    if D is not None:
        D.free()
        del D
        torch.cuda.empty_cache()

    union = down_variants(tw, L.buf, L.Wd, L.y, L.st, flush, stream) if leg_on(args, "down") else None
    memory = None
    if leg_on(args, "memory"):
        del L
        torch.cuda.empty_cache()
        memory = training_memory_leg(tw, inp, L1)
    inference = inference_leg(tw, flush, stream, peaks)[0] if leg_on(args, "inference") else None
    decode = (decode_leg(tw, peaks, flush, stream, batches=tuple(int(m) for m in args.decode_batches.split(",")))
              if leg_on(args, "decode") else None)
    hybrid = hybrid_leg(tw, flush, stream) if leg_on(args, "hybrid") else None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not args.no_extras:
        rate, S, dt, cores, done, one = oracle_rate(inp, args.cpu_budget)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"first {S} of {inp.M} tokens, same weights, fwd + bwd, repeated: {done} tokens in {dt:.1f} s",
               "one_core": one}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded splitmix64/Box-Muller, random-init weights)",
        "config": {"workload": WORKLOAD, "M": inp.M, "d_model": inp.d, "d_ff": inp.F, "T": inp.T, "bias": -2.33,
                   "l1": L1, "l2": "flushed between timed steps (512 MB write, then 512 MB read: clean lines)",
                   "parallelism": f"replicas x{world}", "measured_density": nnz / (inp.M * inp.F),
                   "padding_ratio": slots / max(nnz, 1), "slots": slots},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clocks,
        "fwd": {"value": world * inp.M / (ms_fwd / 1000.0), "unit": UNIT, "ms": ms_fwd,
                "call_roofline": call_roofline((1, 2), ms_fwd, inp, slots, nnz, peaks, ceil)},
        "step_roofline": call_roofline((1, 2, 3, 4, 5, 6), ms_step, inp, slots, nnz, peaks, ceil),
        "stages": stages,
        "kernels": kernels,
        "ceilings": {"fma": fma, "gather_TBs": gath, "hbm_GBs": peaks["hbm"], "bf16_TFLOPs": peaks["bf16"]},
        "dense_tcgen05": dense,
        "sparsity_crossover": crossover,
        "inference_fwd": inference,
        "pages_context": PAGES_CONTEXT,
        "down_projection": union,
        "hybrid": hybrid,
        "energy": energy,
        "memory": memory,
        "decode": decode,
        "wall_s_timed": t_wall,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the e2e, dense and CPU legs (profiling runs)")
    ap.add_argument("--decode-batches", default="1,8,64",
                    help="token counts of the decode leg's gated workloads (of 1, 8, 64)")
    ap.add_argument("--legs", default="all",
                    help="comma list of the extra legs to run: e2e, dense, crossover, inference, energy, memory, down, "
                         "decode, hybrid "
                         "(default all; --no-extras runs none)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1 and args.impl == "ours":
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
