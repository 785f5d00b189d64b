#!/usr/bin/env python3
"""Benchmark of the tensor-parallel MLP block on GB300.

One step = one pass of the whole hot path over one batch: the column-parallel
GEMM with fused bias + erf-GeLU, the row-parallel GEMM with the on-device
shard sum, and the full backward (dH with fused GeLU', dB_i, dA_i, the summed
dX, db1, db2).  The workload is s=2048, b=4, h=5120, ffn=20480, p=4 (bf16,
fp32 accumulation).  The line also carries the forward at the pages' sizing
(s=4096, b=1, h=8192, ffn=32768, p=8).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 (launched by torch.distributed.run) every rank runs an independent
replica of the workload on its own GPU (no exchange between ranks: all p shards
of a block live on one GPU); `value` is the total over ranks divided by the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TP-MLP fwd/bwd TFLOP/s & tokens/s on 1 GB300; % of dense BF16 tensor peak"
NOMINAL_BF16_TFLOPS = 2250.0
WARMUP_SECONDS = 2.0  # default warm-up of the GPU arm (see run_gpu)
# short runs: the end-to-end leg starts after as long an idle as the device-timed region did
# (the buffer set-up), at least E2E_IDLE_SECONDS and at most E2E_IDLE_MAX_SECONDS
E2E_IDLE_SECONDS = 1.0
E2E_IDLE_MAX_SECONDS = 5.0
MAIN_WORKLOAD = 5      # fwd + bwd
FWD_WORKLOAD = 4       # forward at the pages' sizing


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=None,
                    help="untimed warm-up steps (default: steps for about %.0f s, so that the timed region runs at the steady clock the power cap settles to)" % WARMUP_SECONDS)
    ap.add_argument("--impl", default="tpmlp", choices=["tpmlp", "reference"])
    ap.add_argument("--workload", type=int, default=MAIN_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fwd-pages", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true", help="skip the SwiGLU / attention-projection timings")
    ap.add_argument("--next-rows-only", action="store_true",
                    help="time only the SwiGLU and attention-projection steps (for profiling their launches)")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="timed steps of the end-to-end leg (default: as many as the device-timed region, at "
                         "most 60; 0 skips the leg)")
    ap.add_argument("--bwd", action="store_true",
                    help="run forward + backward on a forward-only workload (for profiling its backward GEMMs)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    ap.add_argument("--raster", type=int, default=None,
                    help="M-blocks per raster group of the GEMM tiles (tpmlp_set_gemm_raster; library default 16)")
    ap.add_argument("--no-side-stream", action="store_true",
                    help="do not register a side stream for the backward's column sums (they run in line)")
    ap.add_argument("--tp", action="store_true",
                    help="tensor parallelism across the ranks: each GPU holds p/N shards of the fwd+bwd workload "
                         "and the partial Z and dX are summed with an NCCL All-Reduce (strong scaling)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_max(value: float) -> float:
    """Max of a float over all ranks (the value itself when not distributed).
    Uses the process group's own backend: NCCL on GPUs, gloo on CPU."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step_per_rank: float, world: int, slowest_ms_per_step: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return units_per_step_per_rank * world / (slowest_ms_per_step * 1e-3)


def code_digest(texts):
    """sha256 of source texts with comments and blank space removed."""
    import hashlib
    import re
    h = hashlib.sha256()
    for text in texts:
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [" ".join(line.split()) for line in text.splitlines()]
        h.update("\n".join(line for line in lines if line).encode())
    return h.hexdigest()


def kernel_code_digest():
    """Digest of the GEMM kernel sources (code_digest), so that the committed DRAM capture stays
    valid across comment-only edits but not across code edits."""
    texts = []
    for f in ("gemm_tc.cuh", "gemm_tc.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "megatron_tensor_mlp_gb300", "csrc", f)) as fh:
            texts.append(fh.read())
    return code_digest(texts)


def captured_traffic(kernel_key):
    """DRAM bytes per launch of a forward GEMM at the bench workload, from the committed ncu
    summary, or None when the kernel code has changed since that capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_s2048_b4_h5120_ffn20480_p4.txt")
    try:
        digest = kernel_code_digest()
        recorded, vals = None, {}
        for line in open(path):
            if line.startswith("#"):
                continue
            parts = line.split()
            if not parts:
                continue
            if parts[0] == "kernel_code_sha256":
                recorded = parts[1]
            elif len(parts) >= 3:
                vals[parts[0]] = int(parts[1]) + int(parts[2])
        if recorded != digest:
            return None
        return vals.get(kernel_key)
    except (OSError, ValueError):
        return None


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """SM clock, board power and clock-event (throttle) reasons of one GPU, polled every few
    milliseconds on a background thread through NVML's read-only queries (the driver's
    libnvidia-ml, loaded with ctypes), so that even a timed region of a tenth of a second holds
    dozens of samples.  Windows are marked by name (mark_start / mark_end) and summarised by
    summary(name).  Falls back to `nvidia-smi -lms` when NVML cannot be loaded."""

    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    # NVML clock-event reason bits
    _BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
             "hw_power_brake": 0x80}

    def __init__(self, gpu_index, uuid=None, period_s=0.004):
        import threading
        self.gpu, self.uuid, self.period = gpu_index, uuid, period_s
        self.rows = []        # (perf_counter, sm_mhz, max_mhz, power_w, reason_bits)
        self.windows = {}     # name -> [t0, t1]
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = self._open_nvml()

    def _open_nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        try:
            if lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            ok = False
            if self.uuid:
                for u in (self.uuid, "GPU-" + self.uuid):
                    if lib.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(u.encode()), ctypes.byref(h)) == 0:
                        ok = True
                        break
            if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
                return None
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
            return lib, h, reasons
        except (AttributeError, OSError):
            return None

    def _poll_nvml(self):
        import ctypes
        lib, h, reasons = self._nvml
        clk, mx, pw, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        while not self._stop.is_set():
            t = time.perf_counter()
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                p = pw.value / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
                r = bits.value if (reasons is not None and reasons(h, ctypes.byref(bits)) == 0) else 0
                self.rows.append((t, float(clk.value), float(mx.value), p, int(r)))
            self._stop.wait(self.period)

    def _poll_smi(self):
        fields = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active"
        try:
            proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={fields}",
                                     "--format=csv,noheader,nounits", "-lms", "20"],
                                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        while not self._stop.is_set():
            line = proc.stdout.readline()
            if not line:
                break
            f = [x.strip() for x in line.split(",")]
            try:
                self.rows.append((time.perf_counter(), float(f[0]), float(f[1]), float(f[2]), int(f[3], 16)))
            except (ValueError, IndexError):
                continue
        proc.terminate()

    def start(self):
        import threading
        self.source = "nvml" if self._nvml is not None else "nvidia-smi"
        self._thread = threading.Thread(target=self._poll_nvml if self._nvml is not None else self._poll_smi,
                                        daemon=True)
        self._thread.start()

    def mark_start(self, name="timed"):
        self.windows[name] = [time.perf_counter(), None]

    def mark_end(self, name="timed"):
        self.windows[name][1] = time.perf_counter()

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self, name="timed"):
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"], "samples": 0}
        t0, t1 = self.windows.get(name, (None, None))
        inside = [r for r in self.rows if t0 is not None and t1 is not None and t0 <= r[0] <= t1]
        window = "timed region"
        if len(inside) < 3:  # too few samples inside: every sample of the run, and say so
            inside, window = list(self.rows), "whole run"
        reasons = sorted({n for r in inside for n, bit in self._BITS.items() if r[4] & bit})
        med = lambda xs: statistics.median(xs) if xs else None  # noqa: E731
        return {"sm_mhz": med([r[1] for r in inside]), "sm_max_mhz": max((r[2] for r in inside), default=None),
                "reasons": reasons, "samples": len(inside), "window": window, "source": self.source,
                "seconds": round(t1 - t0, 4) if (t0 is not None and t1 is not None) else None,
                "power_w_median": med([r[3] for r in inside if r[3] is not None])}


def e2e_idle_seconds(setup_s):
    """Idle before a short run's end-to-end leg: as long as the buffer set-up that preceded the
    device-timed region, within [E2E_IDLE_SECONDS, E2E_IDLE_MAX_SECONDS]."""
    return min(max(float(setup_s), E2E_IDLE_SECONDS), E2E_IDLE_MAX_SECONDS)


def e2e_step_count(args):
    """Timed steps of the end-to-end leg: --e2e-steps when given (0 skips the leg), else as many as
    the device-timed region, at most 60."""
    return args.e2e_steps if args.e2e_steps is not None else min(60, args.steps)


def peak_regime(clocks, seconds, peaks):
    """The measured bf16 peak that matches how a timed region ran.  The burst figure (cuBLAS
    best-of-10) applies to a region shorter than about a second or one whose median SM clock is
    within 5 % of the maximum; the sustained figure (cuBLAS looped for seconds at the power cap)
    only to a settled, seconds-long region below that clock."""
    med, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    near_max = med is not None and mx and med >= 0.95 * mx
    if seconds < 1.0 or near_max or med is None:
        why = (f"timed region {seconds:.3f} s" + (f", median SM {med:.0f} of {mx:.0f} MHz" if med else ""))
        return "burst", peaks.get("bf16_tflops", 1900.0), why
    return "sustained", peaks.get("bf16_tflops_sustained", 1700.0), \
        f"timed region {seconds:.3f} s, median SM {med:.0f} of {mx:.0f} MHz"


# --------------------------------------------------------------------------- CPU (oracle) arm
class OracleSample:
    """The oracle (fp64 CPU) on a row sample of the workload: forward (+ backward)
    on the first M' tokens with the full weights.  Inputs are generated once."""

    def __init__(self, wl):
        import oracle
        from megatron_tensor_mlp_gb300 import synth

        self.wl = wl
        self.orc = oracle.get()
        self.synth = synth
        self.A = synth.widen(wl.gen("A"))
        self.B = synth.widen(wl.gen("B"))
        self.b1 = None if wl.sigma_bias == 0 else synth.widen(wl.gen("b1"))
        self.b2 = None if wl.sigma_bias == 0 else synth.widen(wl.gen("b2"))
        self.per_token = (wl.fwd_flops() + (wl.bwd_flops() if wl.backward else 0.0)) / wl.M

    def run(self, tokens):
        """Seconds for one oracle pass over the first `tokens` tokens."""
        wl = self.wl
        X = self.synth.widen(wl.gen("X", 0, tokens))
        dZ = self.synth.widen(wl.gen("dZ", 0, tokens)) if wl.backward else None
        t0 = time.perf_counter()
        H, Y, _ = self.orc.mlp_fwd(X, self.A, self.b1, self.B, self.b2)
        if wl.backward:
            self.orc.mlp_bwd(X, self.A, self.B, H, Y, dZ)
        return time.perf_counter() - t0

    def calibrate(self, target_seconds):
        """Largest power-of-two token count whose pass stays near target_seconds.  One untimed
        pass first: the first call also pays for the oracle's thread start-up and first touches
        of its output arrays, which would otherwise stop the doubling at one token."""
        tokens = 1
        self.run(tokens)
        dt = self.run(tokens)
        while tokens * 2 <= self.wl.M and dt * 2 <= target_seconds:
            tokens *= 2
            dt = self.run(tokens)
        return tokens, dt

    def describe(self, tokens, dt):
        wl = self.wl
        return (f"oracle fp64 {'fwd+bwd' if wl.backward else 'fwd'} on the first {tokens} of {wl.M} tokens "
                f"with the full weights ({dt:.2f} s per pass)")

    def tflops(self, tokens, dt):
        return self.per_token * tokens / dt / 1e12


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from megatron_tensor_mlp_gb300 import synth

    wl = synth.WORKLOADS[args.workload]
    sample = OracleSample(wl)
    if args.warmup is None:
        args.warmup = 3
    per_step = min(30.0, 150.0 / max(1, args.steps + args.warmup))  # whole run within a few minutes
    tokens, _ = sample.calibrate(per_step)
    times = []
    for i in range(args.warmup + args.steps):
        dt = sample.run(tokens)
        if i >= args.warmup:
            times.append(dt)
    dt = statistics.median(times)
    v = sample.tflops(tokens, dt)
    out = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": wl.name, "s": wl.s, "b": wl.b, "h": wl.h, "ffn": wl.ffn, "p": wl.p,
                      "parallelism": "replicas"},
           "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": sample.orc.num_threads(),
                            "kind": "oracle", "sample": sample.describe(tokens, dt)},
           "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# --------------------------------------------------------------------------- GPU arm
def settled_ms(fn, stream, explicit_warmup=None, seconds=0.4, sampler=None, window=None):
    """Milliseconds per call of fn at the settled power-capped clock: warm up for about
    WARMUP_SECONDS (or explicit_warmup calls when given), then time enough calls for about
    `seconds` with CUDA events on `stream` (marked as `window` on the clock sampler, if given)."""
    import torch
    if explicit_warmup is None:
        t_w = time.time()
        while time.time() - t_w < WARMUP_SECONDS:
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
    else:
        for _ in range(max(3, explicit_warmup)):
            fn()
        torch.cuda.synchronize()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(5):
        fn()
    z.record(stream)
    torch.cuda.synchronize()
    n = max(10, int(seconds / max(1e-6, a.elapsed_time(z) / 5e3)))
    if sampler is not None:
        sampler.mark_start(window)
    a.record(stream)
    for _ in range(n):
        fn()
    z.record(stream)
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.mark_end(window)
    return a.elapsed_time(z) / n, n


def graph_ms(fn, explicit_warmup=None, reps=20, seconds=0.4):
    """Milliseconds per call of fn(stream) replayed from a CUDA graph of `reps` calls: the GPU's own
    time for launch-bound work, without the host's per-call cost (a Python loop of ctypes calls).
    Warm-up as in settled_ms; fn launches on the stream it is given (the capture stream here)."""
    import torch
    cur = torch.cuda.current_stream()
    settled_ms(lambda: fn(cur), cur, explicit_warmup, seconds=0.05)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = torch.cuda.current_stream()
        for _ in range(reps):
            fn(cap)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cur)
    g.replay()
    z.record(cur)
    torch.cuda.synchronize()
    n = max(5, int(seconds / max(1e-6, a.elapsed_time(z) / 1e3)))
    a.record(cur)
    for _ in range(n):
        g.replay()
    z.record(cur)
    torch.cuda.synchronize()
    return a.elapsed_time(z) / (n * reps), n * reps


def time_other_configs(stream, explicit_warmup):
    """Forward and forward+backward of the parity-test workloads 2 and 3 (their own shapes,
    seeded synthetic inputs), at the settled clock.  Workload 2 is launch bound (a forward is
    ~40 us of GPU work against ~15-20 us of host work per library call from Python), so the
    headline times come from CUDA-graph replay; the eager loop's times are reported beside them."""
    from megatron_tensor_mlp_gb300 import harness, synth
    from megatron_tensor_mlp_gb300 import tpmlp as T
    import torch
    out = {}
    for cfg in (2, 3):
        wl = synth.WORKLOADS[cfg]
        b_ = harness.MLPBuffers(wl, backward=True)
        ms_f, n_f = graph_ms(lambda s: b_.fwd(stream=s), explicit_warmup)
        ms_fb, n_fb = graph_ms(lambda s: (b_.fwd(stream=s), b_.bwd(stream=s)), explicit_warmup)
        e_f, _ = settled_ms(lambda: b_.fwd(stream=stream), stream, explicit_warmup)
        e_fb, _ = settled_ms(lambda: (b_.fwd(stream=stream), b_.bwd(stream=stream)), stream, explicit_warmup)
        T.tpmlp_device_status()
        f_fwd, f_bwd = wl.fwd_flops(), wl.bwd_flops()
        out[wl.name] = {"fwd_ms": round(ms_f, 5), "fwd_TFLOP/s": round(f_fwd / (ms_f * 1e-3) / 1e12, 1),
                        "fwd_bwd_ms": round(ms_fb, 5),
                        "fwd_bwd_TFLOP/s": round((f_fwd + f_bwd) / (ms_fb * 1e-3) / 1e12, 1),
                        "fwd_tokens_per_s": round(wl.M / (ms_f * 1e-3), 1), "steps": [n_f, n_fb],
                        "timing": "CUDA graph of 20 calls, replayed",
                        "eager_fwd_ms": round(e_f, 5), "eager_fwd_bwd_ms": round(e_fb, 5)}
        del b_
        torch.cuda.empty_cache()
    return out


def time_torch_context(stream, explicit_warmup):
    """Context only: the same fwd+bwd block at the bench workload written with plain PyTorch
    ops on the same GPU -- unsharded torch.matmul (cuBLAS, bf16 in / fp32 accumulate / bf16
    out), bias adds, erf-GeLU and its derivative as separate elementwise kernels -- timed
    like the main line.  Weight gradients come out in bf16 here (fp32 in tpmlp)."""
    import torch
    from megatron_tensor_mlp_gb300 import synth
    wl = synth.WORKLOADS[MAIN_WORKLOAD]
    M, h, f = wl.M, wl.h, wl.ffn
    bf = torch.bfloat16
    gen = lambda sid, shp, sig: torch.from_numpy(  # noqa: E731
        synth.normal(wl.seed, sid, shp, sig, "bf16").view("int16")).view(bf).cuda()
    X, A, B, dZ = gen(1, (M, h), 1.0), gen(2, (h, f), 0.02), gen(3, (f, h), 0.02), gen(6, (M, h), 1.0)
    b1, b2 = torch.zeros(f, dtype=bf, device="cuda"), torch.zeros(h, dtype=bf, device="cuda")
    inv_sqrt_2pi = 0.3989422804014327

    def step():
        H = torch.addmm(b1, X, A)
        Y = torch.nn.functional.gelu(H)
        torch.addmm(b2, Y, B)
        dY = dZ @ B.t()
        Hf = H.float()
        dH = (dY.float() * (torch.special.ndtr(Hf) + Hf * torch.exp(-0.5 * Hf * Hf) * inv_sqrt_2pi)).to(bf)
        Y.t() @ dZ
        X.t() @ dH
        dH @ A.t()
        dH.sum(0, dtype=torch.float32)
        dZ.sum(0, dtype=torch.float32)

    ms, n = settled_ms(step, stream, explicit_warmup, seconds=1.0)  # torch ops run on `stream` (current)
    flops = wl.fwd_flops() + wl.bwd_flops()
    out = {"workload": wl.name, "fwd_bwd_ms": round(ms, 4), "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1),
           "steps": n, "what": "torch.matmul (cuBLAS) + unfused bias / erf-GeLU / GeLU' / column sums, "
                               "one unsharded GPU; context, not a target"}
    del X, A, B, dZ
    torch.cuda.empty_cache()
    return out


def time_next_rows(stream, steps, peaks, explicit_warmup=None):
    """Forward+backward timings of the widened rows at the fwd+bwd workload's sizes
    (s=2048, b=4, h=5120, p=4): the SwiGLU block (ffn=20480 per branch) and the attention
    tensor-parallel projections (QKV column projection over the per-head interleave, 40 heads,
    and the output row projection); then the bandwidth of the two layout kernels at the pages'
    sizing.  Inputs are seeded synthetic bf16."""
    import torch
    from megatron_tensor_mlp_gb300 import synth
    from megatron_tensor_mlp_gb300 import tpmlp as T

    s, b, h, f, p, heads = 2048, 4, 5120, 20480, 4, 40
    M, fs = s * b, f // p
    bf = torch.bfloat16
    gen = lambda stream_id, shp, sig: torch.from_numpy(  # noqa: E731
        synth.normal(11, stream_id, shp, sig, "bf16").view("int16")).view(bf).cuda()
    out = {}

    def timed(fn, n):
        ms, _ = settled_ms(fn, stream, explicit_warmup)
        T.tpmlp_device_status()
        return ms

    n = max(10, steps // 4)
    # SwiGLU block: gate+up column GEMM (2*2*M*h*f), row GEMM (2*M*f*h); backward twice that
    X, dZ = gen(1, (M, h), 1.0), gen(6, (M, h), 1.0)
    W = torch.empty((p, h, 2 * fs), dtype=bf, device="cuda")
    T.tpmlp_swiglu_pack(gen(2, (h, f), 0.02), gen(9, (h, f), 0.02), W, h, f, p)
    B = gen(3, (f, h), 0.02).view(p, fs, h)
    Z, Y = torch.empty((M, h), dtype=bf, device="cuda"), torch.empty((p, M, fs), dtype=bf, device="cuda")
    H = torch.empty((p, M, 2 * fs), dtype=torch.float32, device="cuda")
    dX, dH = torch.empty((M, h), dtype=bf, device="cuda"), torch.empty((p, M, 2 * fs), dtype=bf, device="cuda")
    dW = torch.empty((p, h, 2 * fs), dtype=torch.float32, device="cuda")
    dB = torch.empty((p, fs, h), dtype=torch.float32, device="cuda")
    dbw, db2 = torch.empty((p, 2 * fs), dtype=torch.float32, device="cuda"), torch.empty(h, dtype=torch.float32,
                                                                                         device="cuda")

    def swiglu_step():
        T.tpmlp_swiglu_mlp_fwd(X, W, None, B, None, Z, Y, H, s, b, h, f, p, stream=stream)
        T.tpmlp_swiglu_mlp_bwd(X, W, B, H, Y, dZ, dX, dW, dB, dbw, db2, dH, s, b, h, f, p, stream=stream)

    ms = timed(swiglu_step, n)
    flops = 3 * (2 * 2 * M * h * f + 2 * M * f * h)  # fwd 6 M h f, bwd 12 M h f
    tf = flops / (ms * 1e-3) / 1e12
    out["swiglu_fwd_bwd"] = {"shape": f"s{s} b{b} h{h} ffn{f} p{p}", "ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                             "pct_of_nominal_2250": round(100 * tf / NOMINAL_BF16_TFLOPS, 2)}
    del W, H, dW, dH, Y, dB, dbw
    torch.cuda.empty_cache()

    # attention projections: QKV [h, 3h] column parallel by heads, output [h, h] row parallel
    Wq = torch.empty((h, 3 * h), dtype=bf, device="cuda")
    T.tpmlp_qkv_interleave(gen(12, (h, 3 * h), 0.02), Wq, h, h, heads, p)
    Wq_sh = torch.empty((p, h, 3 * h // p), dtype=bf, device="cuda")
    T.tpmlp_shard_columns(Wq, Wq_sh, h, 3 * h, p)
    Wo = gen(13, (h, h), 0.02).view(p, h // p, h)
    QKV = torch.empty((p, M, 3 * h // p), dtype=bf, device="cuda")
    ctx = gen(14, (p, M, h // p), 1.0)
    dQKV = gen(15, (p, M, 3 * h // p), 1.0)
    dWq = torch.empty((p, h, 3 * h // p), dtype=torch.float32, device="cuda")
    dWo = torch.empty((p, h // p, h), dtype=torch.float32, device="cuda")
    dctx = torch.empty((p, M, h // p), dtype=bf, device="cuda")

    def attn_step():
        T.tpmlp_column_fwd(X, Wq_sh, None, QKV, None, s, b, h, 3 * h, p, act=T.ACT_NONE, stream=stream)
        T.tpmlp_row_fwd(ctx, Wo, None, Z, s, b, h, h, p, stream=stream)
        T.tpmlp_row_bwd(ctx, Wo, dZ, None, dctx, dWo, None, s, b, h, h, p, act=T.ACT_NONE, stream=stream)
        T.tpmlp_column_bwd(X, Wq_sh, dQKV, dX, dWq, None, s, b, h, 3 * h, p, stream=stream)

    ms = timed(attn_step, n)
    flops = 3 * (2 * M * h * 3 * h + 2 * M * h * h)
    tf = flops / (ms * 1e-3) / 1e12
    out["attention_projections_fwd_bwd"] = {"shape": f"s{s} b{b} h{h} heads{heads} p{p}", "ms": round(ms, 4),
                                            "TFLOP/s": round(tf, 1),
                                            "pct_of_nominal_2250": round(100 * tf / NOMINAL_BF16_TFLOPS, 2)}
    del Wq, Wq_sh, Wo, QKV, ctx, dQKV, dWq, dWo, dctx, X, dZ, B, Z, dX
    torch.cuda.empty_cache()

    # The layout kernels (set-up, bit-exact copies) at the pages' sizing (h=8192, ffn=32768, p=8,
    # 64 heads): HBM bound, so the measure is the bytes they move (the tensor read once and
    # written once) against the measured copy bandwidth.
    hp, fp, pp, hd = 8192, 32768, 8, 64
    hbm = peaks.get("hbm_gbs", 6800.0)

    def layout_row(name, shape, fn, nbytes):
        ms = timed(fn, n)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"shape": shape, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                     "frac_of_measured_hbm": round(gbs / hbm, 4)}

    Wa = gen(16, (hp, fp), 0.02)
    Wa_sh = torch.empty((pp, hp, fp // pp), dtype=bf, device="cuda")
    layout_row("shard_columns", f"A [{hp}, {fp}] bf16 -> [{pp}][{hp}][{fp // pp}]",
               lambda: T.tpmlp_shard_columns(Wa, Wa_sh, hp, fp, pp, stream=stream), 2 * Wa.numel() * 2)
    del Wa, Wa_sh
    torch.cuda.empty_cache()
    Wq = gen(17, (hp, 3 * hp), 0.02)
    Wq_out = torch.empty_like(Wq)
    layout_row("qkv_interleave", f"W_qkv [{hp}, {3 * hp}] bf16, {hd} heads, p={pp}",
               lambda: T.tpmlp_qkv_interleave(Wq, Wq_out, hp, hp, hd, pp, stream=stream), 2 * Wq.numel() * 2)
    return out


def run_gpu(args):
    import torch

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    from megatron_tensor_mlp_gb300 import harness, synth
    from megatron_tensor_mlp_gb300 import tpmlp as T

    peaks, peak_kind = load_peaks()
    if args.raster is not None:
        T.tpmlp_set_gemm_raster(args.raster)
    if not args.no_side_stream:
        # the caller's side stream for the fused backwards' column sums (kept for the whole run)
        side = (torch.cuda.Stream(), torch.cuda.Event(), torch.cuda.Event())
        T.tpmlp_set_side_stream(*side)
    if args.tp:
        return run_tp(args, peaks)
    if args.next_rows_only:
        rows = time_next_rows(torch.cuda.current_stream(), args.steps, peaks, args.warmup)
        if rank == 0:
            print(json.dumps({"metric": "widened rows, fwd+bwd TFLOP/s on 1 GB300", "next_rows": rows,
                              "steps": args.steps, "warmup": args.warmup}), flush=True)
        return
    wl = synth.WORKLOADS[args.workload]
    if args.bwd and not wl.backward:
        import dataclasses
        wl = dataclasses.replace(wl, backward=True, name=wl.name.replace("-fwd ", "-fwd-bwd "))
    t_setup = time.time()
    buf = harness.MLPBuffers(wl)
    torch.cuda.synchronize()
    setup_s = time.time() - t_setup  # the GPU idles (but for the input copies) before the timed leg
    s, b, h, f, p = buf.dims()
    M = wl.M
    stream = torch.cuda.current_stream()

    def step():
        T.tpmlp_column_fwd(buf.X, buf.A_sh, buf.b1_sh, buf.Y, buf.H, s, b, h, f, p, stream=stream)
        T.tpmlp_row_fwd(buf.Y, buf.B_sh, buf.b2, buf.Z, s, b, h, f, p, stream=stream)
        if wl.backward:
            buf.bwd(stream=stream)

    props = torch.cuda.get_device_properties(local)
    sampler = ClockSampler(local, uuid=str(getattr(props, "uuid", "") or "") or None)
    sampler.start()
    # Warm-up: the board's power controller allows a higher clock for the first second
    # or so of load and then settles; by default warm up for WARMUP_SECONDS so that the
    # timed region (and the sustained cuBLAS rate it is compared with) sees the settled clock.
    if args.warmup is None:
        n_warm, t_w = 0, time.time()
        while n_warm < 5 or time.time() - t_w < WARMUP_SECONDS:
            for _ in range(5):
                step()
            n_warm += 5
            torch.cuda.synchronize()
    else:
        n_warm = max(3, args.warmup)
        for _ in range(n_warm):
            step()
    torch.cuda.synchronize()
    T.tpmlp_device_status()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    # timed region: per-call events on the launching stream
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler.mark_start()
    n_launch0 = T.tpmlp_launch_count()
    t_start.record(stream)
    per_call = None
    for i in range(K):
        e = ev[i]
        c0 = T.tpmlp_launch_count()
        e[0].record(stream)
        T.tpmlp_column_fwd(buf.X, buf.A_sh, buf.b1_sh, buf.Y, buf.H, s, b, h, f, p, stream=stream)
        e[1].record(stream)
        c1 = T.tpmlp_launch_count()
        T.tpmlp_row_fwd(buf.Y, buf.B_sh, buf.b2, buf.Z, s, b, h, f, p, stream=stream)
        e[2].record(stream)
        c2 = T.tpmlp_launch_count()
        if wl.backward:
            buf.bwd(stream=stream)
        e[3].record(stream)
        if per_call is None:
            per_call = {"column_fwd": c1 - c0, "row_fwd": c2 - c1, "mlp_bwd": T.tpmlp_launch_count() - c2}
    t_end.record(stream)
    n_launch = T.tpmlp_launch_count() - n_launch0  # this library's kernels in the timed region
    torch.cuda.synchronize()
    sampler.mark_end()
    barrier()
    clocks = sampler.summary()
    T.tpmlp_device_status()
    total_ms = dist_max(t_start.elapsed_time(t_end))
    ms_step = total_ms / K
    col_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    row_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    bwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev) if wl.backward else 0.0
    flops_step = wl.fwd_flops() + (wl.bwd_flops() if wl.backward else 0.0)
    value = job_throughput(flops_step, ws, ms_step) / 1e12
    tokens_s = job_throughput(M, ws, ms_step)

    # roofline: the single-launch GEMM with the larger time (column with GeLU, or row with shard sum)
    gemm_flops = 2.0 * M * h * f
    dom_key, dom_name, dom_ms = ("column_fwd", "column_fwd (tcgen05 GEMM + bias + erf-GeLU epilogue)", col_ms) \
        if col_ms >= row_ms else ("row_fwd", "row_fwd (tcgen05 GEMM + in-TMEM shard sum)", row_ms)
    if per_call[dom_key] > 1:
        dom_name += f"; {per_call[dom_key]} launches: full waves on CTA pairs, last partial wave split-K"
    achieved = gemm_flops / (dom_ms * 1e-3) / 1e12
    regime, peak, why = peak_regime(clocks, total_ms / 1e3, peaks)
    burst, sustained = peaks.get("bf16_tflops", 1900.0), peaks.get("bf16_tflops_sustained", 1700.0)
    roofline = {"bound": "tensor", "kernel": dom_name, "achieved": round(achieved, 1), "peak": peak,
                "peak_kind": f"bf16_tflops{'' if regime == 'burst' else '_sustained'} ({regime}, {peak_kind}: "
                             f"{why})",
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "frac_of_measured_burst": round(achieved / burst, 4),
                "frac_of_measured_sustained": round(achieved / sustained, 4),
                "frac_of_nominal_2250": round(achieved / NOMINAL_BF16_TFLOPS, 4),
                "traffic": captured_traffic(dom_key) if args.workload == MAIN_WORKLOAD else None,
                "traffic_algorithmic": {"column_fwd": 964e6, "row_fwd": 629e6}.get(dom_key)
                if args.workload == MAIN_WORKLOAD else None,
                "per_call_ms": {"column_fwd": round(col_ms, 4), "row_fwd": round(row_ms, 4),
                                "mlp_bwd": round(bwd_ms, 4)},
                "launches_per_call": per_call}

    # end to end through the public API with host buffers (pinned), copies inside the timed region.
    # Steps are pipelined the way a caller would run them: step i+1's inputs are copied in and
    # step i-1's results copied out on a copy stream while step i computes (double-buffered
    # device inputs and outputs); every step's copies still happen inside the timed region.
    e2e = None
    n_e2e = e2e_step_count(args)
    if n_e2e > 0:
        X_host = [buf.X.cpu().pin_memory() for _ in range(2)]
        dZ_host = [buf.dZ.cpu().pin_memory() for _ in range(2)] if wl.backward else None
        Z_host = [torch.empty(buf.Z.shape, dtype=buf.Z.dtype).pin_memory() for _ in range(2)]
        dX_host = [torch.empty(buf.dX.shape, dtype=buf.dX.dtype).pin_memory() for _ in range(2)] \
            if wl.backward else None
        Xd = [buf.X, torch.empty_like(buf.X)]
        dZd = [buf.dZ, torch.empty_like(buf.dZ)] if wl.backward else None
        Zd = [buf.Z, torch.empty_like(buf.Z)]
        dXd = [buf.dX, torch.empty_like(buf.dX)] if wl.backward else None
        h2d = X_host[0].numel() * X_host[0].element_size() + \
            (dZ_host[0].numel() * dZ_host[0].element_size() if wl.backward else 0)
        d2h = Z_host[0].numel() * Z_host[0].element_size() + \
            (dX_host[0].numel() * dX_host[0].element_size() if wl.backward else 0)
        copy_stream = torch.cuda.Stream()
        in_ready = [torch.cuda.Event() for _ in range(2)]
        out_ready = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]

        def h2d_copy(i):
            j = i % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(out_done[j])  # buffers of step i-2 are free again
                Xd[j].copy_(X_host[i % 2], non_blocking=True)
                if wl.backward:
                    dZd[j].copy_(dZ_host[i % 2], non_blocking=True)
                in_ready[j].record(copy_stream)

        def compute(i):
            j = i % 2
            stream.wait_event(in_ready[j])
            T.tpmlp_mlp_fwd(Xd[j], buf.A_sh, buf.b1_sh, buf.B_sh, buf.b2, Zd[j], buf.Y, buf.H, s, b, h, f, p,
                            stream=stream)
            if wl.backward:
                T.tpmlp_mlp_bwd(Xd[j], buf.A_sh, buf.B_sh, buf.H, buf.Y, dZd[j], dXd[j], buf.dA_sh, buf.dB_sh,
                                buf.db1_sh, buf.db2, buf.dH, s, b, h, f, p, stream=stream)
            out_ready[j].record(stream)

        def d2h_copy(i):
            j = i % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(out_ready[j])
                Z_host[j].copy_(Zd[j], non_blocking=True)
                if wl.backward:
                    dX_host[j].copy_(dXd[j], non_blocking=True)
                out_done[j].record(copy_stream)

        def run_pipeline(n):
            for i in range(2):
                out_done[i].record(copy_stream)
            h2d_copy(0)
            for i in range(n):
                if i + 1 < n:
                    h2d_copy(i + 1)
                compute(i)
                d2h_copy(i)
            stream.wait_stream(copy_stream)

        # The same clock regime as the device-timed region: by default a settled warm-up; in a
        # short run (explicit --warmup) W pipelined steps after the GPU has been idle as long as
        # before the device-timed region (the buffer set-up), so that the power controller has
        # raised the clock again and neither leg inherits the other's power-capped tail.
        idle_s = 0.0
        if args.warmup is not None:
            torch.cuda.synchronize()
            idle_s = e2e_idle_seconds(setup_s)
            time.sleep(idle_s)
        t_w = time.time()
        n_w = 0
        while True:
            run_pipeline(5)
            n_w += 5
            torch.cuda.synchronize()
            if (args.warmup is not None and n_w >= max(3, args.warmup)) or \
                    (args.warmup is None and time.time() - t_w >= WARMUP_SECONDS):
                break
        barrier()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sampler.mark_start("e2e")
        a.record(stream)
        copy_stream.wait_event(a)  # no copy of the timed steps starts before the timed region
        run_pipeline(n_e2e)
        z.record(stream)
        torch.cuda.synchronize()
        sampler.mark_end("e2e")
        e2e_ms = dist_max(a.elapsed_time(z) / n_e2e)
        ce = sampler.summary("e2e")
        e2e = {"value": round(job_throughput(flops_step, ws, e2e_ms) / 1e12, 2), "unit": "TFLOP/s",
               "ms_per_step": round(e2e_ms, 4), "steps": n_e2e, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "every step copies X, dZ in from pinned host memory and reads Z, dX back, on a copy "
                       "stream overlapped with the neighbouring steps' compute; weights stay resident; "
                       "timed in the device-timed region's clock regime (settled, or after the same idle "
                       "start in a short run)",
               "clocks": {k: ce.get(k) for k in ("sm_mhz", "reasons", "samples", "window", "power_w_median")},
               "idle_before_s": round(idle_s, 2)}
    T.tpmlp_device_status()

    # the forward at the pages' sizing (the >= 60% of dense bf16 target)
    fwd_pages = None
    if not args.no_fwd_pages and args.workload != FWD_WORKLOAD:
        del buf
        torch.cuda.empty_cache()
        w4 = synth.WORKLOADS[FWD_WORKLOAD]
        b4 = harness.MLPBuffers(w4, backward=False)
        # settled clock: building the inputs above left the GPU idle for a while
        ms4, n4 = settled_ms(lambda: b4.fwd(stream=stream), stream, args.warmup, seconds=0.5, sampler=sampler,
                             window="fwd_pages")
        T.tpmlp_device_status()
        tf4 = w4.fwd_flops() / (ms4 * 1e-3) / 1e12
        c4 = sampler.summary("fwd_pages")
        regime4, peak4, why4 = peak_regime(c4, ms4 * n4 / 1e3, peaks)
        fwd_pages = {"workload": w4.name, "ms": round(ms4, 4), "TFLOP/s": round(tf4, 1),
                     "tokens_per_s": round(w4.M / (ms4 * 1e-3), 1),
                     "pct_of_nominal_2250": round(100 * tf4 / NOMINAL_BF16_TFLOPS, 2),
                     "pct_of_measured_peak": round(100 * tf4 / peak4, 2),
                     "measured_peak_kind": f"{regime4} ({why4})",
                     "pct_of_measured_burst": round(100 * tf4 / peaks.get("bf16_tflops", 1900.0), 2),
                     "pct_of_measured_sustained": round(100 * tf4 / peaks.get("bf16_tflops_sustained", 1700.0), 2),
                     "clocks": {k: c4.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "window")},
                     "steps": n4}
        del b4
        torch.cuda.empty_cache()

    other_configs = None
    if not args.no_next_rows and args.workload == MAIN_WORKLOAD:
        other_configs = time_other_configs(stream, args.warmup)

    next_rows = None
    if not args.no_next_rows and args.workload == MAIN_WORKLOAD:
        torch.cuda.empty_cache()
        next_rows = time_next_rows(stream, K, peaks, args.warmup)

    torch_context = None
    if not args.no_next_rows and args.workload == MAIN_WORKLOAD:
        torch_context = time_torch_context(stream, args.warmup)

    sampler.stop()
    device = {"name": props.name, "sm_count": props.multi_processor_count, "cc": f"{props.major}.{props.minor}",
              "torch": torch.__version__, "cuda_runtime": torch.version.cuda}
    try:
        r = subprocess.run(["nvidia-smi", "-i", str(local), "--query-gpu=driver_version", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=20)
        device["driver"] = r.stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        device["driver"] = None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        sample = OracleSample(wl)
        tokens, dt = sample.calibrate(args.cpu_seconds)
        cpu = {"value": round(sample.tflops(tokens, dt), 6), "unit": "TFLOP/s", "cores": sample.orc.num_threads(),
               "kind": "oracle", "sample": sample.describe(tokens, dt)}

    if rank == 0:
        out = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws, "steps": K,
               "warmup": n_warm, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": {"workload": wl.name, "s": s, "b": b, "h": h, "ffn": f, "p": p,
                          "step": "fwd+bwd" if wl.backward else "fwd",
                          "side_stream": not args.no_side_stream,
                          "raster_group_m": T.tpmlp_get_gemm_raster(),
                          "parallelism": f"replicas x{ws} (all p shards on each GPU)",
                          "l2": "inputs larger than L2 (working set > 1 GB per step)"},
               "tokens_per_s": round(tokens_s, 1),
               "pct_of_nominal_bf16_peak": round(100 * value / ws / NOMINAL_BF16_TFLOPS, 2),
               "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
               "gpu_launches": n_launch, "clocks": clocks,
               "fwd_pages_sizing": fwd_pages, "next_rows": next_rows,
               "other_configs": other_configs, "context_torch": torch_context, "device": device}
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_tp(args, peaks):
    """The fwd+bwd workload with its p shards spread over the N ranks (p/N per GPU): each step
    computes the rank-local partials, sums Z and dX over the ranks with an NCCL All-Reduce and
    finishes them (megatron_tensor_mlp_gb300.tp).  Total work is fixed: strong scaling."""
    import numpy as np
    import torch
    from megatron_tensor_mlp_gb300 import harness, synth, tp
    from megatron_tensor_mlp_gb300 import tpmlp as T

    ws, rank, local = dist_env()
    wl = synth.WORKLOADS[MAIN_WORKLOAD]
    s, b, h, f, p = wl.s, wl.b, wl.h, wl.ffn, wl.p
    if p % ws != 0:
        raise SystemExit(f"--tp needs the shard count p={p} to be a multiple of the rank count {ws}")
    if ws > 1:
        import torch.distributed as dist
        all_reduce = tp.process_group_all_reduce()
    else:
        all_reduce = lambda t: None  # noqa: E731  (one rank: the sum is the partial itself)
    lo, hi = tp.feature_range(rank, ws, f)
    fr, pl = hi - lo, p // ws
    X, dZ = harness.to_torch(wl.gen("X")), harness.to_torch(wl.gen("dZ"))
    A = harness.to_torch(np.ascontiguousarray(wl.gen("A")[:, lo:hi]))
    A_sh = torch.empty((pl, h, fr // pl), dtype=torch.bfloat16, device="cuda")
    T.tpmlp_shard_columns(A, A_sh, h, fr, pl)
    del A
    B_sh = harness.to_torch(np.ascontiguousarray(wl.gen("B")[lo:hi])).view(pl, fr // pl, h)
    ops = tp.LibraryRankOps(s, b, h, fr, pl)

    def step():
        Z, Y, H = tp.tp_mlp_fwd(ops, all_reduce, X, A_sh, None, B_sh, None)
        tp.tp_mlp_bwd(ops, all_reduce, X, A_sh, B_sh, H, Y, dZ)

    n_warm = 5 if args.warmup is None else max(3, args.warmup)
    for _ in range(n_warm):
        step()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    stream = torch.cuda.current_stream()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_launch0 = T.tpmlp_launch_count()
    a.record(stream)
    for _ in range(args.steps):
        step()
    z.record(stream)
    n_launch = T.tpmlp_launch_count() - n_launch0
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    T.tpmlp_device_status()
    ms = dist_max(a.elapsed_time(z) / args.steps)
    flops = wl.fwd_flops() + wl.bwd_flops()
    value = flops / (ms * 1e-3) / 1e12  # the whole block, once, over the group
    if rank == 0:
        print(json.dumps({"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws,
                          "steps": args.steps, "warmup": n_warm, "ms_per_step": round(ms, 4),
                          "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
                          "data": "synthetic",
                          "config": {"workload": wl.name, "s": s, "b": b, "h": h, "ffn": f, "p": p,
                                     "parallelism": f"tp{ws} ({pl} of {p} shards per GPU, NCCL All-Reduce of "
                                                    "the fp32 Z and dX partials)"},
                          "all_reduce_bytes_per_step": 2 * s * b * h * 4 if ws > 1 else 0,
                          "gpu_launches": n_launch}), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
