#!/usr/bin/env python3
"""Benchmark of the TurboQuant hot path on B300: quantize K and V of one layer
into the packed cache, then one decode-attention step over that cache.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-e2e] [--no-cpu-baseline]

Prints ONE JSON line on rank 0.  The metric is
the algorithmic HBM traffic of the whole step (bytes the packed format forces
every implementation to move) divided by the device time of the step, in GB/s;
quantize Mrows/s and decode GB/s are reported alongside.  Inputs are synthetic
and resident in HBM; L2 is flushed (a 256 MiB write) before every timed step.
Under torchrun each rank runs the same per-GPU workload on its own device
(weak scaling; no data-path collective) and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synthetic  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
WARM_SECONDS = 1.0
# Kernel launches per library call at d = 128 (quantize: 1; decode: the kernel
# that clears the split tickets, then the split kernel, which rotates the
# queries and merges its splits itself; the decode-step append's decode: the
# split kernel alone, the append having cleared the tickets).
LAUNCHES = {"quantize": 1, "decode": 2, "append_decode": 1}


def kv_one_launch(spec) -> bool:
    """tq_quantize_kv runs K and V in one launch when both are mse with the same
    d in {64, 128}, bits and rotation (otherwise it makes one launch per side)."""
    return (spec["k_variant"] == spec["v_variant"] == "mse" and spec["k_bits"] == spec["v_bits"]
            and spec["d"] in (64, 128))
# The arithmetic the path computes in.
DTYPE_LABEL = "bf16 in, bf16/f16 hi+lo MMA operands, fp32 accumulate and out"
QUANT_SOURCES = ["kv_cache_vector_18_b300/csrc/tq_quantize_tc.cu", "kv_cache_vector_18_b300/csrc/tq_sm100.cuh"]
DECODE_SOURCES = ["kv_cache_vector_18_b300/csrc/tq_decode_mma.cuh", "kv_cache_vector_18_b300/csrc/tq_decode_args.h",
                  "kv_cache_vector_18_b300/csrc/tq_decode.cu"]


# ----------------------------------------------------------------------------- ranks
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, seconds_per_rank: float, world: int, device=None) -> float:
    """Whole-job throughput: all units processed by all ranks / the slowest rank's time."""
    total = sum_over_ranks(units_per_rank, world, device)
    slowest = max_over_ranks(seconds_per_rank, world, device)
    return total / slowest if slowest > 0 else float("nan")


# ----------------------------------------------------------------------------- workload
def workload_spec(name: str) -> dict:
    w = dict(synthetic.WORKLOADS[name])
    if name == "llama70b_layer_kv_quant":
        return dict(name=name, B=1, Hq=w["hq"], Hkv=w["heads"], T=w["tokens"], d=w["d"],
                    k_bits=w["bits"], k_variant=w["variant"], v_bits=w["bits"], v_variant=w["variant"],
                    dist="outliers", lens=None)
    if name == "decode_131k":
        return dict(name=name, B=w["B"], Hq=w["Hq"], Hkv=w["Hkv"], T=w["T"], d=w["d"], k_bits=w["k_bits"],
                    k_variant=w["k_variant"], v_bits=w["v_bits"], v_variant=w["v_variant"], dist="gauss", lens=None)
    if name == "batched_decode_32k":
        return dict(name=name, B=w["B"], Hq=w["Hq"], Hkv=w["Hkv"], T=w["T"], d=w["d"], k_bits=w["k_bits"],
                    k_variant=w["k_variant"], v_bits=w["v_bits"], v_variant=w["v_variant"], dist="t",
                    lens=(w["lo"], w["T"]))
    raise ValueError(name)


def make_inputs(spec: dict):
    """bf16 K, V [B, Hkv, T, d] (host tensors, except the heavy-tailed batched
    workload's, which are drawn on the device), q [B, Hq, d] and int32 lengths."""
    B, Hkv, T, d, Hq = spec["B"], spec["Hkv"], spec["T"], spec["d"], spec["Hq"]
    if spec["dist"] == "outliers":
        ch = synthetic.outlier_channels(d, 4, seed=4)
        K = synthetic.kv_with_outliers(B * Hkv, T, d, seed=0, channels=ch).reshape(B, Hkv, T, d)
        V = synthetic.kv_with_outliers(B * Hkv, T, d, seed=1, channels=ch).reshape(B, Hkv, T, d)
    elif spec["dist"] == "t":
        # 2 x 537 M heavy-tailed values: drawn on the device (a host draw takes minutes)
        K = synthetic.student_t_unit_var_cuda((B, Hkv, T, d), seed=0)
        V = synthetic.student_t_unit_var_cuda((B, Hkv, T, d), seed=1)
    else:
        K = synthetic.gaussian((B, Hkv, T, d), seed=0)
        V = synthetic.gaussian((B, Hkv, T, d), seed=1)
    q = synthetic.gaussian((B, Hq, d), seed=2)
    if spec["lens"] is None:
        lens = torch.full((B,), T, dtype=torch.int32)
    else:
        lens = synthetic.seq_lens_uniform(B, spec["lens"][0], spec["lens"][1], seed=3)
    return K, V, q, lens


def row_bytes(bits: int, variant: str, d: int) -> int:
    b_m = bits if variant == "mse" else bits - 1
    return b_m * d // 8 + 4 + ((d // 8 + 4) if variant == "prod" else 0)


def traffic_model(spec: dict, lens) -> dict:
    """Algorithmic bytes: what the packed format forces any implementation to move."""
    d, B, Hkv, T, Hq = spec["d"], spec["B"], spec["Hkv"], spec["T"], spec["Hq"]
    n_rows = B * Hkv * T
    krb, vrb = row_bytes(spec["k_bits"], spec["k_variant"], d), row_bytes(spec["v_bits"], spec["v_variant"], d)
    qk = n_rows * (2 * d + krb)
    qv = n_rows * (2 * d + vrb)
    ctx = int(sum(int(x) for x in lens)) * Hkv
    dec = ctx * (krb + vrb) + B * Hq * d * 2 + B * Hq * d * 4
    return dict(n_rows=n_rows, quant_k=qk, quant_v=qv, decode=dec, total=qk + qv + dec,
                krb=krb, vrb=vrb, ctx_rows=ctx)


# ----------------------------------------------------------------------------- clocks
REASONS = [(0x4, "sw_power_cap"), (0x8, "hw_slowdown"), (0x20, "sw_thermal_slowdown"),
           (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"), (0x2, "applications_clocks_setting"),
           (0x10, "sync_boost"), (0x100, "display_clock_setting")]


class ClockSampler:
    """Samples the SM clock and clock-event reasons while the timed loop runs:
    NVML through pynvml when importable, else `nvidia-smi -lms` in the background."""

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self.mem_samples = []
        self.period = period_s
        self.mode = None
        self.err = ""
        self.dev = device_index
        try:
            import pynvml as N
            N.nvmlInit()
            self.N = N
            self.h = self._handle(N, device_index)
            self.max_mhz = N.nvmlDeviceGetMaxClockInfo(self.h, N.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:  # pragma: no cover - depends on the box
            self.err = repr(e)
            self.mode = "smi"

    @staticmethod
    def _uuid(device_index):
        try:
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return None

    def _handle(self, N, device_index):
        u = self._uuid(device_index)
        if u is not None:
            try:
                return N.nvmlDeviceGetHandleByUUID(u)
            except Exception:
                pass
        return N.nvmlDeviceGetHandleByIndex(device_index)

    def _run_nvml(self):
        N = self.N
        fn = getattr(N, "nvmlDeviceGetCurrentClocksEventReasons", None) or N.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            try:
                self.samples.append(N.nvmlDeviceGetClockInfo(self.h, N.NVML_CLOCK_SM))
                self.mem_samples.append(N.nvmlDeviceGetClockInfo(self.h, N.NVML_CLOCK_MEM))
                self.reasons |= int(fn(self.h))
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        self._stop = threading.Event()
        if self.mode == "nvml":
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
            self._t.start()
        else:
            import subprocess
            sel = self._uuid(self.dev) or str(self.dev)
            try:
                self._p = subprocess.Popen(
                    ["nvidia-smi", "-i", sel, "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks.mem",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                time.sleep(0.3)  # let the first samples arrive before the loop starts
            except Exception as e:
                self._p = None
                self.err += " " + repr(e)
        return self

    def __exit__(self, *a):
        if self.mode == "nvml":
            self._stop.set()
            self._t.join()
        elif getattr(self, "_p", None) is not None:
            self._p.terminate()
            try:
                out, _ = self._p.communicate(timeout=5)
            except Exception:
                self._p.kill()
                out = ""
            for ln in out.splitlines():
                parts = [x.strip() for x in ln.split(",")]
                try:
                    self.samples.append(float(parts[0]))
                    self.max_mhz = float(parts[1])
                    self.reasons |= int(parts[2], 16)
                    self.mem_samples.append(float(parts[3]))
                except Exception:
                    continue

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": self.err or "no samples"}
        out = {"sm_mhz": float(statistics.median(self.samples)), "sm_max_mhz": float(self.max_mhz),
               "reasons": [n for bit, n in REASONS if self.reasons & bit], "samples": len(self.samples),
               "via": self.mode}
        if self.mem_samples:
            out["mem_mhz"] = float(statistics.median(self.mem_samples))
        return out


# ----------------------------------------------------------------------------- helpers
def keep_busy(fn, min_steps: int, seconds: float) -> int:
    """Run fn back to back for at least min_steps calls and `seconds` of wall time,
    synchronising only every few calls so that the device never idles."""
    t0 = time.perf_counter()
    n = 0
    while n < min_steps or time.perf_counter() - t0 < seconds:
        fn()
        n += 1
        if n % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return n



def load_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def source_hash(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key: str, src_hash: str, units_per_launch: int):
    """DRAM bytes per launch from the committed ncu summary (bytes per row or per
    token-head, scaled to this launch), if it was taken on this source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel_key]
    except Exception:
        return None
    if rec.get("source_hash") != src_hash:
        return None
    return rec["dram_bytes_per_unit"] * units_per_launch


def blas_threads() -> int:
    """Threads of NumPy's BLAS: threadpoolctl when importable, else the thread
    count the environment fixes, else one per host core (OpenBLAS's default)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        return int(max(n)) if n else 1
    except Exception:
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            if os.environ.get(var, "").isdigit():
                return int(os.environ[var])
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- oracle timing
def oracle_sample_run(spec, K, V, q, lens, rows: int, tokens: int, params):
    """The oracle as it stands on a bounded sample of the workload: quantize ``rows``
    K rows and V rows, then decode attention over the first ``tokens`` tokens of
    every (batch, KV head).  Returns the algorithmic bytes of the sample."""
    import oracle as O
    pk, pv = params
    d = spec["d"]
    Kr = K.reshape(-1, d)
    Vr = V.reshape(-1, d)
    O.quantize(pk, Kr[:rows].cpu().double().numpy())
    O.quantize(pv, Vr[:rows].cpu().double().numpy())
    B, Hkv, Hq = spec["B"], spec["Hkv"], spec["Hq"]
    Ks = K[:, :, :tokens].reshape(-1, d).cpu().double().numpy()
    Vs = V[:, :, :tokens].reshape(-1, d).cpu().double().numpy()
    kq = O.quantize(pk, Ks)
    vq = O.quantize(pv, Vs)
    sl = [min(int(x), tokens) for x in lens]
    O.decode_attention(pk, pv, q.double().numpy(), kq, vq, sl, Hkv, tokens)
    krb, vrb = row_bytes(spec["k_bits"], spec["k_variant"], d), row_bytes(spec["v_bits"], spec["v_variant"], d)
    qbytes = rows * (2 * d + krb) + rows * (2 * d + vrb)
    dbytes = sum(sl) * Hkv * (krb + vrb) + B * Hq * d * 6
    return qbytes + dbytes, 2 * rows


def oracle_params(spec):
    import oracle as O
    rot = spec.get("rotation", "qr")
    return (O.make_params(spec["d"], spec["k_bits"], spec["k_variant"], 10, rot),
            O.make_params(spec["d"], spec["v_bits"], spec["v_variant"], 11, rot))


def _oracle_rate(spec, K, V, q, lens, params, rows: int, tokens: int, seconds: float):
    oracle_sample_run(spec, K, V, q, lens, 256, 64, params)  # warm caches / BLAS threads
    t0 = time.perf_counter()
    nbytes = nrows = reps = 0
    while time.perf_counter() - t0 < seconds:
        b, r = oracle_sample_run(spec, K, V, q, lens, rows, tokens, params)
        nbytes += b
        nrows += r
        reps += 1
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, nrows / dt / 1e6, reps, dt


def cpu_baseline(spec, K, V, q, lens, seconds: float = 12.0, seconds_1core: float = 6.0) -> dict:
    """The oracle as it stands on this host's cores: all BLAS threads, then one."""
    params = oracle_params(spec)
    rows, tokens = 4096, 1024
    gbs, mrows, reps, dt = _oracle_rate(spec, K, V, q, lens, params, rows, tokens, seconds)
    out = {"value": gbs, "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
           "sample": f"{reps} x (quantize {rows} K + {rows} V rows, decode over the first {tokens} tokens of "
                     f"all {spec['B']}x{spec['Hkv']} KV heads, {spec['Hq']} query heads); "
                     f"{dt:.1f} s; float64 NumPy",
           "quantize_mrows_s": mrows, "host_cpu_count": os.cpu_count(), "blas_threads": blas_threads()}
    out["one_core"] = oracle_one_core(spec["name"], rows // 4, tokens // 4, seconds_1core)
    return out


def oracle_one_core(workload: str, rows: int, tokens: int, seconds: float) -> dict:
    """The same oracle sample on one core: a fresh interpreter whose BLAS and
    OpenMP pools are limited to one thread before NumPy loads (no GPU use)."""
    import subprocess
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench._one_core_child(%r, %d, %d, %f)))" % (ROOT, workload, rows, tokens, seconds))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as exc:  # pragma: no cover - depends on the host
        return {"note": f"unavailable ({type(exc).__name__})"}


def _one_core_child(workload: str, rows: int, tokens: int, seconds: float) -> dict:
    spec = workload_spec(workload)
    K, V, q, lens = make_inputs(spec) if spec["dist"] != "t" else (None, None, None, None)
    if K is None:
        return {"note": "device-drawn workload; one-core timing runs on the host workloads only"}
    gbs, mrows, reps, dt = _oracle_rate(spec, K, V, q, lens.tolist(), oracle_params(spec), rows, tokens, seconds)
    return {"value": gbs, "unit": "GB/s", "quantize_mrows_s": mrows, "cores": 1, "blas_threads": blas_threads(),
            "sample": f"{reps} x (quantize {rows} K + {rows} V rows, decode over the first {tokens} tokens of "
                      f"every KV head); {dt:.1f} s"}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, spec):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    K, V, q, lens = make_inputs(spec)
    params = oracle_params(spec)
    t0 = time.perf_counter()
    oracle_sample_run(spec, K, V, q, lens, 512, 128, params)
    per_unit = time.perf_counter() - t0
    budget = max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    scale = max(1.0, budget / max(per_unit, 1e-3))
    rows, tokens = int(512 * scale), int(128 * scale)
    rows = min(rows, spec["B"] * spec["Hkv"] * spec["T"])
    tokens = min(tokens, spec["T"])
    for _ in range(args.warmup):
        oracle_sample_run(spec, K, V, q, lens, rows, tokens, params)
    nbytes = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        b, _r = oracle_sample_run(spec, K, V, q, lens, rows, tokens, params)
        nbytes += b
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / max(args.steps, 1) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(spec),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": f"per step: quantize {rows} K + {rows} V rows, decode over the first "
                                       f"{tokens} tokens of every KV head; float64 NumPy"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


METRIC = "compressed-KV decode attention GB/s and quantize Mrows/s, % of B300 HBM peak"


def config_block(spec) -> dict:
    return {"workload": spec["name"], "batch": spec["B"], "kv_heads": spec["Hkv"], "q_heads": spec["Hq"],
            "tokens": spec["T"], "d": spec["d"], "k": f"{spec['k_variant']} b={spec['k_bits']}",
            "v": f"{spec['v_variant']} b={spec['v_bits']}", "rotation": spec.get("rotation", "qr"),
            "step": ("tq_quantize_kv(K, V) (one launch) + tq_decode_attention over the packed cache"
                     if kv_one_launch(spec) else
                     "tq_quantize(K) + tq_quantize(V) + tq_decode_attention over the packed cache"),
            "l2": f"flushed by a {L2_FLUSH_BYTES >> 20} MiB write before every timed step",
            "inputs": "resident in HBM (value); pinned host buffers (e2e)"}


# ----------------------------------------------------------------------------- our arm
def run_ours(args, spec):
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    import kv_cache_vector_18_b300 as tq

    K, V, q, lens = make_inputs(spec)
    d, B, Hq, Hkv, T = spec["d"], spec["B"], spec["Hq"], spec["Hkv"], spec["T"]
    tm = traffic_model(spec, lens.tolist())
    rot = spec.get("rotation", "qr")
    kq = tq.Quantizer(d, spec["k_bits"], spec["k_variant"], seed=10, rotation=rot)
    vq = tq.Quantizer(d, spec["v_bits"], spec["v_variant"], seed=11, rotation=rot)
    Kd, Vd, qd, ld = K.to(dev).reshape(-1, d), V.to(dev).reshape(-1, d), q.to(dev), lens.to(dev)
    kc, vc = kq.empty_planes(tm["n_rows"]), vq.empty_planes(tm["n_rows"])
    ws = torch.empty(tq.decode_workspace_bytes(kq, vq, B, Hq, Hkv, T), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    fused = kv_one_launch(spec)
    dec_call = lambda: tq.decode_attention(kq, vq, qd, kc, vc, ld, Hkv, T, workspace=ws, out=out)
    if fused:  # K and V quantized by one library call and one launch
        names = ["quantize_kv", "decode"]
        calls = [lambda: tq.quantize_kv(kq, vq, Kd, Vd, k_out=kc, v_out=vc), dec_call]
    else:
        names = ["quantize_k", "quantize_v", "decode"]
        calls = [lambda: kq.quantize(Kd, out=kc), lambda: vq.quantize(Vd, out=vc), dec_call]
    for _ in range(max(args.warmup, 0)):
        flush.zero_()
        for fn in calls:
            fn()
    torch.cuda.synchronize()
    # Host cost of one direct library call (argument checks, tensor-map encoding,
    # launch), for the record: it is why the device timing below replays graphs.
    host_us = []
    for fn in calls:
        t = time.perf_counter()
        for _ in range(20):
            fn()
        host_us.append((time.perf_counter() - t) / 20 * 1e6)
        torch.cuda.synchronize()
    # The same calls straight through the C ABI with their arguments marshalled
    # once (what a C or C++ caller pays per call: checks, tensor-map encoding, launch).
    from kv_cache_vector_18_b300 import _lib as _L
    Lb, strm = _L.lib(), torch.cuda.current_stream().cuda_stream
    kps, vps = tq.Quantizer.planes_struct(kc), tq.Quantizer.planes_struct(vc)
    abi_dec = lambda: Lb.tq_decode_attention(kq.handle, vq.handle, qd.data_ptr(), _L.TQ_BF16, kps, vps,
                                             ld.data_ptr(), B, Hq, Hkv, T, 0.0, out.data_ptr(), None, ws.data_ptr(),
                                             ws.numel(), strm)
    if fused:
        abi = [lambda: Lb.tq_quantize_kv(kq.handle, vq.handle, Kd.data_ptr(), Vd.data_ptr(), _L.TQ_BF16, tm["n_rows"],
                                         tm["n_rows"], d, d, kps, vps, strm), abi_dec]
    else:
        abi = [lambda: Lb.tq_quantize(kq.handle, Kd.data_ptr(), _L.TQ_BF16, tm["n_rows"], d, kps, strm),
               lambda: Lb.tq_quantize(vq.handle, Vd.data_ptr(), _L.TQ_BF16, tm["n_rows"], d, vps, strm), abi_dec]
    abi_us = []
    for fn in abi:
        t = time.perf_counter()
        for _ in range(20):
            assert fn() == 0
        abi_us.append((time.perf_counter() - t) / 20 * 1e6)
        torch.cuda.synchronize()
    # One CUDA graph per step holding the library calls back to back (as a
    # serving loop replays them), captured from the same public API: the replay
    # issues exactly the library's kernels with no host work in between, and
    # events around each replay give the step time.  Each call's kernels may
    # start their prologues while the previous call's kernel finishes
    # (programmatic dependent launch), which an event node between the calls
    # would stop; so the per-call device times come from a second graph of the
    # same calls with event record nodes between them, replayed K times right
    # after the timed loop.  If event nodes cannot be captured, one graph per
    # call with events between the replays serves both.
    cap_ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(calls) + 1)]
    step_graph, inst_graph, graphs, graph_note = None, None, [], ""
    try:
        sg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(sg):
            for fn in calls:
                fn()
        ig = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ig):
            cap_ev[0].record()
            for i, fn in enumerate(calls):
                fn()
                cap_ev[i + 1].record()
        sg.replay()
        ig.replay()
        torch.cuda.synchronize()
        _ = cap_ev[0].elapsed_time(cap_ev[-1])
        step_graph, inst_graph = sg, ig
    except Exception as exc:  # fall back to one graph per call
        graph_note = f"step graph unavailable ({type(exc).__name__}); "
        torch.cuda.synchronize()
        for fn in calls:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            graphs.append(g)

    def replay_all():
        if step_graph is not None:
            step_graph.replay()
        else:
            for g in graphs:
                g.replay()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(args.steps)]
    per_call = []
    sampler = ClockSampler(local)
    with sampler:
        # The SM clock idles far below its maximum and takes a sustained load to
        # ramp up; keep the device busy for at least WARM_SECONDS (and W steps)
        # right up to the timed loop so that no idle gap precedes it.
        warm_steps = keep_busy(lambda: (flush.zero_(), replay_all()), args.warmup, args.warm_seconds)
        barrier(world)
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            ev = evs[i]
            if step_graph is not None:
                ev[0].record()
                step_graph.replay()
                ev[-1].record()
            else:
                ev[0].record()
                for k, g in enumerate(graphs):
                    g.replay()
                    ev[k + 1].record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        if inst_graph is not None:  # per-call device times
            for i in range(args.steps):
                flush.zero_()
                inst_graph.replay()
                torch.cuda.synchronize()  # the in-graph events are read before the next replay
                per_call.append([cap_ev[k].elapsed_time(cap_ev[k + 1]) for k in range(len(calls))])
    barrier(world)
    if step_graph is None:
        per_call = [[e[k].elapsed_time(e[k + 1]) for k in range(len(calls))] for e in evs]
    col = {n: [c[k] for c in per_call] for k, n in enumerate(names)}
    dc = col["decode"]
    step_ms = [e[0].elapsed_time(e[-1]) for e in evs]
    t_local = sum(step_ms) / 1e3
    t_step = max_over_ranks(t_local, world, dev)
    value = aggregate_throughput(tm["total"] * args.steps, t_local, world, dev) / 1e9
    quant_s = sum(sum(v) for n, v in col.items() if n != "decode") / 1e3
    quant_mrows = aggregate_throughput(2 * tm["n_rows"] * args.steps, quant_s, world, dev) / 1e6
    dec_gbs = aggregate_throughput(tm["decode"] * args.steps, sum(dc) / 1e3, world, dev) / 1e9

    peaks = load_peaks()
    # one roofline object per library call (K quantize, V quantize, decode), each
    # against the measured HBM copy bandwidth; the dominant one (longest launch)
    # is the line's "roofline"
    qsrc, dsrc = source_hash(QUANT_SOURCES), source_hash(DECODE_SOURCES)

    def hbm_roofline(kernel, ms_list, nbytes, traffic_key, src, units):
        ms = statistics.mean(ms_list)
        achieved = nbytes / (ms / 1e3) / 1e9
        return {"kernel": kernel, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": recorded_traffic(traffic_key, src, units),
                "peak_source": peaks["source"], "bytes_per_launch": nbytes, "launch_ms": ms, "source_hash": src}

    def tensor_info(spec_bits, variant, rows, ms_list):
        """Tensor-pipe view of a quantize call: algorithmic flops (2d² per row for
        the rotation, or d·log2(d) butterfly additions for the Hadamard one, plus
        2d² for the QJL sketch) and the flops the kernel executes (bf16 hi/lo passes
        for Π, one ±1 pass for the Hadamard matrix, 3 f16 passes for the sketch)."""
        ms = statistics.mean(ms_list)
        had = rot == "hadamard"
        alg = ((d * int(math.log2(d))) if had else 2 * d * d) * rows + (2 * d * d * rows if variant == "prod" else 0)
        exe = ((1 if had else 2) + (3 if variant == "prod" else 0)) * 2 * d * d * rows
        peak = peaks.get("bf16_tflops")
        out = {"algorithmic_tflops": alg / (ms / 1e3) / 1e12, "executed_tflops": exe / (ms / 1e3) / 1e12,
               "peak_tflops": peak}
        if peak:
            out["frac_algorithmic"] = out["algorithmic_tflops"] / peak
            out["frac_executed"] = out["executed_tflops"] / peak
        _sustained(out, peaks)
        return out

    wht = "_wht" if rot == "hadamard" else ""
    rl = {}
    if fused:
        rl["quantize_kv"] = hbm_roofline(
            f"tq_quantize_kv (mse b={spec['k_bits']}, K and V rows in one launch)", col["quantize_kv"],
            tm["quant_k"] + tm["quant_v"], f"quantize_mse_b{spec['k_bits']}_d{d}{wht}", qsrc, 2 * tm["n_rows"])
        rl["quantize_kv"]["tensor"] = tensor_info(spec["k_bits"], "mse", 2 * tm["n_rows"], col["quantize_kv"])
    else:
        rl["quantize_k"] = hbm_roofline(f"tq_quantize ({spec['k_variant']} b={spec['k_bits']})", col["quantize_k"],
                                        tm["quant_k"], f"quantize_{spec['k_variant']}_b{spec['k_bits']}_d{d}{wht}",
                                        qsrc, tm["n_rows"])
        rl["quantize_v"] = hbm_roofline(f"tq_quantize ({spec['v_variant']} b={spec['v_bits']})", col["quantize_v"],
                                        tm["quant_v"], f"quantize_{spec['v_variant']}_b{spec['v_bits']}_d{d}{wht}",
                                        qsrc, tm["n_rows"])
        rl["quantize_k"]["tensor"] = tensor_info(spec["k_bits"], spec["k_variant"], tm["n_rows"], col["quantize_k"])
        rl["quantize_v"]["tensor"] = tensor_info(spec["v_bits"], spec["v_variant"], tm["n_rows"], col["quantize_v"])
    for k in rl:  # the binding roofline of each quantize call (HBM or executed tensor flops)
        rl[k]["binding"] = "tensor" if rl[k]["tensor"].get("frac_executed_sustained", 0) > rl[k]["frac"] else "hbm"
    rl["decode"] = hbm_roofline("tq_decode_attention", dc, tm["decode"],
                                f"decode_{spec['k_variant']}_b{spec['k_bits']}_{spec['v_variant']}_b{spec['v_bits']}_d{d}",
                                dsrc, tm["ctx_rows"])
    # score, QJL and value products: 2·d flop each per token-head and query head
    dec_flops = (3 if spec["k_variant"] == "prod" else 2) * 2 * d * (Hq // Hkv) * tm["ctx_rows"]
    rl["decode"]["mma_tflops"] = dec_flops / (statistics.mean(dc) / 1e3) / 1e12
    # dominant kernel: calls of the same kernel (K and V quantize with one
    # configuration) are one kernel; the largest total device time wins
    groups = {}
    for k, v in rl.items():
        groups.setdefault(v["kernel"], []).append(k)
    dom = max(groups, key=lambda kern: sum(rl[k]["launch_ms"] for k in groups[kern]))
    dcalls = groups[dom]
    if len(dcalls) == 1:
        roofline = dict(rl[dcalls[0]], call=dcalls[0])
    else:
        nbytes = sum(rl[k]["bytes_per_launch"] for k in dcalls) / len(dcalls)
        ms = sum(rl[k]["launch_ms"] for k in dcalls) / len(dcalls)
        achieved = nbytes / (ms / 1e3) / 1e9
        roofline = dict(rl[dcalls[0]], call="+".join(dcalls), achieved=achieved, frac=achieved / peaks["hbm_gbs"],
                        bytes_per_launch=nbytes, launch_ms=ms)
    roofline_decode = rl["decode"]

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, spec, tq, kq, vq, K, V, q, ld, kc, vc, ws, out, tm, dev, world)
    append = measure_append(tq, kq, vq, qd, kc, vc, ld, spec, ws, out, flush, dev)

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_step / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_LABEL,
            "data": "synthetic (seeded NumPy draws, bf16)", "config": config_block(spec),
            "quantize_mrows_s": quant_mrows, "decode_gbs": dec_gbs,
            "pct_hbm_peak": value / peaks["hbm_gbs"] * 100.0,
            "pct_nominal_8tbs": value / 8000.0 * 100.0,
            "bytes_per_step": tm["total"],
            "gpu_launches": args.steps * ((1 if fused else 2) * LAUNCHES["quantize"] + LAUNCHES["decode"]),
            "clocks": sampler.summary(), "wall_s_timed_loop": wall, "roofline": roofline,
            "roofline_decode": roofline_decode, "roofline_per_call": rl, "e2e": e2e, "append_step": append,
            "timing": graph_note + (f"one CUDA graph per step holding the {len(calls)} library calls (captured through "
                                    "the public API); step time from CUDA events around each replay; per-call "
                                    "times from event nodes between the calls of a second graph of the same calls, "
                                    "replayed K times after the timed loop (the event nodes stop the calls' "
                                    "programmatic overlap)" if step_graph is not None else
                                    "CUDA events around CUDA-graph replays of each library call (one graph per call)")
                      + "; L2 flushed before every step; after >= %.1f s of back-to-back warm-up (%d steps)"
                      % (args.warm_seconds, warm_steps),
            "host_us_per_direct_call": dict(zip(names, host_us), via="Python binding"),
            "host_us_per_abi_call": dict(zip(names, abi_us), via="C ABI through ctypes, arguments marshalled once")}
    if not args.no_configs and spec["name"] == "llama70b_layer_kv_quant" and spec.get("rotation", "qr") == "qr":
        line["configs"] = measure_configs(tq, flush, dev, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, K, V, q, lens.tolist())
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def time_call(fn, flush, reps: int = 20, warm: int = 3) -> float:
    """Mean device time (ms) of one library call: captured once as a CUDA graph
    through the public API, replayed `reps` times with L2 flushed (a 256 MiB
    write) before each replay, CUDA events on the launching stream around each."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(warm):
        flush.zero_()
        g.replay()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record()
        g.replay()
        e1.record()
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)


def _sustained(t: dict, peaks: dict) -> None:
    """Add the executed flops against the sustained bf16 peak (a kernel timed inside
    a long step runs at the power-capped clock)."""
    ps = peaks.get("bf16_tflops_sustained")
    if ps and t.get("executed_tflops") is not None:
        t["peak_tflops_sustained"] = ps
        t["frac_executed_sustained"] = t["executed_tflops"] / ps


def _rl(kernel, ms, nbytes, peaks, flops=None, exe_flops=None) -> dict:
    """Roofline object of one call: algorithmic bytes (and flops) per launch over
    its mean device time, against the measured HBM copy (and bf16) peaks."""
    gbs = nbytes / (ms / 1e3) / 1e9
    out = {"kernel": kernel, "bound": "hbm", "launch_ms": ms, "bytes_per_launch": nbytes, "achieved": gbs,
           "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "peak_source": peaks["source"]}
    if flops is not None:
        tf = flops / (ms / 1e3) / 1e12
        out["tensor"] = {"algorithmic_tflops": tf, "peak_tflops": peaks.get("bf16_tflops"),
                         "frac_algorithmic": tf / peaks["bf16_tflops"] if peaks.get("bf16_tflops") else None}
        if exe_flops is not None:
            te = exe_flops / (ms / 1e3) / 1e12
            out["tensor"]["executed_tflops"] = te
            out["tensor"]["frac_executed"] = te / peaks["bf16_tflops"] if peaks.get("bf16_tflops") else None
            _sustained(out["tensor"], peaks)
            # the binding roofline: the larger of the HBM fraction and the executed-flops fraction
            out["binding"] = "tensor" if out["tensor"].get("frac_executed_sustained", 0) > out["frac"] else "hbm"
    return out


def _quant_flops(d: int, variant: str, rows: int, rotation: str = "qr"):
    """Algorithmic flops of a quantize call (2d² per row for the rotation, 2d² more
    for the prod sketch) and the flops the tensor-core kernels execute (bf16
    hi/lo passes for Π, or one ±1 pass for the Hadamard matrix, and 3 f16 passes
    for the sketch)."""
    alg = 2 * d * d * rows * (2 if variant == "prod" else 1)
    exe = ((1 if rotation == "hadamard" else 2) + (3 if variant == "prod" else 0)) * 2 * d * d * rows
    return alg, exe


def measure_configs(tq, flush, dev, peaks, reps: int = 20) -> dict:
    """Device time and roofline of every library call of the other workloads the
    metric is quoted on (each call alone, as a CUDA graph, L2 flushed before each
    replay): the 4096-row fp32 case, the 131072-token decode, the batched decode,
    and quantize throughput at every point of the bit-width / head-dim sweep."""
    res = {}
    # 4096 x 128 fp32 rows, mse b = 2: quantize, dequantize, 64 queries scored against all keys
    w = synthetic.WORKLOADS["small_mse_b2"]
    n, d, nq = w["rows"], w["d"], w["queries"]
    X = synthetic.gaussian((n, d), seed=0, dtype="f32").to(dev)
    qz = tq.Quantizer(d, w["bits"], w["variant"], seed=0)
    pl = qz.quantize(X)
    y = torch.empty((n, d), dtype=torch.float32, device=dev)
    q = synthetic.gaussian((1, nq, d), seed=1, dtype="f32").to(dev)
    sl = torch.tensor([n], dtype=torch.int32, device=dev)
    ws = torch.empty(tq.decode_workspace_bytes(qz, qz, 1, nq, 1, n), dtype=torch.uint8, device=dev)
    o = torch.empty((1, nq, d), dtype=torch.float32, device=dev)
    rb = row_bytes(w["bits"], w["variant"], d)

    def dq():
        from kv_cache_vector_18_b300 import _lib
        _lib.check(_lib.lib().tq_dequantize(qz.handle, tq.Quantizer.planes_struct(pl), n, y.data_ptr(),
                                            _lib.TQ_F32, torch.cuda.current_stream().cuda_stream))
    sc = torch.empty((1, nq, n), dtype=torch.float32, device=dev)

    def sc_call():
        from kv_cache_vector_18_b300 import _lib
        _lib.check(_lib.lib().tq_decode_attention(
            qz.handle, qz.handle, q.data_ptr(), _lib.TQ_F32, tq.Quantizer.planes_struct(pl),
            tq.Quantizer.planes_struct(pl), sl.data_ptr(), 1, nq, 1, n, 0.0, o.data_ptr(), sc.data_ptr(),
            ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream))
    a, e = _quant_flops(d, w["variant"], n)
    res["small_mse_b2"] = {
        "quantize": _rl("tq_quantize (fp32 rows, mse b=2)", time_call(lambda: qz.quantize(X, out=pl), flush, reps),
                        n * (4 * d + rb), peaks, a, e),
        "dequantize": _rl("tq_dequantize (fp32 out)", time_call(dq, flush, reps), n * (rb + 4 * d), peaks),
        "decode_scores": _rl("tq_decode_attention (64 queries x 4096 keys, scores out)",
                             time_call(sc_call, flush, reps), 2 * n * rb + nq * d * 8 + nq * n * 4, peaks)}
    del X, pl, y, ws
    # the two decode workloads: both quantize calls and the decode
    for name in ("decode_131k", "batched_decode_32k"):
        spec = workload_spec(name)
        K, V, qh, lens = make_inputs(spec)
        d, B, Hq, Hkv, T = spec["d"], spec["B"], spec["Hq"], spec["Hkv"], spec["T"]
        tm = traffic_model(spec, lens.tolist())
        kq = tq.Quantizer(d, spec["k_bits"], spec["k_variant"], seed=10)
        vq = tq.Quantizer(d, spec["v_bits"], spec["v_variant"], seed=11)
        Kd, Vd, qd, ld = K.to(dev).reshape(-1, d), V.to(dev).reshape(-1, d), qh.to(dev), lens.to(dev)
        del K, V
        kc, vc = kq.empty_planes(tm["n_rows"]), vq.empty_planes(tm["n_rows"])
        ws = torch.empty(tq.decode_workspace_bytes(kq, vq, B, Hq, Hkv, T), dtype=torch.uint8, device=dev)
        o = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
        ka, ke = _quant_flops(d, spec["k_variant"], tm["n_rows"])
        va, ve = _quant_flops(d, spec["v_variant"], tm["n_rows"])
        entry = {
            "quantize_k": _rl(f"tq_quantize ({spec['k_variant']} b={spec['k_bits']})",
                              time_call(lambda: kq.quantize(Kd, out=kc), flush, reps), tm["quant_k"], peaks, ka, ke),
            "quantize_v": _rl(f"tq_quantize ({spec['v_variant']} b={spec['v_bits']})",
                              time_call(lambda: vq.quantize(Vd, out=vc), flush, reps), tm["quant_v"], peaks, va, ve)}
        dms = time_call(lambda: tq.decode_attention(kq, vq, qd, kc, vc, ld, Hkv, T, workspace=ws, out=o), flush, reps)
        entry["decode"] = _rl("tq_decode_attention", dms, tm["decode"], peaks)
        fl = (3 if spec["k_variant"] == "prod" else 2) * 2 * d * (Hq // Hkv) * tm["ctx_rows"]
        entry["decode"]["mma_tflops"] = fl / (dms / 1e3) / 1e12
        entry["decode"]["token_heads"] = tm["ctx_rows"]
        res[name] = entry
        del Kd, Vd, kc, vc, ws
        torch.cuda.empty_cache()
    # bit-width / head-dim sweep: quantize throughput of 2^20 bf16 N(0,1) rows per point
    sw = synthetic.WORKLOADS["sweep"]
    n = sw["rows"]
    pts = []
    for dd in sw["d"]:
        for variant in sw["variants"]:
            for bits in sw["bits"]:
                seed = 100 * dd + 10 * bits + (variant == "prod")
                X = synthetic.gaussian_cuda((n, dd), seed=seed)
                qz = tq.Quantizer(dd, bits, variant, seed=seed)
                pl = qz.empty_planes(n)
                ms = time_call(lambda: qz.quantize(X, out=pl), flush, max(5, reps // 2))
                a, e = _quant_flops(dd, variant, n)
                r = _rl(f"tq_quantize ({variant} b={bits}, d={dd})", ms, n * (2 * dd + row_bytes(bits, variant, dd)),
                        peaks, a, e)
                r.update({"d": dd, "variant": variant, "bits": bits, "mrows_s": n / (ms / 1e3) / 1e6})
                pts.append(r)
                del X, pl, qz
    res["sweep"] = pts
    torch.cuda.empty_cache()
    return res


def measure_append(tq, kq, vq, qd, kc, vc, ld, spec, ws, out, flush, dev, reps: int = 200) -> dict:
    """Device time of one decode step with append (tq_decode_append_attention):
    the new K and V rows of every slab are quantized into token seq_len − 1, the
    lengths bumped back to len, and attention runs over the same tokens as the
    plain decode call.  The lengths are reset to len − 1 before each replay,
    outside the timed region, next to the L2 flush.  The plain decode over the
    same tokens is replayed alternately with it under the same conditions (the
    clock differs between the timed loop and this one), so the overhead is their
    difference.  Runs after the timed loop; it overwrites one cached token per
    slab."""
    B, Hkv, d, T = spec["B"], spec["Hkv"], spec["d"], spec["T"]
    kn = synthetic.gaussian_cuda((B, Hkv, d), seed=20)
    vn = synthetic.gaussian_cuda((B, Hkv, d), seed=21)
    la0 = (ld - 1).clamp_min(0).to(torch.int32)
    la = la0.clone()

    def body():
        tq.decode_append_attention(kq, vq, qd, kn, vn, kc, vc, la, Hkv, T, workspace=ws, out=out)

    body()
    torch.cuda.synchronize()
    la.copy_(la0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    gp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gp):
        tq.decode_attention(kq, vq, qd, kc, vc, ld, Hkv, T, workspace=ws, out=out)
    for _ in range(5):
        la.copy_(la0)
        g.replay()
        gp.replay()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    evs = [(ev(), ev(), ev(), ev()) for _ in range(reps)]
    for e0, e1, e2, e3 in evs:
        flush.zero_()
        la.copy_(la0)
        e0.record()
        g.replay()
        e1.record()
        flush.zero_()
        e2.record()
        gp.replay()
        e3.record()
    torch.cuda.synchronize()
    us = [e0.elapsed_time(e1) * 1e3 for e0, e1, _, _ in evs]
    plain = [e2.elapsed_time(e3) * 1e3 for _, _, e2, e3 in evs]
    return {"us": statistics.mean(us), "decode_us": statistics.mean(plain),
            "append_overhead_us": statistics.mean(us) - statistics.mean(plain), "reps": reps,
            "library_launches": 1 + LAUNCHES["append_decode"],
            "what": "append of K and V (whose last block bumps the lengths and clears the decode's tickets) + "
                    "decode launched as its programmatic dependent, one graph; lengths reset and L2 flushed "
                    "before each replay, outside the timed region; decode_us: the plain decode over the same "
                    "tokens, replayed alternately under the same conditions"}


def score_quality(tq, d: int, bits: int, variant: str, tau: float, B: int = 4, Hq: int = 64, Hkv: int = 8,
                  T: int = 4096, seed: int = 0) -> dict:
    """Attention quality of one key quantizer against exact attention (mse-only
    versus prod keys at the same bits per coordinate).  Keys, values and queries
    are N(0, 1) bf16; the softmax scale τ/√d sets how peaked attention is (logit
    standard deviation ≈ τ).  Scores come from tq_decode_attention (scores_out);
    exact scores, softmax and outputs from the same bf16 rows in fp32."""
    dev = torch.device("cuda")
    K = synthetic.gaussian_cuda((B, Hkv, T, d), seed=seed + 1)
    V = synthetic.gaussian_cuda((B, Hkv, T, d), seed=seed + 2)
    q = synthetic.gaussian_cuda((B, Hq, d), seed=seed + 3)
    kq = tq.Quantizer(d, bits, variant, seed=seed + 11)
    vq = tq.Quantizer(d, 4, "mse", seed=seed + 12)  # values only feed the unused output
    kc = kq.quantize(K.reshape(-1, d))
    vc = vq.quantize(V.reshape(-1, d))
    lens = torch.full((B,), T, dtype=torch.int32, device=dev)
    scale = tau / math.sqrt(d)
    _, sq = tq.decode_attention(kq, vq, q, kc, vc, lens, Hkv, T, scale=scale, return_scores=True)
    G = Hq // Hkv
    Kf = K.float().repeat_interleave(G, dim=1)                # [B, Hq, T, d]
    s = scale * torch.einsum("bhtd,bhd->bht", Kf, q.float())  # exact scores
    p, pq = torch.softmax(s, -1), torch.softmax(sq, -1)
    Vf = V.float().repeat_interleave(G, dim=1)
    o, oq = torch.einsum("bht,bhtd->bhd", p, Vf), torch.einsum("bht,bhtd->bhd", pq, Vf)
    top1 = (s.argmax(-1) == sq.argmax(-1)).double().mean().item()
    t5, t5q = s.topk(5, -1).indices, sq.topk(5, -1).indices
    rec5 = (t5.unsqueeze(-1) == t5q.unsqueeze(-2)).any(-1).double().mean().item()
    kl = (p * (torch.log(p.clamp_min(1e-30)) - torch.log(pq.clamp_min(1e-30)))).sum(-1).mean().item()
    out_rel = ((oq - o).norm() / o.norm()).item()
    sd, sqd = s.double(), sq.double()
    slope = ((sqd * sd).sum() / (sd * sd).sum()).item()
    noise = ((sqd - slope * sd).std() / sd.std()).item()
    return {"d": d, "bits": bits, "keys": variant, "tau": tau, "queries": B * Hq, "tokens": T,
            "top1": top1, "top5_recall": rec5, "kl": kl, "out_rel_l2": out_rel, "score_slope": slope,
            "score_noise": noise}


def run_mixed(args) -> int:
    """Outlier-channel mixed precision on the Llama-3.1-70B layer: the 32 channels
    of largest energy at 3 bits and the other 96 at 2 (mse, K and V), chosen by
    tq_select_outlier_channels from the rows themselves.  Device time per call
    (CUDA graph per call, L2 flushed before each replay), algorithmic bytes ÷ time,
    and the distortion against uniform 2- and 3-bit quantizers on the same rows."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import kv_cache_vector_18_b300 as tq
    spec = workload_spec("llama70b_layer_kv_quant")
    K, V, q, lens = make_inputs(spec)
    d, B, Hq, Hkv, T = spec["d"], spec["B"], spec["Hq"], spec["Hkv"], spec["T"]
    d_o, bo, bn = 32, 3, 2
    Kd, Vd, qd, ld = K.to(dev).reshape(-1, d), V.to(dev).reshape(-1, d), q.to(dev), lens.to(dev)
    n = Kd.shape[0]
    pk, _ = tq.select_outlier_channels(Kd, d_o)
    pv, _ = tq.select_outlier_channels(Vd, d_o)
    mk = tq.MixedQuantizer(pk, d_o, bo, bn, "mse", seed_o=10, seed_n=12)
    mv = tq.MixedQuantizer(pv, d_o, bo, bn, "mse", seed_o=11, seed_n=13)
    kc, vc = mk.empty_planes(n), mv.empty_planes(n)
    ws = torch.empty(tq.mixed_decode_workspace_bytes(mk, mv, B, Hq, Hkv, T), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    def step():
        tq.mixed_quantize_kv(mk, mv, Kd, Vd, kc, vc)
        tq.mixed_decode_attention(mk, mv, qd, kc, vc, ld, Hkv, T, workspace=ws, out=out)
    # the same split with prod key parts (codes of one bit fewer + QJL signs per part)
    mkp = tq.MixedQuantizer(pk, d_o, bo, bn, "prod", seed_o=10, seed_n=12)
    kcp = mkp.quantize(Kd)
    wsp = torch.empty(tq.mixed_decode_workspace_bytes(mkp, mv, B, Hq, Hkv, T), dtype=torch.uint8, device=dev)
    calls = {"quantize_k": lambda: mk.quantize(Kd, out=kc), "quantize_v": lambda: mv.quantize(Vd, out=vc),
             "quantize_kv": lambda: tq.mixed_quantize_kv(mk, mv, Kd, Vd, kc, vc),
             "decode": lambda: tq.mixed_decode_attention(mk, mv, qd, kc, vc, ld, Hkv, T, workspace=ws, out=out),
             "step": step,
             "decode_prod_keys": lambda: tq.mixed_decode_attention(mkp, mv, qd, kcp, vc, ld, Hkv, T, workspace=wsp,
                                                                   out=out)}
    for fn in calls.values():
        fn()
    torch.cuda.synchronize()
    rec = (bo * d_o // 8 + 4) + (bn * (d - d_o) // 8 + 4)  # record bytes of both parts
    nbytes = {"quantize_k": n * (2 * d + rec), "quantize_v": n * (2 * d + rec),
              "quantize_kv": 2 * n * (2 * d + rec), "decode": int(lens.sum()) * Hkv * 2 * rec + B * Hq * d * 6}
    nbytes["step"] = nbytes["quantize_kv"] + nbytes["decode"]
    # prod key parts: codes of one bit fewer plus 32 + 96 sign bits and two residual norms
    rec_kp = ((bo - 1) * d_o // 8 + 4 + d_o // 8 + 4) + ((bn - 1) * (d - d_o) // 8 + 4 + (d - d_o) // 8 + 4)
    nbytes["decode_prod_keys"] = int(lens.sum()) * Hkv * (rec_kp + rec) + B * Hq * d * 6
    peaks = load_peaks()
    res = {}
    for name, fn in calls.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        for _ in range(max(args.warmup, 3)):
            flush.zero_()
            g.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
        for e0, e1 in evs:
            flush.zero_()
            e0.record()
            g.replay()
            e1.record()
        torch.cuda.synchronize()
        ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
        gbs = nbytes[name] / (ms / 1e3) / 1e9
        res[name] = {"us": ms * 1e3, "bytes": nbytes[name], "gbs": gbs, "frac": gbs / peaks["hbm_gbs"]}
    # distortion E‖x − x̃‖²/‖x‖² on the first 65536 K rows: mixed against uniform
    m = 1 << 16
    xs = Kd[:m]
    def dist(y):
        xf = xs.float()
        return float((((xf - y.float()) ** 2).sum(1) / (xf ** 2).sum(1)).double().mean())
    dm = dist(mk.dequantize(mk.quantize(xs)))
    u2, u3 = tq.Quantizer(d, 2, "mse", seed=10), tq.Quantizer(d, 3, "mse", seed=10)
    d2, d3 = dist(u2.dequantize(u2.quantize(xs))), dist(u3.dequantize(u3.quantize(xs)))
    print(json.dumps({"mixed": "outlier channels 32 x 3 bits + 96 x 2 bits, mse, K and V (decode_prod_keys: prod "
                               "key parts of the same bits)",
                      "workload": spec["name"], "code_bits_per_channel": (d_o * bo + (d - d_o) * bn) / d,
                      "record_bytes": rec, "calls": res, "peak_gbs": peaks["hbm_gbs"],
                      "distortion": {"mixed": dm, "uniform_b2": d2, "uniform_b3": d3},
                      "timing": "CUDA graph per call, events around 50 replays, L2 flushed before each"}), flush=True)
    return 0


def run_score_quality_study(args) -> int:
    torch.cuda.set_device(0)
    import kv_cache_vector_18_b300 as tq
    rows = []
    for d in (64, 128):
        for bits in (2, 3, 4):
            for variant in ("mse", "prod"):
                for tau in (1.0, 4.0, 8.0):
                    rows.append(score_quality(tq, d, bits, variant, tau, seed=100 * d + bits))
    print(json.dumps({"study": "score-quality", "data": "synthetic N(0,1) bf16 keys, values and queries",
                      "rows": rows}), flush=True)
    return 0


def measure_e2e(args, spec, tq, kq, vq, K, V, q, ld, kc, vc, ws, out, tm, dev, world):
    """Same metric through the public API with host buffers: pinned H2D of the
    step's K, V and q, the step's library calls, D2H of the packed planes and
    the attention output, all inside the timed region.  Steps are pipelined as a
    serving loop would run them: step i + 1's inputs are copied on a second
    stream into the other of two device buffers while step i's kernels and its
    device-to-host copies run (the two directions of the host link overlap)."""
    d, Hkv, T = spec["d"], spec["Hkv"], spec["T"]
    Kh, Vh, qh = K.reshape(-1, d).cpu().pin_memory(), V.reshape(-1, d).cpu().pin_memory(), q.pin_memory()
    Kd = [torch.empty_like(Kh, device=dev) for _ in range(2)]
    Vd = [torch.empty_like(Vh, device=dev) for _ in range(2)]
    qd = [torch.empty_like(qh, device=dev) for _ in range(2)]
    host_planes = [{k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in p.items()} for p in (kc, vc)]
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = Kh.numel() * Kh.element_size() + Vh.numel() * Vh.element_size() + qh.numel() * qh.element_size()
    d2h = sum(v.numel() * v.element_size() for p in (kc, vc) for v in p.values()) + out.numel() * 4
    main = torch.cuda.current_stream(dev)
    cs = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]  # buffer b holds its step's inputs
    free = [torch.cuda.Event() for _ in range(2)]   # the kernels reading buffer b are done

    def copy_in(i):
        b = i % 2
        cs.wait_event(free[b])
        with torch.cuda.stream(cs):
            Kd[b].copy_(Kh, non_blocking=True)
            Vd[b].copy_(Vh, non_blocking=True)
            qd[b].copy_(qh, non_blocking=True)
        ready[b].record(cs)

    def compute(i):
        b = i % 2
        main.wait_event(ready[b])
        if kv_one_launch(spec):
            tq.quantize_kv(kq, vq, Kd[b], Vd[b], k_out=kc, v_out=vc)
        else:
            kq.quantize(Kd[b], out=kc)
            vq.quantize(Vd[b], out=vc)
        tq.decode_attention(kq, vq, qd[b], kc, vc, ld, Hkv, T, workspace=ws, out=out)
        free[b].record(main)
        for hp, p in zip(host_planes, (kc, vc)):
            for k in p:
                hp[k].copy_(p[k], non_blocking=True)
        out_h.copy_(out, non_blocking=True)

    def run(n, start=None):
        for e in free:
            e.record(main)
        if start is not None:
            start.record(main)
        cs.wait_stream(main)
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)

    n = max(3, min(args.steps, 50))
    run(3)
    torch.cuda.synchronize()
    keep_busy(lambda: run(2), 1, args.warm_seconds)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    run(n, start=e0)
    e1.record(main)
    torch.cuda.synchronize()
    secs = e0.elapsed_time(e1) / 1e3
    value = aggregate_throughput(tm["total"] * n, secs, world, dev) / 1e9
    return {"value": value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "ms_per_step": secs / n * 1e3,
            "pipelining": "step i+1's H2D on a second stream (double-buffered inputs) overlaps step i's kernels and D2H"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama70b_layer_kv_quant",
                    choices=["llama70b_layer_kv_quant", "decode_131k", "batched_decode_32k"])
    ap.add_argument("--rotation", choices=["qr", "hadamard"], default="qr",
                    help="rotation of both quantizers (hadamard: randomised Walsh-Hadamard)")
    ap.add_argument("--study", choices=["score-quality"], default=None,
                    help="print a study's JSON line instead of the benchmark (no timing)")
    ap.add_argument("--mixed", action="store_true",
                    help="time outlier-channel mixed precision on the default workload (own JSON line)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-call timing of the other workloads (configs block)")
    ap.add_argument("--warm-seconds", type=float, default=WARM_SECONDS,
                    help="minimum back-to-back warm-up before timing (0 for profiler launch lists)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.study == "score-quality":
        return run_score_quality_study(args)
    if args.mixed:
        return run_mixed(args)
    spec = workload_spec(args.workload)
    spec["rotation"] = args.rotation
    if args.impl == "reference":
        return run_reference(args, spec)
    return run_ours(args, spec)


if __name__ == "__main__":
    sys.exit(main())
