"""Benchmark: dense-equivalent attention TFLOP/s of the DiT attention forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {ours,reference}] [--no-modes]

One step is one call of the hot path on the headline workload: dense BF16 attention with
B=1, Hq=Hkv=40, Sq=Skv=32768, head_dim 128 (the DiT-shaped workload; K carries a per-channel
offset). Dense-equivalent FLOP per call = 4*B*Hq*Sq*Skv*128. Prints one JSON line.

* value        device-timed throughput: inputs resident in HBM, CUDA events on the launching
               stream around K back-to-back steps (inputs of 1 GiB exceed the 126 MB L2, so no
               flush is needed), max over ranks.
* e2e          the same metric through the public API with pinned host buffers
               (dit_attn_fwd_host): every step copies Q, K, V host->device and O back, overlapped
               with the attention over groups of kv heads; the serial copy-run-copy time is
               reported beside it.
* roofline     the attention kernel against the measured dense BF16 tensor peak.
* cpu_baseline the CPU oracle (float64 NumPy) timed on this host on a bounded sample.
* modes        the other workloads (SAGE INT8, SAGE FP8 with GQA, SAGE INT8 + Skip-Softmax sweep
               on the 75600-token video grid), each against its own instruction peak.
* --impl reference times the oracle (there is no reference implementation to install: the
  pages give no code); it prints the same metric with "impl": "reference".

Multi-GPU (torchrun): every rank runs its own copy of the workload (weak scaling, no
collective on the data path); value = total FLOP of all ranks / the slowest rank's time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

E2E_CHUNKS = 8
HEADLINE = "dit_dense_32k"
METRIC = "dense-equiv attention TFLOPS at B=1,H=40,S=32768,d=128; % of tensor-core peak"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, 1700.0, FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks during the timed region
class ClockSampler:
    """Samples the SM clock, power and clock-event reasons of one GPU while the timed region runs.

    Reads NVML (libnvidia-ml, through ctypes) every 10 ms from a thread, so even a region of a few
    hundred milliseconds gets tens of samples; falls back to ``nvidia-smi -lms 200``. Only queries:
    no clock, power or other setting is touched."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_uuid, period_s: float = 0.01):
        self.uuid = gpu_uuid
        self.period = period_s
        self.rows = []          # (sm_mhz, power_w, reason_bits)
        self.max_mhz = None
        self.proc = None
        self.file = None
        self.thread = None
        self.stop = None
        self.nvml = None

    def _nvml_open(self):
        import ctypes
        import ctypes.util
        name = ctypes.util.find_library("nvidia-ml") or "libnvidia-ml.so.1"
        lib = ctypes.CDLL(name)
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle for this GPU")
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        self.nvml = (lib, h, get_reasons)

    def _nvml_loop(self):
        import ctypes
        lib, h, get_reasons = self.nvml
        mhz, mw, rb = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and
                    lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0 and get_reasons(h, ctypes.byref(rb)) == 0):
                self.rows.append((float(mhz.value), mw.value / 1000.0, int(rb.value)))
            self.stop.wait(self.period)

    def __enter__(self):
        import threading
        try:
            self._nvml_open()
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._nvml_loop, daemon=True)
            self.thread.start()
        except (OSError, AttributeError):
            self.nvml = None
            try:
                self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
                self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.uuid), f"--query-gpu={self.FIELDS}",
                                              "--format=csv,noheader,nounits", "-lms", "200"],
                                             stdout=self.file, stderr=subprocess.DEVNULL)
            except OSError:
                self.proc = None
            time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.nvml is not None:
            # Every NVML sample falls inside the sampled region, which only launches kernels and waits
            # for them, so all count as under load. (NVML's power reading is a moving average that
            # trails a short burst: filtering on it dropped most samples of a sub-second region.)
            load = self.rows
            if not load:
                return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"], "source": "nvml"}
            reasons = sorted({name for _, _, bits in load for bit, name in self.REASONS.items() if bits & bit})
            # the mean of evenly spaced samples is the region's time-averaged clock (cycles / time)
            return {"sm_mhz": statistics.median(r[0] for r in load), "sm_mhz_mean": round(statistics.fmean(
                r[0] for r in load), 1), "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(load),
                "source": "nvml, 10 ms"}
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        load = [r for r in rows if (num(r[3]) or 0) > 300] or rows  # samples under load
        sm = [num(r[1]) for r in load if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in load:
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(load), "source": "nvidia-smi, 200 ms"}


# ------------------------------------------------------------------ distributed helpers
def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest of the ranks' values (the slowest rank's time); x itself on one rank."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(flop_per_step: float, steps: int, elapsed_ms: float, world: int) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` steps of the same workload (weak scaling), and the
    job took as long as its slowest rank."""
    tmax = max_over_ranks(elapsed_ms, world)
    return world * flop_per_step * steps / (tmax * 1e-3) / 1e12


# ------------------------------------------------------------------ CPU oracle sample
def blas_threads():
    """Threads of the BLAS NumPy calls (threadpoolctl when installed, else the bundled OpenBLAS's own
    query through its loaded library), or None when neither is available."""
    try:
        import threadpoolctl
        n = [i["num_threads"] for i in threadpoolctl.threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:  # noqa: BLE001 - optional dependency, any failure means "unknown"
        pass
    import ctypes
    np.ones((2, 2)) @ np.ones((2, 2))  # make sure the BLAS library is loaded
    try:
        with open("/proc/self/maps") as f:
            paths = sorted({ln.split()[-1] for ln in f if "blas" in ln.lower() and ".so" in ln})
    except OSError:
        return None
    for path in paths:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_", "openblas_get_num_threads"):
            fn = getattr(lib, sym, None)
            if fn is not None:
                return int(fn())
    return None


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def oracle_sample(w: workloads.Workload, budget_s: float = 15.0, max_tiles: int = 64, warmup: int = 0,
                  steps: int | None = None, factor: float | None = None):
    """Time the CPU oracle on whole 128-row query tiles of one head of the workload's recipe.

    One sample (a "step") is one query tile against all Skv keys. With ``steps`` given, runs
    ``warmup`` untimed tiles and then exactly ``steps`` timed tiles; otherwise runs tiles until
    ``budget_s`` seconds or ``max_tiles`` (at least two). Quantized recipes first run the oracle's
    quantizer over the whole head (timed separately). Returns a dict: dense-equiv TFLOP/s of the
    sampled tiles, seconds per tile, tiles, the quantizer's seconds for the head, threads,
    description."""
    from oracle import attention as oatt
    from oracle import mx_quant, nvfp4_quant, sage_quant
    one = w.scaled(B=1, Hq=1, Hkv=1)
    q, k, v = workloads.generate(one, seed=0)
    inp = dict(q=q.float().numpy(), k=k.float().numpy(), v=v.float().numpy())
    t0 = time.perf_counter()
    quant = None
    if w.mode == "sage":
        quant = sage_quant.sage_quantize(inp["q"], inp["k"], inp["v"], w.qk_dtype, w.q_block, w.k_block)
    elif w.mode == "qk16pv8":
        quant = sage_quant.qk16pv8_quantize(inp["v"], True)
    elif w.mode == "mxfp8":
        quant = mx_quant.mxfp8_quantize(inp["q"], inp["k"], inp["v"], False)
    elif w.mode == "nvfp4":
        quant = nvfp4_quant.nvfp4_qk_quantize(inp["q"], inp["k"], inp["v"], False)
    quant_s = time.perf_counter() - t0
    if factor is None and w.factors:
        factor = w.factors[len(w.factors) // 2]
    ntiles = math.ceil(w.Sq / 128)
    order = np.random.default_rng(0).permutation(ntiles)

    def tile(n):
        oatt.attention_q_tile(inp, 0, 0, int(order[n % ntiles]), mode=w.mode, qk_dtype=w.qk_dtype,
                              q_block=w.q_block, k_block=w.k_block, factor=factor, quant=quant)
    for n in range(warmup):
        tile(n)
    t0 = time.perf_counter()
    tiles = 0
    while (tiles < steps) if steps is not None else \
            (tiles < 2 or (tiles < max_tiles and time.perf_counter() - t0 < budget_s)):
        tile(warmup + tiles)
        tiles += 1
    dt = time.perf_counter() - t0
    flop = 4.0 * tiles * 128 * w.Skv * 128
    desc = (f"{tiles} query tiles x 128 rows of one head against all {w.Skv} keys, float64 NumPy "
            f"({w.name} recipe" + (f", factor {factor:g}" if factor is not None else "") + ")")
    return {"tflops": flop / dt / 1e12, "s_per_tile": dt / max(tiles, 1), "tiles": tiles, "quant_s": quant_s,
            "threads": host_cores(), "desc": desc}


def oracle_config_baseline(w: workloads.Workload, budget_s: float, factor: float | None = None) -> dict:
    """The oracle on a bounded sample of a large workload: its quantizer over one head and whole query
    tiles of that head, timed on the host cores, with the full call's time extrapolated from them
    (quantizer time x the elements of all heads, attention time x all query tiles of all heads)."""
    r = oracle_sample(w, budget_s=budget_s, max_tiles=16, factor=factor)
    heads_q = w.B * w.Hq
    elems_full = w.B * (w.Sq * w.Hq + 2 * w.Skv * w.Hkv)
    elems_one = w.Sq + 2 * w.Skv
    full_s = r["quant_s"] * elems_full / elems_one + r["s_per_tile"] * heads_q * math.ceil(w.Sq / 128)
    return {"tflops": round(r["tflops"], 5), "tiles": r["tiles"], "s_per_tile": round(r["s_per_tile"], 3),
            "quant_s_one_head": round(r["quant_s"], 3), "full_call_s_extrapolated": round(full_s, 1),
            "full_call_tflops_extrapolated": round(w.dense_equiv_flop / full_s / 1e12, 5)}


def dense_kernel_traffic():
    """DRAM bytes per launch of the dense attention kernel from the committed ncu summary, or None
    when the kernel sources changed since those counters were taken."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", "fmha_dense_bf16_dit32k_traffic.md")
    csrc = os.path.join(ROOT, "diffusion_transformer_attention_gb300", "csrc")
    try:
        text = open(path).read()
        h = hashlib.sha256()
        for name in ("fmha_kernel.cuh", "fmha_common.cuh", "fmha_dense.cu", "sm103_ptx.cuh"):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    m = re.search(r"first 16 hex\): ([0-9a-f]{16})", text)
    t = re.search(r"traffic_bytes_per_launch: (\d+)", text)
    if not m or not t or m.group(1) != h.hexdigest()[:16]:
        return None
    return int(t.group(1))


# ------------------------------------------------------------------ timing helpers
def time_steps(fn, steps, warmup, world, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)  # ms on this rank


def _r(x, nd=3):
    return None if x is None else round(float(x), nd)


def run_recipe(dit, name, steps, warmup, world, stream, peak, hbm_gbs):
    """One quantized workload on the DiT / GQA inputs: the whole call (prepass + attention) through
    dit_attn_fwd, then its two halves through the split entry points: the prepass alone (against the
    measured HBM bandwidth: it is memory-bound) and the attention over precomputed codes (against
    the tensor peak of its operand types)."""
    w = workloads.WORKLOADS[name]
    q, k, v = workloads.generate(w, seed=1, device="cuda")
    qk16, mx, nv = w.mode == "qk16pv8", w.mode == "mxfp8", w.mode == "nvfp4"
    mode = dit.MODE_SAGE | (dit.MODE_V_PER_TENSOR if qk16 else 0)
    ws = torch.empty(dit.dit_attn_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, mode, w.qk_dtype,
                                                  w.q_block, w.k_block), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)

    def step():
        dit.dit_attn_fwd(q, k, v, out, mode=mode, qk_dtype=w.qk_dtype, q_block=w.q_block,
                         k_block=w.k_block, workspace=ws, stream=stream)
    ms = max_over_ranks(time_steps(step, steps, warmup, world, stream), world) / steps
    tf = w.dense_equiv_flop / (ms * 1e-3) / 1e12
    bq, bkv = q.numel() * 2, k.numel() * 2
    # algorithmic prepass bytes (inputs read as often as the passes need them, codes and scales written)
    if qk16:
        pre = lambda: dit.sage_quantize_v(v, per_tensor=True, stream=stream)  # noqa: E731
        pre_bytes = 2 * bkv + bkv // 2                                        # V twice, 1-byte V codes
    elif nv:
        def pre():
            res = dit.nvfp4_quantize_qk(q, k, stream=stream)
            res.update(dit.sage_quantize_v(v, per_tensor=False, stream=stream))
            return res
        # Q, K, V twice; half-byte Q/K codes, 1-byte V codes, 8 scale bytes per 128 Q/K elements
        pre_bytes = 2 * bq + 4 * bkv + (bq + bkv) // 4 + bkv // 2 + (bq + bkv) // 32
    elif mx:
        def pre():
            res = dit.mx_quantize_qk(q, k, stream=stream)
            res.update(dit.sage_quantize_v(v, per_tensor=False, stream=stream))
            return res
        # Q, K once, V twice; 1-byte Q/K/V codes, 4 scale bytes per 128 Q/K elements
        pre_bytes = bq + 3 * bkv + (bq + 2 * bkv) // 2 + (bq + bkv) // 64
    else:
        pre = lambda: dit.sage_quantize_qkv(q, k, v, qk_dtype=w.qk_dtype, q_block=w.q_block,  # noqa: E731
                                            k_block=w.k_block, stream=stream)
        pre_bytes = bq + 4 * bkv + (bq + 2 * bkv) // 2                        # K, V twice, Q once; 1-byte codes
    quant = pre()
    if qk16:
        quant.update(q_codes=q, k_codes=k)
    pre_ms = max_over_ranks(time_steps(pre, steps, warmup, world, stream), world) / steps

    def attn():
        if mx:
            dit.dit_attn_fwd_mxfp8(quant, out, mode=mode, stream=stream)
        elif nv:
            dit.dit_attn_fwd_nvfp4(quant, out, mode=mode, stream=stream)
        else:
            dit.dit_attn_fwd_quantized(quant, out, mode=mode, qk_dtype=w.qk_dtype, q_block=w.q_block,
                                       k_block=w.k_block, stream=stream)
    attn_ms = max_over_ranks(time_steps(attn, steps, warmup, world, stream), world) / steps
    atf = w.dense_equiv_flop / (attn_ms * 1e-3) / 1e12
    pre_gbs = pre_bytes / (pre_ms * 1e-3) / 1e9
    del q, k, v, ws, out, quant
    return {"ms": _r(ms), "tflops": _r(tf, 1), "frac": _r(tf / peak), "peak": _r(peak, 1),
            "pre_ms": _r(pre_ms), "pre_gbs": _r(pre_gbs, 1), "pre_frac_hbm": _r(pre_gbs / hbm_gbs),
            "pre_bytes": int(pre_bytes), "attn_ms": _r(attn_ms), "attn_tflops": _r(atf, 1), "attn_frac": _r(atf / peak)}


def skip_sweep(dit, q, k, v, out, counts, w, factors, steps, warmup, world, stream, dense_ms, *, mode, dt, qb, kb):
    """Time one Skip-Softmax recipe over the threshold factors on the video inputs; returns compact
    lists, one entry per factor: skipped fraction, ms, speedup against dense BF16 on the same inputs."""
    nqt, nkt = math.ceil(w.Sq / 128), math.ceil(w.Skv / 128)
    need = dit.dit_attn_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, mode & ~dit.MODE_SKIP, dt, qb, kb)
    ws = torch.empty(max(1, need), dtype=torch.uint8, device="cuda") if need > 0 else None
    res = {"skip": [], "ms": [], "x": []}
    for factor in factors:
        def step():
            dit.dit_attn_fwd(q, k, v, out, mode=mode, qk_dtype=dt, q_block=qb, k_block=kb,
                             threshold_scale_factor=factor, workspace=ws, skip_counts=counts, stream=stream)
        ms = max_over_ranks(time_steps(step, steps, warmup, world, stream), world) / steps
        frac = float(counts.sum().item()) / (w.B * w.Hq * nqt * nkt)
        res["skip"].append(_r(frac, 4))
        res["ms"].append(_r(ms, 2))
        res["x"].append(_r(dense_ms / ms))
    return res


def run_modes(dit, steps, warmup, world, stream, peak16, hbm_gbs, cpu: bool):
    """The other workloads, in the order the line prints them: the other Q/K formats on the DiT
    inputs, the Skip-Softmax sweeps with FP8-rate BMM1s, then SAGE INT8 on the DiT inputs, SAGE FP8
    with GQA, and the Skip-Softmax curve on the video grid (SAGE INT8, and BF16 without SAGE), each
    against its own instruction peak and, on rank 0, beside the oracle timed on a bounded sample."""
    peak8 = 2.0 * peak16                               # FP8 dense = 2 x BF16 (nominal ratio)
    peak_mix = 2.0 * peak16 * peak8 / (peak16 + peak8)  # BMM1 on 16-bit operands, BMM2 on FP8
    peak4 = 4.0 * peak16                               # FP4 dense = 4 x BF16 (nominal ratio)
    peak_nv = 2.0 * peak4 * peak8 / (peak4 + peak8)     # BMM1 on FP4, BMM2 on FP8
    res = {"peaks": {"bf16": _r(peak16, 1), "f16_e4m3": _r(peak_mix, 1), "e4m3": _r(peak8, 1),
                     "fp4_e4m3": _r(peak_nv, 1)}}
    res["recipes"] = {label: run_recipe(dit, name, steps, warmup, world, stream, peak, hbm_gbs)
                      for label, name, peak in [("qk16pv8", "dit_qk16pv8_32k", peak_mix),
                                                ("mxfp8", "dit_mxfp8_32k", peak8),
                                                ("nvfp4", "dit_nvfp4_32k", peak_nv)]}
    # the video inputs, shared by every sweep
    w = workloads.WORKLOADS["video_skip_int8_75600"]
    q, k, v = workloads.generate(w, seed=1, device="cuda")
    out = torch.empty_like(q)
    counts = torch.zeros((w.B, w.Hq, math.ceil(w.Sq / 128)), dtype=torch.int32, device="cuda")
    s, wu = max(2, steps // 4), min(warmup, 3)

    def dense():
        dit.dit_attn_fwd(q, k, v, out, stream=stream)
    dense_ms = max_over_ranks(time_steps(dense, s, wu, world, stream), world) / s
    sk = dit.MODE_SAGE | dit.MODE_SKIP
    # Q/K formats whose BMM1 runs at the FP8 (or FP4) rate: a skipped tile still costs its BMM1, so the
    # INT8 codes' 16-bit BMM1 caps the INT8 curve's speedup
    short = (0.0, 2.0, 50.0, 3200.0)
    res["video_fp8_rate_bmm1"] = {"f": list(short)}
    res["video_fp8_rate_bmm1"].update({
        label: skip_sweep(dit, q, k, v, out, counts, w, short, s, wu, world, stream, dense_ms, mode=sk, dt=dt, qb=qb,
                          kb=kb)
        for label, dt, qb, kb in [("sage_fp8_1_16", "fp8_e4m3", 1, 16), ("mxfp8", "mxfp8", 0, 0),
                                  ("nvfp4", "nvfp4", 0, 0)]})
    curve = skip_sweep(dit, q, k, v, out, counts, w, w.factors, s, wu, world, stream, dense_ms, mode=sk,
                       dt=w.qk_dtype, qb=w.q_block, kb=w.k_block)
    bf16 = skip_sweep(dit, q, k, v, out, counts, w, w.factors, s, wu, world, stream, dense_ms,
                      mode=dit.MODE_SKIP, dt="bf16", qb=1, kb=1)
    del q, k, v, out, counts
    torch.cuda.empty_cache()
    for label, name, peak in [("dit_sage_int8_32k", "dit_sage_int8_32k", peak_mix),
                              ("gqa_sage_fp8_16k", "gqa_sage_fp8_16k", peak8)]:
        res[label] = run_recipe(dit, name, steps, warmup, world, stream, peak, hbm_gbs)
        if cpu:
            res[label]["cpu"] = oracle_config_baseline(workloads.WORKLOADS[name], budget_s=4.0)
    # INT8 codes run BMM1 at the fp16 tensor rate (there is no INT8 MMA on this part) and BMM2 at the
    # E4M3 rate, half the BF16 time, and a skipped tile still costs its BMM1: at skipped fraction f the
    # tensor time per tile is (1 + (1 - f) / 2) / 2 of dense BF16, so 2 / (1 + (1 - f) / 2) is the
    # most Skip-Softmax with INT8 codes can gain over dense BF16 at equal tensor efficiency
    curve["ceiling_x"] = [_r(2.0 / (1.0 + 0.5 * (1.0 - f))) for f in curve["skip"]]
    vid = {"dense_bf16_ms": _r(dense_ms), "dense_bf16_tflops": _r(w.dense_equiv_flop / (dense_ms * 1e-3) / 1e12, 1),
           "f": list(w.factors), "bf16_skip": bf16, "sage_int8_1_16_skip": curve}
    if cpu:
        vid["cpu"] = oracle_config_baseline(w, budget_s=4.0, factor=50.0)
    res["video_skip_int8_75600"] = vid
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-modes", action="store_true", help="skip the SAGE / Skip-Softmax workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    warmup = max(3, args.warmup)
    w = workloads.WORKLOADS[HEADLINE]
    flop = w.dense_equiv_flop
    config = {"workload": HEADLINE, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Skv": w.Skv, "head_dim": 128,
              "mode": "dense bf16", "l2": "inputs 1.0 GiB > 126 MB L2, no flush"}

    rank, world, local = dist_setup(args.gpus) if args.impl == "ours" else (
        int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), 0)

    if args.impl == "reference":
        if rank != 0:
            return
        r = oracle_sample(w, warmup=warmup, steps=args.steps)
        tf = r["tflops"]
        line = {"metric": METRIC, "value": round(tf, 6), "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": warmup, "ms_per_step": round(r["s_per_tile"] * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "impl": "reference",
                "cpu_baseline": {"value": round(tf, 6), "unit": "TFLOP/s", "cores": r["threads"], "kind": "oracle",
                                 "blas_threads": blas_threads(), "sample": r["desc"]},
                "e2e": {"value": round(tf, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import diffusion_transformer_attention_gb300 as dit
    dit.library()  # raises if the CUDA library is missing: no fallback
    torch.cuda.set_device(local)
    stream = torch.cuda.current_stream()
    peak16, peak16_sus, hbm, peak_src = peaks()

    q, k, v = workloads.generate(w, seed=rank, device="cuda")
    out = torch.empty_like(q)

    def step():
        dit.dit_attn_fwd(q, k, v, out, stream=stream)

    props = torch.cuda.get_device_properties(local)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) is not None else str(local)
    with ClockSampler(gpu_id) as clk:
        elapsed = time_steps(step, args.steps, warmup, world, stream)
    clocks = clk.summary()
    dit.dit_attn_check_errors(stream)
    value = aggregate_value(flop, args.steps, elapsed, world)
    ms = world * flop / (value * 1e12) * 1e3  # the slowest rank's time per step
    kernel_tflops = flop / (elapsed / args.steps * 1e-3) / 1e12  # this rank's launch average

    # end to end through the public API with pinned host buffers
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

    # End to end through the host-buffer entry point: the pinned inputs are copied in and the output
    # copied back every step, overlapped with the attention over 8 groups of kv heads.
    def e2e_step():
        dit.dit_attn_fwd_host(hq, hk, hv, hout, q, k, v, out, chunks=E2E_CHUNKS, stream=stream)
    # Three separately timed runs, the median reported: the host link on a shared machine has slow
    # stretches of a few hundred milliseconds (all three runs are in the line)
    e2e_steps = max(2, args.steps // 2)
    e2e_runs = [max_over_ranks(time_steps(e2e_step, e2e_steps, warmup if i == 0 else 1, world, stream), world)
                / e2e_steps for i in range(3)]
    e2e_ms = sorted(e2e_runs)[1]

    # the same copies and kernel one after the other on one stream, for comparison
    def serial_step():
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        dit.dit_attn_fwd(q, k, v, out, stream=stream)
        hout.copy_(out, non_blocking=True)
    serial_ms = max_over_ranks(time_steps(serial_step, e2e_steps, warmup, world, stream), world) / e2e_steps
    e2e_value = world * flop / (e2e_ms * 1e-3) / 1e12
    h2d = 3 * q.numel() * q.element_size()
    d2h = out.numel() * out.element_size()
    del hq, hk, hv, hout

    modes = None
    if not args.no_modes:
        del q, k, v, out
        torch.cuda.empty_cache()
        modes = run_modes(dit, args.steps, warmup, world, stream, peak16, hbm,
                          cpu=(rank == 0 and not args.no_cpu_baseline))

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        r = oracle_sample(w, budget_s=10.0)
        cpu = {"value": round(r["tflops"], 6), "unit": "TFLOP/s", "cores": r["threads"], "kind": "oracle",
               "blas_threads": blas_threads(), "sample": r["desc"]}
    traffic = dense_kernel_traffic()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) Q/V, K + per-channel offset)",
        "config": config,
        "pct_of_peak": round(100.0 * kernel_tflops / peak16, 1),
        # the same rate over the nominal BF16 tensor rate at the SM clock sampled during the timed region
        # (M128 N128 K16 in 64 clocks = 8192 FLOP per clock per SM): a clock-independent duty estimate,
        # since the measured cuBLAS peak ran at a lower, power-capped clock
        "tensor_duty_at_clock": (round(kernel_tflops * 1e12 / (8192.0 * props.multi_processor_count *
                                                             clocks.get("sm_mhz_mean", clocks["sm_mhz"]) * 1e6), 3)
                                 if clocks.get("sm_mhz") else None),
        "roofline": {"bound": "tensor", "achieved": round(kernel_tflops, 1), "peak": peak16, "unit": "TFLOP/s",
                     "frac": round(kernel_tflops / peak16, 3), "traffic": traffic,
                     "peak_source": f"{peak_src} dense bf16 burst (MEASURED_PEAKS.json bf16_tflops)",
                     "kernel": "fmha_fwd_kernel<bf16,bf16,noskip>", "flop_per_launch": flop},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 1), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                "runs_ms_per_step": [round(x, 3) for x in e2e_runs],
                "statistic": f"median of 3 timed runs of {e2e_steps} steps",
                "api": f"dit_attn_fwd_host, {E2E_CHUNKS} groups of kv heads (copies overlapped with the kernels)",
                "serial_copies_ms_per_step": round(serial_ms, 3)},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if modes is not None:
        line["modes"] = modes
        line["summary"] = summarize(line)
    print(json.dumps(line))


def summarize(line):
    """The numbers the targets are stated in, repeated at the end of the line so that a tail of the
    log still shows every workload: fractions of each workload's peak (whole call; attention alone
    where it differs), and the Skip-Softmax speedups over dense BF16 at the sweep point nearest 65%
    skipped."""
    m = line["modes"]

    def at65(curve):
        k = min(range(len(curve["skip"])), key=lambda i: abs(curve["skip"][i] - 0.65))
        return {"skip": curve["skip"][k], "x": curve["x"][k]}

    vid = m["video_skip_int8_75600"]
    i8 = at65(vid["sage_int8_1_16_skip"])
    i8["ceiling_x"] = vid["sage_int8_1_16_skip"]["ceiling_x"][vid["sage_int8_1_16_skip"]["skip"].index(i8["skip"])]
    return {
        "dit_dense_32k": line["roofline"]["frac"],
        "dit_sage_int8_32k": [m["dit_sage_int8_32k"]["frac"], m["dit_sage_int8_32k"]["attn_frac"]],
        "gqa_sage_fp8_16k": [m["gqa_sage_fp8_16k"]["frac"], m["gqa_sage_fp8_16k"]["attn_frac"]],
        "video_skip_sage_int8": i8,
        "video_skip_sage_fp8": at65(m["video_fp8_rate_bmm1"]["sage_fp8_1_16"]),
        "video_skip_bf16": at65(vid["bf16_skip"]),
    }


if __name__ == "__main__":
    main()
