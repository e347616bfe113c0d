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
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
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
                "reasons": sorted(reasons), "samples": len(load)}


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
def oracle_sample(w: workloads.Workload, budget_s: float = 15.0, max_tiles: int = 64, warmup: int = 0,
                  steps: int | None = None):
    """Time the CPU oracle on whole 128-row query tiles of one head of the workload's recipe.

    One sample (a "step") is one query tile against all Skv keys. With ``steps`` given, runs
    ``warmup`` untimed tiles and then exactly ``steps`` timed tiles; otherwise runs tiles until
    ``budget_s`` seconds or ``max_tiles``. Returns (dense-equiv TFLOP/s, seconds per tile, tiles,
    threads, description)."""
    from oracle import attention as oatt
    from oracle import sage_quant
    one = w.scaled(B=1, Hq=1, Hkv=1)
    q, k, v = workloads.generate(one, seed=0)
    inp = dict(q=q.float().numpy(), k=k.float().numpy(), v=v.float().numpy())
    quant = None
    if w.mode == "sage":
        quant = sage_quant.sage_quantize(inp["q"], inp["k"], inp["v"], w.qk_dtype, w.q_block, w.k_block)
    factor = w.factors[len(w.factors) // 2] if w.factors else None
    ntiles = math.ceil(w.Sq / 128)
    order = np.random.default_rng(0).permutation(ntiles)

    def tile(n):
        oatt.attention_q_tile(inp, 0, 0, int(order[n % ntiles]), mode=w.mode, qk_dtype=w.qk_dtype,
                              q_block=w.q_block, k_block=w.k_block, factor=factor, quant=quant)
    for n in range(warmup):
        tile(n)
    t0 = time.perf_counter()
    tiles = 0
    while (tiles < steps) if steps is not None else (tiles < max_tiles and time.perf_counter() - t0 < budget_s):
        tile(warmup + tiles)
        tiles += 1
    dt = time.perf_counter() - t0
    flop = 4.0 * tiles * 128 * w.Skv * 128
    try:
        threads = len(os.sched_getaffinity(0))
    except AttributeError:
        threads = os.cpu_count()
    desc = (f"{tiles} query tiles x 128 rows of one head against all {w.Skv} keys, float64 NumPy "
            f"({w.name} recipe)")
    return flop / dt / 1e12, dt / max(tiles, 1), tiles, threads, desc


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


def run_modes(dit, steps, warmup, world, stream, peak16, hbm_gbs):
    """The other workloads. Each quantized one is timed as one call of the whole path (prepass +
    attention), and also in its two halves through the split entry points: the prepass alone
    (against the measured HBM bandwidth: it is memory-bound) and the attention over
    precomputed codes (against the tensor peak of its operand types)."""
    res = {}
    peak8 = 2.0 * peak16                               # FP8 dense = 2 x BF16 (nominal ratio)
    peak_mix = 2.0 * peak16 * peak8 / (peak16 + peak8)  # BMM1 on 16-bit operands, BMM2 on FP8
    peak4 = 4.0 * peak16                               # FP4 dense = 4 x BF16 (nominal ratio)
    peak_nv = 2.0 * peak4 * peak8 / (peak4 + peak8)     # BMM1 on FP4, BMM2 on FP8
    table = [("dit_sage_int8_32k", peak_mix, "BMM1 f16 + BMM2 e4m3 harmonic peak"),
             ("gqa_sage_fp8_16k", peak8, "2 x measured bf16 (e4m3 nominal ratio)"),
             ("dit_qk16pv8_32k", peak_mix, "BMM1 bf16 + BMM2 e4m3 harmonic peak"),
             ("dit_mxfp8_32k", peak8, "2 x measured bf16 (e4m3 nominal ratio; BMM1 block-scaled)"),
             ("dit_nvfp4_32k", peak_nv, "BMM1 fp4 (4 x bf16) + BMM2 e4m3 (2 x bf16) harmonic peak")]
    for name, peak, peak_desc in table:
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
        entry = {"ms": round(ms, 3), "tflops": round(tf, 1), "peak_tflops": round(peak, 1),
                 "frac": round(tf / peak, 3), "peak": peak_desc,
                 "launches_per_step": 4 if qk16 else 6 if mx else 9 if nv else 5}
        # the two halves, through the split entry points
        bq, bkv = q.numel() * 2, k.numel() * 2
        if qk16:
            pre = lambda: dit.sage_quantize_v(v, per_tensor=True, stream=stream)  # noqa: E731
            # V read twice (absmax, then codes), 1-byte codes written
            pre_bytes, pre_desc = 2 * bkv + bkv // 2, "V read twice, 1-byte V codes written"
        elif nv:
            def pre():
                res = dit.nvfp4_quantize_qk(q, k, stream=stream)
                res.update(dit.sage_quantize_v(v, per_tensor=False, stream=stream))
                return res
            # Q, K read twice (tensor max, then codes), V twice; half-byte Q/K codes, 1-byte V codes and
            # 8 scale bytes per 128 Q/K elements written
            pre_bytes = 2 * bq + 4 * bkv + (bq + bkv) // 4 + bkv // 2 + (bq + bkv) // 32
            pre_desc = "Q, K, V read twice, half-byte Q/K codes, 1-byte V codes and E4M3 block scales written"
        elif mx:
            def pre():
                res = dit.mx_quantize_qk(q, k, stream=stream)
                res.update(dit.sage_quantize_v(v, per_tensor=False, stream=stream))
                return res
            # Q, K read once and V twice; 1-byte Q/K/V codes and 4 scale bytes per 128 Q/K elements written
            pre_bytes = bq + 3 * bkv + (bq + 2 * bkv) // 2 + (bq + bkv) // 64
            pre_desc = "Q, K read once, V twice, 1-byte Q/K/V codes and E8M0 bytes written"
        else:
            pre = lambda: dit.sage_quantize_qkv(q, k, v, qk_dtype=w.qk_dtype, q_block=w.q_block,  # noqa: E731
                                                k_block=w.k_block, stream=stream)
            # K, V read in the stats pass and again with Q in the code pass; 1-byte codes written
            pre_bytes = bq + 4 * bkv + (bq + 2 * bkv) // 2
            pre_desc = "K, V read twice, Q once, 1-byte Q/K/V codes written"
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
        entry["prepass"] = {"ms": round(pre_ms, 3), "gbs": round(pre_bytes / (pre_ms * 1e-3) / 1e9, 1),
                            "frac_hbm": round(pre_bytes / (pre_ms * 1e-3) / 1e9 / hbm_gbs, 3),
                            "bytes": int(pre_bytes), "bytes_desc": pre_desc}
        entry["attention"] = {"ms": round(attn_ms, 3), "tflops": round(atf, 1), "frac": round(atf / peak, 3),
                              "note": "INT8 codes are widened to fp16 inside this call" if w.qk_dtype == "int8"
                              else "the attention kernel alone"}
        res[name] = entry
        del q, k, v, ws, out, quant
    # Skip-Softmax sweep on the video grid, against dense BF16 on the same shape
    w = workloads.WORKLOADS["video_skip_int8_75600"]
    q, k, v = workloads.generate(w, seed=1, device="cuda")
    out = torch.empty_like(q)
    nqt = math.ceil(w.Sq / 128)
    counts = torch.zeros((w.B, w.Hq, nqt), dtype=torch.int32, device="cuda")
    ws = torch.empty(dit.dit_attn_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, dit.MODE_SAGE, w.qk_dtype,
                                                  w.q_block, w.k_block), dtype=torch.uint8, device="cuda")
    s = max(2, steps // 4)

    def dense():
        dit.dit_attn_fwd(q, k, v, out, stream=stream)
    dense_ms = max_over_ranks(time_steps(dense, s, min(warmup, 3), world, stream), world) / s
    sweep = {}
    nkt = math.ceil(w.Skv / 128)
    for factor in w.factors:
        def step():
            dit.dit_attn_fwd(q, k, v, out, mode=dit.MODE_SAGE | dit.MODE_SKIP, qk_dtype=w.qk_dtype,
                             q_block=w.q_block, k_block=w.k_block, threshold_scale_factor=factor, workspace=ws,
                             skip_counts=counts, stream=stream)
        ms = max_over_ranks(time_steps(step, s, min(warmup, 3), world, stream), world) / s
        frac = float(counts.sum().item()) / (w.B * w.Hq * nqt * nkt)
        sweep[str(factor)] = {"ms": round(ms, 3), "skip_fraction": round(frac, 4),
                              "speedup_vs_dense_bf16": round(dense_ms / ms, 3),
                              "dense_equiv_tflops": round(w.dense_equiv_flop / (ms * 1e-3) / 1e12, 1)}
    # The same inputs and sweep points with Q/K formats whose BMM1 runs at the FP8 (or FP4) rate: a skipped
    # tile still costs its BMM1, so the INT8 codes' 16-bit BMM1 caps the INT8 sweep's speedup
    fast = {}
    for label, dt, qb, kb in [("sage_fp8_1_16", "fp8_e4m3", 1, 16), ("mxfp8", "mxfp8", 0, 0),
                              ("nvfp4", "nvfp4", 0, 0)]:
        ws2 = torch.empty(max(1, dit.dit_attn_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, dit.MODE_SAGE, dt, qb, kb)),
                          dtype=torch.uint8, device="cuda")
        pts = {}
        for factor in (0.0, 50.0, 3200.0):
            def step2():
                dit.dit_attn_fwd(q, k, v, out, mode=dit.MODE_SAGE | dit.MODE_SKIP, qk_dtype=dt, q_block=qb, k_block=kb,
                                 threshold_scale_factor=factor, workspace=ws2, skip_counts=counts, stream=stream)
            ms = max_over_ranks(time_steps(step2, s, min(warmup, 3), world, stream), world) / s
            frac = float(counts.sum().item()) / (w.B * w.Hq * nqt * nkt)
            pts[str(factor)] = {"ms": round(ms, 3), "skip_fraction": round(frac, 4),
                                "speedup_vs_dense_bf16": round(dense_ms / ms, 3)}
        fast[label] = pts
        del ws2
    res["video_skip_int8_75600"] = {"dense_bf16_ms": round(dense_ms, 3),
                                    "dense_bf16_tflops": round(w.dense_equiv_flop / (dense_ms * 1e-3) / 1e12, 1),
                                    "sweep": sweep, "fp8_rate_bmm1_sweeps": fast}
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
        tf, per_tile, tiles, threads, desc = oracle_sample(w, warmup=warmup, steps=args.steps)
        line = {"metric": METRIC, "value": round(tf, 6), "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": warmup, "ms_per_step": round(per_tile * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "impl": "reference",
                "cpu_baseline": {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                 "sample": desc},
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
        modes = run_modes(dit, args.steps, warmup, world, stream, peak16, hbm)

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        tf, _, tiles, threads, desc = oracle_sample(w)
        cpu = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc}
    traffic = dense_kernel_traffic()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) Q/V, K + per-channel offset)",
        "config": config,
        "pct_of_peak": round(100.0 * kernel_tflops / peak16, 1),
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
    print(json.dumps(line))


if __name__ == "__main__":
    main()
