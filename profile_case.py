"""Run one attention configuration a few times, for profiling under ncu.

    python profile_case.py --mode dense --B 1 --H 16 --S 16384 \
        --warmup 1 --launches 2

Inputs are drawn on the device with the DiT recipe (K with a per-channel offset; the video
recipe for --kind video). The process exits non-zero if any call reports an error.
"""

from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import diffusion_transformer_attention_gb300 as dit  # noqa: E402
import workloads  # noqa: E402

MODES = {
    "dense": (dit.MODE_DENSE, "bf16"),
    "sage_int8": (dit.MODE_SAGE, "int8"),
    "sage_fp8": (dit.MODE_SAGE, "fp8_e4m3"),
    "skip_dense": (dit.MODE_SKIP, "bf16"),
    "skip_sage_int8": (dit.MODE_SAGE | dit.MODE_SKIP, "int8"),
    "skip_sage_fp8": (dit.MODE_SAGE | dit.MODE_SKIP, "fp8_e4m3"),
    "qk16pv8": (dit.MODE_SAGE | dit.MODE_V_PER_TENSOR, "bf16"),
    "mxfp8": (dit.MODE_SAGE, "mxfp8"),
    "nvfp4": (dit.MODE_SAGE, "nvfp4"),
    "skip_mxfp8": (dit.MODE_SAGE | dit.MODE_SKIP, "mxfp8"),
}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--mode", choices=sorted(MODES), default="dense")
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--Hkv", type=int, default=0, help="kv heads (default: H)")
    ap.add_argument("--S", type=int, default=16384)
    ap.add_argument("--kind", default="koffset")
    ap.add_argument("--grid", default="", help="T,H,W for --kind video")
    ap.add_argument("--q-block", type=int, default=1)
    ap.add_argument("--k-block", type=int, default=16)
    ap.add_argument("--factor", type=float, default=0.0)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--launches", type=int, default=2)
    ap.add_argument("--prepass", action="store_true",
                    help="run only the SAGE quantize prepass (sage_quantize_qkv) for a quantized --mode")
    args = ap.parse_args()
    mode, dt = MODES[args.mode]
    if dt in ("bf16", "mxfp8", "nvfp4") and mode & dit.MODE_SAGE:  # these recipes have no token blocks
        args.q_block = args.k_block = 0
    grid = tuple(int(x) for x in args.grid.split(",")) if args.grid else ()
    S = args.S if not grid else grid[0] * grid[1] * grid[2]
    w = workloads.Workload("profile", args.B, args.H, args.Hkv or args.H, S, S, kind=args.kind, grid=grid)
    q, k, v = workloads.generate(w, seed=0, device="cuda")
    if args.prepass:
        if dt == "bf16":
            raise SystemExit("--prepass needs a SAGE --mode with int8, fp8, mxfp8 or nvfp4 Q/K")
        for _ in range(args.warmup + args.launches):
            if dt in ("mxfp8", "nvfp4"):
                (dit.mx_quantize_qk if dt == "mxfp8" else dit.nvfp4_quantize_qk)(q, k)
                dit.sage_quantize_v(v)
            else:
                dit.sage_quantize_qkv(q, k, v, qk_dtype=dt, q_block=args.q_block, k_block=args.k_block)
        dit.dit_attn_check_errors()
        torch.cuda.synchronize()
        print(f"ok: prepass {args.mode} B={w.B} H={w.Hq}/{w.Hkv} S={S} calls={args.warmup + args.launches}")
        return
    out = torch.empty_like(q)
    ws_bytes = dit.dit_attn_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, mode, dt, args.q_block, args.k_block)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup + args.launches):
        dit.dit_attn_fwd(q, k, v, out, mode=mode, qk_dtype=dt, q_block=args.q_block, k_block=args.k_block,
                         threshold_scale_factor=args.factor, workspace=ws)
    dit.dit_attn_check_errors()
    torch.cuda.synchronize()
    print(f"ok: {args.mode} B={w.B} H={w.Hq}/{w.Hkv} S={S} launches={args.warmup + args.launches}")


if __name__ == "__main__":
    main()
